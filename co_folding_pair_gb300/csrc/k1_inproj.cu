// k1_inproj.cu -- LayerNorm(z) + gated input projection + pair mask, stored channel-major.
//
// fold-cp-ops README, "Use": norm_in = LayerNorm(D); p_in, g_in = Linear(D, 2D,
// bias=False) produce the value and gate of a (first half) and b (second half);
// the (B, N, N) pair mask multiplies them.  Per pair p and channel c:
//     a[b, c, p] = sigmoid(z'_p . W_ga[c]) * (z'_p . W_a[c]) * m_p,  z'_p = LN_in(z_p)
// and the same for b.  The result is written channel-major ([B][C][N*N]) so the
// triangle GEMM reads each channel plane contiguously; no separate permute runs.
//
// The GEMM is computed transposed, weight rows x pairs, so the accumulator's
// TMEM lanes are weight rows and its columns consecutive pairs.  A CTA pair
// takes a tile of 256 pairs: each CTA loads and normalises its own 128 (half
// of the MMA's N = 256 operand) and stages 128 weight rows of every chunk of
// 128 output channels (half of the M = 256 operand); the even CTA issues
// tcgen05.mma.cta_group::2 (M = 256, N = 256, K = 16).  The weight rows come in
// groups of 16: the value rows of 8 channels, then their gate rows.  A
// 16-lane tcgen05.ld.16x256b then hands each thread the value and the gate of
// one channel for the same pairs (lanes base + t/4 and base + 8 + t/4), so
// one accumulator of 256 columns holds both, and two of them double-buffer
// TMEM.
//
// LN_in's affine is folded into the weights: the LayerNorm warps write the
// bare normalised rows zh = (z - mean) rstd and the host stores
// W~ = W diag(gamma_in) / 2 with the bias W beta_in / 2 per row, so the
// accumulators plus bias hold v/2 and g/2 and the epilogue evaluates
//     sigmoid(g) * v * m = (v/2) m (1 + tanh(g/2))
// with one tanh per two outputs (tanh.approx.f16x2).
//
// Structure per CTA (one persistent CTA pair per two SMs, 480 threads each):
//   warp 0       TMA producer of this CTA's z half-tiles (128 pairs x D, bf16)
//                into a ring of 2 to 4 buffers
//   warp 1       TMEM (512 columns, allocated pairwise); in the even CTA, lane 0
//                issues the MMAs
//   warp 2       TMA producer of this CTA's weight slabs (128 rows x 64 K,
//                fp16) into a ring, signalled to the even CTA; when all of the
//                CTA's slabs fit in the ring they are loaded once and kept
//   warps 3..6   LayerNorm of the CTA's 128 pairs, one thread per pair, zh
//                written back in place as fp16; then one release arrival on
//                the even CTA's z-ready barrier
//   warps 7..22  epilogue: warp (h, q) takes TMEM quadrant q (16 channels) and
//                pairs h*64 .. h*64+63 of each chunk's accumulator:
//                sigmoid(gate) * value * mask -> fp16, staged in shared memory
//                and written by one TMA store of the 16-channel x 64-pair box
//                (two 8-channel boxes where it straddles the a / b boundary).
//                The CTA's epilogue warps meet at a named barrier after their
//                accumulator reads, and one thread per CTA signals the even CTA
//                that the buffer is free.  Sixteen warps (four per SMSP) keep
//                enough TMEM loads and arithmetic in flight to match the MMAs;
//                the tile's mask values are staged in shared memory one tile
//                ahead by the first 128 epilogue threads.
#include "kernels.h"
#include "sm103_ptx.cuh"

namespace trimul {

namespace {
constexpr int TP = INPROJ_TILE_PAIRS;       // pairs per tile (per CTA pair)
constexpr int HALF = INPROJ_HALF_PAIRS;     // pairs per CTA
constexpr int CH = 64;                      // output channels per CTA per chunk (128 weight rows)
constexpr uint32_t Z_SLAB = HALF * 128;     // 16 KB: 128 pair rows x 64 K
constexpr uint32_t W_SLAB = 2 * CH * 128;   // 16 KB: 128 weight rows x 64 K
constexpr uint32_t STAGE_OUT = 16 * 128;    // per epilogue warp: one box of 16 channel rows x 64 pairs
constexpr uint32_t MASK_SLOT = TP * 2;      // one tile's mask values (fp16)
constexpr uint32_t BAR_BYTES = 512;
constexpr uint32_t TMEM_COLS = 512;
constexpr int EPI_WARPS = 16;               // four per TMEM quadrant, 64 pairs each
constexpr int LN_THREADS = HALF;            // one thread per pair row
constexpr int THREADS = 96 + LN_THREADS + 32 * EPI_WARPS;
constexpr int MAX_W_STAGES = INPROJ_MAX_W_STAGES;
constexpr int MAX_Z_BUFS = INPROJ_MAX_Z_BUFS;
static_assert(24 * MAX_Z_BUFS + 16 * MAX_W_STAGES + 48 <= BAR_BYTES, "barrier block too small");

struct Layout {
  uint32_t z, w, stage, mask, bars, total;
};

__host__ __device__ inline Layout layout(int k_slabs, int w_stages, int z_bufs) {
  Layout L;
  uint32_t o = 0;
  L.z = o;  // z_bufs buffers of k_slabs slabs
  o += z_bufs * k_slabs * Z_SLAB;
  L.w = o;
  o += w_stages * W_SLAB;
  L.stage = o;
  o += EPI_WARPS * STAGE_OUT;
  L.mask = o;  // two tile slots of mask values, by tile parity
  o += 2 * MASK_SLOT;
  L.bars = o;
  o += BAR_BYTES;
  L.total = o + 1024;  // slack for aligning the base to 1024 bytes
  return L;
}
}  // namespace

size_t inproj_smem_bytes(int k_slabs, int w_stages, int z_bufs) { return layout(k_slabs, w_stages, z_bufs).total; }

// kResident: all of the CTA's weight slabs stay in the ring (loaded once).
// A compile-time switch: the streaming loop is the hot path at C = 256.
// kOut: how a and b are stored.  INPROJ_OUT_F16 (the forward); INPROJ_OUT_BF16
// (the backward pass's planes, which meet bf16 gradients in the tensor cores);
// INPROJ_OUT_E4M3 (the opt-in 8-bit triangle path: a * fp8_scale rounded to
// e4m3, saturating; each staged box row is 64 bytes, stored unswizzled).
template <bool kResident, int kOut>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(THREADS, 1)
    k1_inproj(const __grid_constant__ CUtensorMap tm_z, const __grid_constant__ CUtensorMap tm_w,
              const __grid_constant__ CUtensorMap tm_a, const __grid_constant__ CUtensorMap tm_b,
              const __grid_constant__ CUtensorMap tm_a8, const __grid_constant__ CUtensorMap tm_b8,
              const __grid_constant__ CUtensorMap tm_zh, const InprojArgs p) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_addr(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* const base_ptr = smem_raw + (base - raw);
  const Layout L = layout(p.k_slabs, p.w_stages, p.z_bufs);
  const uint32_t z_buf_bytes = p.k_slabs * Z_SLAB;
  const uint32_t zbuf0 = base + L.z, wring = base + L.w, bars = base + L.bars;
  const uint32_t zfull0 = bars, zready0 = zfull0 + 8 * MAX_Z_BUFS, zempty0 = zready0 + 8 * MAX_Z_BUFS;
  const uint32_t wfull0 = zempty0 + 8 * MAX_Z_BUFS, wempty0 = wfull0 + 8 * MAX_W_STAGES;
  const uint32_t tfull0 = wempty0 + 8 * MAX_W_STAGES, tempty0 = tfull0 + 16;
  const uint32_t drain = tempty0 + 16, tmem_slot = drain + 8;
  volatile uint32_t* tmem_slot_ptr = reinterpret_cast<volatile uint32_t*>(base_ptr + (tmem_slot - base));

  const KStatus st{p.status, p.timeout_ns};
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();  // 0: issues the MMAs
  // the backward's recompute (bf16 a, b): bf16 LayerNorm output and weights,
  // and optionally the normalised z itself stored as zh
  const bool zh_out = kOut == INPROJ_OUT_BF16 && p.write_zhat != 0;
  const bool leader = rank == 0;

  if (threadIdx.x == 0) {
    for (int i = 0; i < p.z_bufs; ++i) {
      mbar_init(zfull0 + 8 * i, 1);           // this CTA's z loads
      mbar_init(zready0 + 8 * i, 2);          // leader only: one arrival from the LayerNorm of each CTA
      // one multicast commit per phase, and with zh stores the LayerNorm's
      // arrival once its store has read the buffer
      mbar_init(zempty0 + 8 * i, zh_out ? 2 : 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(tfull0 + 8 * i, 1);           // one multicast commit per phase
      mbar_init(tempty0 + 8 * i, 2);          // leader only: one arrival from the epilogue of each CTA
    }
    for (int s = 0; s < p.w_stages; ++s) {
      mbar_init(wfull0 + 8 * s, 1);   // leader only: one expect_tx arrival; bytes of both CTAs
      mbar_init(wempty0 + 8 * s, 1);  // one multicast commit per phase
    }
    mbar_init(drain, 1);
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc_pair(tmem_slot, TMEM_COLS);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  cluster_sync_all();  // barriers of both CTAs initialised before any remote signal
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot_ptr;

  const int total = p.tile_end;
  const int cluster = p.tile_begin + (blockIdx.x >> 1), n_clusters = gridDim.x >> 1;
  const int n_cc = p.n_chunks;  // chunks of 128 channels (64 per CTA)

  if (warp == 0) {
    // ------------------------------------------------------------ z producer (both CTAs)
    if (lane == 0 && !p.inject_stall) {
      tma_prefetch_desc(&tm_z);
      long long z_issued = 0;
      int zb = 0;
      uint32_t zph = 0;
      for (int tile = cluster; tile < total; tile += n_clusters) {
        if (!mbar_wait(zempty0 + 8 * zb, zph ^ 1u, st, SITE_PRODUCER)) break;
        const int bb = tile / p.tiles_per_batch;
        // a half-tile wholly past N*N loads rows 0.. instead: its pairs are not stored
        long long prow = static_cast<long long>(tile - bb * p.tiles_per_batch) * TP + rank * HALF;
        if (prow >= p.NN) prow = 0;
        const uint32_t fb = zfull0 + 8 * zb;
        mbar_arrive_expect_tx(fb, z_buf_bytes);
        for (int s = 0; s < p.k_slabs; ++s)
          tma_load_3d(zbuf0 + zb * z_buf_bytes + s * Z_SLAB, &tm_z, fb, s * 64, static_cast<int>(prow), bb);
        ++z_issued;
        if (++zb == p.z_bufs) {
          zb = 0;
          zph ^= 1u;
        }
      }
      if (status_failed(st))
        for (long long i = (z_issued > p.z_bufs ? z_issued - p.z_bufs : 0); i < z_issued; ++i)
          mbar_wait_drain(zfull0 + 8 * static_cast<int>(i % p.z_bufs),
                          static_cast<uint32_t>(i / p.z_bufs) & 1u, p.timeout_ns);
    }
  } else if (warp == 2) {
    // ------------------------------------------------------------ weight producer (both CTAs)
    if (lane == 0 && !p.inject_stall) {
      tma_prefetch_desc(&tm_w);
      int ws = 0;
      uint32_t wph = 0;
      long long w_issued = 0;
      bool ok = true;
      // resident weights: one pass over the chunks (stage cc * k_slabs + s)
      const int tile_end_w = kResident ? min(total, cluster + 1) : total;
      for (int tile = cluster; tile < tile_end_w && ok; tile += n_clusters) {
        for (int cc = 0; cc < n_cc && ok; ++cc) {
          for (int s = 0; s < p.k_slabs; ++s) {
            if (!mbar_wait(wempty0 + 8 * ws, wph ^ 1u, st, SITE_PRODUCER)) {
              ok = false;
              break;
            }
            if (leader) mbar_arrive_expect_tx(wfull0 + 8 * ws, 2 * W_SLAB);
            tma_load_2d_pair(wring + ws * W_SLAB, &tm_w, mapa_shared(wfull0 + 8 * ws, 0), s * 64,
                             cc * 4 * CH + static_cast<int>(rank) * 2 * CH);
            ++w_issued;
            if (++ws == p.w_stages) {
              ws = 0;
              wph ^= 1u;
            }
          }
        }
      }
      if (!ok && leader) {
        int s = ws;
        uint32_t ph = wph;
        for (long long i = 0; i < w_issued && i < p.w_stages; ++i) {
          if (--s < 0) {
            s = p.w_stages - 1;
            ph ^= 1u;
          }
          mbar_wait_drain(wfull0 + 8 * s, ph, p.timeout_ns);
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer (even CTA)
    if (lane == 0 && leader) {
      const uint32_t idesc = kOut == INPROJ_OUT_BF16 ? idesc_bf16_f32(4 * CH, TP, 0, 0) : idesc_f16_f32(4 * CH, TP, 0, 0);
      // Descriptors of buffer / stage 0; a buffer, stage, slab or K step is a
      // plain add to the start address field (every address stays below 256 KB,
      // so the field cannot carry out).  Both CTAs hold their halves at the same
      // offsets.
      const uint64_t zdesc0 = sdesc_sw128(zbuf0, 16, 1024);
      const uint64_t wdesc0 = sdesc_sw128(wring, 16, 1024);
      int ws = 0, acc = 0;
      uint32_t wph = 0, aph = 0;
      bool ok = true;
      int zb = 0;
      uint32_t zph = 0;
      // resident weights: every stage lands once, before the first tile
      constexpr bool w_ready = kResident;
      if (w_ready && cluster < total)
        for (int i = 0; i < n_cc * p.k_slabs && ok; ++i) ok = mbar_wait(wfull0 + 8 * i, 0, st, SITE_MMA);
      for (int tile = cluster; tile < total && ok; tile += n_clusters) {
        if (!mbar_wait_cluster(zready0 + 8 * zb, zph, st, SITE_MMA)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint64_t zdesc = zdesc0 + ((zb * z_buf_bytes) >> 4);
        for (int cc = 0; cc < n_cc && ok; ++cc) {
          if (!mbar_wait_cluster(tempty0 + 8 * acc, aph ^ 1u, st, SITE_MMA)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t d = tmem_base + acc * TP;
          for (int s = 0; s < p.k_slabs; ++s) {
            if (kResident) ws = cc * p.k_slabs + s;  // each stage holds one slab for good
            if (!w_ready && !mbar_wait(wfull0 + 8 * ws, wph, st, SITE_MMA)) {
              ok = false;
              break;
            }
            tc_fence_after();
            const uint64_t bd = zdesc + ((s * Z_SLAB) >> 4), ad = wdesc0 + ((ws * W_SLAB) >> 4);
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) mma_f16_ss_pair(d, ad + 2 * kk, bd + 2 * kk, idesc, (s | kk) != 0);
            if (!kResident) {
              mma_commit_pair(wempty0 + 8 * ws, 0x3);
              if (++ws == p.w_stages) {
                ws = 0;
                wph ^= 1u;
              }
            }
          }
          if (!ok) break;
          mma_commit_pair(tfull0 + 8 * acc, 0x3);
          if (++acc == 2) {
            acc = 0;
            aph ^= 1u;
          }
        }
        if (!ok) break;
        mma_commit_pair(zempty0 + 8 * zb, 0x3);
        if (++zb == p.z_bufs) {
          zb = 0;
          zph ^= 1u;
        }
      }
      if (!ok) {
        mma_commit_pair(drain, 0x1);
        mbar_wait_drain(drain, 0, p.timeout_ns);
      }
    }
  } else if (warp < 3 + LN_THREADS / 32) {
    // ------------------------------------------------------------ LayerNorm (in place; fp16 out, bf16 for the backward's recompute)
    const uint32_t r = threadIdx.x - 96;  // pair row of this CTA's half tile
    const float inv_d = 1.0f / static_cast<float>(p.D);
    const int n8 = p.D >> 3;  // 8-element chunks per row
    const uint32_t zready_leader = mapa_shared(zready0, 0);
    int zb = 0;
    uint32_t zph = 0;
    int zh_pending = -1;  // buffer whose zh store has not been confirmed read yet
    for (int tile = cluster; tile < total; tile += n_clusters) {
      if (zh_out && r == 0 && zh_pending >= 0) {  // the previous tile's zh store has read its buffer
        tma_store_wait_read<0>();
        mbar_arrive(zempty0 + 8 * zh_pending);
        zh_pending = -1;
      }
      if (!named_bar_and(1, LN_THREADS, mbar_wait(zfull0 + 8 * zb, zph, st, SITE_XFORM))) break;
      uint8_t* const zrow = base_ptr + L.z + zb * z_buf_bytes;
      // One pass for the statistics, shifted by the row's first element so
      // that a large common offset does not cancel in E[(v-K)^2] - E[v-K]^2.
      const float shift = bf16_lo(*reinterpret_cast<const uint32_t*>(zrow + sw128_offset(r, 0)));
      float2 s1[4], s2[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) s1[e] = s2[e] = make_float2(0.f, 0.f);
      const float2 nsh = make_float2(-shift, -shift);
#pragma unroll 4
      for (int c8 = 0; c8 < n8; ++c8) {
        const uint4 v = *reinterpret_cast<const uint4*>(zrow + (c8 >> 3) * Z_SLAB + sw128_offset(r, (c8 & 7) * 8));
        const uint32_t w4[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float2 d = __fadd2_rn(make_float2(bf16_lo(w4[e]), bf16_hi(w4[e])), nsh);
          s1[e] = __fadd2_rn(s1[e], d);
          s2[e] = __ffma2_rn(d, d, s2[e]);
        }
      }
      float t1 = 0.f, t2 = 0.f;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        t1 += s1[e].x + s1[e].y;
        t2 += s2[e].x + s2[e].y;
      }
      const float m1 = t1 * inv_d;
      const float mu = shift + m1;
      const float rstd = rsqrtf(fmaxf(t2 * inv_d - m1 * m1, 0.f) + p.eps);
      if (p.zstats) {
        const int bb = tile / p.tiles_per_batch;
        const long long pidx = static_cast<long long>(tile - bb * p.tiles_per_batch) * TP + rank * HALF + r;
        if (pidx < p.NN) p.zstats[bb * p.NN + pidx] = make_float2(mu, rstd);
      }
      // zh = (z - mean) rstd = z rstd - mean rstd, two elements per packed FMA
      const float2 r2 = make_float2(rstd, rstd), nmr2 = make_float2(-mu * rstd, -mu * rstd);
#pragma unroll 4
      for (int c8 = 0; c8 < n8; ++c8) {
        uint4* const ptr = reinterpret_cast<uint4*>(zrow + (c8 >> 3) * Z_SLAB + sw128_offset(r, (c8 & 7) * 8));
        const uint4 v = *ptr;
        const uint32_t w4[4] = {v.x, v.y, v.z, v.w};
        uint32_t o4[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float2 y = __ffma2_rn(make_float2(bf16_lo(w4[e]), bf16_hi(w4[e])), r2, nmr2);
          o4[e] = kOut == INPROJ_OUT_BF16 ? pack_bf162(y.x, y.y) : pack_half2(y.x, y.y);
        }
        *ptr = make_uint4(o4[0], o4[1], o4[2], o4[3]);
      }
      // The leader's tensor cores read this buffer: make the generic writes
      // visible to the async proxy, gather the LayerNorm threads, then one
      // release arrival (cluster scope) on the leader's z-ready barrier.
      fence_proxy_async_all();
      named_bar_sync(3, LN_THREADS);
      if (r == 0) {
        mbar_arrive_cluster(zready_leader + 8 * zb);
        if (zh_out) {
          // zh: the normalised half tile, stored slab by slab from the buffer
          // (rows past N*N are clipped; a half tile wholly past them, which
          // was loaded from rows 0.., is not stored)
          const int bb = tile / p.tiles_per_batch;
          const long long prow = static_cast<long long>(tile - bb * p.tiles_per_batch) * TP + rank * HALF;
          if (prow < p.NN)
            for (int s = 0; s < p.k_slabs; ++s)
              tma_store_3d(&tm_zh, zbuf0 + zb * z_buf_bytes + s * Z_SLAB, s * 64, static_cast<int>(prow), bb);
          tma_store_commit();
          zh_pending = zb;
        }
      }
      if (++zb == p.z_bufs) {
        zb = 0;
        zph ^= 1u;
      }
    }
    if (zh_out && r == 0) tma_store_wait_all();  // the zh stores have completed before the CTA exits
  } else {
    // ------------------------------------------------------------ epilogue (both CTAs)
    // Warp (hc, q): TMEM quadrant q, i.e. the CTA's weight rows q*32 .. q*32+31
    // of a chunk = channels q*16 .. q*16+15 of the CTA's 64 (two 16-lane
    // groups g of 8 channels), and the pairs hc*64 .. hc*64+63 of the tile.
    // Thread t holds channel g*8 + t/4 of the warp's 16 and, in each 32-pair
    // block j, the pairs 8k + 2(t%4) and 8k + 2(t%4) + 1 (k = 0..3).
    const int ew = warp - 3 - LN_THREADS / 32;  // 0..15
    const int e = ew * 32 + lane;                 // epilogue thread index
    const int q = warp & 3;                       // TMEM lane quadrant
    const int hc = ew >> 2;                       // 64-pair quarter of the tile
    const uint32_t stage = base + L.stage + ew * STAGE_OUT;
    const uint32_t lrow = static_cast<uint32_t>(lane) >> 2;  // row within an 8-row group
    const uint32_t cpair = 2u * (lane & 3);                  // pair offset within an 8-pair group
    const uint32_t tempty_leader = mapa_shared(tempty0, 0);
    const bool track = p.ab_max != nullptr;
    constexpr int EPI_THREADS = 32 * EPI_WARPS;
    // Mask staging: thread e < TP / 2 owns the pairs 2e, 2e + 1 of every tile.
    // Slot n % 2 holds tile n's values (fp16 pairs); the raw bf16 pair of the
    // tile after next waits in a register, loaded a whole tile ahead.
    uint32_t* const mslot = reinterpret_cast<uint32_t*>(base_ptr + L.mask);
    auto mask_word = [&](int t) -> uint32_t {  // raw bf16 pair of tile t, or two ones
      if (!p.mask || e >= TP / 2 || t >= total) return 0x3F803F80u;
      const int tb = t / p.tiles_per_batch;
      const long long pm = static_cast<long long>(t - tb * p.tiles_per_batch) * TP + 2 * e;
      // NN is a multiple of 64: both pairs are in or out together
      return pm < p.NN ? __ldg(reinterpret_cast<const unsigned int*>(p.mask + tb * p.NN + pm)) : 0x3F803F80u;
    };
    auto stage_mask = [&](int slot, uint32_t raw) {
      if (e >= TP / 2) return;
      const float m0 = bf16_lo(raw), m1 = bf16_hi(raw);
      // the binary16 range of a and b assumes 0 <= m <= 1 (NaN fails the test too)
      if (!(m0 >= 0.f && m0 <= 1.f && m1 >= 0.f && m1 <= 1.f) && p.mask_flag) atomicOr(p.mask_flag, 1);
      mslot[slot * (TP / 2) + e] = pack_half2(m0, m1);
    };
    stage_mask(0, mask_word(cluster));
    uint32_t mnext = mask_word(cluster + n_clusters);
    int acc = 0;
    uint32_t aph = 0;
    bool ok = true;
    // running max of |a|, |b| over this thread's stored values (for the call's x scale)
    __half2 vmax = __float2half2_rn(0.f);
    int n = 0;
    for (int tile = cluster; tile < total && ok; tile += n_clusters, ++n) {
      const int bb = tile / p.tiles_per_batch;
      const long long pb = static_cast<long long>(tile - bb * p.tiles_per_batch) * TP + hc * 64;
      // every epilogue warp is done with tile n - 1 (whose slot is refilled now)
      // and sees slot n % 2 complete
      named_bar_sync(5, EPI_THREADS);
      stage_mask((n + 1) & 1, mnext);
      mnext = mask_word(tile + 2 * n_clusters);
      const uint32_t* const mrow = mslot + (n & 1) * (TP / 2) + (hc * 64 + cpair) / 2;
      for (int cc = 0; cc < n_cc; ++cc) {
        // every warp reaches the named barrier below (its wait is bounded) and
        // the barrier's AND makes the bail-out uniform across the warps
        const bool got = __all_sync(0xffffffffu, mbar_wait(tfull0 + 8 * acc, aph, st, SITE_EPI));
        tc_fence_after();
        const int ob = cc * 2 * CH + static_cast<int>(rank) * CH + q * 16;  // first output channel of the warp
        const int rw = cc * 4 * CH + static_cast<int>(rank) * 2 * CH + q * 32 + static_cast<int>(lrow);
        float2 bv2[2], bg2[2];  // biases of this thread's channel in lane group g (value row, gate row)
#pragma unroll
        for (int g = 0; g < 2; ++g) {
          const float bv = __ldg(p.bias + rw + g * 16), bg = __ldg(p.bias + rw + g * 16 + 8);
          bv2[g] = make_float2(bv, bv);
          bg2[g] = make_float2(bg, bg);
        }
        const uint32_t t_addr = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + acc * TP + hc * 64;
        // step i: lane group g = i / 2, 32-pair block j = i % 2; the loads run one step ahead
        auto step_addr = [&](int i) -> uint32_t {
          return t_addr + (static_cast<uint32_t>((i >> 1) * 16) << 16) + static_cast<uint32_t>((i & 1) * 32);
        };
        uint32_t ra[16], rb[16];
        if (got) tmem_ld16x256b_x4(step_addr(0), ra);
        // the previous store has read the staging box
        if (lane == 0) tma_store_wait_read<0>();
        __syncwarp();
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int g = i >> 1, j = i & 1;
          uint32_t(&cur)[16] = (i & 1) ? rb : ra;
          if (got) tmem_ld_wait();
          if (i < 3 && got) tmem_ld16x256b_x4(step_addr(i + 1), (i & 1) ? ra : rb);
          if (i == 3) {
            // the accumulator is in registers now: once every epilogue warp of
            // the CTA is done with it, one thread hands it back to the MMA warp
            tc_fence_before();
            if (!named_bar_and(4, EPI_THREADS, got)) ok = false;
            if (ok && ew == 0 && lane == 0) mbar_arrive_remote(tempty_leader + 8 * acc);
          }
          if (!ok) break;
          // staged row g*8 + t/4; this thread's 4 bytes sit at byte 2 * cpair
          // of each 16-byte chunk (e4m3: its 2 bytes at byte j*32 + 8k + cpair
          // of a 64-byte row)
          uint8_t* const srow = base_ptr + L.stage + ew * STAGE_OUT +
                                (g * 8 + lrow) * (kOut == INPROJ_OUT_E4M3 ? 64u : 128u) +
                                cpair * (kOut == INPROJ_OUT_E4M3 ? 1u : 2u);
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const uint32_t m2 = mrow[(j * 32 + 8 * k) / 2];  // fp16 mask pair
            // accumulator + bias = v/2 and g/2 (the host halved the weights)
            const float2 v2 = __fadd2_rn(make_float2(__uint_as_float(cur[4 * k]), __uint_as_float(cur[4 * k + 1])), bv2[g]);
            const float2 g2 =
                __fadd2_rn(make_float2(__uint_as_float(cur[4 * k + 2]), __uint_as_float(cur[4 * k + 3])), bg2[g]);
            const __half2 g16 = __float22half2_rn(g2);
            const uint32_t th16 = tanh_h2(*reinterpret_cast<const uint32_t*>(&g16));
            uint32_t packed;
            if (kOut == INPROJ_OUT_E4M3) {
              const float2 th = __half22float2(*reinterpret_cast<const __half2*>(&th16));
              const float2 y = __ffma2_rn(v2, th, v2);
              const float2 mf = __half22float2(*reinterpret_cast<const __half2*>(&m2));
              const float2 ym = make_float2(y.x * mf.x, y.y * mf.y);
              // the max of the values before rounding sets the x scale, as in fp16
              if (track) vmax = __hmax2(vmax, __habs2(__floats2half2_rn(ym.x, ym.y)));
              const __nv_fp8x2_storage_t q = __nv_cvt_float2_to_fp8x2(
                  make_float2(ym.x * p.fp8_scale, ym.y * p.fp8_scale), __NV_SATFINITE, __NV_E4M3);
              *reinterpret_cast<__nv_fp8x2_storage_t*>(srow + j * 32 + 8 * k) = q;
              continue;
            } else if (kOut == INPROJ_OUT_BF16) {
              const float2 th = __half22float2(*reinterpret_cast<const __half2*>(&th16));
              const float2 y = __ffma2_rn(v2, th, v2);
              const float2 mf = __half22float2(*reinterpret_cast<const __half2*>(&m2));
              packed = pack_bf162(y.x * mf.x, y.y * mf.y);
              // |a|, |b| <= 65504 (checked at create), so fp16 holds them
              if (track) vmax = __hmax2(vmax, __habs2(__floats2half2_rn(bf16_lo(packed), bf16_hi(packed))));
            } else {
              // (v/2)(1 + tanh(g/2)) m in fp16: v/2 rounded once, one fma, one product
              const __half2 v16 = __float22half2_rn(v2);
              const __half2 yh = __hmul2(__hfma2(v16, *reinterpret_cast<const __half2*>(&th16), v16),
                                         *reinterpret_cast<const __half2*>(&m2));
              packed = *reinterpret_cast<const uint32_t*>(&yh);
              if (track) vmax = __hmax2(vmax, __habs2(yh));
            }
            // 16-byte chunk 4j + k of the staged row, 128-byte swizzle
            *reinterpret_cast<uint32_t*>(srow + (((static_cast<uint32_t>(4 * j + k) ^ lrow) & 7u) << 4)) = packed;
          }
        }
        if (!ok) break;
        // the box is complete: one store (16 channels x 64 pairs)
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          if (got && pb < p.NN && ob < 2 * p.C) {
            if (ob + 16 <= p.C) {
              tma_store_3d(&tm_a, stage, static_cast<int>(pb), ob, bb);
            } else if (ob >= p.C) {
              tma_store_3d(&tm_b, stage, static_cast<int>(pb), ob - p.C, bb);
            } else {  // C = ob + 8: the first 8 channels are a's, the last 8 b's
              tma_store_3d(&tm_a8, stage, static_cast<int>(pb), ob, bb);
              tma_store_3d(&tm_b8, stage + (kOut == INPROJ_OUT_E4M3 ? 512 : 1024), static_cast<int>(pb), 0, bb);
            }
          }
          tma_store_commit();
        }
        if (++acc == 2) {
          acc = 0;
          aph ^= 1u;
        }
      }
    }
    if (lane == 0) tma_store_wait_all();
    if (track) {
      // Values computed but not stored (pairs past N*N, from zero-filled or
      // redirected z rows; channels past 2C, from zero weight rows) are outputs
      // of the same layer too, so they can only raise the max to another valid
      // bound.  The bits of non-negative floats order like the floats, so an
      // unsigned max works.
      float m = fmaxf(__low2float(vmax), __high2float(vmax));
#pragma unroll
      for (int o = 16; o >= 1; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
      if (lane == 0) atomicMax(p.ab_max, __float_as_uint(m));
    }
  }

  tc_fence_before();
  __syncthreads();
  cluster_sync_all();  // no CTA leaves while its peer may still signal it
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem_base, TMEM_COLS);
  }
}

cudaError_t launch_inproj(const InprojArgs& a, const CUtensorMap& tm_z, const CUtensorMap& tm_w,
                          const CUtensorMap& tm_a, const CUtensorMap& tm_b, const CUtensorMap& tm_a8,
                          const CUtensorMap& tm_b8, const CUtensorMap& tm_zh, int grid, cudaStream_t s) {
  if (a.w_stages < (a.w_resident ? 1 : 2) || a.w_stages > MAX_W_STAGES || a.z_bufs < 2 || a.z_bufs > MAX_Z_BUFS)
    return cudaErrorInvalidValue;
  const size_t smem = inproj_smem_bytes(a.k_slabs, a.w_stages, a.z_bufs);
  auto* const kern =
      a.out_kind == INPROJ_OUT_BF16   ? (a.w_resident ? k1_inproj<true, INPROJ_OUT_BF16> : k1_inproj<false, INPROJ_OUT_BF16>)
      : a.out_kind == INPROJ_OUT_E4M3 ? (a.w_resident ? k1_inproj<true, INPROJ_OUT_E4M3> : k1_inproj<false, INPROJ_OUT_E4M3>)
                                      : (a.w_resident ? k1_inproj<true, INPROJ_OUT_F16> : k1_inproj<false, INPROJ_OUT_F16>);
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  grid &= ~1;  // whole CTA pairs
  if (grid < 2) grid = 2;
  kern<<<grid, THREADS, smem, s>>>(tm_z, tm_w, tm_a, tm_b, tm_a8, tm_b8, tm_zh, a);
  return cudaGetLastError();
}

int inproj_max_pairs(int num_sms, int k_slabs, int w_stages, int z_bufs) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(num_sms & ~1, 1, 1);
  cfg.blockDim = dim3(THREADS, 1, 1);
  cfg.dynamicSmemBytes = inproj_smem_bytes(k_slabs, w_stages, z_bufs);
  cudaLaunchAttribute attr;
  attr.id = cudaLaunchAttributeClusterDimension;
  attr.val.clusterDim.x = 2;
  attr.val.clusterDim.y = 1;
  attr.val.clusterDim.z = 1;
  cfg.attrs = &attr;
  cfg.numAttrs = 1;
  // every instantiation has the same footprint and cluster shape
  cudaFuncSetAttribute(k1_inproj<false, INPROJ_OUT_F16>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                       static_cast<int>(cfg.dynamicSmemBytes));
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, k1_inproj<false, INPROJ_OUT_F16>, &cfg) != cudaSuccess || n < 1) {
    cudaGetLastError();
    return num_sms / 2;
  }
  return n;
}

}  // namespace trimul
