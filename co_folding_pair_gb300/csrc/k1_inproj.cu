// k1_inproj.cu -- LayerNorm(z) + gated input projection + pair mask, stored channel-major.
//
// fold-cp-ops README, "Use": norm_in = LayerNorm(D); p_in, g_in = Linear(D, 2D,
// bias=False) produce the value and gate of a (first half) and b (second half);
// the (B, N, N) pair mask multiplies them.  Per pair p and channel c:
//     a[b, c, p] = sigmoid(z'_p . W_ga[c]) * (z'_p . W_a[c]) * m_p,  z'_p = LN_in(z_p)
// and the same for b.  The result is written channel-major ([B][C][N*N]) so the
// triangle GEMM reads each channel plane contiguously; no separate permute runs.
//
// The GEMM is computed transposed, channels x pairs, so the accumulator's TMEM
// lanes are channels and its columns are consecutive pairs: each epilogue
// lane owns one channel row and 64 consecutive pairs of it, 128 contiguous
// bytes of a channel plane.
//
// CTA pairs: a cluster of two CTAs takes a tile of 128 pairs.  Each CTA loads
// and normalises its own 64 pairs (half of the MMA's B operand) and stages the
// weights of its own 128 channels of every 256-channel chunk (half of the A
// operand); the even CTA issues tcgen05.mma.cta_group::2 (M = 256 channels,
// N = 128 pairs, K = 16), which leaves each CTA the accumulators of its own
// channels for all 128 pairs.  LN_in's affine is folded into the weights:
// the LayerNorm warps write the bare normalised rows zh = (z - mean) rstd and
// the host stores W~ = W diag(gamma_in) / 2 with the bias W beta_in / 2 per
// row, so the accumulators plus bias hold v/2 and g/2 and the epilogue
// evaluates
//     sigmoid(g) * v * m = (v/2) m (1 + tanh(g/2))
// with one tanh per two outputs (tanh.approx.f16x2).
//
// Structure per CTA (one persistent CTA pair per two SMs, 480 threads each):
//   warp 0       TMA producer of this CTA's z half-tiles (64 pairs x D, bf16)
//                into a ring of 2 to 8 buffers
//   warp 1       TMEM (512 columns, allocated pairwise); in the even CTA, lane 0
//                issues the MMAs
//   warp 2       TMA producer of this CTA's weight slabs (128 value rows + their
//                128 gate rows, x 64 K, fp16) into a ring, signalled to the even
//                CTA; when all of the CTA's slabs fit in the ring (C <= 128 with
//                few enough K slabs), they are loaded once and kept
//   warps 3..6   LayerNorm of the CTA's 64 pairs, two adjacent lanes per pair, zh
//                written back in place as fp16; then one release arrival on
//                the even CTA's z-ready barrier
//   warps 7..14  epilogue: per chunk, warp (h, q) takes the 32 channels of TMEM
//                quadrant q and pairs h*64 .. h*64+63: sigmoid(gate) * value *
//                mask -> fp16, staged in shared memory and written by one TMA
//                store of the 32 x 64 block (four 8-channel boxes where the
//                block straddles the a / b boundary).  The CTA's epilogue warps
//                meet at a named barrier after their accumulator reads, and one
//                thread per CTA signals the even CTA that the buffer is free.
// The accumulator pair (128 value + 128 gate columns) is double-buffered.
#include "kernels.h"
#include "sm103_ptx.cuh"

namespace trimul {

namespace {
constexpr int BM = 128;                     // pairs per tile (per CTA pair)
constexpr int HALF = INPROJ_HALF_PAIRS;     // pairs per CTA
constexpr int CH = 128;                     // output channels per CTA per chunk
constexpr uint32_t Z_SLAB = HALF * 128;     // 8 KB: 64 pair rows x 64 K
constexpr uint32_t W_SLAB = 2 * CH * 128;   // 32 KB: 128 value + 128 gate rows x 64 K
constexpr uint32_t STAGE_OUT = 4096;        // per epilogue warp: 32 channel rows x 128 B
constexpr uint32_t BAR_BYTES = 512;
constexpr uint32_t TMEM_COLS = 512;
constexpr int EPI_WARPS = 8;
constexpr int LN_THREADS = 128;
constexpr int THREADS = 96 + LN_THREADS + 32 * EPI_WARPS;
constexpr int MAX_W_STAGES = 4;
constexpr int MAX_Z_BUFS = 8;
static_assert(24 * MAX_Z_BUFS + 16 * MAX_W_STAGES + 40 <= BAR_BYTES, "barrier block too small");

struct Layout {
  uint32_t z, w, stage, maskh, bars, total;
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
  L.maskh = o;  // [EPI_WARPS][64] fp16: this warp's mask values of the tile
  o += EPI_WARPS * HALF * 2;
  L.bars = o;
  o += BAR_BYTES;
  L.total = o + 1024;  // slack for aligning the base to 1024 bytes
  return L;
}
}  // namespace

size_t inproj_smem_bytes(int k_slabs, int w_stages, int z_bufs) { return layout(k_slabs, w_stages, z_bufs).total; }

// kResident: all of the CTA's weight slabs stay in the ring (loaded once).
// A compile-time switch: the streaming loop is the hot path at C = 256 and
// measured slower with the residency tests made at run time.
// kBf16Out: a and b are stored as bf16 instead of fp16 (the backward pass's
// planes, which meet bf16 gradients in the tensor cores).
template <bool kResident, bool kBf16Out>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(THREADS, 1)
    k1_inproj(const __grid_constant__ CUtensorMap tm_z, const __grid_constant__ CUtensorMap tm_w,
              const __grid_constant__ CUtensorMap tm_a, const __grid_constant__ CUtensorMap tm_b,
              const __grid_constant__ CUtensorMap tm_a8, const __grid_constant__ CUtensorMap tm_b8,
              const InprojArgs p) {
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
  const bool leader = rank == 0;

  if (threadIdx.x == 0) {
    for (int i = 0; i < p.z_bufs; ++i) {
      mbar_init(zfull0 + 8 * i, 1);           // this CTA's z loads
      mbar_init(zready0 + 8 * i, 2);          // leader only: one arrival from the LayerNorm of each CTA
      mbar_init(zempty0 + 8 * i, 1);          // one multicast commit per phase
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
  const int n_cchunks = (p.n_chunks + 1) >> 1;  // chunks of 256 channels (128 per CTA)
  const int C2 = 2 * p.C;

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
        long long prow = static_cast<long long>(tile - bb * p.tiles_per_batch) * BM + rank * HALF;
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
        for (int cc = 0; cc < n_cchunks && ok; ++cc) {
          // this CTA's 128-channel group of the chunk; a group past the weights
          // loads group 0 instead (its channels are not stored)
          int grp = 2 * cc + static_cast<int>(rank);
          if (grp >= p.n_chunks) grp = 0;
          for (int s = 0; s < p.k_slabs; ++s) {
            if (!mbar_wait(wempty0 + 8 * ws, wph ^ 1u, st, SITE_PRODUCER)) {
              ok = false;
              break;
            }
            if (leader) mbar_arrive_expect_tx(wfull0 + 8 * ws, 2 * W_SLAB);
            tma_load_2d_pair(wring + ws * W_SLAB, &tm_w, mapa_shared(wfull0 + 8 * ws, 0), s * 64, grp * 2 * CH);
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
      const uint32_t idesc = idesc_f16_f32(2 * CH, BM, 0, 0);
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
        for (int i = 0; i < n_cchunks * p.k_slabs && ok; ++i) ok = mbar_wait(wfull0 + 8 * i, 0, st, SITE_MMA);
      for (int tile = cluster; tile < total && ok; tile += n_clusters) {
        if (!mbar_wait_cluster(zready0 + 8 * zb, zph, st, SITE_MMA)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint64_t zdesc = zdesc0 + ((zb * z_buf_bytes) >> 4);
        for (int cc = 0; cc < n_cchunks && ok; ++cc) {
          if (!mbar_wait_cluster(tempty0 + 8 * acc, aph ^ 1u, st, SITE_MMA)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t d_val = tmem_base + acc * 256, d_gate = d_val + 128;
          for (int s = 0; s < p.k_slabs; ++s) {
            if (kResident) ws = cc * p.k_slabs + s;  // each stage holds one slab for good
            if (!w_ready && !mbar_wait(wfull0 + 8 * ws, wph, st, SITE_MMA)) {
              ok = false;
              break;
            }
            tc_fence_after();
            const uint64_t bd = zdesc + ((s * Z_SLAB) >> 4), ad = wdesc0 + ((ws * W_SLAB) >> 4);
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
              mma_f16_ss_pair(d_val, ad + 2 * kk, bd + 2 * kk, idesc, (s | kk) != 0);
              mma_f16_ss_pair(d_gate, ad + ((CH * 128) >> 4) + 2 * kk, bd + 2 * kk, idesc, (s | kk) != 0);
            }
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
    // ------------------------------------------------------------ LayerNorm (in place, fp16 out)
    const uint32_t t = threadIdx.x - 96;
    const uint32_t r = t >> 1, hh = t & 1;  // pair row of this CTA's half, half of the row (adjacent lanes)
    const float inv_d = 1.0f / static_cast<float>(p.D);
    const int n8 = p.D >> 3;  // 8-element chunks per row
    const int c8_lo = hh ? n8 / 2 : 0, c8_hi = hh ? n8 : n8 / 2;
    const uint32_t zready_leader = mapa_shared(zready0, 0);
    int zb = 0;
    uint32_t zph = 0;
    for (int tile = cluster; tile < total; tile += n_clusters) {
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
      for (int c8 = c8_lo; c8 < c8_hi; ++c8) {
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
      t1 += __shfl_xor_sync(0xffffffffu, t1, 1);  // the other half of the row
      t2 += __shfl_xor_sync(0xffffffffu, t2, 1);
      const float m1 = t1 * inv_d;
      const float mu = shift + m1;
      const float rstd = rsqrtf(fmaxf(t2 * inv_d - m1 * m1, 0.f) + p.eps);
      if (p.zstats && hh == 0) {
        const int bb = tile / p.tiles_per_batch;
        const long long pidx = static_cast<long long>(tile - bb * p.tiles_per_batch) * BM + rank * HALF + r;
        if (pidx < p.NN) p.zstats[bb * p.NN + pidx] = make_float2(mu, rstd);
      }
      // zh = (z - mean) rstd = z rstd - mean rstd, two elements per packed FMA
      const float2 r2 = make_float2(rstd, rstd), nmr2 = make_float2(-mu * rstd, -mu * rstd);
#pragma unroll 4
      for (int c8 = c8_lo; c8 < c8_hi; ++c8) {
        uint4* const ptr = reinterpret_cast<uint4*>(zrow + (c8 >> 3) * Z_SLAB + sw128_offset(r, (c8 & 7) * 8));
        const uint4 v = *ptr;
        const uint32_t w4[4] = {v.x, v.y, v.z, v.w};
        uint32_t o4[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float2 y = __ffma2_rn(make_float2(bf16_lo(w4[e]), bf16_hi(w4[e])), r2, nmr2);
          o4[e] = pack_half2(y.x, y.y);
        }
        *ptr = make_uint4(o4[0], o4[1], o4[2], o4[3]);
      }
      // The leader's tensor cores read this buffer: make the generic writes
      // visible to the async proxy, gather the LayerNorm threads, then one
      // release arrival (cluster scope) on the leader's z-ready barrier.
      fence_proxy_async_all();
      named_bar_sync(3, LN_THREADS);
      if (t == 0) mbar_arrive_cluster(zready_leader + 8 * zb);
      if (++zb == p.z_bufs) {
        zb = 0;
        zph ^= 1u;
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue (both CTAs)
    const int ew = warp - 3 - LN_THREADS / 32;  // 0..7
    const int q = warp & 3;                       // TMEM lane quadrant = channels q*32 .. q*32+31
    const int colhalf = ew >> 2;                  // pairs colhalf*64 .. +63 of the tile
    const uint32_t stage = base + L.stage + ew * STAGE_OUT;
    uint4* const srow = reinterpret_cast<uint4*>(base_ptr + L.stage + ew * STAGE_OUT + lane * 128);
    uint32_t* const mh = reinterpret_cast<uint32_t*>(base_ptr + L.maskh + ew * HALF * 2);  // 32 half2
    const uint32_t sw = lane & 7;
    const uint32_t tempty_leader = mapa_shared(tempty0, 0);
    int acc = 0;
    uint32_t aph = 0;
    bool ok = true;
    // running max of |a|, |b| over this lane's stored values (for the call's x scale)
    __half2 vmax = __float2half2_rn(0.f);
    for (int tile = cluster; tile < total && ok; tile += n_clusters) {
      const int bb = tile / p.tiles_per_batch;
      const long long pp0 = static_cast<long long>(tile - bb * p.tiles_per_batch) * BM + colhalf * 64;
      // this warp's 64 mask values, as fp16 pairs in shared memory (two per lane)
      {
        const long long pm = pp0 + 2 * lane;
        float m0 = 1.f, m1 = 1.f;
        if (p.mask && pm < p.NN) {  // NN is even: both pairs are in or out together
          const uint32_t mv = __ldg(reinterpret_cast<const unsigned int*>(p.mask + bb * p.NN + pm));
          m0 = bf16_lo(mv);
          m1 = bf16_hi(mv);
        }
        // the binary16 range of a and b assumes 0 <= m <= 1 (NaN fails the test too)
        const bool bad = !(m0 >= 0.f && m0 <= 1.f && m1 >= 0.f && m1 <= 1.f);
        if (__any_sync(0xffffffffu, bad) && lane == 0 && p.mask_flag) atomicOr(p.mask_flag, 1);
        __syncwarp();
        mh[lane] = pack_half2(m0, m1);
        __syncwarp();
      }
      for (int cc = 0; cc < n_cchunks; ++cc) {
        // every warp reaches the named barrier below (its wait is bounded) and
        // the barrier's AND makes the bail-out uniform across the 8 warps
        const bool got = __all_sync(0xffffffffu, mbar_wait(tfull0 + 8 * acc, aph, st, SITE_EPI));
        tc_fence_after();
        const uint32_t t_addr = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + acc * 256 + colhalf * 64;
        // this lane's weight rows: value row grp*256 + q*32 + lane, gate row +128
        const int wrow = (2 * cc + static_cast<int>(rank)) * 2 * CH + q * 32 + lane;
        const bool grp_ok = 2 * cc + static_cast<int>(rank) < p.n_chunks;
        const float bv = grp_ok ? __ldg(p.bias + wrow) : 0.f, bg = grp_ok ? __ldg(p.bias + wrow + CH) : 0.f;
        const float2 bv2 = make_float2(bv, bv), bg2 = make_float2(bg, bg);
        // this lane's channel, the warp's 64 pairs: 8 chunks of 8 fp16
        uint4 R[8];
#pragma unroll
        for (int blk = 0; blk < 4 && got; ++blk) {  // 16 pairs at a time keeps the register footprint small
          uint32_t v[16], g[16];
          tmem_ld16(t_addr + blk * 16, v);
          tmem_ld16(t_addr + 128 + blk * 16, g);
          tmem_ld_wait();
#pragma unroll
          for (int u = 0; u < 2; ++u) {
            const uint4 m8 = *reinterpret_cast<const uint4*>(mh + (blk * 16 + u * 8) / 2);  // 8 fp16 mask values
            const uint32_t mm[4] = {m8.x, m8.y, m8.z, m8.w};
            uint32_t packed[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              // accumulator + bias = g/2 and v/2 (the host halved the weights)
              const float2 g2 = __fadd2_rn(
                  make_float2(__uint_as_float(g[u * 8 + 2 * e]), __uint_as_float(g[u * 8 + 2 * e + 1])), bg2);
              const float2 v2 = __fadd2_rn(
                  make_float2(__uint_as_float(v[u * 8 + 2 * e]), __uint_as_float(v[u * 8 + 2 * e + 1])), bv2);
              const __half2 g16 = __float22half2_rn(g2);
              const uint32_t th16 = tanh_h2(*reinterpret_cast<const uint32_t*>(&g16));
              const float2 th = __half22float2(*reinterpret_cast<const __half2*>(&th16));
              const float2 y = __ffma2_rn(v2, th, v2);
              if (kBf16Out) {
                const float2 mf = __half22float2(*reinterpret_cast<const __half2*>(&mm[e]));
                packed[e] = pack_bf162(y.x * mf.x, y.y * mf.y);
              } else {
                const __half2 yh = __hmul2(__floats2half2_rn(y.x, y.y), *reinterpret_cast<const __half2*>(&mm[e]));
                packed[e] = *reinterpret_cast<const uint32_t*>(&yh);
              }
            }
            R[blk * 2 + u] = make_uint4(packed[0], packed[1], packed[2], packed[3]);
          }
        }
        // the accumulator is in registers now: once every epilogue warp of the
        // CTA is done with it, one thread hands it back to the MMA warp
        tc_fence_before();
        if (!named_bar_and(4, 32 * EPI_WARPS, got)) {
          ok = false;
          break;
        }
        if (ew == 0 && lane == 0) mbar_arrive_cluster(tempty_leader + 8 * acc);
        const int grp = 2 * cc + static_cast<int>(rank);  // this CTA's 128-channel group
        if (++acc == 2) {
          acc = 0;
          aph ^= 1u;
        }
        // stage the 32 x 64 block (row = channel, 128-byte swizzle) and store it:
        // one 32-channel box when it lies wholly in a or in b, else four
        // 8-channel boxes (C is a multiple of 8, so those never straddle)
        if (p.ab_max) {
#pragma unroll
          for (int c = 0; c < 8; ++c) {
            const uint32_t w4[4] = {R[c].x, R[c].y, R[c].z, R[c].w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              if (kBf16Out)  // |a|, |b| <= 65504 (checked at create), so fp16 holds them
                vmax = __hmax2(vmax, __habs2(__floats2half2_rn(bf16_lo(w4[e]), bf16_hi(w4[e]))));
              else
                vmax = __hmax2(vmax, __habs2(*reinterpret_cast<const __half2*>(&w4[e])));
            }
          }
        }
        if (lane == 0) tma_store_wait_read<0>();  // the previous stores have read the buffer
        __syncwarp();
#pragma unroll
        for (int c = 0; c < 8; ++c) srow[c ^ sw] = R[c];
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0 && pp0 < p.NN) {
          const int ob = grp * CH + q * 32;  // first output channel of the block
          if (ob + 32 <= p.C) {
            tma_store_3d(&tm_a, stage, static_cast<int>(pp0), ob, bb);
          } else if (ob >= p.C && ob + 32 <= C2) {
            tma_store_3d(&tm_b, stage, static_cast<int>(pp0), ob - p.C, bb);
          } else {
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              const int o0 = ob + 8 * k;
              if (o0 < p.C)
                tma_store_3d(&tm_a8, stage + k * 1024, static_cast<int>(pp0), o0, bb);
              else if (o0 < C2)
                tma_store_3d(&tm_b8, stage + k * 1024, static_cast<int>(pp0), o0 - p.C, bb);
            }
          }
          tma_store_commit();
        }
      }
    }
    if (lane == 0) tma_store_wait_all();
    if (p.ab_max) {
      // Values computed but not stored (pairs past N*N, from zero-filled or
      // redirected z rows; channel groups past the weights, which repeat group
      // 0) are outputs of the same layer too, so they can only raise the max
      // to another valid bound.  The bits of non-negative floats order like
      // the floats, so an unsigned max works.
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
                          const CUtensorMap& tm_b8, int grid, cudaStream_t s) {
  if (a.w_stages < (a.w_resident ? 1 : 2) || a.w_stages > MAX_W_STAGES || a.z_bufs < 2 || a.z_bufs > MAX_Z_BUFS)
    return cudaErrorInvalidValue;
  const size_t smem = inproj_smem_bytes(a.k_slabs, a.w_stages, a.z_bufs);
  auto* const kern = a.out_bf16 ? (a.w_resident ? k1_inproj<true, true> : k1_inproj<false, true>)
                                : (a.w_resident ? k1_inproj<true, false> : k1_inproj<false, false>);
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  grid &= ~1;  // whole CTA pairs
  if (grid < 2) grid = 2;
  kern<<<grid, THREADS, smem, s>>>(tm_z, tm_w, tm_a, tm_b, tm_a8, tm_b8, a);
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
  cudaFuncSetAttribute(k1_inproj<false, false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                       static_cast<int>(cfg.dynamicSmemBytes));
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, k1_inproj<false, false>, &cfg) != cudaSuccess || n < 1) {
    cudaGetLastError();
    return num_sms / 2;
  }
  return n;
}

}  // namespace trimul
