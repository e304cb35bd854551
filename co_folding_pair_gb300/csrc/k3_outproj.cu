// k3_outproj.cu -- LayerNorm over channels of x, output projection, output gate.
//
// fold-cp-ops README, "Use": norm_out = LayerNorm, p_out = Linear(., D, bias=False),
// g_out = Linear(D, D, bias=False) applied to the normalised input z' = LN_in(z):
//     out[p, :] = sigmoid(z'_p W_g^T) * (LN_out(x_p) W_o^T)
//
// Both LayerNorms are folded into the projections.  For a row v with mean m
// and rstd r,  LN(v) W^T = r (v W~^T) - r m s + t  with  W~ = W diag(gamma),
// s = W~ 1 and t = W beta  (prepared once by the handle).  So the raw tiles
// feed the tensor cores as they land: z (bf16) against W~_g (bf16), and x
// (stored by the triangle GEMM as fp16 x * 2^-s, channel-major, i.e. an
// MN-major A operand) against W~_o (fp16).  The per-pair statistics are
// accumulated slab by slab by read-only passes off the MMA's path (or, for z,
// handed over by the input projection) and applied in the epilogue together
// with s and t.
//
// Each tile is 128 pairs x all D outputs: one M=128, N=D MMA per 16-wide K
// step, the gate accumulator in TMEM columns [0, D) and the value accumulator
// in [256, 256 + D).  The activations stream through a ring of 16 KB slabs
// (128 pairs x 64 channels): the D/64 z slabs of a tile, then its C/64 x
// slabs.  At D = 256 the two accumulators fill TMEM, so the epilogue works in
// two phases that hand the halves back one at a time: it turns the gate
// accumulator into tanh(gate/2) held in registers (fp16) and returns it, which
// lets the next tile's gate MMAs run while this tile's value MMAs finish; then
// it reads the value accumulator, forms the output and returns that half,
// which the next tile's value MMAs wait for.  Without the split a tile's MMAs
// waited for the whole previous epilogue.
//
// Structure (one persistent CTA per SM, 736 threads):
//   warp 0       TMA producer of the activation slabs
//   warp 1       TMEM (512 columns) + tcgen05.mma, one lane
//   warp 2       TMA producer of the weight slabs (D rows x 64 K), in MMA order
//   warps 3..6   statistics: per x slab the shifted sums of 8 pairs over a
//                channel phase; per z slab (only when the z statistics are not
//                handed in) the sums of one pair; the z and the x statistics
//                of a tile are published separately (double-buffered by tile
//                parity) as soon as each is complete.  Every statistics thread
//                waits for and releases every slab, so no thread ever waits
//                on a phase more than one ahead of a barrier.
//   warps 7..22  epilogue: warp (b, q) takes TMEM lane quadrant q (32 pairs)
//                and the 64-column block b of D: folded affines,
//                sigmoid(gate) * value -> bf16, staged in shared memory per
//                32 columns and written by TMA stores
#include "kernels.h"
#include "sm103_ptx.cuh"

namespace trimul {

namespace {
constexpr int BM = 128;                 // pairs per tile
constexpr int MAX_D = 256;
constexpr uint32_t SLAB = BM * 128;     // 16 KB activation slab: 128 pairs x 64 K
constexpr uint32_t BAR_BYTES = 512;
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t VAL_COL = 256;       // value accumulator columns [256, 256 + D)
constexpr int STAT_THREADS = 128;
constexpr int EPI_WARPS = 16;           // four per TMEM lane quadrant, one 64-column block each
constexpr uint32_t STAGE_W = 2048;      // per epilogue warp: 32 pair rows x 32 outputs (bf16), 64-byte swizzle
constexpr int THREADS = 96 + STAT_THREADS + 32 * EPI_WARPS;
constexpr int X_PHASES = 8;             // channel phases of the x statistics

struct Layout {
  uint32_t act, w, stage, xred, sbuf, colc, bars, total;
};

__host__ __device__ inline Layout layout(int a_stages, int w_stages, uint32_t w_stage_bytes) {
  Layout L;
  uint32_t o = 0;
  L.act = o;
  o += a_stages * SLAB;
  L.w = o;
  o += w_stages * w_stage_bytes;
  L.stage = o;  // [EPI_WARPS][32 rows x 64 B]: output staging for the TMA stores (64-byte swizzle)
  o += EPI_WARPS * STAGE_W;
  L.xred = o;  // [2][X_PHASES][128]: shifted sums and sums of squares per phase
  o += 2 * X_PHASES * BM * 4;
  L.sbuf = o;  // [2][128] float4 (z mean, z rstd, x mean, x rstd), by tile parity
  o += 2 * BM * 16;
  L.colc = o;  // [4][MAX_D] float: s_g, t_g / 2, s_o, t_o / 2 per output feature
  o += MAX_D * 16;
  L.bars = o;
  o += BAR_BYTES;
  L.total = o + 1024;  // slack for aligning the base to 1024 bytes
  return L;
}

}  // namespace

uint32_t outproj_w_stage_bytes(int D) { return static_cast<uint32_t>((D + 15) / 16 * 16) * 128u; }

size_t outproj_smem_bytes(int a_stages, int w_stages, int D) {
  return layout(a_stages, w_stages, outproj_w_stage_bytes(D)).total;
}

__global__ void __launch_bounds__(THREADS, 1)
    k3_outproj(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_z,
               const __grid_constant__ CUtensorMap tm_wg, const __grid_constant__ CUtensorMap tm_wo,
               const __grid_constant__ CUtensorMap tm_out, const OutprojArgs p) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_addr(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* const base_ptr = smem_raw + (base - raw);
  const uint32_t npad = static_cast<uint32_t>((p.D + 15) / 16 * 16);
  const uint32_t wsb = npad * 128u;  // bytes of one weight slab (npad rows x 64 K)
  const Layout L = layout(p.a_stages, p.w_stages, wsb);
  const uint32_t act = base + L.act, wring = base + L.w, bars = base + L.bars;
  const uint32_t afull0 = bars, aempty0 = afull0 + 8 * MAX_OUTPROJ_A_STAGES;
  const uint32_t wfull0 = aempty0 + 8 * MAX_OUTPROJ_A_STAGES, wempty0 = wfull0 + 8 * MAX_OUTPROJ_W_STAGES;
  // gate / value accumulator full (MMA commit) and empty (every epilogue warp)
  const uint32_t gfull = wempty0 + 8 * MAX_OUTPROJ_W_STAGES, gempty = gfull + 8;
  const uint32_t vfull = gempty + 8, vempty = vfull + 8;
  // statistics: z and x halves ready, slot free (by tile parity)
  const uint32_t zready0 = vempty + 8, xready0 = zready0 + 16, sfree0 = xready0 + 16;
  const uint32_t drain = sfree0 + 16, tmem_slot = drain + 8;
  volatile uint32_t* tmem_slot_ptr = reinterpret_cast<volatile uint32_t*>(base_ptr + (tmem_slot - base));
  float4* const sbuf = reinterpret_cast<float4*>(base_ptr + L.sbuf);
  float* const cs = reinterpret_cast<float*>(base_ptr + L.colc);

  const KStatus st{p.status, p.timeout_ns};
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int z_slabs = p.z_slabs, x_slabs = p.x_slabs, nk = z_slabs + x_slabs;  // slabs per tile: z first, then x

  if (threadIdx.x == 0) {
    for (int s = 0; s < p.a_stages; ++s) {
      mbar_init(afull0 + 8 * s, 1);
      mbar_init(aempty0 + 8 * s, 1 + STAT_THREADS);  // the MMAs' commit and every statistics thread
    }
    for (int s = 0; s < p.w_stages; ++s) {
      mbar_init(wfull0 + 8 * s, 1);
      mbar_init(wempty0 + 8 * s, 1);
    }
    mbar_init(gfull, 1);
    mbar_init(gempty, EPI_WARPS);
    mbar_init(vfull, 1);
    mbar_init(vempty, EPI_WARPS);
    for (int a = 0; a < 2; ++a) {
      mbar_init(zready0 + 8 * a, STAT_THREADS);
      mbar_init(xready0 + 8 * a, STAT_THREADS);
      mbar_init(sfree0 + 8 * a, EPI_WARPS);
    }
    mbar_init(drain, 1);
    fence_mbar_init();
  }
  for (int d = threadIdx.x; d < MAX_D; d += THREADS) {
    const float4 c = d < p.D ? p.colc[d] : make_float4(0.f, 0.f, 0.f, 0.f);
    cs[d] = c.x;
    cs[MAX_D + d] = c.y;
    cs[2 * MAX_D + d] = c.z;
    cs[3 * MAX_D + d] = c.w;
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot_ptr;
  const int total = p.tile_end;
  const int first = p.tile_begin + static_cast<int>(blockIdx.x);

  if (warp == 0) {
    // ------------------------------------------------------------ activation producer
    if (lane == 0 && !p.inject_stall) {
      tma_prefetch_desc(&tm_x);
      tma_prefetch_desc(&tm_z);
      int as = 0;
      uint32_t aph = 0;
      long long issued = 0;
      bool ok = true;
      for (int tile = first; tile < total && ok; tile += gridDim.x) {
        const int bb = tile / p.tiles_per_batch;
        const int pair0 = (tile - bb * p.tiles_per_batch) * BM;
        for (int k = 0; k < nk; ++k) {
          if (!mbar_wait(aempty0 + 8 * as, aph ^ 1u, st, SITE_PRODUCER)) { ok = false; break; }
          const uint32_t full = afull0 + 8 * as, dst = act + as * SLAB;
          mbar_arrive_expect_tx(full, SLAB);
          if (k < z_slabs) {
            tma_load_3d(dst, &tm_z, full, k * 64, pair0, bb);
          } else {
            tma_load_3d(dst, &tm_x, full, pair0, (k - z_slabs) * 64, bb);
            tma_load_3d(dst + 8192, &tm_x, full, pair0 + 64, (k - z_slabs) * 64, bb);
          }
          ++issued;
          if (++as == p.a_stages) { as = 0; aph ^= 1u; }
        }
      }
      if (!ok) {
        int s = as;
        uint32_t ph = aph;
        for (long long i = 0; i < issued && i < p.a_stages; ++i) {
          if (--s < 0) { s = p.a_stages - 1; ph ^= 1u; }
          mbar_wait_drain(afull0 + 8 * s, ph, p.timeout_ns);
        }
      }
    }
  } else if (warp == 2) {
    // ------------------------------------------------------------ weight producer
    if (lane == 0 && !p.inject_stall) {
      tma_prefetch_desc(&tm_wg);
      tma_prefetch_desc(&tm_wo);
      int ws = 0;
      uint32_t wph = 0;
      long long issued = 0;
      bool ok = true;
      for (int tile = first; tile < total && ok; tile += gridDim.x) {
        for (int k = 0; k < nk; ++k) {  // W~_g slabs (K = D), then W~_o slabs (K = C)
          if (!mbar_wait(wempty0 + 8 * ws, wph ^ 1u, st, SITE_PRODUCER)) { ok = false; break; }
          mbar_arrive_expect_tx(wfull0 + 8 * ws, wsb);
          if (k < z_slabs)
            tma_load_2d(wring + ws * wsb, &tm_wg, wfull0 + 8 * ws, k * 64, 0);
          else
            tma_load_2d(wring + ws * wsb, &tm_wo, wfull0 + 8 * ws, (k - z_slabs) * 64, 0);
          ++issued;
          if (++ws == p.w_stages) { ws = 0; wph ^= 1u; }
        }
      }
      if (!ok) {
        int s = ws;
        uint32_t ph = wph;
        for (long long i = 0; i < issued && i < p.w_stages; ++i) {
          if (--s < 0) { s = p.w_stages - 1; ph ^= 1u; }
          mbar_wait_drain(wfull0 + 8 * s, ph, p.timeout_ns);
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t idesc_gate = idesc_bf16_f32(BM, npad, 0, 0);  // z (bf16) K-major, W~_g bf16
      const uint32_t idesc_val = idesc_f16_f32(BM, npad, 1, 0);    // x (fp16) MN-major, W~_o fp16
      // Descriptors of stage 0; a stage or K step is a plain add to the start
      // address field (every address stays below 256 KB, so it cannot carry out).
      const uint64_t zdesc0 = sdesc_sw128(act, 16, 1024);
      const uint64_t xdesc0 = sdesc_sw128(act, 8192, 1024);
      const uint64_t wdesc0 = sdesc_sw128(wring, 16, 1024);
      const uint32_t d_gate = tmem_base, d_val = tmem_base + VAL_COL;
      int as = 0, ws = 0;
      uint32_t aph = 0, wph = 0;
      bool ok = true;
      int n = 0;
      for (int tile = first; tile < total && ok; tile += gridDim.x, ++n) {
        const uint32_t free_ph = (static_cast<uint32_t>(n) & 1u) ^ 1u;
        for (int k = 0; k < nk; ++k) {
          // each accumulator is free once the epilogue has read the previous tile's
          if (k == 0 || k == z_slabs) {
            if (!mbar_wait(k == 0 ? gempty : vempty, free_ph, st, SITE_MMA)) { ok = false; break; }
            tc_fence_after();
          }
          if (!mbar_wait(afull0 + 8 * as, aph, st, SITE_MMA) || !mbar_wait(wfull0 + 8 * ws, wph, st, SITE_MMA)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t bd = wdesc0 + ((ws * wsb) >> 4);
          if (k < z_slabs) {
            const uint64_t ad = zdesc0 + ((as * SLAB) >> 4);
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
              mma_f16_ss(d_gate, ad + 2 * kk, bd + 2 * kk, idesc_gate, (k | kk) != 0);
          } else {
            const uint64_t ad = xdesc0 + ((as * SLAB) >> 4);
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
              mma_f16_ss(d_val, ad + 128 * kk, bd + 2 * kk, idesc_val, ((k - z_slabs) | kk) != 0);
          }
          mma_commit(wempty0 + 8 * ws);
          mma_commit(aempty0 + 8 * as);
          if (++ws == p.w_stages) { ws = 0; wph ^= 1u; }
          if (++as == p.a_stages) { as = 0; aph ^= 1u; }
          if (k == z_slabs - 1) mma_commit(gfull);
          if (k == nk - 1) mma_commit(vfull);
        }
      }
      if (!ok) {
        mma_commit(drain);
        mbar_wait_drain(drain, 0, p.timeout_ns);
      }
    }
  } else if (warp < 3 + STAT_THREADS / 32) {
    // ------------------------------------------------------------ statistics (read-only)
    const uint32_t t = threadIdx.x - 96;  // pair t of the tile
    // LayerNorm eps of the stored x * 2^-s: eps * 4^-s, with s the caller's or
    // this call's (from max |a|, |b|, as the triangle GEMM derived it)
    const float eps_x =
        p.ab_max ? p.eps * exp2_neg(2 * x_scale_log2_from_max(__uint_as_float(*p.ab_max), p.N)) : p.eps_x;
    const float inv_d = 1.0f / static_cast<float>(p.D);
    const float inv_c = 1.0f / static_cast<float>(p.C);
    float* const xred1 = reinterpret_cast<float*>(base_ptr + L.xred);
    float* const xred2 = xred1 + X_PHASES * BM;
    // x: thread (pc, hp) owns pairs 8pc..8pc+7 and, in every slab, channels
    // hp, hp+8, ...; every one of those channels has (c & 7) == hp, so its
    // 16-byte chunk sits at the same swizzled position in every channel row.
    const uint32_t pc = t & 15, hp = t >> 4;
    const uint32_t x_chunk = (pc >> 3) * 8192u + ((((pc & 7u) ^ hp) & 7u) << 4);
    int as = 0;
    uint32_t aph = 0;
    bool ok = true;
    int n = 0;
    float2* const sbuf2 = reinterpret_cast<float2*>(sbuf);  // per pair: (z mean, z rstd), (x mean, x rstd)
    for (int tile = first; tile < total && ok; tile += gridDim.x, ++n) {
      const int bb = tile / p.tiles_per_batch;
      const long long pidx = static_cast<long long>(tile - bb * p.tiles_per_batch) * BM + t;
      float2 s1[4], s2[4], nk2[4];  // pairs of the 8 pairs (x) or of the 8 lanes of a chunk (z)
#pragma unroll
      for (int e = 0; e < 4; ++e) s1[e] = s2[e] = nk2[e] = make_float2(0.f, 0.f);
      float kt = 0.f;
      const int j = n & 1;
      const uint32_t use = static_cast<uint32_t>(n >> 1) & 1u;
      float2* const slot = sbuf2 + 2 * (j * BM + t);
      // the z statistics (handed in by the input projection) are loaded
      // before the wait below, so their DRAM latency overlaps it
      const float2 zst = (p.zstats && pidx < p.NN) ? p.zstats[bb * p.NN + pidx] : make_float2(0.f, 1.f);
      // slot j is free once the epilogue has read tile n - 2's statistics
      if (!named_bar_and(3, STAT_THREADS, mbar_wait(sfree0 + 8 * j, use ^ 1u, st, SITE_XFORM))) break;
      if (p.zstats) {
        slot[0] = zst;
        mbar_arrive(zready0 + 8 * j);
      }
      for (int k = 0; k < nk; ++k) {
        if (!named_bar_and(1, STAT_THREADS, mbar_wait(afull0 + 8 * as, aph, st, SITE_XFORM))) { ok = false; break; }
        const uint8_t* const slab = base_ptr + L.act + as * SLAB;
        if (k >= z_slabs) {
          const int kx = k - z_slabs;
          if (kx == 0) {  // shifts: the channel-0 values of the pairs
            const uint4 k8 = *reinterpret_cast<const uint4*>(slab + (pc >> 3) * 8192u + ((pc & 7u) << 4));
            const uint32_t kw[4] = {k8.x, k8.y, k8.z, k8.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&kw[e]));
              nk2[e] = make_float2(-f.x, -f.y);
            }
            kt = __half2float(*reinterpret_cast<const __half*>(slab + (t >> 6) * 8192u +
                                                                ((((t & 63u) >> 3) & 7u) << 4) + ((t & 7u) << 1)));
          }
          const int cn = min(64, p.C - kx * 64);  // channels of this slab
          uint4 v[64 / X_PHASES];
#pragma unroll
          for (int i = 0; i < 64 / X_PHASES; ++i) {
            const int c = static_cast<int>(hp) + X_PHASES * i;
            v[i] = c < cn ? *reinterpret_cast<const uint4*>(slab + c * 128 + x_chunk) : make_uint4(0u, 0u, 0u, 0u);
          }
#pragma unroll
          for (int i = 0; i < 64 / X_PHASES; ++i) {
            const bool in = static_cast<int>(hp) + X_PHASES * i < cn;
            const uint32_t w4[4] = {v[i].x, v[i].y, v[i].z, v[i].w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              float2 d = __fadd2_rn(__half22float2(*reinterpret_cast<const __half2*>(&w4[e])), nk2[e]);
              d = in ? d : make_float2(0.f, 0.f);
              s1[e] = __fadd2_rn(s1[e], d);
              s2[e] = __ffma2_rn(d, d, s2[e]);
            }
          }
          if (kx == x_slabs - 1) {  // reduce the channel phases: x mean and rstd of pair t
            float* const r1 = xred1 + hp * BM + pc * 8;
            float* const r2 = xred2 + hp * BM + pc * 8;
            reinterpret_cast<float4*>(r1)[0] = make_float4(s1[0].x, s1[0].y, s1[1].x, s1[1].y);
            reinterpret_cast<float4*>(r1)[1] = make_float4(s1[2].x, s1[2].y, s1[3].x, s1[3].y);
            reinterpret_cast<float4*>(r2)[0] = make_float4(s2[0].x, s2[0].y, s2[1].x, s2[1].y);
            reinterpret_cast<float4*>(r2)[1] = make_float4(s2[2].x, s2[2].y, s2[3].x, s2[3].y);
            named_bar_sync(2, STAT_THREADS);
            float t1 = 0.f, t2 = 0.f;
#pragma unroll
            for (int h = 0; h < X_PHASES; ++h) {
              t1 += xred1[h * BM + t];
              t2 += xred2[h * BM + t];
            }
            const float m1 = t1 * inv_c;
            slot[1] = make_float2(kt + m1, rsqrtf(fmaxf(t2 * inv_c - m1 * m1, 0.f) + eps_x));
            mbar_arrive(xready0 + 8 * j);
          }
        } else if (!p.zstats) {  // z row of pair t: channels k*64 .. k*64+63, shifted by its first element
          if (k == 0) {
            const float sh = bf16_lo(*reinterpret_cast<const uint32_t*>(slab + sw128_offset(t, 0)));
#pragma unroll
            for (int e = 0; e < 4; ++e) nk2[e] = make_float2(-sh, -sh);
          }
          const int n8 = min(8, (p.D - k * 64) >> 3);
#pragma unroll
          for (int c8 = 0; c8 < 8; ++c8) {
            if (c8 >= n8) break;
            const uint4 v = *reinterpret_cast<const uint4*>(slab + sw128_offset(t, c8 * 8));
            const uint32_t w4[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const float2 f = make_float2(bf16_lo(w4[e]), bf16_hi(w4[e]));
              const float2 d = __fadd2_rn(f, nk2[e]);
              s1[e] = __fadd2_rn(s1[e], d);
              s2[e] = __ffma2_rn(d, d, s2[e]);
            }
          }
          if (k == z_slabs - 1) {
            float t1 = 0.f, t2 = 0.f;
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              t1 += s1[e].x + s1[e].y;
              t2 += s2[e].x + s2[e].y;
            }
            const float m1 = t1 * inv_d;
            slot[0] = make_float2(-nk2[0].x + m1, rsqrtf(fmaxf(t2 * inv_d - m1 * m1, 0.f) + p.eps));
            mbar_arrive(zready0 + 8 * j);
#pragma unroll
            for (int e = 0; e < 4; ++e) s1[e] = s2[e] = make_float2(0.f, 0.f);
          }
        }
        mbar_arrive(aempty0 + 8 * as);  // last read of this slab
        if (++as == p.a_stages) { as = 0; aph ^= 1u; }
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue
    // Warp ew (0..15) takes TMEM lane quadrant q = warp % 4 (pair rows
    // q*32 .. q*32+31, one per lane) and the 64-column block cb = ew / 4.
    // With the constants colc = (s_g, t_g/2, s_o, t_o/2):
    //   gate/2  = (zr/2) acc_g + (t_g/2 - (zr/2) zm s_g)
    //   value/2 = (xr/2) acc_v + (t_o/2 - (xr/2) xm s_o)
    //   out = sigmoid(gate) * value = value/2 + value/2 * tanh(gate/2),
    // with tanh.approx.f16x2 on the fp16 rounding of gate/2.
    // Phase 1 (gate MMAs done): tanh(gate/2) of the warp's 32 x 64 block into
    // 32 registers (fp16 pairs), then the gate half of TMEM is handed back.
    // Phase 2 (value MMAs done): the outputs, 8 columns per TMEM load, into
    // the registers of the tanh pairs they consume; the value half is handed
    // back after the last load, before any store.  Then each 32-column half
    // is staged in the warp's 2 KB buffer (row r's 16-byte chunk c at position
    // c ^ ((r / 2) % 4), the 64-byte swizzle) and written by one TMA store of
    // the 32 x 32 box.  Rows past N*N are not written by the store.
    const int ew = warp - 3 - STAT_THREADS / 32;
    const int cb = ew >> 2;
    const int q = warp & 3;
    const bool active = cb * 64 < p.D;
    const uint32_t t_row = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + static_cast<uint32_t>(cb * 64);
    const uint32_t stage = base + L.stage + ew * STAGE_W;
    uint8_t* const srow = base_ptr + L.stage + ew * STAGE_W + lane * 64;
    const uint32_t sw = (lane >> 1) & 3u;
    const float2* const sbuf2 = reinterpret_cast<const float2*>(sbuf);
    int n = 0;
    for (int tile = first; tile < total; tile += gridDim.x, ++n) {
      const uint32_t ph = static_cast<uint32_t>(n) & 1u;
      const int bb = tile / p.tiles_per_batch;
      const int prow = (tile - bb * p.tiles_per_batch) * BM + q * 32;  // this warp's first pair row
      const int j = n & 1;
      const uint32_t use = static_cast<uint32_t>(n >> 1) & 1u;
      const float2* const slot = sbuf2 + 2 * (j * BM + q * 32 + lane);
      // ---- phase 1: gate
      if (!__all_sync(0xffffffffu, mbar_wait(zready0 + 8 * j, use, st, SITE_EPI))) break;
      const float2 zs = slot[0];
      const float ga = 0.5f * zs.y, gbv = -ga * zs.x;
      const float2 ga2 = make_float2(ga, ga), gb2 = make_float2(gbv, gbv);
      if (!__all_sync(0xffffffffu, mbar_wait(gfull, ph, st, SITE_EPI))) break;
      tc_fence_after();
      uint32_t th[32];  // tanh(gate/2) of columns 2i, 2i+1 of the block (fp16 pairs)
      if (active) {
        uint32_t ra[8], rb[8];
        tmem_ld8(t_row, ra);
#pragma unroll
        for (int s8 = 0; s8 < 8; ++s8) {
          tmem_ld_wait();
          uint32_t(&cur)[8] = (s8 & 1) ? rb : ra;
          if (s8 < 7) tmem_ld8(t_row + (s8 + 1) * 8, (s8 & 1) ? ra : rb);
          const int c = cb * 64 + s8 * 8;
          const float4* const c4 = reinterpret_cast<const float4*>(cs + c);
          const float4 sg[2] = {c4[0], c4[1]}, tg[2] = {c4[MAX_D / 4], c4[MAX_D / 4 + 1]};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float4& sgq = sg[e >> 1];
            const float4& tgq = tg[e >> 1];
            const bool hi = e & 1;
            const float2 sg2 = hi ? make_float2(sgq.z, sgq.w) : make_float2(sgq.x, sgq.y);
            const float2 tg2 = hi ? make_float2(tgq.z, tgq.w) : make_float2(tgq.x, tgq.y);
            const float2 g2 = make_float2(__uint_as_float(cur[2 * e]), __uint_as_float(cur[2 * e + 1]));
            const float2 gh = __ffma2_rn(ga2, g2, __ffma2_rn(gb2, sg2, tg2));  // gate / 2
            const __half2 gh16 = __float22half2_rn(gh);
            th[s8 * 4 + e] = tanh_h2(*reinterpret_cast<const uint32_t*>(&gh16));
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(gempty);
      // ---- phase 2: value and output
      if (!__all_sync(0xffffffffu, mbar_wait(xready0 + 8 * j, use, st, SITE_EPI))) break;
      const float2 xs = slot[1];
      __syncwarp();
      if (lane == 0) mbar_arrive(sfree0 + 8 * j);
      const float va = 0.5f * xs.y, vbv = -va * xs.x;
      const float2 va2 = make_float2(va, va), vb2 = make_float2(vbv, vbv);
      if (!__all_sync(0xffffffffu, mbar_wait(vfull, ph, st, SITE_EPI))) break;
      tc_fence_after();
      if (active) {
        uint32_t ra[8], rb[8];
        tmem_ld8(t_row + VAL_COL, ra);
#pragma unroll
        for (int s8 = 0; s8 < 8; ++s8) {
          tmem_ld_wait();
          uint32_t(&cur)[8] = (s8 & 1) ? rb : ra;
          if (s8 < 7) {
            tmem_ld8(t_row + VAL_COL + (s8 + 1) * 8, (s8 & 1) ? ra : rb);
          } else {  // this warp's last read of the accumulators: hand the value half back
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(vempty);
          }
          const int c = cb * 64 + s8 * 8;
          const float4* const c4 = reinterpret_cast<const float4*>(cs + c);
          const float4 so[2] = {c4[MAX_D / 2], c4[MAX_D / 2 + 1]}, to[2] = {c4[3 * MAX_D / 4], c4[3 * MAX_D / 4 + 1]};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float4& soq = so[e >> 1];
            const float4& toq = to[e >> 1];
            const bool hi = e & 1;
            const float2 so2 = hi ? make_float2(soq.z, soq.w) : make_float2(soq.x, soq.y);
            const float2 to2 = hi ? make_float2(toq.z, toq.w) : make_float2(toq.x, toq.y);
            const float2 v2 = make_float2(__uint_as_float(cur[2 * e]), __uint_as_float(cur[2 * e + 1]));
            const float2 vh = __ffma2_rn(va2, v2, __ffma2_rn(vb2, so2, to2));  // value / 2
            const float2 t2 = __half22float2(*reinterpret_cast<const __half2*>(&th[s8 * 4 + e]));
            const float2 o = __ffma2_rn(vh, t2, vh);
            th[s8 * 4 + e] = pack_bf162(o.x, o.y);  // the output pair replaces its tanh pair
          }
        }
        // the accumulators are handed back; stage and store the two 32-column halves
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          if (lane == 0) tma_store_wait_read<0>();  // the previous store has read the staging buffer
          __syncwarp();
#pragma unroll
          for (int c16 = 0; c16 < 4; ++c16)
            *reinterpret_cast<uint4*>(srow + (((static_cast<uint32_t>(c16) ^ sw) & 3u) << 4)) =
                make_uint4(th[hh * 16 + c16 * 4], th[hh * 16 + c16 * 4 + 1], th[hh * 16 + c16 * 4 + 2],
                           th[hh * 16 + c16 * 4 + 3]);
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0 && prow < p.NN && cb * 64 + hh * 32 < p.D) {
            tma_store_3d(&tm_out, stage, cb * 64 + hh * 32, prow, bb);
            tma_store_commit();
          }
        }
      } else {
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(vempty);
      }
    }
    if (lane == 0) tma_store_wait_all();
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, TMEM_COLS);
  }
}

cudaError_t launch_outproj(const OutprojArgs& a, const CUtensorMap& tm_x, const CUtensorMap& tm_z,
                           const CUtensorMap& tm_wg, const CUtensorMap& tm_wo, const CUtensorMap& tm_out, int grid,
                           cudaStream_t s) {
  if (a.a_stages < 2 || a.a_stages > MAX_OUTPROJ_A_STAGES || a.w_stages < 2 || a.w_stages > MAX_OUTPROJ_W_STAGES ||
      a.D > MAX_D || a.D < 8)
    return cudaErrorInvalidValue;
  const size_t smem = outproj_smem_bytes(a.a_stages, a.w_stages, a.D);
  cudaError_t e = cudaFuncSetAttribute(k3_outproj, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  k3_outproj<<<grid, THREADS, smem, s>>>(tm_x, tm_z, tm_wg, tm_wo, tm_out, a);
  return cudaGetLastError();
}

}  // namespace trimul
