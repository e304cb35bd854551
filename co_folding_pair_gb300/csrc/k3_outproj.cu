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
// computed by read-only passes off the MMA's path (or, for z, handed over by
// the input projection) and applied in the epilogue together with s and t.
//
// Structure (one persistent CTA per SM, 480 threads):
//   warp 0       TMA producer of the activations: z tile and x tile (one
//                buffer each), each re-filled as soon as its MMAs and its
//                statistics pass are done with it
//   warp 1       TMEM (512 columns) + tcgen05.mma.  Per tile, the gate phase
//                (z W~_g^T, K = D) then the value phase (x W~_o^T, K = C), each
//                for both 128-column halves of D
//   warp 2       TMA producer of the weight slabs (128 rows x 64 K), in MMA order
//   warps 3..6   statistics: mean and rstd per pair of x (over C) and, when not
//                handed in, of z (over D); one shifted pass, published per tile
//                through a double-buffered shared array
//   warps 7..14  epilogue, one group of four warps per 128-column half of D:
//                folded affines, sigmoid(gate) * value -> bf16; an 8x8 transpose
//                of 16-byte chunks inside groups of 8 lanes makes every store
//                instruction write four whole 128-byte row segments
// Each half of D has its own accumulator pair in TMEM (value 128 + gate 128
// columns), so one half's epilogue runs under the other half's MMAs.
#include "kernels.h"
#include "sm103_ptx.cuh"

namespace trimul {

namespace {
constexpr int BM = 128;                 // pairs per tile
constexpr int BN = 128;                 // output columns per half
constexpr int MAX_D = 256;
constexpr uint32_t SLAB = BM * 128;     // 16 KB: 128 pairs x 64 K
constexpr uint32_t W_SLAB = BN * 128;   // 16 KB: 128 rows x 64 K
constexpr uint32_t BAR_BYTES = 256;
constexpr uint32_t TMEM_COLS = 512;
constexpr int STAT_THREADS = 128;
constexpr int EPI_WARPS = 8;
constexpr int THREADS = 96 + STAT_THREADS + 32 * EPI_WARPS;
constexpr int MAX_W_STAGES = 6;
constexpr int X_PHASES = 8;             // channel phases of the x statistics

struct Layout {
  uint32_t x, z, w, xred, sbuf, colc, bars, total;
};

__host__ __device__ inline Layout layout(int x_slabs, int z_slabs, int w_stages) {
  Layout L;
  uint32_t o = 0;
  L.x = o;
  o += x_slabs * SLAB;
  L.z = o;
  o += z_slabs * SLAB;
  L.w = o;
  o += w_stages * W_SLAB;
  L.xred = o;  // [2][X_PHASES][128]: shifted sums and sums of squares per phase
  o += 2 * X_PHASES * BM * 4;
  L.sbuf = o;  // [2][128] float4 (z mean, z rstd, x mean, x rstd), by tile parity
  o += 2 * BM * 16;
  L.colc = o;  // [MAX_D] float4 (s_g, t_g, s_o, t_o)
  o += MAX_D * 16;
  L.bars = o;
  o += BAR_BYTES;
  L.total = o + 1024;  // slack for aligning the base to 1024 bytes
  return L;
}

__device__ __forceinline__ float h2f_lo(uint32_t v) { return __low2float(*reinterpret_cast<const __half2*>(&v)); }
__device__ __forceinline__ float h2f_hi(uint32_t v) { return __high2float(*reinterpret_cast<const __half2*>(&v)); }
}  // namespace

size_t outproj_smem_bytes(int x_slabs, int z_slabs, int w_stages) {
  return layout(x_slabs, z_slabs, w_stages).total;
}

__global__ void __launch_bounds__(THREADS, 1)
    k3_outproj(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_z,
               const __grid_constant__ CUtensorMap tm_wg, const __grid_constant__ CUtensorMap tm_wo,
               const OutprojArgs p) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_addr(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* const base_ptr = smem_raw + (base - raw);
  const Layout L = layout(p.x_slabs, p.z_slabs, p.w_stages);
  const uint32_t xbuf = base + L.x, zbuf = base + L.z, wring = base + L.w, bars = base + L.bars;
  const uint32_t zfull = bars, zempty = bars + 8, xfull = bars + 16, xempty = bars + 24;
  const uint32_t wfull0 = bars + 32, wempty0 = wfull0 + 8 * MAX_W_STAGES;
  const uint32_t tfull0 = wempty0 + 8 * MAX_W_STAGES, tempty0 = tfull0 + 16;
  const uint32_t sready0 = tempty0 + 16, sfree0 = sready0 + 16;
  const uint32_t drain = sfree0 + 16, tmem_slot = drain + 8;
  volatile uint32_t* tmem_slot_ptr = reinterpret_cast<volatile uint32_t*>(base_ptr + (tmem_slot - base));
  float4* const sbuf = reinterpret_cast<float4*>(base_ptr + L.sbuf);
  float4* const colc = reinterpret_cast<float4*>(base_ptr + L.colc);

  const KStatus st{p.status, p.timeout_ns};
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    mbar_init(zfull, 1);
    // The gate MMAs' commit, plus every statistics thread when it reads the z
    // tile (no statistics pass over z when the input projection hands them in:
    // an arrival that is not ordered after the tile's zfull would let the
    // producer refill z under the gate MMAs and re-arm zfull early).
    mbar_init(zempty, 1 + (p.zstats ? 0 : STAT_THREADS));
    mbar_init(xfull, 1);
    mbar_init(xempty, 1 + STAT_THREADS);  // the value MMAs' commit and every statistics thread
    for (int s = 0; s < p.w_stages; ++s) {
      mbar_init(wfull0 + 8 * s, 1);
      mbar_init(wempty0 + 8 * s, 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(tfull0 + 8 * a, 1);
      mbar_init(tempty0 + 8 * a, 4);          // the four epilogue warps of that half
      mbar_init(sready0 + 8 * a, STAT_THREADS);
      mbar_init(sfree0 + 8 * a, EPI_WARPS);
    }
    mbar_init(drain, 1);
    fence_mbar_init();
  }
  for (int d = threadIdx.x; d < MAX_D; d += THREADS) colc[d] = d < p.D ? p.colc[d] : make_float4(0.f, 0.f, 0.f, 0.f);
  if (warp == 1) {
    tmem_alloc(tmem_slot, TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot_ptr;
  const int total = p.total_tiles;

  if (warp == 0) {
    // ------------------------------------------------------------ activation producer
    if (lane == 0 && !p.inject_stall) {
      tma_prefetch_desc(&tm_x);
      tma_prefetch_desc(&tm_z);
      long long z_issued = 0, x_issued = 0;
      bool ok = true;
      int n = 0;
      for (int tile = blockIdx.x; tile < total && ok; tile += gridDim.x, ++n) {
        const uint32_t ph = static_cast<uint32_t>(n) & 1u;
        const int bb = tile / p.tiles_per_batch;
        const int pair0 = (tile - bb * p.tiles_per_batch) * BM;
        if (!mbar_wait(zempty, ph ^ 1u, st, SITE_PRODUCER)) { ok = false; break; }
        mbar_arrive_expect_tx(zfull, p.z_slabs * SLAB);
        for (int s = 0; s < p.z_slabs; ++s) tma_load_3d(zbuf + s * SLAB, &tm_z, zfull, s * 64, pair0, bb);
        ++z_issued;
        if (!mbar_wait(xempty, ph ^ 1u, st, SITE_PRODUCER)) { ok = false; break; }
        mbar_arrive_expect_tx(xfull, p.x_slabs * SLAB);
        for (int s = 0; s < p.x_slabs; ++s)
          for (int h = 0; h < 2; ++h)
            tma_load_3d(xbuf + s * SLAB + h * 8192, &tm_x, xfull, pair0 + h * 64, s * 64, bb);
        ++x_issued;
      }
      if (!ok) {
        if (z_issued > 0) mbar_wait_drain(zfull, static_cast<uint32_t>(z_issued - 1) & 1u, p.timeout_ns);
        if (x_issued > 0) mbar_wait_drain(xfull, static_cast<uint32_t>(x_issued - 1) & 1u, p.timeout_ns);
      }
    }
  } else if (warp == 2) {
    // ------------------------------------------------------------ weight producer
    if (lane == 0 && !p.inject_stall) {
      tma_prefetch_desc(&tm_wg);
      tma_prefetch_desc(&tm_wo);
      int ws = 0;
      uint32_t wph = 0;
      long long w_issued = 0;
      bool ok = true;
      for (int tile = blockIdx.x; tile < total && ok; tile += gridDim.x) {
        for (int part = 0; part < 2 && ok; ++part) {  // 0: W~_g slabs (K = D), 1: W~_o slabs (K = C)
          const int nsl = part == 0 ? p.z_slabs : p.x_slabs;
          const CUtensorMap* tm = part == 0 ? &tm_wg : &tm_wo;
          for (int hh = 0; hh < p.n_halves && ok; ++hh) {
            for (int s = 0; s < nsl; ++s) {
              if (!mbar_wait(wempty0 + 8 * ws, wph ^ 1u, st, SITE_PRODUCER)) { ok = false; break; }
              mbar_arrive_expect_tx(wfull0 + 8 * ws, W_SLAB);
              tma_load_2d(wring + ws * W_SLAB, tm, wfull0 + 8 * ws, s * 64, hh * BN);
              ++w_issued;
              if (++ws == p.w_stages) { ws = 0; wph ^= 1u; }
            }
          }
        }
      }
      if (!ok) {
        int s = ws;
        uint32_t ph = wph;
        for (long long i = 0; i < w_issued && i < p.w_stages; ++i) {
          if (--s < 0) { s = p.w_stages - 1; ph ^= 1u; }
          mbar_wait_drain(wfull0 + 8 * s, ph, p.timeout_ns);
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    // Half hh uses TMEM columns [hh*256, hh*256+256): value at +0, gate at +128.
    if (lane == 0) {
      const uint32_t idesc_gate = idesc_bf16_f32(BM, BN, 0, 0);  // z (bf16) K-major, W~_g bf16
      const uint32_t idesc_val = idesc_f16_f32(BM, BN, 1, 0);    // x (fp16) MN-major, W~_o fp16
      int ws = 0;
      uint32_t wph = 0;
      bool ok = true;
      int n = 0;
      for (int tile = blockIdx.x; tile < total && ok; tile += gridDim.x, ++n) {
        const uint32_t ph = static_cast<uint32_t>(n) & 1u;
        for (int part = 0; part < 2 && ok; ++part) {
          if (!mbar_wait(part == 0 ? zfull : xfull, ph, st, SITE_MMA)) { ok = false; break; }
          tc_fence_after();
          const int nsl = part == 0 ? p.z_slabs : p.x_slabs;
          for (int hh = 0; hh < p.n_halves && ok; ++hh) {
            if (part == 0) {  // first use of this half's accumulator in the tile
              if (!mbar_wait(tempty0 + 8 * hh, ph ^ 1u, st, SITE_MMA)) { ok = false; break; }
              tc_fence_after();
            }
            const uint32_t d = tmem_base + hh * 256 + (part == 0 ? 128 : 0);
            for (int s = 0; s < nsl; ++s) {
              if (!mbar_wait(wfull0 + 8 * ws, wph, st, SITE_MMA)) { ok = false; break; }
              tc_fence_after();
              const uint32_t wb = wring + ws * W_SLAB;
#pragma unroll
              for (int kk = 0; kk < 4; ++kk) {
                if (part == 0)
                  mma_f16_ss(d, sdesc_sw128(zbuf + s * SLAB + kk * 32, 16, 1024), sdesc_sw128(wb + kk * 32, 16, 1024),
                             idesc_gate, (s | kk) != 0);
                else
                  mma_f16_ss(d, sdesc_sw128(xbuf + s * SLAB + kk * 2048, 8192, 1024),
                             sdesc_sw128(wb + kk * 32, 16, 1024), idesc_val, (s | kk) != 0);
              }
              mma_commit(wempty0 + 8 * ws);
              if (++ws == p.w_stages) { ws = 0; wph ^= 1u; }
            }
            if (ok && part == 1) mma_commit(tfull0 + 8 * hh);
          }
          if (ok) mma_commit(part == 0 ? zempty : xempty);
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
    const float inv_d = 1.0f / static_cast<float>(p.D);
    const float inv_c = 1.0f / static_cast<float>(p.C);
    const uint8_t* const zt = base_ptr + L.z;
    const uint8_t* const xt = base_ptr + L.x;
    float* const xred1 = reinterpret_cast<float*>(base_ptr + L.xred);
    float* const xred2 = xred1 + X_PHASES * BM;
    const int n8 = p.D >> 3;
    // x: thread (pc, hp) owns pairs 8pc..8pc+7 and channels hp, hp+8, ...; every
    // one of those channels has (c & 7) == hp, so its 16-byte chunk sits at the
    // same swizzled position in every channel row.
    const uint32_t pc = t & 15, hp = t >> 4;
    const uint32_t x_chunk = (pc >> 3) * 8192u + ((((pc & 7u) ^ hp) & 7u) << 4);
    int n = 0;
    for (int tile = blockIdx.x; tile < total; tile += gridDim.x, ++n) {
      const uint32_t ph = static_cast<uint32_t>(n) & 1u;
      const int bb = tile / p.tiles_per_batch;
      const long long pidx = static_cast<long long>(tile - bb * p.tiles_per_batch) * BM + t;
      // ---- z statistics of pair t
      float zm = 0.f, zr = 1.f;
      if (p.zstats) {
        if (pidx < p.NN) {
          const float2 ms = p.zstats[bb * p.NN + pidx];
          zm = ms.x;
          zr = ms.y;
        }
      } else {
        if (!named_bar_and(1, STAT_THREADS, mbar_wait(zfull, ph, st, SITE_XFORM))) break;
        // one pass, shifted by the row's first element
        const float shift = bf16_lo(*reinterpret_cast<const uint32_t*>(zt + sw128_offset(t, 0)));
        float s1[8], s2[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) s1[e] = s2[e] = 0.f;
        for (int c8 = 0; c8 < n8; ++c8) {
          const uint4 v = *reinterpret_cast<const uint4*>(zt + (c8 >> 3) * SLAB + sw128_offset(t, (c8 & 7) * 8));
          const float f[8] = {bf16_lo(v.x), bf16_hi(v.x), bf16_lo(v.y), bf16_hi(v.y),
                              bf16_lo(v.z), bf16_hi(v.z), bf16_lo(v.w), bf16_hi(v.w)};
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            const float d = f[e] - shift;
            s1[e] += d;
            s2[e] = fmaf(d, d, s2[e]);
          }
        }
        float t1 = 0.f, t2 = 0.f;
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          t1 += s1[e];
          t2 += s2[e];
        }
        const float m1 = t1 * inv_d;
        zm = shift + m1;
        zr = rsqrtf(fmaxf(t2 * inv_d - m1 * m1, 0.f) + p.eps);
        mbar_arrive(zempty);  // last read of this tile's z
      }
      // ---- x statistics: one pass, shifted per pair by its channel-0 value
      if (!named_bar_and(2, STAT_THREADS, mbar_wait(xfull, ph, st, SITE_XFORM))) break;
      {
        const uint4 k8 = *reinterpret_cast<const uint4*>(xt + (pc >> 3) * 8192u + ((pc & 7u) << 4));
        const float kx[8] = {h2f_lo(k8.x), h2f_hi(k8.x), h2f_lo(k8.y), h2f_hi(k8.y),
                             h2f_lo(k8.z), h2f_hi(k8.z), h2f_lo(k8.w), h2f_hi(k8.w)};
        float s1[8], s2[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) s1[e] = s2[e] = 0.f;
        for (int c = hp; c < p.C; c += X_PHASES) {
          const uint4 v = *reinterpret_cast<const uint4*>(xt + (c >> 6) * SLAB + (c & 63) * 128 + x_chunk);
          const float f[8] = {h2f_lo(v.x), h2f_hi(v.x), h2f_lo(v.y), h2f_hi(v.y),
                              h2f_lo(v.z), h2f_hi(v.z), h2f_lo(v.w), h2f_hi(v.w)};
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            const float d = f[e] - kx[e];
            s1[e] += d;
            s2[e] = fmaf(d, d, s2[e]);
          }
        }
        float* const r1 = xred1 + hp * BM + pc * 8;
        float* const r2 = xred2 + hp * BM + pc * 8;
        reinterpret_cast<float4*>(r1)[0] = make_float4(s1[0], s1[1], s1[2], s1[3]);
        reinterpret_cast<float4*>(r1)[1] = make_float4(s1[4], s1[5], s1[6], s1[7]);
        reinterpret_cast<float4*>(r2)[0] = make_float4(s2[0], s2[1], s2[2], s2[3]);
        reinterpret_cast<float4*>(r2)[1] = make_float4(s2[4], s2[5], s2[6], s2[7]);
      }
      named_bar_sync(2, STAT_THREADS);
      float t1 = 0.f, t2 = 0.f;
#pragma unroll
      for (int h = 0; h < X_PHASES; ++h) {
        t1 += xred1[h * BM + t];
        t2 += xred2[h * BM + t];
      }
      const float kt = __half2float(
          *reinterpret_cast<const __half*>(xt + (t >> 6) * 8192u + ((((t & 63u) >> 3) & 7u) << 4) + ((t & 7u) << 1)));
      mbar_arrive(xempty);  // last read of this tile's x
      const float m1 = t1 * inv_c;
      const float xm = kt + m1;
      const float xr = rsqrtf(fmaxf(t2 * inv_c - m1 * m1, 0.f) + p.eps_x);
      // ---- publish (double-buffered by tile parity)
      const int j = n & 1;
      const uint32_t use = static_cast<uint32_t>(n >> 1) & 1u;
      if (!mbar_wait(sfree0 + 8 * j, use ^ 1u, st, SITE_XFORM)) break;
      sbuf[j * BM + t] = make_float4(zm, zr, xm, xr);
      mbar_arrive(sready0 + 8 * j);
    }
  } else {
    // ------------------------------------------------------------ epilogue
    // Group hh (warps 7..10: half 0, warps 11..14: half 1); lane r of quadrant q
    // holds pair row q*32+r.  gate = zr*acc_g + (t_g - zr*zm*s_g),
    // value = xr*acc_v + (t_o - xr*xm*s_o), out = sigmoid(gate) * value.
    const int e = warp - 3 - STAT_THREADS / 32;
    const int hh = e >> 2;
    const int q = warp & 3;
    const uint32_t gb = lane & 7, ga = lane >> 3;
    bool ok = true;
    int n = 0;
    for (int tile = blockIdx.x; tile < total && ok; tile += gridDim.x, ++n) {
      const uint32_t ph = static_cast<uint32_t>(n) & 1u;
      const int bb = tile / p.tiles_per_batch;
      const long long row0 = static_cast<long long>(tile - bb * p.tiles_per_batch) * BM + q * 32 + ga * 8;
      const int j = n & 1;
      const uint32_t use = static_cast<uint32_t>(n >> 1) & 1u;
      if (!__all_sync(0xffffffffu, mbar_wait(sready0 + 8 * j, use, st, SITE_EPI))) break;
      const float4 s4 = sbuf[j * BM + q * 32 + lane];
      __syncwarp();
      if (lane == 0) mbar_arrive(sfree0 + 8 * j);
      if (hh >= p.n_halves) continue;
      if (!__all_sync(0xffffffffu, mbar_wait(tfull0 + 8 * hh, ph, st, SITE_EPI))) {
        ok = false;
        break;
      }
      tc_fence_after();
      const float ga_z = s4.y, gb_z = -s4.y * s4.x;  // gate  = zr*acc + (t_g + gb_z*s_g)
      const float va_x = s4.w, vb_x = -s4.w * s4.z;  // value = xr*acc + (t_o + vb_x*s_o)
      const uint32_t t_addr = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + hh * 256;
      const int n_cb = (hh * BN + 64 < p.D) ? 2 : 1;  // 64-column blocks in this half
#pragma unroll 1
      for (int cb = 0; cb < n_cb; ++cb) {
        const int col0 = hh * BN + cb * 64;
        uint4 R[8];
#pragma unroll
        for (int blk = 0; blk < 4; ++blk) {
          uint32_t v[16], g[16];
          tmem_ld16(t_addr + cb * 64 + blk * 16, v);
          tmem_ld16(t_addr + 128 + cb * 64 + blk * 16, g);
          tmem_ld_wait();
#pragma unroll
          for (int u = 0; u < 2; ++u) {
            float o[8];
#pragma unroll
            for (int k = 0; k < 8; ++k) {
              const float4 cc = colc[col0 + blk * 16 + u * 8 + k];
              const float gate = fmaf(ga_z, __uint_as_float(g[u * 8 + k]), fmaf(gb_z, cc.x, cc.y));
              const float val = fmaf(va_x, __uint_as_float(v[u * 8 + k]), fmaf(vb_x, cc.z, cc.w));
              o[k] = sigmoid_fast(gate) * val;
            }
            R[blk * 2 + u] = make_uint4(pack_bf162(o[0], o[1]), pack_bf162(o[2], o[3]), pack_bf162(o[4], o[5]),
                                        pack_bf162(o[6], o[7]));
          }
        }
        if (cb == n_cb - 1) {  // accumulator fully read: hand it back
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(tempty0 + 8 * hh);
        }
#pragma unroll
        for (int k = 4; k >= 1; k >>= 1) {
          const bool upper = (gb & k) != 0;
#pragma unroll
          for (int jj = 0; jj < 8; ++jj) {
            if (jj & k) continue;
            const uint4 lo = R[jj], hi = R[jj | k];
            const uint4 send = upper ? lo : hi;
            uint4 recv;
            recv.x = __shfl_xor_sync(0xffffffffu, send.x, k);
            recv.y = __shfl_xor_sync(0xffffffffu, send.y, k);
            recv.z = __shfl_xor_sync(0xffffffffu, send.z, k);
            recv.w = __shfl_xor_sync(0xffffffffu, send.w, k);
            R[jj] = upper ? recv : lo;
            R[jj | k] = upper ? hi : recv;
          }
        }
        const int col = col0 + static_cast<int>(gb) * 8;
        if (col < p.D) {
#pragma unroll
          for (int s8 = 0; s8 < 8; ++s8) {
            const long long row = row0 + s8;
            if (row < p.NN)
              *reinterpret_cast<uint4*>(p.out + (static_cast<size_t>(bb) * p.NN + row) * p.D + col) = R[s8];
          }
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, TMEM_COLS);
  }
}

cudaError_t launch_outproj(const OutprojArgs& a, const CUtensorMap& tm_x, const CUtensorMap& tm_z,
                           const CUtensorMap& tm_wg, const CUtensorMap& tm_wo, int grid, cudaStream_t s) {
  if (a.w_stages < 1 || a.w_stages > MAX_W_STAGES || a.D > MAX_D) return cudaErrorInvalidValue;
  const size_t smem = outproj_smem_bytes(a.x_slabs, a.z_slabs, a.w_stages);
  cudaError_t e = cudaFuncSetAttribute(k3_outproj, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  k3_outproj<<<grid, THREADS, smem, s>>>(tm_x, tm_z, tm_wg, tm_wo, a);
  return cudaGetLastError();
}

}  // namespace trimul
