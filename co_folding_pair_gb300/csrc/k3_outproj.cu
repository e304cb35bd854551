// k3_outproj.cu -- LayerNorm over channels of x, output projection, output gate.
//
// fold-cp-ops README, "Use": norm_out = LayerNorm, p_out = Linear(., D, bias=False),
// g_out = Linear(D, D, bias=False) applied to the normalised input z' = LN_in(z):
//     out[p, :] = sigmoid(z'_p W_g^T) * (LN_out(x_p) W_o^T)
// x arrives channel-major ([B][C][N*N], bf16, from the triangle GEMM), so one
// 128-pair tile of x is a [C x 128] block with the pairs contiguous: it is the
// MMA's A operand in MN-major form.  z is re-read pair-major and normalised
// again (cheaper than storing and re-reading z').
//
// Structure (one persistent CTA per SM, 480 threads):
//   warp 0       TMA producer of the activations: z tile and x tile (one
//                buffer each)
//   warp 1       TMEM (512 columns) + tcgen05.mma.  Per tile, first the gate
//                phase (z' W_g^T, K = D, both 128-column halves of D), then the
//                value phase (LN(x) W_o^T, K = C).  z's buffer is released
//                after the gate phase and x's after the value phase, so the
//                next tile's z load and LayerNorm run under this tile's value
//                MMAs and the next x load runs under the next gate MMAs.
//   warp 2       TMA producer of the weight slabs (128 rows x 64 K, fp16), in
//                MMA order, through a ring
//   warps 3..10  LayerNorms, 256 threads cooperating through shared memory:
//                z rows (two threads per pair) and x columns (16 channel
//                phases x 16 chunks of 8 pairs, 16-byte reads); fp32
//                statistics in two passes, results written in place as fp16
//   warps 11..14 epilogue: sigmoid(gate) * value -> bf16, 16-byte stores
// Each 128-column half of D has its own accumulator pair in TMEM (value 128 +
// gate 128 columns), so one half's epilogue runs under the other's MMAs.
#include "kernels.h"
#include "sm103_ptx.cuh"

namespace trimul {

namespace {
constexpr int BM = 128;                 // pairs per tile
constexpr int BN = 128;                 // output columns per half
constexpr uint32_t SLAB = BM * 128;     // 16 KB: 128 pairs x 64 K
constexpr uint32_t W_SLAB = BN * 128;   // 16 KB: 128 rows x 64 K
constexpr uint32_t BAR_BYTES = 256;
constexpr uint32_t TMEM_COLS = 512;
constexpr int XFORM_THREADS = 256;
constexpr int THREADS = 96 + XFORM_THREADS + 128;
constexpr int MAX_W_STAGES = 6;
constexpr int X_PHASES = 16;            // channel phases of the x-column LayerNorm

struct Layout {
  uint32_t x, z, w, xred, zred, stat, bars, total;
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
  L.xred = o;  // [X_PHASES][128] partial sums over channel phases
  o += X_PHASES * BM * 4;
  L.zred = o;  // [2 sums | 2 squares][128] partials of the two half-rows
  o += 4 * BM * 4;
  L.stat = o;  // x mean[128], x rstd[128]
  o += 2 * BM * 4;
  L.bars = o;
  o += BAR_BYTES;
  L.total = o + 1024;  // slack for aligning the base to 1024 bytes
  return L;
}
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
  const uint32_t xfull = bars, xready = bars + 8, xempty = bars + 16;
  const uint32_t zfull = bars + 24, zready = bars + 32, zempty = bars + 40;
  const uint32_t wfull0 = bars + 48, wempty0 = wfull0 + 8 * MAX_W_STAGES;
  const uint32_t tfull0 = wempty0 + 8 * MAX_W_STAGES, tempty0 = tfull0 + 16;
  const uint32_t drain = tempty0 + 16, tmem_slot = drain + 8;
  volatile uint32_t* tmem_slot_ptr = reinterpret_cast<volatile uint32_t*>(base_ptr + (tmem_slot - base));

  const KStatus st{p.status, p.timeout_ns};
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    mbar_init(xfull, 1);
    mbar_init(xready, XFORM_THREADS);
    mbar_init(xempty, 1);
    mbar_init(zfull, 1);
    mbar_init(zready, XFORM_THREADS);
    mbar_init(zempty, 1);
    for (int s = 0; s < p.w_stages; ++s) {
      mbar_init(wfull0 + 8 * s, 1);
      mbar_init(wempty0 + 8 * s, 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(tfull0 + 8 * a, 1);
      mbar_init(tempty0 + 8 * a, 4);
    }
    mbar_init(drain, 1);
    fence_mbar_init();
  }
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
    // z and x tiles, each single-buffered.  z(n+1) is issued as soon as the
    // gate MMAs of tile n are done with z(n); x(n+1) as soon as the value MMAs
    // are done with x(n).
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
    // Slabs in the order the MMA warp consumes them: per tile, W_g for every
    // 128-column half (K = D), then W_o for every half (K = C).
    if (lane == 0 && !p.inject_stall) {
      tma_prefetch_desc(&tm_wg);
      tma_prefetch_desc(&tm_wo);
      int ws = 0;
      uint32_t wph = 0;
      long long w_issued = 0;
      bool ok = true;
      for (int tile = blockIdx.x; tile < total && ok; tile += gridDim.x) {
        for (int part = 0; part < 2 && ok; ++part) {  // 0: W_g slabs, 1: W_o slabs
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
    // Per tile: gate phase (z' W_g^T into the gate columns of each half's
    // accumulator), then value phase (LN(x) W_o^T into the value columns).
    // Half hh uses TMEM columns [hh*256, hh*256+256): value at +0, gate at +128.
    if (lane == 0) {
      const uint32_t idesc_gate = idesc_f16_f32(BM, BN, 0, 0);  // z' K-major
      const uint32_t idesc_val = idesc_f16_f32(BM, BN, 1, 0);   // LN(x) MN-major
      int ws = 0;
      uint32_t wph = 0;
      bool ok = true;
      int n = 0;
      for (int tile = blockIdx.x; tile < total && ok; tile += gridDim.x, ++n) {
        const uint32_t ph = static_cast<uint32_t>(n) & 1u;
        for (int part = 0; part < 2 && ok; ++part) {
          if (!mbar_wait(part == 0 ? zready : xready, ph, st, SITE_MMA)) { ok = false; break; }
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
  } else if (warp < 3 + XFORM_THREADS / 32) {
    // ------------------------------------------------------------ LayerNorms (in place, fp16 out)
    const uint32_t t = threadIdx.x - 96;
    const float inv_d = 1.0f / static_cast<float>(p.D);
    const float inv_c = 1.0f / static_cast<float>(p.C);
    uint8_t* const zt = base_ptr + L.z;
    uint8_t* const xt = base_ptr + L.x;
    float* const xred = reinterpret_cast<float*>(base_ptr + L.xred);
    float* const zred = reinterpret_cast<float*>(base_ptr + L.zred);
    float* const xmu = reinterpret_cast<float*>(base_ptr + L.stat);
    float* const xrs = xmu + BM;
    // z: two threads per pair row, each owning half of the 8-element chunks
    const uint32_t zr = t & (BM - 1), zh = t >> 7;
    const int n8 = p.D >> 3;
    const int c8_lo = zh ? n8 / 2 : 0, c8_hi = zh ? n8 : n8 / 2;
    // x: chunk of 8 pairs and channel phase
    const uint32_t pc = t & 15, hp = t >> 4;
    const uint32_t x_chunk = (pc >> 3) * 8192u + ((((pc & 7u) ^ (hp & 7u)) & 7u) << 4);
    int n = 0;
    for (int tile = blockIdx.x; tile < total; tile += gridDim.x, ++n) {
      const uint32_t ph = static_cast<uint32_t>(n) & 1u;
      // ---- z row: LN over D (statistics from the input projection when given)
      if (!named_bar_and(1, XFORM_THREADS, mbar_wait(zfull, ph, st, SITE_XFORM))) break;
      float mu, rstd;
      if (p.zstats) {
        const int bb = tile / p.tiles_per_batch;
        const long long pidx = static_cast<long long>(tile - bb * p.tiles_per_batch) * BM + zr;
        const float2 ms = pidx < p.NN ? p.zstats[bb * p.NN + pidx] : make_float2(0.f, 1.f);
        mu = ms.x;
        rstd = ms.y;
      } else {
        // one pass, shifted by the row's first element (both half-row threads use it)
        const float shift = bf16_lo(*reinterpret_cast<const uint32_t*>(zt + sw128_offset(zr, 0)));
        float s1[8], s2[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) s1[e] = s2[e] = 0.f;
        for (int c8 = c8_lo; c8 < c8_hi; ++c8) {
          const uint4 v = *reinterpret_cast<const uint4*>(zt + (c8 >> 3) * SLAB + sw128_offset(zr, (c8 & 7) * 8));
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
        zred[zh * BM + zr] = t1;
        zred[(2 + zh) * BM + zr] = t2;
        named_bar_sync(1, XFORM_THREADS);
        const float m1 = (zred[zr] + zred[BM + zr]) * inv_d;
        mu = shift + m1;
        rstd = rsqrtf(fmaxf((zred[2 * BM + zr] + zred[3 * BM + zr]) * inv_d - m1 * m1, 0.f) + p.eps);
      }
      for (int c8 = c8_lo; c8 < c8_hi; ++c8) {
        uint4* const ptr = reinterpret_cast<uint4*>(zt + (c8 >> 3) * SLAB + sw128_offset(zr, (c8 & 7) * 8));
        const uint4 v = *ptr;
        const float4 g0 = __ldg(reinterpret_cast<const float4*>(p.ln_in_gamma) + 2 * c8);
        const float4 g1 = __ldg(reinterpret_cast<const float4*>(p.ln_in_gamma) + 2 * c8 + 1);
        const float4 b0 = __ldg(reinterpret_cast<const float4*>(p.ln_in_beta) + 2 * c8);
        const float4 b1 = __ldg(reinterpret_cast<const float4*>(p.ln_in_beta) + 2 * c8 + 1);
        uint4 o;
        o.x = pack_half2(fmaf((bf16_lo(v.x) - mu) * rstd, g0.x, b0.x), fmaf((bf16_hi(v.x) - mu) * rstd, g0.y, b0.y));
        o.y = pack_half2(fmaf((bf16_lo(v.y) - mu) * rstd, g0.z, b0.z), fmaf((bf16_hi(v.y) - mu) * rstd, g0.w, b0.w));
        o.z = pack_half2(fmaf((bf16_lo(v.z) - mu) * rstd, g1.x, b1.x), fmaf((bf16_hi(v.z) - mu) * rstd, g1.y, b1.y));
        o.w = pack_half2(fmaf((bf16_lo(v.w) - mu) * rstd, g1.z, b1.z), fmaf((bf16_hi(v.w) - mu) * rstd, g1.w, b1.w));
        *ptr = o;
      }
      fence_proxy_async_smem();
      mbar_arrive(zready);

      // ---- x columns: LN over C.  Thread (pc, hp) owns pairs 8pc..8pc+7 and
      // channels hp, hp+16, ...; every channel it owns has (c & 7) == (hp & 7),
      // so its 16-byte chunk sits at the same swizzled position in every row.
      if (!named_bar_and(2, XFORM_THREADS, mbar_wait(xfull, ph, st, SITE_XFORM))) break;
      // one pass, shifted per pair by its channel-0 value (the 16-byte chunk
      // of channel row 0 holding this thread's 8 pairs)
      const uint4 k8 = *reinterpret_cast<const uint4*>(xt + (pc >> 3) * 8192u + ((pc & 7u) << 4));
      const float kx[8] = {bf16_lo(k8.x), bf16_hi(k8.x), bf16_lo(k8.y), bf16_hi(k8.y),
                           bf16_lo(k8.z), bf16_hi(k8.z), bf16_lo(k8.w), bf16_hi(k8.w)};
      float s1[8], s2[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) s1[e] = s2[e] = 0.f;
      for (int c = hp; c < p.C; c += X_PHASES) {
        const uint4 v = *reinterpret_cast<const uint4*>(xt + (c >> 6) * SLAB + (c & 63) * 128 + x_chunk);
        const float f[8] = {bf16_lo(v.x), bf16_hi(v.x), bf16_lo(v.y), bf16_hi(v.y),
                            bf16_lo(v.z), bf16_hi(v.z), bf16_lo(v.w), bf16_hi(v.w)};
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const float d = f[e] - kx[e];
          s1[e] += d;
          s2[e] = fmaf(d, d, s2[e]);
        }
      }
      // lanes l and l^16 hold the same 8 pairs for two channel phases
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        s1[e] += __shfl_xor_sync(0xffffffffu, s1[e], 16);
        s2[e] += __shfl_xor_sync(0xffffffffu, s2[e], 16);
      }
      float* const xred2 = xred + (X_PHASES / 2) * BM;
      if ((hp & 1u) == 0) {
        float* const r1 = xred + (hp >> 1) * BM + pc * 8;
        float* const r2 = xred2 + (hp >> 1) * BM + pc * 8;
        reinterpret_cast<float4*>(r1)[0] = make_float4(s1[0], s1[1], s1[2], s1[3]);
        reinterpret_cast<float4*>(r1)[1] = make_float4(s1[4], s1[5], s1[6], s1[7]);
        reinterpret_cast<float4*>(r2)[0] = make_float4(s2[0], s2[1], s2[2], s2[3]);
        reinterpret_cast<float4*>(r2)[1] = make_float4(s2[4], s2[5], s2[6], s2[7]);
      }
      named_bar_sync(2, XFORM_THREADS);
      if (t < BM) {
        float t1 = 0.f, t2 = 0.f;
#pragma unroll
        for (int h = 0; h < X_PHASES / 2; ++h) {
          t1 += xred[h * BM + t];
          t2 += xred2[h * BM + t];
        }
        // shift of pair t: x(channel 0, pair t)
        const float kt = __bfloat162float(*reinterpret_cast<const __nv_bfloat16*>(
            xt + (t >> 6) * 8192u + ((((t & 63u) >> 3) & 7u) << 4) + ((t & 7u) << 1)));
        const float m1 = t1 * inv_c;
        xmu[t] = kt + m1;
        xrs[t] = rsqrtf(fmaxf(t2 * inv_c - m1 * m1, 0.f) + p.eps);
      }
      named_bar_sync(2, XFORM_THREADS);
      float mu8[8];
      {
        const float4 m0 = reinterpret_cast<const float4*>(xmu + pc * 8)[0];
        const float4 m1 = reinterpret_cast<const float4*>(xmu + pc * 8)[1];
        mu8[0] = m0.x; mu8[1] = m0.y; mu8[2] = m0.z; mu8[3] = m0.w;
        mu8[4] = m1.x; mu8[5] = m1.y; mu8[6] = m1.z; mu8[7] = m1.w;
      }
      float rs8[8];
      {
        const float4 r0 = reinterpret_cast<const float4*>(xrs + pc * 8)[0];
        const float4 r1 = reinterpret_cast<const float4*>(xrs + pc * 8)[1];
        rs8[0] = r0.x; rs8[1] = r0.y; rs8[2] = r0.z; rs8[3] = r0.w;
        rs8[4] = r1.x; rs8[5] = r1.y; rs8[6] = r1.z; rs8[7] = r1.w;
      }
      for (int c = hp; c < p.C; c += X_PHASES) {
        uint4* const ptr = reinterpret_cast<uint4*>(xt + (c >> 6) * SLAB + (c & 63) * 128 + x_chunk);
        const uint4 v = *ptr;
        const float g = __ldg(p.ln_out_gamma + c), b = __ldg(p.ln_out_beta + c);
        uint4 o;
        o.x = pack_half2(fmaf((bf16_lo(v.x) - mu8[0]) * rs8[0], g, b), fmaf((bf16_hi(v.x) - mu8[1]) * rs8[1], g, b));
        o.y = pack_half2(fmaf((bf16_lo(v.y) - mu8[2]) * rs8[2], g, b), fmaf((bf16_hi(v.y) - mu8[3]) * rs8[3], g, b));
        o.z = pack_half2(fmaf((bf16_lo(v.z) - mu8[4]) * rs8[4], g, b), fmaf((bf16_hi(v.z) - mu8[5]) * rs8[5], g, b));
        o.w = pack_half2(fmaf((bf16_lo(v.w) - mu8[6]) * rs8[6], g, b), fmaf((bf16_hi(v.w) - mu8[7]) * rs8[7], g, b));
        *ptr = o;
      }
      fence_proxy_async_smem();
      mbar_arrive(xready);
    }
  } else {
    // ------------------------------------------------------------ epilogue
    // Lane r of quadrant q holds pair row q*32+r.  Per block of 64 output
    // columns the lane computes 8 chunks of 8 bf16, then an 8x8 transpose of
    // chunks inside each group of 8 lanes (three butterfly rounds) leaves lane
    // 8a+b with chunk b of rows 8a..8a+7, so every store instruction writes
    // four whole 128-byte row segments.
    const int q = warp & 3;
    const uint32_t gb = lane & 7, ga = lane >> 3;
    bool ok = true;
    int n = 0;
    for (int tile = blockIdx.x; tile < total && ok; tile += gridDim.x, ++n) {
      const uint32_t aph = static_cast<uint32_t>(n) & 1u;  // each half's accumulator is used once per tile
      const int bb = tile / p.tiles_per_batch;
      const long long row0 = static_cast<long long>(tile - bb * p.tiles_per_batch) * BM + q * 32 + ga * 8;
      for (int hh = 0; hh < p.n_halves; ++hh) {
        const int acc = hh;
        if (!__all_sync(0xffffffffu, mbar_wait(tfull0 + 8 * acc, aph, st, SITE_EPI))) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t t_addr = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + acc * 256;
        const int n_cb = (hh * BN + 64 < p.D) ? 2 : 1;  // 64-column blocks in this half
#pragma unroll 1
        for (int cb = 0; cb < n_cb; ++cb) {
          const int col0 = hh * BN + cb * 64;
          uint4 R[8];
#pragma unroll
          for (int blk = 0; blk < 2; ++blk) {
            uint32_t v[32], g[32];
            tmem_ld32(t_addr + cb * 64 + blk * 32, v);
            tmem_ld32(t_addr + 128 + cb * 64 + blk * 32, g);
            tmem_ld_wait();
#pragma unroll
            for (int u = 0; u < 4; ++u) {
              float o[8];
#pragma unroll
              for (int e = 0; e < 8; ++e)
                o[e] = sigmoid_fast(__uint_as_float(g[u * 8 + e])) * __uint_as_float(v[u * 8 + e]);
              R[blk * 4 + u] = make_uint4(pack_bf162(o[0], o[1]), pack_bf162(o[2], o[3]), pack_bf162(o[4], o[5]),
                                          pack_bf162(o[6], o[7]));
            }
          }
          if (cb == n_cb - 1) {  // accumulator fully read: hand it back
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(tempty0 + 8 * acc);
          }
#pragma unroll
          for (int k = 4; k >= 1; k >>= 1) {
            const bool upper = (gb & k) != 0;
#pragma unroll
            for (int j = 0; j < 8; ++j) {
              if (j & k) continue;
              const uint4 lo = R[j], hi = R[j | k];
              const uint4 send = upper ? lo : hi;
              uint4 recv;
              recv.x = __shfl_xor_sync(0xffffffffu, send.x, k);
              recv.y = __shfl_xor_sync(0xffffffffu, send.y, k);
              recv.z = __shfl_xor_sync(0xffffffffu, send.z, k);
              recv.w = __shfl_xor_sync(0xffffffffu, send.w, k);
              R[j] = upper ? recv : lo;
              R[j | k] = upper ? hi : recv;
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
  if (a.w_stages < 1 || a.w_stages > MAX_W_STAGES) return cudaErrorInvalidValue;
  const size_t smem = outproj_smem_bytes(a.x_slabs, a.z_slabs, a.w_stages);
  cudaError_t e = cudaFuncSetAttribute(k3_outproj, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  k3_outproj<<<grid, THREADS, smem, s>>>(tm_x, tm_z, tm_wg, tm_wo, a);
  return cudaGetLastError();
}

}  // namespace trimul
