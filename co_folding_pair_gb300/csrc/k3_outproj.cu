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
// Structure (one persistent CTA per SM, 320 threads):
//   warp 0      TMA producer: x tile, z tile (single buffers), weight slabs
//               (128 rows x 64 K, fp16) into a ring
//   warp 1      TMEM (512 columns) + tcgen05.mma: per 128-column half of D,
//               gate = z' W_g^T (K = D) and value = LN(x) W_o^T (K = C)
//   warps 2..5  LayerNorm: row p of z (over D) and column p of x (over C),
//               fp32 statistics, results written in place as fp16
//   warps 6..9  epilogue: sigmoid(gate) * value -> bf16, 16-byte stores
// The accumulator pair (value 128 + gate 128 columns) is double-buffered.
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
constexpr int THREADS = 320;
constexpr int MAX_W_STAGES = 6;
}  // namespace

size_t outproj_smem_bytes(int x_slabs, int z_slabs, int w_stages) {
  return 1024 + static_cast<size_t>(x_slabs + z_slabs) * SLAB + static_cast<size_t>(w_stages) * W_SLAB + BAR_BYTES;
}

// Byte offset of x element (channel c, pair r) in an MN-major 128B-swizzled
// tile: 64-channel slabs of two 64-pair blocks, one 128-byte row per channel.
__device__ __forceinline__ uint32_t x_tile_offset(uint32_t c, uint32_t r) {
  const uint32_t cr = c & 63u, pr = r & 63u;
  return (c >> 6) * SLAB + (r >> 6) * 8192u + cr * 128u + ((((pr >> 3) ^ (cr & 7u)) & 7u) << 4) + ((pr & 7u) << 1);
}

__global__ void __launch_bounds__(THREADS, 1)
    k3_outproj(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_z,
               const __grid_constant__ CUtensorMap tm_wg, const __grid_constant__ CUtensorMap tm_wo,
               const OutprojArgs p) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_addr(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* const base_ptr = smem_raw + (base - raw);
  const uint32_t xbuf = base;
  const uint32_t zbuf = xbuf + p.x_slabs * SLAB;
  const uint32_t wring = zbuf + p.z_slabs * SLAB;
  const uint32_t bars = wring + p.w_stages * W_SLAB;
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
    mbar_init(xready, 128);
    mbar_init(xempty, 1);
    mbar_init(zfull, 1);
    mbar_init(zready, 128);
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
    // ------------------------------------------------------------ producer
    if (lane == 0 && !p.inject_stall) {
      tma_prefetch_desc(&tm_x);
      tma_prefetch_desc(&tm_z);
      tma_prefetch_desc(&tm_wg);
      tma_prefetch_desc(&tm_wo);
      int ws = 0;
      uint32_t wph = 0;
      long long w_issued = 0, n_issued = 0;
      bool ok = true;
      int n = 0;
      for (int tile = blockIdx.x; tile < total && ok; tile += gridDim.x, ++n) {
        const uint32_t ph = static_cast<uint32_t>(n) & 1u;
        const int bb = tile / p.tiles_per_batch;
        const int pair0 = (tile - bb * p.tiles_per_batch) * BM;
        if (!mbar_wait(zempty, ph ^ 1u, st, SITE_PRODUCER)) { ok = false; break; }
        mbar_arrive_expect_tx(zfull, p.z_slabs * SLAB);
        for (int s = 0; s < p.z_slabs; ++s) tma_load_3d(zbuf + s * SLAB, &tm_z, zfull, s * 64, pair0, bb);
        if (!mbar_wait(xempty, ph ^ 1u, st, SITE_PRODUCER)) { ok = false; ++n_issued; break; }
        mbar_arrive_expect_tx(xfull, p.x_slabs * SLAB);
        for (int s = 0; s < p.x_slabs; ++s)
          for (int h = 0; h < 2; ++h)
            tma_load_3d(xbuf + s * SLAB + h * 8192, &tm_x, xfull, pair0 + h * 64, s * 64, bb);
        ++n_issued;
        for (int hh = 0; hh < p.n_halves && ok; ++hh) {
          for (int part = 0; part < 2 && ok; ++part) {  // 0: W_g slabs (K = D), 1: W_o slabs (K = C)
            const int nsl = part == 0 ? p.z_slabs : p.x_slabs;
            const CUtensorMap* tm = part == 0 ? &tm_wg : &tm_wo;
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
        if (n_issued > 0) {
          const uint32_t ph_last = static_cast<uint32_t>(n_issued - 1) & 1u;
          mbar_wait_drain(zfull, ph_last, p.timeout_ns);
          mbar_wait_drain(xfull, ph_last, p.timeout_ns);
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t idesc_gate = idesc_f16_f32(BM, BN, 0, 0);  // z' K-major
      const uint32_t idesc_val = idesc_f16_f32(BM, BN, 1, 0);   // LN(x) MN-major
      int ws = 0, acc = 0;
      uint32_t wph = 0, aph = 0;
      bool ok = true;
      int n = 0;
      for (int tile = blockIdx.x; tile < total && ok; tile += gridDim.x, ++n) {
        const uint32_t ph = static_cast<uint32_t>(n) & 1u;
        for (int hh = 0; hh < p.n_halves && ok; ++hh) {
          if (!mbar_wait(tempty0 + 8 * acc, aph ^ 1u, st, SITE_MMA)) { ok = false; break; }
          tc_fence_after();
          const uint32_t d_val = tmem_base + acc * 256, d_gate = d_val + 128;
          for (int part = 0; part < 2 && ok; ++part) {
            if (hh == 0) {
              if (!mbar_wait(part == 0 ? zready : xready, ph, st, SITE_MMA)) { ok = false; break; }
              tc_fence_after();
            }
            const int nsl = part == 0 ? p.z_slabs : p.x_slabs;
            for (int s = 0; s < nsl; ++s) {
              if (!mbar_wait(wfull0 + 8 * ws, wph, st, SITE_MMA)) { ok = false; break; }
              tc_fence_after();
              const uint32_t wb = wring + ws * W_SLAB;
#pragma unroll
              for (int kk = 0; kk < 4; ++kk) {
                if (part == 0)
                  mma_f16_ss(d_gate, sdesc_sw128(zbuf + s * SLAB + kk * 32, 16, 1024),
                             sdesc_sw128(wb + kk * 32, 16, 1024), idesc_gate, (s | kk) != 0);
                else
                  mma_f16_ss(d_val, sdesc_sw128(xbuf + s * SLAB + kk * 2048, 8192, 1024),
                             sdesc_sw128(wb + kk * 32, 16, 1024), idesc_val, (s | kk) != 0);
              }
              mma_commit(wempty0 + 8 * ws);
              if (++ws == p.w_stages) { ws = 0; wph ^= 1u; }
            }
          }
          if (!ok) break;
          mma_commit(tfull0 + 8 * acc);
          if (++acc == 2) { acc = 0; aph ^= 1u; }
        }
        if (!ok) break;
        mma_commit(zempty);
        mma_commit(xempty);
      }
      if (!ok) {
        mma_commit(drain);
        mbar_wait_drain(drain, 0, p.timeout_ns);
      }
    }
  } else if (warp < 6) {
    // ------------------------------------------------------------ LayerNorms (in place, fp16 out)
    const uint32_t r = threadIdx.x - 64;
    const float inv_d = 1.0f / static_cast<float>(p.D);
    const float inv_c = 1.0f / static_cast<float>(p.C);
    const int n8 = p.D >> 3;
    uint8_t* const zt = base_ptr + (zbuf - base);
    uint8_t* const xt = base_ptr + (xbuf - base);
    int n = 0;
    for (int tile = blockIdx.x; tile < total; tile += gridDim.x, ++n) {
      const uint32_t ph = static_cast<uint32_t>(n) & 1u;
      // z row r: LN over D
      if (!__all_sync(0xffffffffu, mbar_wait(zfull, ph, st, SITE_XFORM))) break;
      float sum = 0.f;
      for (int c8 = 0; c8 < n8; ++c8) {
        const uint4 v = *reinterpret_cast<const uint4*>(zt + (c8 >> 3) * SLAB + sw128_offset(r, (c8 & 7) * 8));
        sum += bf16_lo(v.x) + bf16_hi(v.x) + bf16_lo(v.y) + bf16_hi(v.y) + bf16_lo(v.z) + bf16_hi(v.z) +
               bf16_lo(v.w) + bf16_hi(v.w);
      }
      const float mu = sum * inv_d;
      float ss = 0.f;
      for (int c8 = 0; c8 < n8; ++c8) {
        const uint4 v = *reinterpret_cast<const uint4*>(zt + (c8 >> 3) * SLAB + sw128_offset(r, (c8 & 7) * 8));
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float d0 = bf16_lo(w[e]) - mu, d1 = bf16_hi(w[e]) - mu;
          ss = fmaf(d0, d0, ss);
          ss = fmaf(d1, d1, ss);
        }
      }
      const float rstd = rsqrtf(ss * inv_d + p.eps);
      for (int c8 = 0; c8 < n8; ++c8) {
        uint4* const ptr = reinterpret_cast<uint4*>(zt + (c8 >> 3) * SLAB + sw128_offset(r, (c8 & 7) * 8));
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

      // x column r: LN over C
      if (!__all_sync(0xffffffffu, mbar_wait(xfull, ph, st, SITE_XFORM))) break;
      float xs = 0.f;
      for (int c = 0; c < p.C; ++c)
        xs += __bfloat162float(*reinterpret_cast<const __nv_bfloat16*>(xt + x_tile_offset(c, r)));
      const float xmu = xs * inv_c;
      float xss = 0.f;
      for (int c = 0; c < p.C; ++c) {
        const float d = __bfloat162float(*reinterpret_cast<const __nv_bfloat16*>(xt + x_tile_offset(c, r))) - xmu;
        xss = fmaf(d, d, xss);
      }
      const float xrstd = rsqrtf(xss * inv_c + p.eps);
      for (int c = 0; c < p.C; ++c) {
        __half* const ptr = reinterpret_cast<__half*>(xt + x_tile_offset(c, r));
        const float v = __bfloat162float(*reinterpret_cast<const __nv_bfloat16*>(ptr));
        *ptr = __float2half_rn(fmaf((v - xmu) * xrstd, __ldg(p.ln_out_gamma + c), __ldg(p.ln_out_beta + c)));
      }
      fence_proxy_async_smem();
      mbar_arrive(xready);
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;
    const int r = q * 32 + lane;
    int acc = 0;
    uint32_t aph = 0;
    bool ok = true;
    for (int tile = blockIdx.x; tile < total && ok; tile += gridDim.x) {
      const int bb = tile / p.tiles_per_batch;
      const long long pidx = static_cast<long long>(tile - bb * p.tiles_per_batch) * BM + r;
      const bool valid = pidx < p.NN;
      __nv_bfloat16* const orow = p.out + (static_cast<size_t>(bb) * p.NN + (valid ? pidx : 0)) * p.D;
      for (int hh = 0; hh < p.n_halves; ++hh) {
        if (!__all_sync(0xffffffffu, mbar_wait(tfull0 + 8 * acc, aph, st, SITE_EPI))) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t t_addr = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + acc * 256;
#pragma unroll 1
        for (int blk = 0; blk < BN / 32; ++blk) {
          const int col0 = hh * BN + blk * 32;
          if (col0 >= p.D) break;
          uint32_t v[32], g[32];
          tmem_ld32(t_addr + blk * 32, v);
          tmem_ld32(t_addr + 128 + blk * 32, g);
          tmem_ld_wait();
          if (valid) {
#pragma unroll
            for (int u = 0; u < 4; ++u) {
              if (col0 + u * 8 < p.D) {
                float o[8];
#pragma unroll
                for (int e = 0; e < 8; ++e)
                  o[e] = sigmoid_fast(__uint_as_float(g[u * 8 + e])) * __uint_as_float(v[u * 8 + e]);
                uint4 pk;
                pk.x = pack_bf162(o[0], o[1]);
                pk.y = pack_bf162(o[2], o[3]);
                pk.z = pack_bf162(o[4], o[5]);
                pk.w = pack_bf162(o[6], o[7]);
                *reinterpret_cast<uint4*>(orow + col0 + u * 8) = pk;
              }
            }
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(tempty0 + 8 * acc);
        if (++acc == 2) { acc = 0; aph ^= 1u; }
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
