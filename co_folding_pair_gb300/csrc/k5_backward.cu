// k5_backward.cu -- the per-pair (CUDA-core) steps of the TriMul backward pass.
//
// The backward of the update takes the forward's steps in reverse order; the
// contractions run in k4_gemm.cu and k2_triangle.cu, and these kernels do the
// per-pair work between them, each one streaming pass over its planes (zh =
// (z - mean) rstd, the normalised input rows, is stored by the input
// projection's recompute):
//
//   k5_xhat       statistics of x over C per pair and xh = (x - mean) rstd,
//                 channel-major like x
//   k5_dout       output gate and value from their projections (fp16): with
//                 g = zh W~_g^T + t_g and v = xh W~_o^T + t_o,
//                 dv = dout sigmoid(g), dg = dout v sigmoid(g) (1 - sigmoid(g)),
//                 and the column sums of dv and dg over all pairs
//   k5_lnout_bwd  dx = r (dy^ - mean(dy^) - xh mean(dy^ xh)), dy^ = dy gamma_out
//   k5_lnin_bwd   dz = r (dz^ - mean(dz^) - zh mean(dz^ zh)), dz^ = dz' gamma_in,
//                 and the column sums of dz' zh and dz' (d gamma_in, d beta_in)
//   k5_sum, k5_assemble  the reductions of the per-block partial sums and the
//                 final parameter gradients
//
// LayerNorm gamma and beta are folded out of the stored planes (zh and xh are
// bare normalised rows): with y = yh gamma + beta and u = y W^T,
//   dW = (du^T yh) diag(gamma) + (sum_p du_p) beta^T,
//   d gamma_out[c] = sum_d W_o[d][c] (dv^T xh)[d][c],  d beta_out[c] = sum_d W_o[d][c] (sum_p dv_p)[d],
// so every sum over pairs is either a tensor-core GEMM or a column / row sum
// that one thread keeps for a fixed feature.  All partial sums are per block
// and reduced in a fixed order: the results are deterministic.
#include <algorithm>

#include "kernels.h"
#include "sm103_ptx.cuh"

namespace trimul {

namespace {

__device__ __forceinline__ float sigmoidf_(float x) { return 1.0f / (1.0f + __expf(-x)); }

__device__ __forceinline__ void unpack_bf16x8(const uint4 v, float (&f)[8]) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    f[2 * e] = bf16_lo(w[e]);
    f[2 * e + 1] = bf16_hi(w[e]);
  }
}

__device__ __forceinline__ uint4 pack_bf16x8(const float (&f)[8]) {
  return make_uint4(pack_bf162(f[0], f[1]), pack_bf162(f[2], f[3]), pack_bf162(f[4], f[5]), pack_bf162(f[6], f[7]));
}

// 16-byte asynchronous copy global -> shared (both 16-byte aligned), and the
// wait for all of this thread's outstanding copies.
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }
// Close this thread's group of copies issued since the last commit (an empty
// group when there were none), and wait until at most one group is pending.
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_one_pending() { asm volatile("cp.async.wait_group 1;" ::: "memory"); }

__device__ __forceinline__ float x_scale_of(const unsigned* ab_max, int N) {
  return exp2_neg(x_scale_log2_from_max(__uint_as_float(*ab_max), N));
}

}  // namespace

// ------------------------------------------------------------------ xh
// x holds x * 2^-s; its statistics are taken in those units with
// eps * 4^-s, which normalises x exactly as LN_out does with eps.  Tiles of
// 64 consecutive pairs of one batch element, staged in shared memory (C x 64
// fp16) so x is read from DRAM once; two buffers, so that the next tile's
// copies are in flight while this one is normalised.  Thread (g, p): pair p
// of the tile, channels c = g, g + 4, ... (32 consecutive pairs per warp, so
// the shared-memory accesses of a warp fall in distinct banks).
constexpr int XH_PAIRS = 64;
constexpr int XH_THREADS = 256;
constexpr int XH_GROUPS = XH_THREADS / XH_PAIRS;

__global__ void __launch_bounds__(XH_THREADS)
    k5_xhat(const __half* __restrict__ x, __nv_bfloat16* __restrict__ xh, float2* __restrict__ xstats,
            const unsigned* ab_max, int B, int N, int C, float eps) {
  extern __shared__ float4 xh_smem[];
  __half* const sx0 = reinterpret_cast<__half*>(xh_smem);                   // [2][C][64]
  float* const red = reinterpret_cast<float*>(sx0 + 2 * C * XH_PAIRS);      // [2][4][64] sums
  const long long P = static_cast<long long>(N) * N;
  const long long tiles_per_b = P / XH_PAIRS;
  const long long total = B * tiles_per_b;
  const float xs = x_scale_of(ab_max, N);
  const float eps_s = eps * xs * xs;
  const float inv_c = 1.0f / static_cast<float>(C);
  const int g = threadIdx.x / XH_PAIRS, p = threadIdx.x % XH_PAIRS;
  // copies of tile t into buffer buf, one commit group per thread
  auto issue = [&](long long t, int buf) {
    if (t < total) {
      const long long b = t / tiles_per_b, p0 = (t - b * tiles_per_b) * XH_PAIRS;
      const __half* xb = x + b * C * P + p0;
      __half* const dst = sx0 + buf * C * XH_PAIRS;
      for (int i = threadIdx.x; i < C * 8; i += blockDim.x) {
        const int c = i >> 3, k = i & 7;
        cp_async16(smem_addr(dst + i * 8), xb + static_cast<size_t>(c) * P + k * 8);
      }
    }
    cp_async_commit();
  };
  int buf = 0;
  issue(blockIdx.x, 0);
  for (long long tile = blockIdx.x; tile < total; tile += gridDim.x, buf ^= 1) {
    issue(tile + gridDim.x, buf ^ 1);  // the other buffer was released at the end of the last iteration
    cp_async_wait_one_pending();       // this tile's copies have landed
    __syncthreads();
    const __half* const sx = sx0 + buf * C * XH_PAIRS;
    const long long b = tile / tiles_per_b, p0 = (tile - b * tiles_per_b) * XH_PAIRS;
    // shifted sums (shift: the pair's channel-0 value, read by every group)
    const float k0 = __half2float(sx[p]);
    float s1 = 0.f, s2 = 0.f;
    for (int c = g; c < C; c += XH_GROUPS) {
      const float d = __half2float(sx[c * XH_PAIRS + p]) - k0;
      s1 += d;
      s2 = fmaf(d, d, s2);
    }
    red[g * XH_PAIRS + p] = s1;
    red[(XH_GROUPS + g) * XH_PAIRS + p] = s2;
    __syncthreads();
    float t1 = 0.f, t2 = 0.f;
#pragma unroll
    for (int k = 0; k < XH_GROUPS; ++k) {
      t1 += red[k * XH_PAIRS + p];
      t2 += red[(XH_GROUPS + k) * XH_PAIRS + p];
    }
    const float m1 = t1 * inv_c;
    const float mu = k0 + m1;
    const float r = rsqrtf(fmaxf(t2 * inv_c - m1 * m1, 0.f) + eps_s);
    if (g == 0) xstats[b * P + p0 + p] = make_float2(mu, r);
    __nv_bfloat16* const ob = xh + b * C * P + p0 + p;
    for (int c = g; c < C; c += XH_GROUPS)
      ob[static_cast<size_t>(c) * P] = __float2bfloat16_rn((__half2float(sx[c * XH_PAIRS + p]) - mu) * r);
    __syncthreads();  // every thread is done with this buffer and with red
  }
  cp_async_wait_all();
}

// ------------------------------------------------------------------ output gate
// Thread (c8, r): features c8*8 .. c8*8+7 of pairs r, r + Rb, ... of its block's
// stride; it keeps the column sums of those 8 features.  Partials:
// part[block][0][D] (dv) and part[block][1][D] (dg).
__global__ void k5_dout(const __nv_bfloat16* __restrict__ dout, const __half* __restrict__ gacc,
                        const __half* __restrict__ vacc, const float* __restrict__ tg, const float* __restrict__ to,
                        __nv_bfloat16* __restrict__ dv, __nv_bfloat16* __restrict__ dg, float* __restrict__ part,
                        long long n_pairs, int D) {
  extern __shared__ float red[];  // [Rb][2][D]
  const int d8 = D >> 3, rb = blockDim.x / d8;
  const int c8 = threadIdx.x % d8, r = threadIdx.x / d8;
  float sv[8], sg[8], t_g[8], t_o[8];
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    sv[e] = sg[e] = 0.f;
    t_g[e] = tg[c8 * 8 + e];
    t_o[e] = to[c8 * 8 + e];
  }
  if (r < rb) {
    for (long long pr = blockIdx.x * static_cast<long long>(rb) + r; pr < n_pairs;
         pr += static_cast<long long>(gridDim.x) * rb) {
      const long long i = pr * d8 + c8;
      float o[8], g[8], v[8], a[8], b[8];
      unpack_bf16x8(reinterpret_cast<const uint4*>(dout)[i], o);
      const uint4 g8 = reinterpret_cast<const uint4*>(gacc)[i], v8 = reinterpret_cast<const uint4*>(vacc)[i];
      const uint32_t gw[4] = {g8.x, g8.y, g8.z, g8.w}, vw[4] = {v8.x, v8.y, v8.z, v8.w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float2 gf = __half22float2(*reinterpret_cast<const __half2*>(&gw[e]));
        const float2 vf = __half22float2(*reinterpret_cast<const __half2*>(&vw[e]));
        g[2 * e] = gf.x;
        g[2 * e + 1] = gf.y;
        v[2 * e] = vf.x;
        v[2 * e + 1] = vf.y;
      }
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const float s = sigmoidf_(g[e] + t_g[e]);
        const float val = v[e] + t_o[e];
        a[e] = o[e] * s;
        b[e] = o[e] * val * s * (1.0f - s);
      }
      const uint4 pa = pack_bf16x8(a), pb = pack_bf16x8(b);
      reinterpret_cast<uint4*>(dv)[i] = pa;
      reinterpret_cast<uint4*>(dg)[i] = pb;
      // sums of the stored (rounded) values, as the GEMMs see them
      float ra[8], rb2[8];
      unpack_bf16x8(pa, ra);
      unpack_bf16x8(pb, rb2);
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        sv[e] += ra[e];
        sg[e] += rb2[e];
      }
    }
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      red[(r * 2 + 0) * D + c8 * 8 + e] = sv[e];
      red[(r * 2 + 1) * D + c8 * 8 + e] = sg[e];
    }
  }
  __syncthreads();
  for (int k = threadIdx.x; k < 2 * D; k += blockDim.x) {
    float s = 0.f;
    for (int rr = 0; rr < rb; ++rr) s += red[rr * 2 * D + k];
    part[static_cast<size_t>(blockIdx.x) * 2 * D + k] = s;
  }
}

// ------------------------------------------------------------------ LN_out backward
// dy holds dy^T (bf16 [B][C][P]); x, xstats as k5_xhat; dx bf16 [B][C][P].
// A block takes tiles of LNO_PAIRS consecutive pairs of one batch element: it
// stages the tile's dy and x rows (C x 64 each) in shared memory with 16-byte
// loads, so each value comes from DRAM once although the formula needs two
// passes over the row.  Thread (g, p): pair p of the tile, channels
// c = g, g + 4, ... (4 channel groups, 32 consecutive pairs per warp, so the
// shared-memory accesses of a warp fall in distinct banks).
constexpr int LNO_PAIRS = 64;
constexpr int LNO_THREADS = 256;

__global__ void __launch_bounds__(LNO_THREADS)
    k5_lnout_bwd(const __nv_bfloat16* __restrict__ dy, const __half* __restrict__ x, const float2* __restrict__ xstats,
                 const float* __restrict__ gamma, __nv_bfloat16* __restrict__ dx, const unsigned* ab_max, int B, int N,
                 int C) {
  extern __shared__ float4 lno_smem[];
  __nv_bfloat16* const sdy = reinterpret_cast<__nv_bfloat16*>(lno_smem);  // [C][64]
  __half* const sx = reinterpret_cast<__half*>(sdy + C * LNO_PAIRS);       // [C][64]
  float* const gam = reinterpret_cast<float*>(sx + C * LNO_PAIRS);       // [C]
  float* const red = gam + C;                                            // [2][4][64]
  for (int c = threadIdx.x; c < C; c += blockDim.x) gam[c] = gamma[c];
  const long long P = static_cast<long long>(N) * N;
  const long long tiles_per_b = P / LNO_PAIRS;  // P is a multiple of 64
  const float xs = x_scale_of(ab_max, N);       // r of x = r of x * 2^-s, times 2^-s
  const float inv_c = 1.0f / static_cast<float>(C);
  const int g = threadIdx.x >> 6, p = threadIdx.x & 63;
  for (long long tile = blockIdx.x; tile < B * tiles_per_b; tile += gridDim.x) {
    const long long b = tile / tiles_per_b, p0 = (tile - b * tiles_per_b) * LNO_PAIRS;
    const __nv_bfloat16* dyb = dy + b * C * P + p0;
    const __half* xb = x + b * C * P + p0;
    __syncthreads();  // the previous tile's readers are done
    // dy and x rows: 64 16-bit values = 8 chunks of 16 bytes.  Asynchronous
    // copies: every chunk of the tile is in flight at once.
    for (int i = threadIdx.x; i < C * 8; i += blockDim.x) {
      const int c = i >> 3, k = i & 7;
      cp_async16(smem_addr(sdy + i * 8), dyb + static_cast<size_t>(c) * P + k * 8);
    }
    for (int i = threadIdx.x; i < C * 8; i += blockDim.x) {
      const int c = i >> 3, k = i & 7;
      cp_async16(smem_addr(sx + i * 8), xb + static_cast<size_t>(c) * P + k * 8);
    }
    cp_async_wait_all();
    __syncthreads();
    const float2 st = xstats[b * P + p0 + p];
    float s1 = 0.f, s2 = 0.f;
    for (int c = g; c < C; c += 4) {
      const float h = (__half2float(sx[c * LNO_PAIRS + p]) - st.x) * st.y;
      const float d = __bfloat162float(sdy[c * LNO_PAIRS + p]) * gam[c];
      s1 += d;
      s2 = fmaf(d, h, s2);
    }
    red[g * LNO_PAIRS + p] = s1;
    red[(4 + g) * LNO_PAIRS + p] = s2;
    __syncthreads();
    float m1 = 0.f, m2 = 0.f;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      m1 += red[k * LNO_PAIRS + p];
      m2 += red[(4 + k) * LNO_PAIRS + p];
    }
    m1 *= inv_c;
    m2 *= inv_c;
    const float r = st.y * xs;
    __nv_bfloat16* const ob = dx + b * C * P + p0 + p;
    for (int c = g; c < C; c += 4) {
      const float h = (__half2float(sx[c * LNO_PAIRS + p]) - st.x) * st.y;
      const float d = __bfloat162float(sdy[c * LNO_PAIRS + p]) * gam[c];
      ob[static_cast<size_t>(c) * P] = __float2bfloat16_rn(r * (d - m1 - h * m2));
    }
  }
}

// ------------------------------------------------------------------ gated input projections
// Rows rc = b * C + c (one channel row of a and b) from grid.y in steps of
// gridDim.y, grid.x = segments of the pairs.  pt: [B][4C][P] pre-activations without their biases (rows: value a,
// gate a, value b, gate b; t_in holds the biases), overwritten in place with
// their gradients.  part[(b * C + c) * gridDim.x + segment][4]: row sums.

// ------------------------------------------------------------------ LN_in backward
// One warp per pair; lane l < D / 8 owns features 8l .. 8l+7 and keeps their
// sums of dz' zh and dz' over the warp's pairs.  dz' = dzp + dzq (its gate
// and input-projection parts).  part[block][2][D].
__global__ void k5_lnin_bwd(const __nv_bfloat16* __restrict__ dzp, const __nv_bfloat16* __restrict__ dzq,
                            const __nv_bfloat16* __restrict__ z,
                            const float2* __restrict__ zstats, const float* __restrict__ gamma,
                            __nv_bfloat16* __restrict__ dz, float* __restrict__ part, long long n_pairs, int D) {
  extern __shared__ float red[];  // [warps][2][D]
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5, nw = blockDim.x >> 5;
  const int d8 = D >> 3;
  const bool on = lane < d8;
  float gm[8], sgam[8], sbet[8];
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    gm[e] = on ? gamma[lane * 8 + e] : 0.f;
    sgam[e] = sbet[e] = 0.f;
  }
  const float inv_d = 1.0f / static_cast<float>(D);
  for (long long pr = blockIdx.x * static_cast<long long>(nw) + wid; pr < n_pairs;
       pr += static_cast<long long>(gridDim.x) * nw) {
    const float2 ms = zstats[pr];
    float g[8], zz[8], h[8], dh[8];
    float s1 = 0.f, s2 = 0.f;
    const long long i = pr * d8 + lane;
    if (on) {
      float gq[8];
      unpack_bf16x8(reinterpret_cast<const uint4*>(dzp)[i], g);
      unpack_bf16x8(reinterpret_cast<const uint4*>(dzq)[i], gq);
#pragma unroll
      for (int e = 0; e < 8; ++e) g[e] += gq[e];
      unpack_bf16x8(reinterpret_cast<const uint4*>(z)[i], zz);
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        h[e] = (zz[e] - ms.x) * ms.y;
        dh[e] = g[e] * gm[e];
        s1 += dh[e];
        s2 = fmaf(dh[e], h[e], s2);
        sgam[e] = fmaf(g[e], h[e], sgam[e]);
        sbet[e] += g[e];
      }
    }
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) {
      s1 += __shfl_xor_sync(0xffffffffu, s1, o);
      s2 += __shfl_xor_sync(0xffffffffu, s2, o);
    }
    if (on) {
      const float m1 = s1 * inv_d, m2 = s2 * inv_d;
      float o8[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) o8[e] = ms.y * (dh[e] - m1 - h[e] * m2);
      reinterpret_cast<uint4*>(dz)[i] = pack_bf16x8(o8);
    }
  }
  if (on) {
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      red[(wid * 2 + 0) * D + lane * 8 + e] = sgam[e];
      red[(wid * 2 + 1) * D + lane * 8 + e] = sbet[e];
    }
  }
  __syncthreads();
  for (int k = threadIdx.x; k < 2 * D; k += blockDim.x) {
    float s = 0.f;
    for (int w = 0; w < nw; ++w) s += red[w * 2 * D + k];
    part[static_cast<size_t>(blockIdx.x) * 2 * D + k] = s;
  }
}

// ------------------------------------------------------------------ reductions
// out[i] = sum_j part[j * n + i], j < count (a fixed order).
__global__ void k5_sum(const float* __restrict__ part, float* __restrict__ out, long long n, int count) {
  for (long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; i < n;
       i += static_cast<long long>(gridDim.x) * blockDim.x) {
    float s = 0.f;
    for (int j = 0; j < count; ++j) s += part[static_cast<size_t>(j) * n + i];
    out[i] = s;
  }
}

// The parameter gradients from the reduced sums.  m_o [D][C] = dv^T xh,
// m_g [D][D] = dg^T zh, m_in [4C][D] = dP^T zh, cs [2][D] = column sums of dv
// and dg, gp = the gate kernel's partials (rows b * C + c, nseg segments,
// 4 sums each), ln_in [2][D] = d gamma_in, d beta_in.
__global__ void k5_assemble(const float* __restrict__ m_o, const float* __restrict__ m_g,
                            const float* __restrict__ m_in, const float* __restrict__ cs,
                            const float* __restrict__ gp, int nseg, const float* __restrict__ ln_in,
                            const float* __restrict__ w_o, const float* __restrict__ g_in,
                            const float* __restrict__ b_in, const float* __restrict__ g_out,
                            const float* __restrict__ b_out, TrimulGradPtrs out, int B, int D, int C) {
  const int tid = blockIdx.x * blockDim.x + threadIdx.x, nt = gridDim.x * blockDim.x;
  for (int i = tid; i < D * C; i += nt) {  // dW_o [D][C]
    const int d = i / C, c = i - d * C;
    out.w_o[i] = m_o[i] * g_out[c] + cs[d] * b_out[c];
  }
  for (int i = tid; i < D * D; i += nt) {  // dW_g [D][D]
    const int d = i / D, e = i - d * D;
    out.w_g[i] = m_g[i] * g_in[e] + cs[D + d] * b_in[e];
  }
  for (int i = tid; i < 4 * C * D; i += nt) {  // dW_a, dW_ga, dW_b, dW_gb [C][D] each
    const int f = i / D, e = i - f * D, k = f / C, c = f - k * C;
    float rs = 0.f;
    for (int b = 0; b < B; ++b)
      for (int s = 0; s < nseg; ++s) rs += gp[((static_cast<size_t>(b) * C + c) * nseg + s) * 4 + k];
    float* const dst = k == 0 ? out.w_a : k == 1 ? out.w_ga : k == 2 ? out.w_b : out.w_gb;
    dst[c * D + e] = m_in[i] * g_in[e] + rs * b_in[e];
  }
  for (int c = tid; c < C; c += nt) {  // d gamma_out, d beta_out
    float sg = 0.f, sb = 0.f;
    for (int d = 0; d < D; ++d) {
      sg = fmaf(w_o[d * C + c], m_o[d * C + c], sg);
      sb = fmaf(w_o[d * C + c], cs[d], sb);
    }
    out.ln_out_gamma[c] = sg;
    out.ln_out_beta[c] = sb;
  }
  for (int d = tid; d < D; d += nt) {
    out.ln_in_gamma[d] = ln_in[d];
    out.ln_in_beta[d] = ln_in[D + d];
  }
}

// ------------------------------------------------------------------ launchers
namespace {
int stream_blocks(long long items, int per_block, int num_sms) {
  const long long want = (items + per_block - 1) / per_block;
  return static_cast<int>(std::max<long long>(1, std::min<long long>(want, 8ll * num_sms)));
}
}  // namespace


cudaError_t launch_xhat(const __half* x, __nv_bfloat16* xh, float2* xstats, const unsigned* ab_max, int B, int N,
                        int C, float eps, int num_sms, cudaStream_t s) {
  const size_t smem = 2 * static_cast<size_t>(C) * XH_PAIRS * 2 + 2 * XH_GROUPS * XH_PAIRS * 4;
  cudaError_t e =
      cudaFuncSetAttribute(k5_xhat, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  const long long tiles = static_cast<long long>(B) * N * N / XH_PAIRS;
  // as many resident blocks as shared memory allows: each keeps its next tile's
  // loads in flight
  int per_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k5_xhat, XH_THREADS, smem) != cudaSuccess || per_sm < 1) {
    cudaGetLastError();
    per_sm = 4;
  }
  const int grid = static_cast<int>(std::max<long long>(1, std::min<long long>(tiles, 1ll * per_sm * num_sms)));
  k5_xhat<<<grid, XH_THREADS, smem, s>>>(x, xh, xstats, ab_max, B, N, C, eps);
  return cudaGetLastError();
}

int dout_blocks(long long n_pairs, int D, int num_sms) {
  const int d8 = D / 8, rb = 256 / d8;
  return stream_blocks(n_pairs, rb, num_sms);
}

cudaError_t launch_dout(const __nv_bfloat16* dout, const __half* gacc, const __half* vacc, const float* tg,
                        const float* to, __nv_bfloat16* dv, __nv_bfloat16* dg, float* part, long long n_pairs, int D,
                        int num_sms, cudaStream_t s) {
  const int d8 = D / 8, rb = 256 / d8;
  const size_t smem = static_cast<size_t>(rb) * 2 * D * sizeof(float);
  k5_dout<<<dout_blocks(n_pairs, D, num_sms), d8 * rb, smem, s>>>(dout, gacc, vacc, tg, to, dv, dg, part, n_pairs, D);
  return cudaGetLastError();
}

cudaError_t launch_lnout_bwd(const __nv_bfloat16* dy, const __half* x, const float2* xstats, const float* gamma,
                             __nv_bfloat16* dx, const unsigned* ab_max, int B, int N, int C, int num_sms,
                             cudaStream_t s) {
  const size_t smem = static_cast<size_t>(C) * LNO_PAIRS * (2 + 2) + C * 4 + 8 * LNO_PAIRS * 4;
  cudaError_t e = cudaFuncSetAttribute(k5_lnout_bwd, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  const long long tiles = static_cast<long long>(B) * N * N / LNO_PAIRS;
  int per_sm = 0;  // as many resident blocks as shared memory allows (as for xh)
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k5_lnout_bwd, LNO_THREADS, smem) != cudaSuccess ||
      per_sm < 1) {
    cudaGetLastError();
    per_sm = 2;
  }
  const int grid = static_cast<int>(std::max<long long>(1, std::min<long long>(tiles, 1ll * per_sm * num_sms)));
  k5_lnout_bwd<<<grid, LNO_THREADS, smem, s>>>(dy, x, xstats, gamma, dx, ab_max, B, N, C);
  return cudaGetLastError();
}



int lnin_blocks(long long n_pairs, int num_sms) { return stream_blocks(n_pairs, 8, num_sms); }

cudaError_t launch_lnin_bwd(const __nv_bfloat16* dzp, const __nv_bfloat16* dzq, const __nv_bfloat16* z, const float2* zstats,
                            const float* gamma, __nv_bfloat16* dz, float* part, long long n_pairs, int D, int num_sms,
                            cudaStream_t s) {
  k5_lnin_bwd<<<lnin_blocks(n_pairs, num_sms), 256, 8 * 2 * D * sizeof(float), s>>>(dzp, dzq, z, zstats, gamma, dz,
                                                                                      part, n_pairs, D);
  return cudaGetLastError();
}

cudaError_t launch_sum(const float* part, float* out, long long n, int count, int num_sms, cudaStream_t s) {
  k5_sum<<<stream_blocks(n, 256, num_sms), 256, 0, s>>>(part, out, n, count);
  return cudaGetLastError();
}

cudaError_t launch_assemble(const float* m_o, const float* m_g, const float* m_in, const float* cs, const float* gp,
                            int nseg, const float* ln_in, const float* w_o, const float* g_in, const float* b_in,
                            const float* g_out, const float* b_out, const TrimulGradPtrs& out, int B, int D, int C,
                            int num_sms, cudaStream_t s) {
  k5_assemble<<<stream_blocks(4ll * C * D, 256, num_sms), 256, 0, s>>>(m_o, m_g, m_in, cs, gp, nseg, ln_in, w_o, g_in,
                                                                        b_in, g_out, b_out, out, B, D, C);
  return cudaGetLastError();
}

}  // namespace trimul
