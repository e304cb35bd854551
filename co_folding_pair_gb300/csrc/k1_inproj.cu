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
// thread owns one channel plane and writes runs of pairs with 16-byte stores.
//
// Structure (one persistent CTA per SM, 448 threads):
//   warp 0       TMA producer: z tiles (128 pairs x D, bf16) into 2 buffers,
//                weight slabs (128 value rows + their 128 gate rows, x 64 K,
//                fp16) into a ring
//   warp 1       allocates 512 TMEM columns and issues tcgen05.mma: per chunk of
//                128 output channels, value = W_v z'^T and gate = W_g z'^T
//                (M = 128 channels, N = 128 pairs, K = D in slabs of 64)
//   warps 2..5   LayerNorm: one pair row per thread, fp32 statistics (two
//                passes), z' written back in place as fp16 in the same
//                swizzled layout, which the MMA then reads as its B operand
//   warps 6..13  epilogue: sigmoid(gate) * value * mask -> fp16, two warps per
//                TMEM lane quadrant, 64 pairs each
// The accumulator pair (128 value + 128 gate columns) is double-buffered.
#include "kernels.h"
#include "sm103_ptx.cuh"

namespace trimul {

namespace {
constexpr int BM = 128;                     // pairs per tile
constexpr int CH = 128;                     // output channels per chunk
constexpr uint32_t Z_SLAB = BM * 128;       // 16 KB: 128 pair rows x 64 K
constexpr uint32_t W_SLAB = 2 * CH * 128;   // 32 KB: 128 value + 128 gate rows x 64 K
constexpr uint32_t BAR_BYTES = 256;
constexpr uint32_t TMEM_COLS = 512;
constexpr int EPI_WARPS = 8;
constexpr int THREADS = 64 + 128 + 32 * EPI_WARPS;
constexpr int MAX_W_STAGES = 4;
}  // namespace

size_t inproj_smem_bytes(int k_slabs, int w_stages) {
  return 1024 + 2 * static_cast<size_t>(k_slabs) * Z_SLAB + static_cast<size_t>(w_stages) * W_SLAB + BAR_BYTES;
}

__global__ void __launch_bounds__(THREADS, 1)
    k1_inproj(const __grid_constant__ CUtensorMap tm_z, const __grid_constant__ CUtensorMap tm_w,
              const InprojArgs p) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_addr(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* const base_ptr = smem_raw + (base - raw);
  const uint32_t z_buf_bytes = p.k_slabs * Z_SLAB;
  const uint32_t zbuf0 = base;                      // 2 z buffers
  const uint32_t wring = base + 2 * z_buf_bytes;    // weight ring
  const uint32_t bars = wring + p.w_stages * W_SLAB;
  // barriers: zfull[2] zready[2] zempty[2] wfull[4] wempty[4] tfull[2] tempty[2] drain, tmem slot
  const uint32_t zfull0 = bars, zready0 = bars + 16, zempty0 = bars + 32;
  const uint32_t wfull0 = bars + 48, wempty0 = wfull0 + 8 * MAX_W_STAGES;
  const uint32_t tfull0 = wempty0 + 8 * MAX_W_STAGES, tempty0 = tfull0 + 16;
  const uint32_t drain = tempty0 + 16, tmem_slot = drain + 8;
  volatile uint32_t* tmem_slot_ptr = reinterpret_cast<volatile uint32_t*>(base_ptr + (tmem_slot - base));

  const KStatus st{p.status, p.timeout_ns};
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int i = 0; i < 2; ++i) {
      mbar_init(zfull0 + 8 * i, 1);
      mbar_init(zready0 + 8 * i, 128);
      mbar_init(zempty0 + 8 * i, 1);
      mbar_init(tfull0 + 8 * i, 1);
      mbar_init(tempty0 + 8 * i, EPI_WARPS);
    }
    for (int s = 0; s < p.w_stages; ++s) {
      mbar_init(wfull0 + 8 * s, 1);
      mbar_init(wempty0 + 8 * s, 1);
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
  const int C2 = 2 * p.C;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0 && !p.inject_stall) {
      tma_prefetch_desc(&tm_z);
      tma_prefetch_desc(&tm_w);
      int ws = 0;
      uint32_t wph = 0;
      long long w_issued = 0, z_issued = 0;
      bool ok = true;
      auto issue_z = [&](int tile, int n) -> bool {
        const int zb = n & 1;
        const uint32_t zph = static_cast<uint32_t>(n >> 1) & 1u;
        if (!mbar_wait(zempty0 + 8 * zb, zph ^ 1u, st, SITE_PRODUCER)) return false;
        const int bb = tile / p.tiles_per_batch;
        const int pair0 = (tile - bb * p.tiles_per_batch) * BM;
        const uint32_t fb = zfull0 + 8 * zb;
        mbar_arrive_expect_tx(fb, z_buf_bytes);
        for (int s = 0; s < p.k_slabs; ++s)
          tma_load_3d(zbuf0 + zb * z_buf_bytes + s * Z_SLAB, &tm_z, fb, s * 64, pair0, bb);
        ++z_issued;
        return true;
      };
      int n = 0;
      if (static_cast<int>(blockIdx.x) < total) ok = issue_z(blockIdx.x, 0);
      for (int tile = blockIdx.x; tile < total && ok; tile += gridDim.x, ++n) {
        const int next = tile + gridDim.x;
        if (next < total && !issue_z(next, n + 1)) {
          ok = false;
          break;
        }
        for (int qc = 0; qc < p.n_chunks && ok; ++qc) {
          for (int s = 0; s < p.k_slabs; ++s) {
            if (!mbar_wait(wempty0 + 8 * ws, wph ^ 1u, st, SITE_PRODUCER)) {
              ok = false;
              break;
            }
            mbar_arrive_expect_tx(wfull0 + 8 * ws, W_SLAB);
            tma_load_2d(wring + ws * W_SLAB, &tm_w, wfull0 + 8 * ws, s * 64, qc * 2 * CH);
            ++w_issued;
            if (++ws == p.w_stages) {
              ws = 0;
              wph ^= 1u;
            }
          }
        }
      }
      if (!ok) {
        int s = ws;
        uint32_t ph = wph;
        for (long long i = 0; i < w_issued && i < p.w_stages; ++i) {
          if (--s < 0) {
            s = p.w_stages - 1;
            ph ^= 1u;
          }
          mbar_wait_drain(wfull0 + 8 * s, ph, p.timeout_ns);
        }
        for (long long i = (z_issued > 2 ? z_issued - 2 : 0); i < z_issued; ++i)
          mbar_wait_drain(zfull0 + 8 * (i & 1), static_cast<uint32_t>(i >> 1) & 1u, p.timeout_ns);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t idesc = idesc_f16_f32(CH, BM, 0, 0);
      // Descriptors of buffer / stage 0; a buffer, stage, slab or K step is a
      // plain add to the start address field (every address stays below 256 KB,
      // so the field cannot carry out).
      const uint64_t zdesc0 = sdesc_sw128(zbuf0, 16, 1024);
      const uint64_t wdesc0 = sdesc_sw128(wring, 16, 1024);
      int ws = 0, acc = 0;
      uint32_t wph = 0, aph = 0;
      bool ok = true;
      int n = 0;
      for (int tile = blockIdx.x; tile < total && ok; tile += gridDim.x, ++n) {
        const int zb = n & 1;
        const uint32_t zph = static_cast<uint32_t>(n >> 1) & 1u;
        if (!mbar_wait(zready0 + 8 * zb, zph, st, SITE_MMA)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint64_t zdesc = zdesc0 + ((zb * z_buf_bytes) >> 4);
        for (int qc = 0; qc < p.n_chunks && ok; ++qc) {
          if (!mbar_wait(tempty0 + 8 * acc, aph ^ 1u, st, SITE_MMA)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t d_val = tmem_base + acc * 256, d_gate = d_val + 128;
          for (int s = 0; s < p.k_slabs; ++s) {
            if (!mbar_wait(wfull0 + 8 * ws, wph, st, SITE_MMA)) {
              ok = false;
              break;
            }
            tc_fence_after();
            const uint64_t bd = zdesc + ((s * Z_SLAB) >> 4), ad = wdesc0 + ((ws * W_SLAB) >> 4);
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
              mma_f16_ss(d_val, ad + 2 * kk, bd + 2 * kk, idesc, (s | kk) != 0);
              mma_f16_ss(d_gate, ad + ((CH * 128) >> 4) + 2 * kk, bd + 2 * kk, idesc, (s | kk) != 0);
            }
            mma_commit(wempty0 + 8 * ws);
            if (++ws == p.w_stages) {
              ws = 0;
              wph ^= 1u;
            }
          }
          if (!ok) break;
          mma_commit(tfull0 + 8 * acc);
          if (++acc == 2) {
            acc = 0;
            aph ^= 1u;
          }
        }
        if (!ok) break;
        mma_commit(zempty0 + 8 * zb);
      }
      if (!ok) {
        mma_commit(drain);
        mbar_wait_drain(drain, 0, p.timeout_ns);
      }
    }
  } else if (warp < 6) {
    // ------------------------------------------------------------ LayerNorm (in place, fp16 out)
    const uint32_t r = threadIdx.x - 64;  // pair row of the tile
    const float inv_d = 1.0f / static_cast<float>(p.D);
    const int n8 = p.D >> 3;              // 8-element chunks per row
    int n = 0;
    for (int tile = blockIdx.x; tile < total; tile += gridDim.x, ++n) {
      const int zb = n & 1;
      const uint32_t zph = static_cast<uint32_t>(n >> 1) & 1u;
      if (!named_bar_and(1, 128, mbar_wait(zfull0 + 8 * zb, zph, st, SITE_XFORM))) break;
      uint8_t* const zrow = base_ptr + (zbuf0 - base) + zb * z_buf_bytes;
      // One pass for the statistics, shifted by the row's first element so
      // that a large common offset does not cancel in E[(v-K)^2] - E[v-K]^2.
      const float shift = bf16_lo(*reinterpret_cast<const uint32_t*>(zrow + sw128_offset(r, 0)));
      float s1[8], s2[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) s1[e] = s2[e] = 0.f;
      for (int c8 = 0; c8 < n8; ++c8) {
        const uint4 v = *reinterpret_cast<const uint4*>(zrow + (c8 >> 3) * Z_SLAB + sw128_offset(r, (c8 & 7) * 8));
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
      const float mu = shift + m1;
      const float rstd = rsqrtf(fmaxf(t2 * inv_d - m1 * m1, 0.f) + p.eps);
      if (p.zstats) {
        const int bb = tile / p.tiles_per_batch;
        const long long pidx = static_cast<long long>(tile - bb * p.tiles_per_batch) * BM + r;
        if (pidx < p.NN) p.zstats[bb * p.NN + pidx] = make_float2(mu, rstd);
      }
      for (int c8 = 0; c8 < n8; ++c8) {
        uint4* const ptr = reinterpret_cast<uint4*>(zrow + (c8 >> 3) * Z_SLAB + sw128_offset(r, (c8 & 7) * 8));
        const uint4 v = *ptr;
        const float4 g0 = __ldg(reinterpret_cast<const float4*>(p.gamma) + 2 * c8);
        const float4 g1 = __ldg(reinterpret_cast<const float4*>(p.gamma) + 2 * c8 + 1);
        const float4 b0 = __ldg(reinterpret_cast<const float4*>(p.beta) + 2 * c8);
        const float4 b1 = __ldg(reinterpret_cast<const float4*>(p.beta) + 2 * c8 + 1);
        uint4 o;
        o.x = pack_half2(fmaf((bf16_lo(v.x) - mu) * rstd, g0.x, b0.x), fmaf((bf16_hi(v.x) - mu) * rstd, g0.y, b0.y));
        o.y = pack_half2(fmaf((bf16_lo(v.y) - mu) * rstd, g0.z, b0.z), fmaf((bf16_hi(v.y) - mu) * rstd, g0.w, b0.w));
        o.z = pack_half2(fmaf((bf16_lo(v.z) - mu) * rstd, g1.x, b1.x), fmaf((bf16_hi(v.z) - mu) * rstd, g1.y, b1.y));
        o.w = pack_half2(fmaf((bf16_lo(v.w) - mu) * rstd, g1.z, b1.z), fmaf((bf16_hi(v.w) - mu) * rstd, g1.w, b1.w));
        *ptr = o;
      }
      fence_proxy_async_smem();
      mbar_arrive(zready0 + 8 * zb);
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;              // TMEM lane quadrant = channels q*32 .. q*32+31
    const int colhalf = (warp - 6) >> 2;  // pairs colhalf*64 .. +63 of the tile
    int acc = 0;
    uint32_t aph = 0;
    bool ok = true;
    for (int tile = blockIdx.x; tile < total && ok; tile += gridDim.x) {
      const int bb = tile / p.tiles_per_batch;
      const long long pair0 = static_cast<long long>(tile - bb * p.tiles_per_batch) * BM;
      // this warp's 64 mask values (128 bytes): pulled into L1 once per tile,
      // ahead of the accumulator wait, and read from there per chunk
      const long long mp0 = pair0 + colhalf * 64;
      const __nv_bfloat16* const mrow = (p.mask && mp0 < p.NN) ? p.mask + bb * p.NN + mp0 : nullptr;
      if (mrow) asm volatile("prefetch.global.L1 [%0];" ::"l"(mrow));
      for (int qc = 0; qc < p.n_chunks; ++qc) {
        if (!__all_sync(0xffffffffu, mbar_wait(tfull0 + 8 * acc, aph, st, SITE_EPI))) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t t_addr = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + acc * 256;
        // this lane's channel, the warp's 64 pairs: 8 chunks of 8 fp16
        uint4 R[8];
#pragma unroll
        for (int blk = 0; blk < 4; ++blk) {  // 16 pairs at a time keeps the register footprint small
          const int pcol = colhalf * 64 + blk * 16;
          uint32_t v[16], g[16];
          tmem_ld16(t_addr + pcol, v);
          tmem_ld16(t_addr + 128 + pcol, g);
          tmem_ld_wait();
#pragma unroll
          for (int u = 0; u < 2; ++u) {
            const bool m_in = mrow && mp0 + blk * 16 + u * 8 < p.NN;
            const uint4 m = m_in ? __ldg(reinterpret_cast<const uint4*>(mrow + blk * 16 + u * 8))
                                 : make_uint4(0x3F803F80u, 0x3F803F80u, 0x3F803F80u, 0x3F803F80u);
            const float mf[8] = {bf16_lo(m.x), bf16_hi(m.x), bf16_lo(m.y), bf16_hi(m.y),
                                 bf16_lo(m.z), bf16_hi(m.z), bf16_lo(m.w), bf16_hi(m.w)};
            float y[8];
#pragma unroll
            for (int e = 0; e < 8; ++e)
              y[e] = sigmoid_fast(__uint_as_float(g[u * 8 + e])) * __uint_as_float(v[u * 8 + e]) * mf[e];
            R[blk * 2 + u] = make_uint4(pack_half2(y[0], y[1]), pack_half2(y[2], y[3]), pack_half2(y[4], y[5]),
                                        pack_half2(y[6], y[7]));
          }
        }
        // the accumulator is in registers now: hand it back to the MMA warp
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(tempty0 + 8 * acc);
        if (++acc == 2) {
          acc = 0;
          aph ^= 1u;
        }
        // 8x8 transpose of 16-byte chunks inside each group of 8 lanes (three
        // butterfly rounds): afterwards lane 8a+b holds chunk b of channels
        // 8a+0 .. 8a+7, so each store instruction below writes four whole
        // 128-byte runs (one channel per group) instead of 32 scattered pieces.
        const uint32_t gb = lane & 7, ga = lane >> 3;
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
        const long long pp = pair0 + colhalf * 64 + gb * 8;
        if (pp < p.NN) {  // NN is a multiple of 8: a chunk is all in or all out
#pragma unroll
          for (int s8 = 0; s8 < 8; ++s8) {
            const int o = qc * CH + q * 32 + ga * 8 + s8;  // output channel (a: 0..C-1, b: C..2C-1)
            if (o < C2) {
              __half* const plane = o < p.C ? p.a + (static_cast<size_t>(bb) * p.C + o) * p.NN
                                            : p.b + (static_cast<size_t>(bb) * p.C + (o - p.C)) * p.NN;
              *reinterpret_cast<uint4*>(plane + pp) = R[s8];
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

cudaError_t launch_inproj(const InprojArgs& a, const CUtensorMap& tm_z, const CUtensorMap& tm_w, int grid,
                          cudaStream_t s) {
  if (a.w_stages < 1 || a.w_stages > MAX_W_STAGES) return cudaErrorInvalidValue;
  const size_t smem = inproj_smem_bytes(a.k_slabs, a.w_stages);
  cudaError_t e = cudaFuncSetAttribute(k1_inproj, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  k1_inproj<<<grid, THREADS, smem, s>>>(tm_z, tm_w, a);
  return cudaGetLastError();
}

}  // namespace trimul
