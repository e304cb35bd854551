// k2_triangle.cu -- the triangle contraction of TriMul as a per-channel batched GEMM.
//
// fold-cp-ops README, "Use": the layer takes direction = "outgoing" | "incoming".
// For each plane (batch b, channel c) with A = a[b, c] and B = b[b, c] (N x N):
//     outgoing  X = A B^T    (x[i,j] = sum_k a[i,k] b[j,k]; both operands K-major)
//     incoming  X = A^T B    (x[i,j] = sum_k a[k,i] b[k,j]; both operands MN-major)
// The incoming case reads the same planes; only the operand major-ness in the
// MMA descriptors and the TMA boxes change, so no transposed copy is made.
//
// Structure (one persistent CTA per SM, 192 threads):
//   warp 0      TMA producer: 128x64 A and 256x64 B fp16 tiles into a 4-stage ring
//   warp 1      allocates 512 TMEM columns, issues tcgen05.mma (M=128, N=256, K=16)
//   warps 2..5  epilogue: TMEM -> registers -> bf16 -> global x, one row per thread
// The fp32 accumulator is double-buffered in TMEM (2 x 256 columns) so the
// epilogue of one tile overlaps the main loop of the next.  Tiles are visited
// plane by plane, so every CTA works on the same plane at about the same time
// and each plane's operands (2 x N^2 x 2 bytes) are read from HBM about once.
#include "kernels.h"
#include "sm103_ptx.cuh"

namespace trimul {

namespace {
constexpr int BM = 128, BN = 256, BK = 64, STAGES = 4;
constexpr uint32_t A_BYTES = BM * BK * 2;  // 16 KB
constexpr uint32_t B_BYTES = BN * BK * 2;  // 32 KB
constexpr uint32_t STAGE_BYTES = A_BYTES + B_BYTES;
constexpr uint32_t BAR_BYTES = 256;
constexpr uint32_t TMEM_COLS = 512;
constexpr int THREADS = 192;
}  // namespace

size_t triangle_smem_bytes() { return 1024 + STAGES * STAGE_BYTES + BAR_BYTES; }

__global__ void __launch_bounds__(THREADS, 1)
    k2_triangle(const __grid_constant__ CUtensorMap tm_a, const __grid_constant__ CUtensorMap tm_b,
                const TriangleArgs p) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_addr(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* const base_ptr = smem_raw + (base - raw);
  const uint32_t bars = base + STAGES * STAGE_BYTES;
  // barrier slots: full[STAGES] empty[STAGES] tfull[2] tempty[2] drain, then the TMEM base word
  const uint32_t full0 = bars, empty0 = bars + 8 * STAGES, tfull0 = bars + 16 * STAGES;
  const uint32_t tempty0 = tfull0 + 16, drain = tempty0 + 16;
  const uint32_t tmem_slot = drain + 8;
  volatile uint32_t* tmem_slot_ptr = reinterpret_cast<volatile uint32_t*>(base_ptr + (tmem_slot - base));

  const KStatus st{p.status, p.timeout_ns};
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(full0 + 8 * s, 1);
      mbar_init(empty0 + 8 * s, 1);
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

  const int tiles_per_plane = p.tiles_m * p.tiles_n;
  const int total = p.planes * tiles_per_plane;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0 && !p.inject_stall) {
      tma_prefetch_desc(&tm_a);
      tma_prefetch_desc(&tm_b);
      int stage = 0;
      uint32_t phase = 0;
      long long issued = 0;
      bool ok = true;
      for (int tile = blockIdx.x; tile < total && ok; tile += gridDim.x) {
        const int plane = tile / tiles_per_plane, rem = tile - plane * tiles_per_plane;
        const int tm = rem / p.tiles_n, tn = rem - tm * p.tiles_n;
        for (int kb = 0; kb < p.k_iters; ++kb) {
          if (!mbar_wait(empty0 + 8 * stage, phase ^ 1u, st, SITE_PRODUCER)) {
            ok = false;
            break;
          }
          const uint32_t sa = base + stage * STAGE_BYTES, sb = sa + A_BYTES, fb = full0 + 8 * stage;
          mbar_arrive_expect_tx(fb, STAGE_BYTES);
          if (!p.incoming) {
            tma_load_3d(sa, &tm_a, fb, kb * BK, tm * BM, plane);
            tma_load_3d(sb, &tm_b, fb, kb * BK, tn * BN, plane);
          } else {
            // MN-major: 64-wide runs of i (resp. j), one per k row of the stage
            for (int h = 0; h < BM / 64; ++h) tma_load_3d(sa + h * 8192, &tm_a, fb, tm * BM + h * 64, kb * BK, plane);
            for (int h = 0; h < BN / 64; ++h) tma_load_3d(sb + h * 8192, &tm_b, fb, tn * BN + h * 64, kb * BK, plane);
          }
          ++issued;
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      if (!ok) {
        // let the copies already in flight land before the CTA goes away
        int s = stage;
        uint32_t ph = phase;
        for (long long i = 0; i < issued && i < STAGES; ++i) {
          if (--s < 0) {
            s = STAGES - 1;
            ph ^= 1u;
          }
          mbar_wait_drain(full0 + 8 * s, ph, p.timeout_ns);
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t idesc = idesc_f16_f32(BM, BN, p.incoming, p.incoming);
      int stage = 0, acc = 0;
      uint32_t phase = 0, aphase = 0;
      bool ok = true;
      for (int tile = blockIdx.x; tile < total && ok; tile += gridDim.x) {
        if (!mbar_wait(tempty0 + 8 * acc, aphase ^ 1u, st, SITE_MMA)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + acc * BN;
        for (int kb = 0; kb < p.k_iters; ++kb) {
          if (!mbar_wait(full0 + 8 * stage, phase, st, SITE_MMA)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sa = base + stage * STAGE_BYTES, sb = sa + A_BYTES;
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk) {
            uint64_t ad, bd;
            if (!p.incoming) {
              ad = sdesc_sw128(sa + kk * 32, 16, 1024);
              bd = sdesc_sw128(sb + kk * 32, 16, 1024);
            } else {
              ad = sdesc_sw128(sa + kk * 2048, 8192, 1024);
              bd = sdesc_sw128(sb + kk * 2048, 8192, 1024);
            }
            mma_f16_ss(d_tmem, ad, bd, idesc, (kb | kk) != 0);
          }
          mma_commit(empty0 + 8 * stage);
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        mma_commit(tfull0 + 8 * acc);
        if (++acc == 2) {
          acc = 0;
          aphase ^= 1u;
        }
      }
      if (!ok) {
        mma_commit(drain);
        mbar_wait_drain(drain, 0, p.timeout_ns);
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;  // TMEM lane quadrant this warp may access
    int acc = 0;
    uint32_t aphase = 0;
    for (int tile = blockIdx.x; tile < total; tile += gridDim.x) {
      const bool ok = __all_sync(0xffffffffu, mbar_wait(tfull0 + 8 * acc, aphase, st, SITE_EPI));
      if (!ok) break;
      tc_fence_after();
      const int plane = tile / tiles_per_plane, rem = tile - plane * tiles_per_plane;
      const int tm = rem / p.tiles_n, tn = rem - tm * p.tiles_n;
      const int row = tm * BM + q * 32 + lane;
      const bool row_ok = row < p.N;
      __nv_bfloat16* xrow = p.x + (static_cast<size_t>(plane) * p.N + (row_ok ? row : 0)) * p.N + tn * BN;
      const uint32_t t_addr = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + acc * BN;
#pragma unroll 1
      for (int c0 = 0; c0 < BN; c0 += 32) {
        uint32_t r[32];
        tmem_ld32(t_addr + c0, r);
        tmem_ld_wait();
        if (row_ok) {
#pragma unroll
          for (int v = 0; v < 4; ++v) {
            if (tn * BN + c0 + v * 8 < p.N) {
              uint4 pk;
              pk.x = pack_bf162(__uint_as_float(r[v * 8 + 0]), __uint_as_float(r[v * 8 + 1]));
              pk.y = pack_bf162(__uint_as_float(r[v * 8 + 2]), __uint_as_float(r[v * 8 + 3]));
              pk.z = pack_bf162(__uint_as_float(r[v * 8 + 4]), __uint_as_float(r[v * 8 + 5]));
              pk.w = pack_bf162(__uint_as_float(r[v * 8 + 6]), __uint_as_float(r[v * 8 + 7]));
              *reinterpret_cast<uint4*>(xrow + c0 + v * 8) = pk;
            }
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(tempty0 + 8 * acc);
      if (++acc == 2) {
        acc = 0;
        aphase ^= 1u;
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

cudaError_t launch_triangle(const TriangleArgs& a, const CUtensorMap& tm_a, const CUtensorMap& tm_b, int grid,
                            cudaStream_t s) {
  static bool attr_set = false;
  const size_t smem = triangle_smem_bytes();
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(k2_triangle, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  k2_triangle<<<grid, THREADS, smem, s>>>(tm_a, tm_b, a);
  return cudaGetLastError();
}

}  // namespace trimul
