// k4_gemm.cu -- batched / split-K tcgen05 GEMM for the TriMul backward pass.
//
// C[z] = sum_k A(m, k) B(n, k) per z slice, with fp32 accumulation in TMEM.
// Each operand is a bf16 or fp16 matrix (both the same type), K-major
// ([rows][K], K contiguous) or MN-major ([K][rows], rows contiguous), either
// one matrix per batch (a 3-D tensor map over batches) or one matrix shared by
// every batch (a weight, 2-D map).  The K loop runs over "global" K blocks of
// 64: block g is block g % kpb of batch g / kpb, so a z slice is either one
// batch (a batched GEMM: the per-pair projections) or a range of blocks that
// spans batches (split-K: the weight gradients, sums over every pair of every
// batch element, each slice writing fp32 partials).
//
// The projections and weight gradients mix weights with pair-major or
// channel-major planes, so both operand majors occur.  (The triangle
// gradients, per-channel N x N products, run on the triangle kernel.)
//
// Tiles are visited slice by slice, and within a slice with the N tile
// fastest (consecutive pairs share A's panel) or, for a GEMM with a few M
// tiles and many N tiles, the M tile fastest (consecutive pairs share B's
// panel, which is then read from DRAM once).
//
// Tile and pipeline as in the triangle kernel: a CTA pair computes one
// 256 x 256 tile with tcgen05.mma.cta_group::2 (M = 256, N = 256, K = 16); each
// CTA stages its own 128 rows of A and of B per K block through a 6-stage TMA
// ring; the fp32 accumulator is double-buffered in TMEM (2 x 256 columns), so
// a tile's epilogue overlaps the next tile's MMAs.  Rows of a box that lie
// past M or N are filled with zeros by the tensor-memory-access engine (a box
// wholly past them loads row 0, whose products are never stored), and the
// epilogue stores only rows < M and columns < N.
//
// Epilogue (16 warps per CTA: warp (cb, q) takes TMEM quadrant q, i.e. 32 of
// the CTA's 128 rows, and the 64-column block cb; lane = one row): TMEM ->
// registers -> packed chunks of 16 bytes, an 8 x 8 transpose of chunks inside
// each group of 8 lanes, then stores of whole 128-byte row segments: bf16
// (GEMM_OUT_BF16), fp16 (GEMM_OUT_F16), fp32 (GEMM_OUT_F32) or fp32 added to
// what C holds (GEMM_OUT_F32_ADD).  A GEMM with a short K (the per-pair projections, K of
// 256) gives each tile's epilogue about a microsecond; one warp per quadrant
// and column block keeps enough TMEM loads and stores in flight for that,
// where four warps walking all columns could not (a TMEM load barely overlaps
// the arithmetic of its own warp).
#include "kernels.h"
#include "sm103_ptx.cuh"

namespace trimul {

namespace {
constexpr int ROWS = 128;  // rows of A (and of B) per CTA
constexpr int BK = 64;
constexpr int STAGES = 6;
constexpr uint32_t A_BYTES = ROWS * BK * 2;  // 16 KB
constexpr uint32_t B_BYTES = ROWS * BK * 2;  // 16 KB
constexpr uint32_t STAGE_BYTES = A_BYTES + B_BYTES;
constexpr uint32_t BAR_BYTES = 256;
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t ACC_COLS = 256;
constexpr int EPI_WARPS = 16;  // four per TMEM lane quadrant
constexpr int THREADS = 64 + 32 * EPI_WARPS;
constexpr int TILE = 256;

size_t gemm_smem_bytes() { return 1024 + STAGES * STAGE_BYTES + BAR_BYTES; }

// Transpose 8 x 8 chunks of 16 bytes inside each group of 8 lanes: lane 8a+b
// holds chunks R[0..7] of its row; afterwards it holds chunk b of rows
// 8a..8a+7 (three butterfly rounds).
__device__ __forceinline__ void transpose8(uint4 (&R)[8], uint32_t gb) {
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
}
}  // namespace

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(THREADS, 1)
    k4_gemm(const __grid_constant__ CUtensorMap tm_a, const __grid_constant__ CUtensorMap tm_b, const GemmArgs p) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_addr(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* const base_ptr = smem_raw + (base - raw);
  const uint32_t bars = base + STAGES * STAGE_BYTES;
  const uint32_t full0 = bars, empty0 = bars + 8 * STAGES, tfull0 = bars + 16 * STAGES;
  const uint32_t tempty0 = tfull0 + 16, drain = tempty0 + 16;
  const uint32_t tmem_slot = drain + 8;
  volatile uint32_t* tmem_slot_ptr = reinterpret_cast<volatile uint32_t*>(base_ptr + (tmem_slot - base));

  const KStatus st{p.status, p.timeout_ns};
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();  // 0: issues the MMAs
  const bool leader = rank == 0;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(full0 + 8 * s, 1);   // leader only: one expect_tx arrival; bytes of both CTAs
      mbar_init(empty0 + 8 * s, 1);  // one multicast commit per phase
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(tfull0 + 8 * a, 1);   // one multicast commit per phase
      mbar_init(tempty0 + 8 * a, 2 * EPI_WARPS);  // leader only: every epilogue warp of each CTA
    }
    mbar_init(drain, 1);
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc_pair(tmem_slot, TMEM_COLS);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  cluster_sync_all();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot_ptr;

  const int tiles_per_z = p.tiles_m * p.tiles_n;
  const int total = p.tile_end;
  const int cluster = p.tile_begin + static_cast<int>(blockIdx.x >> 1), n_clusters = gridDim.x >> 1;
  const long long kb_total = static_cast<long long>(p.batches) * p.kpb;
  // the global K blocks of slice z
  auto k_range = [&](int z, long long* g0, long long* g1) {
    *g0 = static_cast<long long>(z) * p.kb_per_z;
    *g1 = min(*g0 + p.kb_per_z, kb_total);
  };

  if (warp == 0) {
    // ------------------------------------------------------------ producer (both CTAs)
    if (lane == 0) {
      tma_prefetch_desc(&tm_a);
      tma_prefetch_desc(&tm_b);
      int stage = 0;
      uint32_t phase = 0;
      long long issued = 0;
      bool ok = true;
      for (int tile = cluster; tile < total && ok; tile += n_clusters) {
        const int z = tile / tiles_per_z, rem = tile - z * tiles_per_z;
        const int tm = p.m_fastest ? rem % p.tiles_m : rem / p.tiles_n;
        const int tn = p.m_fastest ? rem / p.tiles_m : rem % p.tiles_n;
        // a box wholly past M (N) may not complete its bytes: it loads row 0
        // instead, whose products land only in rows / columns that are not stored
        const int ra = tm * TILE + static_cast<int>(rank) * ROWS, rb = tn * TILE + static_cast<int>(rank) * ROWS;
        long long g0, g1;
        k_range(z, &g0, &g1);
        for (long long g = g0; g < g1; ++g) {
          if (!mbar_wait(empty0 + 8 * stage, phase ^ 1u, st, SITE_PRODUCER)) {
            ok = false;
            break;
          }
          const int batch = static_cast<int>(g / p.kpb), k0 = static_cast<int>(g - static_cast<long long>(batch) * p.kpb) * BK;
          const uint32_t sa = base + stage * STAGE_BYTES, sb = sa + A_BYTES;
          const uint32_t fb = mapa_shared(full0 + 8 * stage, 0);
          if (leader) mbar_arrive_expect_tx(full0 + 8 * stage, 2 * STAGE_BYTES);
          if (!p.a_mn) {
            const int r = ra < p.M ? ra : 0;
            if (p.a_batched) tma_load_3d_pair(sa, &tm_a, fb, k0, r, batch);
            else tma_load_2d_pair(sa, &tm_a, fb, k0, r);
          } else {
            for (int h = 0; h < ROWS / 64; ++h) {
              const int r = ra + h * 64 < p.M ? ra + h * 64 : 0;
              if (p.a_batched) tma_load_3d_pair(sa + h * 8192, &tm_a, fb, r, k0, batch);
              else tma_load_2d_pair(sa + h * 8192, &tm_a, fb, r, k0);
            }
          }
          if (!p.b_mn) {
            const int r = rb < p.N ? rb : 0;
            if (p.b_batched) tma_load_3d_pair(sb, &tm_b, fb, k0, r, batch);
            else tma_load_2d_pair(sb, &tm_b, fb, k0, r);
          } else {
            for (int h = 0; h < ROWS / 64; ++h) {
              const int r = rb + h * 64 < p.N ? rb + h * 64 : 0;
              if (p.b_batched) tma_load_3d_pair(sb + h * 8192, &tm_b, fb, r, k0, batch);
              else tma_load_2d_pair(sb + h * 8192, &tm_b, fb, r, k0);
            }
          }
          ++issued;
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      if (!ok && leader) {
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
    // ------------------------------------------------------------ MMA issuer (even CTA)
    if (lane == 0 && leader) {
      const uint32_t idesc = p.bf16 ? idesc_bf16_f32(2 * ROWS, 2 * ROWS, p.a_mn, p.b_mn)
                                    : idesc_f16_f32(2 * ROWS, 2 * ROWS, p.a_mn, p.b_mn);
      const uint64_t adesc0 = p.a_mn ? sdesc_sw128(base, 8192, 1024) : sdesc_sw128(base, 16, 1024);
      const uint64_t bdesc0 = p.b_mn ? sdesc_sw128(base + A_BYTES, 8192, 1024) : sdesc_sw128(base + A_BYTES, 16, 1024);
      const uint32_t astep = p.a_mn ? 2048u >> 4 : 32u >> 4;  // one K step of 16, in descriptor units
      const uint32_t bstep = p.b_mn ? 2048u >> 4 : 32u >> 4;
      int stage = 0, acc = 0;
      uint32_t phase = 0, aphase = 0;
      bool ok = true;
      for (int tile = cluster; tile < total && ok; tile += n_clusters) {
        if (!mbar_wait(tempty0 + 8 * acc, aphase ^ 1u, st, SITE_MMA)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + acc * ACC_COLS;
        const int z = tile / tiles_per_z;
        long long g0, g1;
        k_range(z, &g0, &g1);
        for (long long g = g0; g < g1; ++g) {
          if (!mbar_wait(full0 + 8 * stage, phase, st, SITE_MMA)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t soff = (stage * STAGE_BYTES) >> 4;
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk)
            mma_f16_ss_pair(d_tmem, adesc0 + soff + kk * astep, bdesc0 + soff + kk * bstep, idesc,
                            (g != g0 || kk != 0) ? 1u : 0u);
          mma_commit_pair(empty0 + 8 * stage, 0x3);
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        mma_commit_pair(tfull0 + 8 * acc, 0x3);
        if (++acc == 2) {
          acc = 0;
          aphase ^= 1u;
        }
      }
      if (!ok) {
        mma_commit_pair(drain, 0x1);
        mbar_wait_drain(drain, 0, p.timeout_ns);
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue (both CTAs)
    const int q = warp & 3;  // TMEM lane quadrant of this warp
    const int cb = (warp - 2) >> 2;  // first 64-column block of this warp
    const uint32_t gb = lane & 7, ga = lane >> 3;
    int acc = 0;
    uint32_t aphase = 0;
    for (int tile = cluster; tile < total; tile += n_clusters) {
      const bool ok = __all_sync(0xffffffffu, mbar_wait(tfull0 + 8 * acc, aphase, st, SITE_EPI));
      if (!ok) break;
      tc_fence_after();
      const int z = tile / tiles_per_z, rem = tile - z * tiles_per_z;
      const int tm = p.m_fastest ? rem % p.tiles_m : rem / p.tiles_n;
      const int tn = p.m_fastest ? rem / p.tiles_m : rem % p.tiles_n;
      const int row0 = tm * TILE + static_cast<int>(rank) * ROWS + q * 32 + static_cast<int>(ga) * 8;
      const uint32_t t_addr = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + acc * ACC_COLS;
      const bool half_out = p.out_mode == GEMM_OUT_BF16 || p.out_mode == GEMM_OUT_F16;
      char* const cz = static_cast<char*>(p.c) + static_cast<size_t>(z) * p.c_zstride * (half_out ? 2 : 4);
      static_assert(EPI_WARPS == 16, "one 64-column block per epilogue warp");
      {
        const int c0 = cb * 64;
        if (half_out) {
          const bool f16 = p.out_mode == GEMM_OUT_F16;
          auto pack = [f16](uint32_t lo, uint32_t hi) {
            return f16 ? pack_half2(__uint_as_float(lo), __uint_as_float(hi))
                       : pack_bf162(__uint_as_float(lo), __uint_as_float(hi));
          };
          uint4 R[8];
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            uint32_t r[32];
            tmem_ld32(t_addr + c0 + h * 32, r);
            tmem_ld_wait();
#pragma unroll
            for (int v = 0; v < 4; ++v)
              R[h * 4 + v] = make_uint4(pack(r[v * 8 + 0], r[v * 8 + 1]), pack(r[v * 8 + 2], r[v * 8 + 3]),
                                        pack(r[v * 8 + 4], r[v * 8 + 5]), pack(r[v * 8 + 6], r[v * 8 + 7]));
          }
          transpose8(R, gb);
          const int col = tn * TILE + c0 + static_cast<int>(gb) * 8;
          if (col < p.N) {  // N is a multiple of 8: a chunk is all in or all out
#pragma unroll
            for (int s8 = 0; s8 < 8; ++s8) {
              const int row = row0 + s8;
              if (row < p.M)
                *reinterpret_cast<uint4*>(cz + (static_cast<size_t>(row) * p.ldc + col) * 2) = R[s8];
            }
          }
        } else {
#pragma unroll
          for (int h = 0; h < 2; ++h) {  // 32 columns: 8 chunks of 4 fp32
            uint32_t r[32];
            tmem_ld32(t_addr + c0 + h * 32, r);
            tmem_ld_wait();
            uint4 R[8];
#pragma unroll
            for (int v = 0; v < 8; ++v) R[v] = make_uint4(r[v * 4 + 0], r[v * 4 + 1], r[v * 4 + 2], r[v * 4 + 3]);
            transpose8(R, gb);
            const int col = tn * TILE + c0 + h * 32 + static_cast<int>(gb) * 4;
            if (col < p.N) {  // N is a multiple of 8, so of 4
#pragma unroll
              for (int s8 = 0; s8 < 8; ++s8) {
                const int row = row0 + s8;
                if (row < p.M) {
                  float4* const dst = reinterpret_cast<float4*>(cz + (static_cast<size_t>(row) * p.ldc + col) * 4);
                  float4 v = make_float4(__uint_as_float(R[s8].x), __uint_as_float(R[s8].y),
                                         __uint_as_float(R[s8].z), __uint_as_float(R[s8].w));
                  if (p.out_mode == GEMM_OUT_F32_ADD) {
                    const float4 o = *dst;
                    v.x += o.x;
                    v.y += o.y;
                    v.z += o.z;
                    v.w += o.w;
                  }
                  *dst = v;
                }
              }
            }
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_remote(mapa_shared(tempty0 + 8 * acc, 0));
      if (++acc == 2) {
        acc = 0;
        aphase ^= 1u;
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  cluster_sync_all();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem_base, TMEM_COLS);
  }
}

size_t gemm_smem_size() { return gemm_smem_bytes(); }

cudaError_t launch_gemm(const GemmArgs& a, const CUtensorMap& tm_a, const CUtensorMap& tm_b, int grid,
                        cudaStream_t s) {
  const size_t smem = gemm_smem_bytes();
  cudaError_t e = cudaFuncSetAttribute(k4_gemm, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  grid &= ~1;
  if (grid < 2) grid = 2;
  k4_gemm<<<grid, THREADS, smem, s>>>(tm_a, tm_b, a);
  return cudaGetLastError();
}

int gemm_max_pairs(int num_sms) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(num_sms & ~1, 1, 1);
  cfg.blockDim = dim3(THREADS, 1, 1);
  cfg.dynamicSmemBytes = gemm_smem_bytes();
  cudaLaunchAttribute attr;
  attr.id = cudaLaunchAttributeClusterDimension;
  attr.val.clusterDim.x = 2;
  attr.val.clusterDim.y = 1;
  attr.val.clusterDim.z = 1;
  cfg.attrs = &attr;
  cfg.numAttrs = 1;
  cudaFuncSetAttribute(k4_gemm, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(cfg.dynamicSmemBytes));
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, k4_gemm, &cfg) != cudaSuccess || n < 1) {
    cudaGetLastError();
    return num_sms / 2;
  }
  return n;
}

}  // namespace trimul
