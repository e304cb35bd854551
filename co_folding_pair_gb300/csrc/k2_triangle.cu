// k2_triangle.cu -- the triangle contraction of TriMul as a per-channel batched GEMM.
//
// fold-cp-ops README, "Use": the layer takes direction = "outgoing" | "incoming".
// For each plane (batch b, channel c) with A = a[b, c] and B = b[b, c] (N x N):
//     outgoing  X = A B^T    (x[i,j] = sum_k a[i,k] b[j,k]; both operands K-major)
//     incoming  X = A^T B    (x[i,j] = sum_k a[k,i] b[k,j]; both operands MN-major)
// The incoming case reads the same planes; only the operand major-ness in the
// MMA descriptors and the TMA boxes change, so no transposed copy is made.
//
// With 8-bit operands (the opt-in e4m3 path, outgoing only) the same stage of
// 128 rows x 128 bytes holds 128 K elements, and the MMAs are
// tcgen05.mma.kind::f8f6f4 with K = 32: the same descriptors and the same four
// K steps per stage, twice the K per stage, half the K blocks.
//
// CTA pairs: a cluster of two CTAs computes one 256 x 256 tile of X with
// tcgen05.mma.cta_group::2 (M = 256, N = 256, K = 16).  Each CTA stages its own
// 128 rows of A and 128 rows (columns of X) of B, so each shared memory feeds
// the tensor cores half the B operand it would for a one-CTA 128 x 256 tile.
// The even CTA issues the MMAs; TMA completions of both CTAs are counted on
// its barriers, and its commits are multicast to both CTAs.
//
// Structure per CTA (one persistent CTA pair per two SMs, 192 threads each):
//   warp 0      TMA producer: 128 x 64 A and 128 x 64 B fp16 tiles, 6-stage ring
//   warp 1      TMEM (512 columns, allocated pairwise); in the even CTA, lane 0
//               issues the MMAs
//   warps 2..5  epilogue: TMEM -> registers -> fp16 x * 2^-s -> global x (the
//               power-of-two scale keeps the sum within binary16 range), or
//               bf16 x unscaled (the backward's triangle gradients: each
//               operand's major-ness is a launch argument, so dA = dX B
//               (K-major, MN-major), dB = dX^T A (MN, MN), and the incoming
//               dA = B dX^T (K, K), dB = A dX (K, MN) all run here)
// The fp32 accumulator is double-buffered in TMEM (2 x 256 columns).  Tiles
// are visited plane by plane, so the pairs work on the same plane at about
// the same time and each plane's operands are read from HBM about once.
#include "kernels.h"
#include "sm103_ptx.cuh"

namespace trimul {

namespace {
constexpr int BM = TRI_ROWS;  // rows of A per CTA (256 per pair)
constexpr int BN = TRI_ROWS;  // rows of B per CTA (256 columns of X per pair)
constexpr int BK = TRI_BK;
constexpr int STAGES = 6;
constexpr uint32_t A_BYTES = BM * BK * 2;  // 16 KB
constexpr uint32_t B_BYTES = BN * BK * 2;  // 16 KB
constexpr uint32_t STAGE_BYTES = A_BYTES + B_BYTES;
static_assert(STAGE_BYTES == TRI_STAGE_BYTES, "stage size must match the host's TMA boxes");
constexpr uint32_t BAR_BYTES = 256;
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t ACC_COLS = 256;
constexpr int THREADS = 192;
constexpr int TILE = 256;  // X tile edge per CTA pair
}  // namespace

size_t triangle_smem_bytes() { return 1024 + STAGES * STAGE_BYTES + BAR_BYTES; }

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(THREADS, 1)
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
  const uint32_t rank = cluster_ctarank();  // 0: issues the MMAs
  const bool leader = rank == 0;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(full0 + 8 * s, 1);   // leader only: one expect_tx arrival; bytes of both CTAs
      mbar_init(empty0 + 8 * s, 1);  // one multicast commit per phase
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(tfull0 + 8 * a, 1);  // one multicast commit per phase
      mbar_init(tempty0 + 8 * a, 8); // leader only: 4 epilogue warps of each CTA
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

  const int tiles_per_plane = p.tiles_m * p.tiles_n;
  const int total = p.tile_end;
  const int cluster = p.tile_begin + static_cast<int>(blockIdx.x >> 1), n_clusters = gridDim.x >> 1;

  if (warp == 0) {
    // ------------------------------------------------------------ producer (both CTAs)
    if (lane == 0 && !p.inject_stall) {
      tma_prefetch_desc(&tm_a);
      tma_prefetch_desc(&tm_b);
      int stage = 0;
      uint32_t phase = 0;
      long long issued = 0;
      bool ok = true;
      for (int tile = cluster; tile < total && ok; tile += n_clusters) {
        const int plane = tile / tiles_per_plane, rem = tile - plane * tiles_per_plane;
        const int tm = rem / p.tiles_n, tn = rem - tm * p.tiles_n;
        // A box that lies wholly outside the tensor may not complete its bytes:
        // such boxes (this CTA's half lies past N) load rows 0.. instead.  Those
        // rows only feed rows / columns of X at or past N, which are not stored.
        const int row_a = tm * TILE + rank * BM, row_b = tn * TILE + rank * BN;
        auto clamp = [&](int r) { return r < p.N ? r : 0; };
        const int bk = p.fp8 ? 2 * BK : BK;  // K elements per stage
        for (int kb = 0; kb < p.k_iters; ++kb) {
          if (!mbar_wait(empty0 + 8 * stage, phase ^ 1u, st, SITE_PRODUCER)) {
            ok = false;
            break;
          }
          const uint32_t sa = base + stage * STAGE_BYTES, sb = sa + A_BYTES;
          const uint32_t fb = mapa_shared(full0 + 8 * stage, 0);  // the leader's full barrier
          if (leader) mbar_arrive_expect_tx(full0 + 8 * stage, 2 * STAGE_BYTES);
          // K-major: one box of the CTA's rows x the stage's K; MN-major:
          // 64-wide runs of the rows, one per K row of the stage
          if (!p.a_mn) {
            tma_load_3d_pair(sa, &tm_a, fb, kb * bk, clamp(row_a), plane);
          } else {
            for (int h = 0; h < BM / 64; ++h)
              tma_load_3d_pair(sa + h * 8192, &tm_a, fb, clamp(row_a + h * 64), kb * BK, plane);
          }
          if (!p.b_mn) {
            tma_load_3d_pair(sb, &tm_b, fb, kb * bk, clamp(row_b), plane);
          } else {
            for (int h = 0; h < BN / 64; ++h)
              tma_load_3d_pair(sb + h * 8192, &tm_b, fb, clamp(row_b + h * 64), kb * BK, plane);
          }
          ++issued;
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      if (!ok && leader) {
        // let the copies already in flight (both CTAs' bytes count here) land before the pair goes away
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
      const uint32_t idesc = p.bf16 ? idesc_bf16_f32(2 * BM, 2 * BN, p.a_mn, p.b_mn)
                                    : idesc_f16_f32(2 * BM, 2 * BN, p.a_mn, p.b_mn);
      // Descriptors of stage 0 (K-major for outgoing, MN-major for incoming); a
      // stage or K step is a plain add to the start address field (every
      // address stays below 256 KB, so the field cannot carry out).
      const uint64_t adesc0 = p.a_mn ? sdesc_sw128(base, 8192, 1024) : sdesc_sw128(base, 16, 1024);
      const uint64_t bdesc0 = p.b_mn ? sdesc_sw128(base + A_BYTES, 8192, 1024) : sdesc_sw128(base + A_BYTES, 16, 1024);
      // one K step of 16, in descriptor units
      const uint32_t astep = p.a_mn ? 2048u >> 4 : 32u >> 4, bstep = p.b_mn ? 2048u >> 4 : 32u >> 4;
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
        for (int kb = 0; kb < p.k_iters; ++kb) {
          if (!mbar_wait(full0 + 8 * stage, phase, st, SITE_MMA)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t soff = (stage * STAGE_BYTES) >> 4;
          if (p.fp8) {
#pragma unroll
            for (int kk = 0; kk < BK / 16; ++kk)
              mma_f8_ss_pair(d_tmem, adesc0 + soff + kk * astep, bdesc0 + soff + kk * bstep, idesc, (kb | kk) != 0);
          } else {
#pragma unroll
            for (int kk = 0; kk < BK / 16; ++kk)
              mma_f16_ss_pair(d_tmem, adesc0 + soff + kk * astep, bdesc0 + soff + kk * bstep, idesc, (kb | kk) != 0);
          }
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
    const int q = warp & 3;  // TMEM lane quadrant this warp may access
    // x is stored as fp16 x * xs: the caller's power of two, or one from this
    // call's max |a|, |b| (written by the input projection before this launch)
    float xs = p.ab_max ? exp2_neg(x_scale_log2_from_max(__uint_as_float(*p.ab_max), p.N)) : p.x_scale;
    if (p.fp8) xs *= p.fp8_descale;
    const bool out_bf16 = p.out_bf16 != 0;  // bf16 x, unscaled
    auto pack = [&](uint32_t lo, uint32_t hi) {
      return out_bf16 ? pack_bf162(__uint_as_float(lo), __uint_as_float(hi))
                      : pack_half2(xs * __uint_as_float(lo), xs * __uint_as_float(hi));
    };
    int acc = 0;
    uint32_t aphase = 0;
    for (int tile = cluster; tile < total; tile += n_clusters) {
      const bool ok = __all_sync(0xffffffffu, mbar_wait(tfull0 + 8 * acc, aphase, st, SITE_EPI));
      if (!ok) break;
      tc_fence_after();
      const int plane = tile / tiles_per_plane, rem = tile - plane * tiles_per_plane;
      const int tm = rem / p.tiles_n, tn = rem - tm * p.tiles_n;
      // Lane r holds row q*32+r of this CTA's half.  Per block of 64 columns it
      // packs 8 chunks of 8 bf16; an 8x8 transpose of chunks inside each group of
      // 8 lanes (three butterfly rounds) then leaves lane 8a+b with chunk b of
      // rows 8a..8a+7, so each store instruction writes four whole 128-byte row
      // segments instead of 32 scattered 16-byte pieces.
      const uint32_t gb = lane & 7, ga = lane >> 3;
      const int row0 = tm * TILE + rank * BM + q * 32 + static_cast<int>(ga) * 8;
      const uint32_t t_addr = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + acc * ACC_COLS;
#pragma unroll 1
      for (int c0 = 0; c0 < TILE; c0 += 64) {
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
        const int col = tn * TILE + c0 + static_cast<int>(gb) * 8;
        if (col < p.N) {  // N is a multiple of 8: a chunk is all in or all out
#pragma unroll
          for (int s8 = 0; s8 < 8; ++s8) {
            const int row = row0 + s8;
            if (row < p.N) *reinterpret_cast<uint4*>(p.x + (static_cast<size_t>(plane) * p.N + row) * p.N + col) = R[s8];
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_remote(mapa_shared(tempty0 + 8 * acc, 0));  // the leader's barrier
      if (++acc == 2) {
        acc = 0;
        aphase ^= 1u;
      }
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

cudaError_t launch_triangle(const TriangleArgs& a, const CUtensorMap& tm_a, const CUtensorMap& tm_b, int grid,
                            cudaStream_t s) {
  const size_t smem = triangle_smem_bytes();
  cudaError_t e = cudaFuncSetAttribute(k2_triangle, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  grid &= ~1;  // whole CTA pairs
  if (grid < 2) grid = 2;
  k2_triangle<<<grid, THREADS, smem, s>>>(tm_a, tm_b, a);
  return cudaGetLastError();
}

int triangle_max_pairs(int num_sms) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(num_sms & ~1, 1, 1);
  cfg.blockDim = dim3(THREADS, 1, 1);
  cfg.dynamicSmemBytes = triangle_smem_bytes();
  cudaLaunchAttribute attr;
  attr.id = cudaLaunchAttributeClusterDimension;
  attr.val.clusterDim.x = 2;
  attr.val.clusterDim.y = 1;
  attr.val.clusterDim.z = 1;
  cfg.attrs = &attr;
  cfg.numAttrs = 1;
  cudaFuncSetAttribute(k2_triangle, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(cfg.dynamicSmemBytes));
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, k2_triangle, &cfg) != cudaSuccess || n < 1) {
    cudaGetLastError();
    return num_sms / 2;
  }
  return n;
}

}  // namespace trimul
