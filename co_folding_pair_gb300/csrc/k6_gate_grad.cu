// k6_gate_grad.cu -- backward of the gated input projections, fused with the
// recomputation of their pre-activations.
//
// fold-cp-ops README, "Use": a = sigmoid(z' W_ga^T) * (z' W_a^T) * m and the
// same for b.  With the pre-activations v = z' W_a^T, g = z' W_ga^T of a
// channel and the incoming gradient da of a, the chain rule gives
//     dv = da m sigmoid(g),    dg = da m v sigmoid(g) (1 - sigmoid(g)),
// i.e. with t = tanh(g/2):  dv = (da m / 2)(1 + t),  dg = (da m / 2)(v/2)(1 + t)(1 - t).
// The kernel writes dv and dg (bf16) into the rows of dP [B][4C][P]
// (a values, a gates, b values, b gates; C rows each) that the projections'
// weight and input gradients read, so the pre-activations never reach HBM.
//
// Pipeline as in the input projection (k1_inproj.cu): a CTA pair takes 256
// pairs, each CTA loads its 128 rows of the normalised z (zh, bf16, already
// in memory for the other backward GEMMs, so there is no LayerNorm here) and
// 128 weight rows of each chunk of 128 channels (bf16 W~ = W diag(gamma_in)/2,
// value and gate rows interleaved in groups of 16, the same order as the
// forward's fp16 weights); the even CTA issues tcgen05.mma.cta_group::2
// (M = 256, N = 256, K = 16) and 16 epilogue warps read the accumulators with
// tcgen05.ld.16x256b, which gives each thread the value and the gate of one
// channel for the same pairs.
//
// Epilogue, warp (hc, q) = TMEM quadrant q (16 channels), pairs hc*64 ..
// hc*64+63: per chunk and lane group g (8 channels, all of a or all of b) it
// stages dv and dg as two 8-row x 64-pair boxes and stores them.  The
// row sums of dv and dg over pairs (for the bias part of the weight
// gradients) are summed per thread over its pairs (in fp32, before the values
// are rounded for storing), reduced over the 4 threads
// of a channel and written per tile to `rowpart` (32 floats per warp and
// chunk); k6_rowsum_* reduce them in a fixed order, so the gradients are
// deterministic.
#include "kernels.h"
#include "sm103_ptx.cuh"

namespace trimul {

namespace {
constexpr int TP = INPROJ_TILE_PAIRS;       // pairs per tile (per CTA pair)
constexpr int HALF = INPROJ_HALF_PAIRS;     // pairs per CTA
constexpr int CH = 64;                      // output channels per CTA per chunk (128 weight rows)
constexpr uint32_t Z_SLAB = HALF * 128;     // 16 KB: 128 pair rows x 64 K
constexpr uint32_t W_SLAB = 2 * CH * 128;   // 16 KB: 128 weight rows x 64 K
constexpr uint32_t STAGE_OUT = 16 * 128;    // per epilogue warp: one box of 16 rows x 64 pairs
constexpr uint32_t MASK_SLOT = TP * 2;      // one tile's mask values (fp16)
constexpr uint32_t BAR_BYTES = 512;
constexpr uint32_t TMEM_COLS = 512;
constexpr int EPI_WARPS = 16;               // four per TMEM quadrant, 64 pairs each
constexpr int THREADS = 96 + 32 * EPI_WARPS;
constexpr int MAX_W_STAGES = INPROJ_MAX_W_STAGES;
constexpr int MAX_Z_BUFS = INPROJ_MAX_Z_BUFS;
static_assert(16 * MAX_Z_BUFS + 16 * MAX_W_STAGES + 48 <= BAR_BYTES, "barrier block too small");

struct Layout {
  uint32_t z, w, stage, mask, bars, total;
};

__host__ __device__ inline Layout layout(int k_slabs, int w_stages, int z_bufs) {
  Layout L;
  uint32_t o = 0;
  L.z = o;
  o += z_bufs * k_slabs * Z_SLAB;
  L.w = o;
  o += w_stages * W_SLAB;
  L.stage = o;
  o += EPI_WARPS * STAGE_OUT;
  L.mask = o;
  o += 2 * MASK_SLOT;
  L.bars = o;
  o += BAR_BYTES;
  L.total = o + 1024;
  return L;
}
}  // namespace

size_t gategrad_smem_bytes(int k_slabs, int w_stages, int z_bufs) { return layout(k_slabs, w_stages, z_bufs).total; }

// Bring the 128-byte line holding p into L2 (no register, no wait).
__device__ __forceinline__ void prefetch_l2(const void* p) {
  asm volatile("prefetch.global.L2 [%0];" ::"l"(p) : "memory");
}

template <bool kResident>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(THREADS, 1)
    k6_gate_grad(const __grid_constant__ CUtensorMap tm_z, const __grid_constant__ CUtensorMap tm_w,
                 const __grid_constant__ CUtensorMap tm_p8, const GateGradArgs p) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_addr(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* const base_ptr = smem_raw + (base - raw);
  const Layout L = layout(p.k_slabs, p.w_stages, p.z_bufs);
  const uint32_t z_buf_bytes = p.k_slabs * Z_SLAB;
  const uint32_t zbuf0 = base + L.z, wring = base + L.w, bars = base + L.bars;
  const uint32_t zfull0 = bars, zempty0 = zfull0 + 8 * MAX_Z_BUFS;
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
      mbar_init(zfull0 + 8 * i, 1);   // leader only: one expect_tx arrival; bytes of both CTAs
      mbar_init(zempty0 + 8 * i, 1);  // one multicast commit per phase
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(tfull0 + 8 * i, 1);   // one multicast commit per phase
      mbar_init(tempty0 + 8 * i, 2);  // leader only: one arrival from the epilogue of each CTA
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
  const int n_cc = p.n_chunks;

  if (warp == 0) {
    // ------------------------------------------------------------ zh producer (both CTAs)
    if (lane == 0) {
      tma_prefetch_desc(&tm_z);
      long long z_issued = 0;
      int zb = 0;
      uint32_t zph = 0;
      bool ok = true;
      for (int tile = cluster; tile < total; tile += n_clusters) {
        if (!mbar_wait(zempty0 + 8 * zb, zph ^ 1u, st, SITE_PRODUCER)) {
          ok = false;
          break;
        }
        const int bb = tile / p.tiles_per_batch;
        // a half-tile wholly past N*N loads rows 0.. instead: its pairs are not stored
        long long prow = static_cast<long long>(tile - bb * p.tiles_per_batch) * TP + rank * HALF;
        if (prow >= p.NN) prow = 0;
        if (leader) mbar_arrive_expect_tx(zfull0 + 8 * zb, 2 * z_buf_bytes);
        const uint32_t fb = mapa_shared(zfull0 + 8 * zb, 0);
        for (int s = 0; s < p.k_slabs; ++s)
          tma_load_3d_pair(zbuf0 + zb * z_buf_bytes + s * Z_SLAB, &tm_z, fb, s * 64, static_cast<int>(prow), bb);
        ++z_issued;
        if (++zb == p.z_bufs) {
          zb = 0;
          zph ^= 1u;
        }
      }
      if (!ok && leader) {
        int s = zb;
        uint32_t ph = zph;
        for (long long i = 0; i < z_issued && i < p.z_bufs; ++i) {
          if (--s < 0) {
            s = p.z_bufs - 1;
            ph ^= 1u;
          }
          mbar_wait_drain(zfull0 + 8 * s, ph, p.timeout_ns);
        }
      }
    }
  } else if (warp == 2) {
    // ------------------------------------------------------------ weight producer (both CTAs)
    if (lane == 0) {
      tma_prefetch_desc(&tm_w);
      int ws = 0;
      uint32_t wph = 0;
      long long w_issued = 0;
      bool ok = true;
      const int tile_end_w = kResident ? min(total, cluster + 1) : total;
      for (int tile = cluster; tile < tile_end_w && ok; tile += n_clusters) {
        for (int cc = 0; cc < n_cc && ok; ++cc) {
          for (int s = 0; s < p.k_slabs; ++s) {
            if (!mbar_wait(wempty0 + 8 * ws, wph ^ 1u, st, SITE_PRODUCER)) {
              ok = false;
              break;
            }
            if (leader) mbar_arrive_expect_tx(wfull0 + 8 * ws, 2 * W_SLAB);
            tma_load_2d_pair(wring + ws * W_SLAB, &tm_w, mapa_shared(wfull0 + 8 * ws, 0), s * 64,
                             cc * 4 * CH + static_cast<int>(rank) * 2 * CH);
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
      const uint32_t idesc = idesc_bf16_f32(4 * CH, TP, 0, 0);
      const uint64_t zdesc0 = sdesc_sw128(zbuf0, 16, 1024);
      const uint64_t wdesc0 = sdesc_sw128(wring, 16, 1024);
      int ws = 0, acc = 0;
      uint32_t wph = 0, aph = 0;
      bool ok = true;
      int zb = 0;
      uint32_t zph = 0;
      constexpr bool w_ready = kResident;
      if (w_ready && cluster < total)
        for (int i = 0; i < n_cc * p.k_slabs && ok; ++i) ok = mbar_wait(wfull0 + 8 * i, 0, st, SITE_MMA);
      for (int tile = cluster; tile < total && ok; tile += n_clusters) {
        if (!mbar_wait(zfull0 + 8 * zb, zph, st, SITE_MMA)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint64_t zdesc = zdesc0 + ((zb * z_buf_bytes) >> 4);
        for (int cc = 0; cc < n_cc && ok; ++cc) {
          if (!mbar_wait_cluster(tempty0 + 8 * acc, aph ^ 1u, st, SITE_MMA)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t d = tmem_base + acc * TP;
          for (int s = 0; s < p.k_slabs; ++s) {
            if (kResident) ws = cc * p.k_slabs + s;
            if (!w_ready && !mbar_wait(wfull0 + 8 * ws, wph, st, SITE_MMA)) {
              ok = false;
              break;
            }
            tc_fence_after();
            const uint64_t bd = zdesc + ((s * Z_SLAB) >> 4), ad = wdesc0 + ((ws * W_SLAB) >> 4);
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) mma_f16_ss_pair(d, ad + 2 * kk, bd + 2 * kk, idesc, (s | kk) != 0);
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
  } else {
    // ------------------------------------------------------------ epilogue (both CTAs)
    // Thread t of warp (hc, q) holds channel g*8 + t/4 of the warp's 16 (lane
    // group g) and, in each 32-pair block j, the pairs 8k + 2(t%4), +1.
    const int ew = warp - 3;  // 0..15
    const int e = ew * 32 + lane;
    const int q = warp & 3;
    const int hc = ew >> 2;
    const uint32_t stage = base + L.stage + ew * STAGE_OUT;
    uint8_t* const stage_ptr = base_ptr + L.stage + ew * STAGE_OUT;
    const uint32_t lrow = static_cast<uint32_t>(lane) >> 2;
    const uint32_t cpair = 2u * (lane & 3);
    const uint32_t tempty_leader = mapa_shared(tempty0, 0);
    constexpr int EPI_THREADS = 32 * EPI_WARPS;
    uint32_t* const mslot = reinterpret_cast<uint32_t*>(base_ptr + L.mask);
    auto mask_word = [&](int t) -> uint32_t {  // raw bf16 pair of tile t, or two ones
      if (!p.mask || e >= TP / 2 || t >= total) return 0x3F803F80u;
      const int tb = t / p.tiles_per_batch;
      const long long pm = static_cast<long long>(t - tb * p.tiles_per_batch) * TP + 2 * e;
      return pm < p.NN ? __ldg(reinterpret_cast<const unsigned int*>(p.mask + tb * p.NN + pm)) : 0x3F803F80u;
    };
    auto stage_mask = [&](int slot, uint32_t raw) {  // staged as m / 2 (exact)
      if (e < TP / 2) mslot[slot * (TP / 2) + e] = pack_half2(0.5f * bf16_lo(raw), 0.5f * bf16_hi(raw));
    };
    stage_mask(0, mask_word(cluster));
    uint32_t mnext = mask_word(cluster + n_clusters);
    int acc = 0;
    uint32_t aph = 0;
    bool ok = true;
    int n = 0;
    for (int tile = cluster; tile < total && ok; tile += n_clusters, ++n) {
      const int bb = tile / p.tiles_per_batch;
      const long long pb = static_cast<long long>(tile - bb * p.tiles_per_batch) * TP + hc * 64;
      named_bar_sync(5, EPI_THREADS);
      stage_mask((n + 1) & 1, mnext);
      mnext = mask_word(tile + 2 * n_clusters);
      const uint32_t* const mrow = mslot + (n & 1) * (TP / 2) + (hc * 64 + cpair) / 2;
      for (int cc = 0; cc < n_cc; ++cc) {
        const int ob = cc * 2 * CH + static_cast<int>(rank) * CH + q * 16;  // first channel of the warp
        const int rw = cc * 4 * CH + static_cast<int>(rank) * 2 * CH + q * 32 + static_cast<int>(lrow);
        // step i: lane group g = i / 2, 32-pair block j = i % 2; the thread's
        // da / db row of that lane group (none past 2C)
        auto da_row = [&](int o) -> const uint16_t* {
          const int c = o < p.C ? o : o - p.C;
          return reinterpret_cast<const uint16_t*>(o < p.C ? p.da : p.db) + (static_cast<long long>(bb) * p.C + c) * p.NN;
        };
        auto da_load = [&](int i, uint32_t (&d)[4]) {
          const int o = ob + (i >> 1) * 8 + static_cast<int>(lrow);
          const bool in = o < 2 * p.C;
          const uint16_t* const r = da_row(o);
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const long long pr = pb + (i & 1) * 32 + 8 * k + cpair;
            d[k] = (in && pr < p.NN) ? __ldg(reinterpret_cast<const unsigned int*>(r + pr)) : 0u;
          }
        };
        // The da / db values do not depend on the accumulator: the first two
        // steps' loads are issued before waiting for it, each later step's two
        // steps ahead, and the next chunk's 16 rows (128 bytes each) are
        // prefetched into L2, so the loads' DRAM latency overlaps the MMAs.
        uint32_t ra[16], rb[16], da_a[4], da_b[4];
        da_load(0, da_a);
        da_load(1, da_b);
        if (cc + 1 < n_cc && lane < 16 && pb < p.NN) {
          const int o = ob + 2 * CH + lane;  // the next chunk's rows of this warp
          if (o < 2 * p.C) prefetch_l2(da_row(o) + pb);
        }
        float bv[2], bg[2];  // biases of this thread's channel in lane group g (value row, gate row)
#pragma unroll
        for (int g = 0; g < 2; ++g) {
          bv[g] = __ldg(p.bias + rw + g * 16);
          bg[g] = __ldg(p.bias + rw + g * 16 + 8);
        }
        const bool got = __all_sync(0xffffffffu, mbar_wait(tfull0 + 8 * acc, aph, st, SITE_EPI));
        tc_fence_after();
        const uint32_t t_addr = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + acc * TP + hc * 64;
        auto step_addr = [&](int i) -> uint32_t {
          return t_addr + (static_cast<uint32_t>((i >> 1) * 16) << 16) + static_cast<uint32_t>((i & 1) * 32);
        };
        float rs[4] = {0.f, 0.f, 0.f, 0.f};  // row sums: (g, value / gate)
        if (got) tmem_ld16x256b_x4(step_addr(0), ra);
        // rows of dP: a values [0, C), a gates [C, 2C), b values [2C, 3C), b gates [3C, 4C);
        // lane group g's 8 channels are all a's or all b's (C is a multiple of 8)
        auto store_group = [&](int g) {
          if (lane == 0) {
            const int o0 = ob + g * 8;
            if (got && pb < p.NN && o0 < 2 * p.C) {
              const int vrow = o0 < p.C ? o0 : o0 + p.C;
              tma_store_3d(&tm_p8, stage, static_cast<int>(pb), vrow, bb);
              tma_store_3d(&tm_p8, stage + 1024, static_cast<int>(pb), vrow + p.C, bb);
            }
            tma_store_commit();
          }
        };
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int g = i >> 1, j = i & 1;
          uint32_t(&cur)[16] = (i & 1) ? rb : ra;
          uint32_t(&dcur)[4] = (i & 1) ? da_b : da_a;
          if (got) tmem_ld_wait();
          if (i < 3 && got) tmem_ld16x256b_x4(step_addr(i + 1), (i & 1) ? ra : rb);
          if (i == 3) {
            tc_fence_before();
            if (!named_bar_and(4, EPI_THREADS, got)) ok = false;
            if (ok && ew == 0 && lane == 0) mbar_arrive_remote(tempty_leader + 8 * acc);
          }
          if (!ok) break;
          // the step's results go to registers first, so that the wait for the
          // previous stores to read the staging box overlaps this arithmetic
          uint32_t pvk[4], pgk[4];
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const uint32_t m2 = mrow[(j * 32 + 8 * k) / 2];  // m / 2
            const float2 mf = __half22float2(*reinterpret_cast<const __half2*>(&m2));
            // v/2 and g/2 (the host halved the weights)
            const float2 v2 = __fadd2_rn(make_float2(__uint_as_float(cur[4 * k]), __uint_as_float(cur[4 * k + 1])),
                                         make_float2(bv[g], bv[g]));
            const float2 g2 = __fadd2_rn(make_float2(__uint_as_float(cur[4 * k + 2]), __uint_as_float(cur[4 * k + 3])),
                                         make_float2(bg[g], bg[g]));
            const float2 th = make_float2(tanh_fast(g2.x), tanh_fast(g2.y));
            const float2 dm = __fmul2_rn(make_float2(bf16_lo(dcur[k]), bf16_hi(dcur[k])), mf);  // da m / 2
            const float2 dv = __ffma2_rn(dm, th, dm);                                            // dm (1 + t)
            const float2 u = __fmul2_rn(dv, v2);
            const float2 dg = __ffma2_rn(make_float2(-u.x, -u.y), th, u);                        // u (1 - t)
            pvk[k] = pack_bf162(dv.x, dv.y);
            pgk[k] = pack_bf162(dg.x, dg.y);
            rs[2 * g] += dv.x + dv.y;
            rs[2 * g + 1] += dg.x + dg.y;
          }
          if (j == 0) {  // the staging box is free again: the previous stores have read it
            if (lane == 0) tma_store_wait_read<0>();
            __syncwarp();
          }
          // dv in rows 0..7, dg in rows 8..15 (both lrow = t / 4 of this lane group)
          uint8_t* const srow = stage_ptr + lrow * 128u + cpair * 2u;
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            *reinterpret_cast<uint32_t*>(srow + (((static_cast<uint32_t>(4 * j + k) ^ lrow) & 7u) << 4)) = pvk[k];
            *reinterpret_cast<uint32_t*>(srow + 1024 + (((static_cast<uint32_t>(4 * j + k) ^ lrow) & 7u) << 4)) = pgk[k];
          }
          if (i < 2) da_load(i + 2, dcur);  // its buffer is free again
          if (j == 1) {
            fence_proxy_async_smem();
            __syncwarp();
            store_group(g);
          }
        }
        if (!ok) break;
        // row sums: reduce over the 4 threads of a channel; lane t writes sum (t % 4) of row t / 4
#pragma unroll
        for (int v = 0; v < 4; ++v) {
          rs[v] += __shfl_xor_sync(0xffffffffu, rs[v], 1);
          rs[v] += __shfl_xor_sync(0xffffffffu, rs[v], 2);
        }
        const int sel = lane & 3;
        const float mine = sel == 0 ? rs[0] : sel == 1 ? rs[1] : sel == 2 ? rs[2] : rs[3];
        if (got)
          p.rowpart[((((static_cast<long long>(tile) * n_cc + cc) * 2 + rank) * 4 + q) * 4 + hc) * 32 + sel * 8 + lrow] =
              mine;
        if (++acc == 2) {
          acc = 0;
          aph ^= 1u;
        }
      }
    }
    if (lane == 0) tma_store_wait_all();
  }

  tc_fence_before();
  __syncthreads();
  cluster_sync_all();  // no CTA leaves while its peer may still signal it
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem_base, TMEM_COLS);
  }
}

// Row sums, stage 1: rowpart [tiles][n_cc * 1024] -> tmp [B][nslice][n_cc * 1024],
// block (slice, b) summing the tiles slice*per .. of batch b, in order.
__global__ void k6_rowsum_tiles(const float* __restrict__ rowpart, float* __restrict__ tmp, int tiles_per_batch,
                                int per, int width) {
  const int slice = blockIdx.x, b = blockIdx.y, nslice = gridDim.x;
  const int t0 = slice * per, t1 = min(tiles_per_batch, t0 + per);
  for (int j = threadIdx.x; j < width; j += blockDim.x) {
    float s = 0.f;
    for (int t = t0; t < t1; ++t) s += rowpart[(static_cast<long long>(b) * tiles_per_batch + t) * width + j];
    tmp[(static_cast<long long>(b) * nslice + slice) * width + j] = s;
  }
}

// Row sums, stage 2: for output channel o (a channels, then b) and kind
// (value, gate) of batch b, the sum over slices and column quarters, into the
// gradient assembly's layout gp[(b * C + c) * 4 + k] (k: a value, a gate,
// b value, b gate).
__global__ void k6_rowsum_rows(const float* __restrict__ tmp, float* __restrict__ gp, int nslice, int width, int C,
                               int B) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= B * 2 * C * 2) return;
  const int kind = i & 1, o = (i >> 1) % (2 * C), b = (i >> 1) / (2 * C);
  const int cc = o / 128, r = (o / 64) & 1, q = (o / 16) & 3, g = (o / 8) & 1, lrow = o & 7;
  float s = 0.f;
  for (int sl = 0; sl < nslice; ++sl)
    for (int hc = 0; hc < 4; ++hc)
      s += tmp[(static_cast<long long>(b) * nslice + sl) * width + ((((cc * 2 + r) * 4 + q) * 4 + hc) * 32) +
               (g * 2 + kind) * 8 + lrow];
  const int c = o < C ? o : o - C, k = kind + (o < C ? 0 : 2);
  gp[(static_cast<long long>(b) * C + c) * 4 + k] = s;
}

cudaError_t launch_gate_grad(const GateGradArgs& a, const CUtensorMap& tm_z, const CUtensorMap& tm_w,
                             const CUtensorMap& tm_p8, int grid, cudaStream_t s) {
  if (a.w_stages < (a.w_resident ? 1 : 2) || a.w_stages > MAX_W_STAGES || a.z_bufs < 2 || a.z_bufs > MAX_Z_BUFS)
    return cudaErrorInvalidValue;
  const size_t smem = gategrad_smem_bytes(a.k_slabs, a.w_stages, a.z_bufs);
  auto* const kern = a.w_resident ? k6_gate_grad<true> : k6_gate_grad<false>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  grid &= ~1;
  if (grid < 2) grid = 2;
  kern<<<grid, THREADS, smem, s>>>(tm_z, tm_w, tm_p8, a);
  return cudaGetLastError();
}

cudaError_t launch_gate_rowsums(const float* rowpart, float* tmp, float* gp, int B, int tiles_per_batch, int n_cc,
                                int C, int nslice, cudaStream_t s) {
  const int width = n_cc * 1024;
  const int per = (tiles_per_batch + nslice - 1) / nslice;
  k6_rowsum_tiles<<<dim3(nslice, B), 256, 0, s>>>(rowpart, tmp, tiles_per_batch, per, width);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const int n = B * 2 * C * 2;
  k6_rowsum_rows<<<(n + 255) / 256, 256, 0, s>>>(tmp, gp, nslice, width, C, B);
  return cudaGetLastError();
}

int gategrad_max_pairs(int num_sms, int k_slabs, int w_stages, int z_bufs) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(num_sms & ~1, 1, 1);
  cfg.blockDim = dim3(THREADS, 1, 1);
  cfg.dynamicSmemBytes = gategrad_smem_bytes(k_slabs, w_stages, z_bufs);
  cudaLaunchAttribute attr;
  attr.id = cudaLaunchAttributeClusterDimension;
  attr.val.clusterDim.x = 2;
  attr.val.clusterDim.y = 1;
  attr.val.clusterDim.z = 1;
  cfg.attrs = &attr;
  cfg.numAttrs = 1;
  cudaFuncSetAttribute(k6_gate_grad<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                       static_cast<int>(cfg.dynamicSmemBytes));
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, k6_gate_grad<false>, &cfg) != cudaSuccess || n < 1) {
    cudaGetLastError();
    return num_sms / 2;
  }
  return n;
}

}  // namespace trimul
