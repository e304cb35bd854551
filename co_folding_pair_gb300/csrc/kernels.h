// kernels.h -- argument blocks and launchers of the three TriMul kernels (internal).
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>

#include <cstdint>

namespace trimul {

// ---------------------------------------------------------------- stage 1
// LN_in + gated input projection + mask -> a, b channel-major planes (fp16).
// One tile = 256 consecutive pairs of one batch element, taken by a CTA pair
// (128 pairs per CTA).  The weight matrix holds n_chunks chunks of 256 rows,
// one per 128 output channels (a channels 0..C-1, then b channels 0..C-1):
// for output channel o and kind k (0 value, 1 gate) the row is
//     (o / 8) * 16 + k * 8 + o % 8,
// so every 16 rows hold the value rows of 8 channels then their gate rows;
// rows of channels past 2C are zero.
constexpr int INPROJ_TILE_PAIRS = 256;
constexpr int INPROJ_HALF_PAIRS = INPROJ_TILE_PAIRS / 2;  // the host's z box has exactly this many rows
constexpr int INPROJ_MAX_Z_BUFS = 4;
constexpr int INPROJ_MAX_W_STAGES = 16;
enum : int { INPROJ_OUT_F16 = 0, INPROJ_OUT_BF16 = 1, INPROJ_OUT_E4M3 = 2 };

struct InprojArgs {
  int B, N, D, C;
  long long NN;          // N * N pairs per batch element
  int k_slabs;           // ceil(D / 64)
  int n_chunks;          // ceil(2C / 128)
  int tiles_per_batch;   // ceil(NN / INPROJ_TILE_PAIRS)
  int tile_begin, tile_end;  // the launch covers tiles [tile_begin, tile_end) of all B * tiles_per_batch
  int w_stages;          // depth of the weight ring (2..INPROJ_MAX_W_STAGES; resident weights: their slab count)
  int z_bufs;            // z half-tile buffers (2..INPROJ_MAX_Z_BUFS)
  int w_resident;        // 1: all of a CTA's weight slabs fit the ring and are loaded once
  int inject_stall;      // test hook: producer issues nothing
  int out_kind;          // INPROJ_OUT_*: how a and b are stored
  float fp8_scale;       // INPROJ_OUT_E4M3: a power of two with max |a|, |b| * fp8_scale <= 448
  const __nv_bfloat16* mask;  // [B][NN] or nullptr (all ones)
  const float* bias;          // [n_chunks * 256]: W beta_in / 2 per weight row (same row order as the weights)
  float eps;
  __half* a;                  // [B][C][NN] (bf16 bits, or bytes, by out_kind)
  __half* b;                  // [B][C][NN]
  float2* zstats;             // [B][NN] (mean, rstd) of LN_in per pair, written when non-null
  int write_zhat;             // INPROJ_OUT_BF16 only: also store zh = (z - mean) rstd (bf16 [B][NN][D], tm_zh)
  unsigned* ab_max;           // when non-null: atomicMax of the bits of max |a|, |b| (fp16 values as stored)
  int* mask_flag;             // when non-null: set to 1 if a mask value lies outside [0, 1] (or is NaN)
  int* status;
  unsigned long long timeout_ns;
};

// ---------------------------------------------------------------- stage 2
// Per-plane triangle GEMM, plane = b * C + c; one 256 x 256 tile of X per CTA pair.
// Each CTA stages TRI_ROWS rows of A and TRI_ROWS rows of B per K block of
// TRI_BK: the host's TMA boxes must move exactly TRI_STAGE_BYTES per CTA and stage.
constexpr int TRI_ROWS = 128;
constexpr int TRI_BK = 64;
constexpr unsigned TRI_STAGE_BYTES = 2u * TRI_ROWS * TRI_BK * 2u;
struct TriangleArgs {
  int N;
  int planes;
  int tiles_m, tiles_n, k_iters;  // tiles of 256 rows / 256 columns; K blocks of 64
  int tile_begin, tile_end;  // the launch covers tiles [tile_begin, tile_end), plane-major
  int a_mn, b_mn;    // 1: the operand is MN-major ([K][rows], rows contiguous), 0: K-major
                     // (the forward: both 0 outgoing, both 1 incoming)
  int inject_stall;
  int bf16;          // 1: a and b are bf16 (else fp16)
  int fp8;           // 1: a and b are e4m3 (outgoing only; K blocks of 2 * TRI_BK elements)
  int out_bf16;      // 1: x is stored as bf16, unscaled (the backward's triangle gradients)
  float fp8_descale; // with fp8: 1 / (scale of a * scale of b), applied with x_scale
  __half* x;         // [planes][N][N]: x * x_scale (fp16), or x (bf16 bits) with out_bf16
  float x_scale;     // a power of two that keeps |x| * x_scale within binary16
  const unsigned* ab_max;  // when non-null, x_scale = 2^-x_scale_log2_from_max(max |a|, |b| of this call, N) instead
  int* status;
  unsigned long long timeout_ns;
};

// ---------------------------------------------------------------- stage 3
// LN_out(x) W_o^T gated by sigmoid(LN_in(z) W_g^T), per pair tile of 128, with
// both LayerNorms folded into the weights (W~ = W diag(gamma), see colc).
constexpr int MAX_OUTPROJ_A_STAGES = 8;  // activation slabs (16 KB) in the ring
constexpr int MAX_OUTPROJ_W_STAGES = 8;  // weight slabs (round16(D) rows x 64 K) in the ring

struct OutprojArgs {
  int B, N, D, C;        // 8 <= D <= 256
  long long NN;
  int x_slabs;           // ceil(C / 64)
  int z_slabs;           // ceil(D / 64)
  int tiles_per_batch;
  int tile_begin, tile_end;  // the launch covers tiles [tile_begin, tile_end) of all B * tiles_per_batch
  int a_stages;          // 2 .. MAX_OUTPROJ_A_STAGES
  int w_stages;          // 2 .. MAX_OUTPROJ_W_STAGES
  int inject_stall;
  float eps;             // LayerNorm eps of z
  __nv_bfloat16* out;    // [B][NN][D]
  const float2* zstats;  // [B][NN] (mean, rstd) of LN_in per pair, or nullptr (then computed here)
  const float4* colc;    // [D]: (s_g, t_g / 2, s_o, t_o / 2) of the folded LayerNorm affines
  float eps_x;           // LayerNorm eps for the stored (scaled) x
  const unsigned* ab_max;  // when non-null, eps_x = eps * 4^-x_scale_log2_from_max(max |a|, |b| of this call, N) instead
  int* status;
  unsigned long long timeout_ns;
};

// ---------------------------------------------------------------- backward GEMM
// C[z] (M x N, row-major, ldc) = sum over the global K blocks of slice z of
// A(m, k) B(n, k); see k4_gemm.cu.
enum : int { GEMM_OUT_BF16 = 0, GEMM_OUT_F32 = 1, GEMM_OUT_F32_ADD = 2, GEMM_OUT_F16 = 3 };

struct GemmArgs {
  int M, N;               // output rows and columns (multiples of 8)
  int kpb;                // K blocks of 64 per operand batch
  int batches;            // operand batches (1 when neither operand is batched)
  int n_z;                // z slices: one per batch, or split-K slices over batches * kpb blocks
  long long kb_per_z;     // global K blocks per slice (every slice gets at least one)
  int tiles_m, tiles_n;   // ceil(M / 256), ceil(N / 256)
  int tile_begin, tile_end;  // tiles [tile_begin, tile_end) of n_z * tiles_m * tiles_n, slice-major
  int a_mn, b_mn;         // 1: the operand is MN-major ([K][rows]), 0: K-major ([rows][K])
  int a_batched, b_batched;  // 1: a 3-D tensor map over batches; 0: one 2-D matrix for all
  int bf16;               // operand type: 1 bf16, 0 fp16
  int out_mode;           // GEMM_OUT_*
  int m_fastest;          // 1: a slice's tiles are visited with the M tile fastest (else the N tile)
  void* c;                // output base: slice z at c + z * c_zstride elements
  long long ldc, c_zstride;
  int* status;
  unsigned long long timeout_ns;
};

size_t gemm_smem_size();
int gemm_max_pairs(int num_sms);
cudaError_t launch_gemm(const GemmArgs& a, const CUtensorMap& tm_a, const CUtensorMap& tm_b, int grid,
                        cudaStream_t s);

// ---------------------------------------------------------------- backward per-pair steps (k5_backward.cu)
struct TrimulGradPtrs {
  float *w_a, *w_ga, *w_b, *w_gb;  // [C][D]
  float *w_o;                      // [D][C]
  float *w_g;                      // [D][D]
  float *ln_in_gamma, *ln_in_beta, *ln_out_gamma, *ln_out_beta;
};


cudaError_t launch_xhat(const __half* x, __nv_bfloat16* xh, float2* xstats, const unsigned* ab_max, int B, int N,
                        int C, float eps, int num_sms, cudaStream_t s);
int dout_blocks(long long n_pairs, int D, int num_sms);
cudaError_t launch_dout(const __nv_bfloat16* dout, const __half* gacc, const __half* vacc, const float* tg,
                        const float* to, __nv_bfloat16* dv, __nv_bfloat16* dg, float* part, long long n_pairs, int D,
                        int num_sms, cudaStream_t s);
cudaError_t launch_lnout_bwd(const __nv_bfloat16* dy, const __half* x, const float2* xstats, const float* gamma,
                             __nv_bfloat16* dx, const unsigned* ab_max, int B, int N, int C, int num_sms,
                             cudaStream_t s);
// Backward of the gated input projections fused with their pre-activations
// (k6_gate_grad.cu): same tiles, rings and weight row order as the input
// projection, operands zh (bf16 [B][NN][D]) and bf16 weights; writes dP
// (bf16 [B][4C][NN]: a values, a gates, b values, b gates) and per-tile row
// sums rowpart [tiles][n_chunks * 1024].
struct GateGradArgs {
  int B, N, D, C;
  long long NN;
  int k_slabs, n_chunks, tiles_per_batch;
  int tile_begin, tile_end;
  int w_stages, z_bufs, w_resident;
  const __nv_bfloat16* mask;  // [B][NN] or nullptr
  const float* bias;          // W beta_in / 2 per weight row (the input projection's)
  const __nv_bfloat16* da;    // [B][C][NN]
  const __nv_bfloat16* db;    // [B][C][NN]
  float* rowpart;
  int* status;
  unsigned long long timeout_ns;
};
size_t gategrad_smem_bytes(int k_slabs, int w_stages, int z_bufs);
int gategrad_max_pairs(int num_sms, int k_slabs, int w_stages, int z_bufs);
cudaError_t launch_gate_grad(const GateGradArgs& a, const CUtensorMap& tm_z, const CUtensorMap& tm_w,
                             const CUtensorMap& tm_p8, int grid, cudaStream_t s);
// rowpart -> gp[(b * C + c) * 4 + k] (the assembly's layout with one segment),
// through tmp [B][nslice][n_chunks * 1024]
cudaError_t launch_gate_rowsums(const float* rowpart, float* tmp, float* gp, int B, int tiles_per_batch, int n_cc,
                                int C, int nslice, cudaStream_t s);
int lnin_blocks(long long n_pairs, int num_sms);
cudaError_t launch_lnin_bwd(const __nv_bfloat16* dzp, const __nv_bfloat16* dzq, const __nv_bfloat16* z, const float2* zstats,
                            const float* gamma, __nv_bfloat16* dz, float* part, long long n_pairs, int D, int num_sms,
                            cudaStream_t s);
cudaError_t launch_sum(const float* part, float* out, long long n, int count, int num_sms, cudaStream_t s);
cudaError_t launch_assemble(const float* m_o, const float* m_g, const float* m_in, const float* cs, const float* gp,
                            int nseg, const float* ln_in, const float* w_o, const float* g_in, const float* b_in,
                            const float* g_out, const float* b_out, const TrimulGradPtrs& out, int B, int D, int C,
                            int num_sms, cudaStream_t s);

// The power of two s with which the triangle GEMM stores x as fp16 x * 2^-s,
// from m = max |a|, |b| of the call: |x| <= N m^2 (a sum of N products), so s
// is the smallest with N m^2 2^-s <= 32768 (half the binary16 maximum).  The
// triangle kernel and the output projection evaluate it alike from the same word.
__host__ __device__ inline int x_scale_log2_from_max(float m, int N) {
  const float bound = static_cast<float>(N) * m * m;
  int s = 0;
  float v = bound;
  while (s < 40 && v > 32768.0f) {
    v *= 0.5f;
    ++s;
  }
  return s;
}

// 2^-k as a float, exactly, for 0 <= k <= 126.
__host__ __device__ inline float exp2_neg(int k) {
  union {
    uint32_t u;
    float f;
  } v;
  v.u = static_cast<uint32_t>(127 - k) << 23;
  return v.f;
}

// Co-resident CTA pairs (clusters of two) the triangle kernel can run on this device.
int triangle_max_pairs(int num_sms);

// Shared-memory footprints (bytes of dynamic shared memory per CTA).
size_t inproj_smem_bytes(int k_slabs, int w_stages, int z_bufs);
size_t triangle_smem_bytes();
size_t outproj_smem_bytes(int a_stages, int w_stages, int D);
uint32_t outproj_w_stage_bytes(int D);

// Launchers: set the shared-memory attribute once, then launch `grid` CTAs.
// tm_a / tm_b: 64-pair x 32-channel store boxes; tm_a8 / tm_b8: 64 x 8.
cudaError_t launch_inproj(const InprojArgs& a, const CUtensorMap& tm_z, const CUtensorMap& tm_w,
                          const CUtensorMap& tm_a, const CUtensorMap& tm_b, const CUtensorMap& tm_a8,
                          const CUtensorMap& tm_b8, const CUtensorMap& tm_zh, int grid, cudaStream_t s);
// Co-resident CTA pairs (clusters of two) the input projection can run on this device.
int inproj_max_pairs(int num_sms, int k_slabs, int w_stages, int z_bufs);
cudaError_t launch_triangle(const TriangleArgs& a, const CUtensorMap& tm_a, const CUtensorMap& tm_b, int grid,
                            cudaStream_t s);
cudaError_t launch_outproj(const OutprojArgs& a, const CUtensorMap& tm_x, const CUtensorMap& tm_z,
                           const CUtensorMap& tm_wg, const CUtensorMap& tm_wo, const CUtensorMap& tm_out, int grid,
                           cudaStream_t s);

}  // namespace trimul
