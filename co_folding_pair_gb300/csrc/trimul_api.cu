// trimul_api.cu -- the C ABI declared in include/trimul.h: handle life cycle,
// weight re-layout, workspace, tensor maps and the launch sequence.
//
// The life cycle mirrors the fold-cp-ops README ("Use"): construct (fix the
// layer's weights), optional prepare (front-load allocation), call, free.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <vector>

#include "trimul.h"
#include "kernels.h"

using namespace trimul;

namespace {

thread_local char g_err[512] = "";

trimul_status fail(trimul_status s, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_err, sizeof(g_err), fmt, ap);
  va_end(ap);
  return s;
}

trimul_status cuda_fail(cudaError_t e, const char* what) {
  return fail(e == cudaErrorMemoryAllocation ? TRIMUL_ERR_OOM : TRIMUL_ERR_CUDA, "%s: %s (%s)", what,
              cudaGetErrorName(e), cudaGetErrorString(e));
}

#define TRY_CUDA(expr, what)                      \
  do {                                            \
    cudaError_t e_ = (expr);                      \
    if (e_ != cudaSuccess) return cuda_fail(e_, what); \
  } while (0)

// ------------------------------------------------------------------ tensor maps
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

// A row-major tensor of 16-bit elements: dims[0] is the contiguous axis.
// Tiled tensor map over a dense row-major tensor of 2-byte elements (bf16 or
// fp16) with the 128-byte swizzle, or (make_map_u8) of bytes without swizzle.
trimul_status make_map_any(CUtensorMap* m, CUtensorMapDataType dtype, unsigned elem_bytes, CUtensorMapSwizzle swz,
                           int rank, const void* ptr, const uint64_t* dims, const uint32_t* box, const char* what) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return fail(TRIMUL_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
  cuuint64_t gdim[3], gstride[2];
  cuuint32_t bdim[3], estride[3] = {1, 1, 1};
  uint64_t stride = elem_bytes;
  for (int i = 0; i < rank; ++i) {
    gdim[i] = dims[i];
    bdim[i] = box[i];
    if (i > 0) gstride[i - 1] = stride;
    stride *= dims[i];
  }
  CUresult r = fn(m, dtype, static_cast<cuuint32_t>(rank), const_cast<void*>(ptr), gdim, gstride, bdim, estride,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(TRIMUL_ERR_CUDA, "tensor map for %s rejected (CUresult %d)", what, (int)r);
  return TRIMUL_OK;
}

trimul_status make_map(CUtensorMap* m, bool is_bf16, int rank, const void* ptr, const uint64_t* dims,
                       const uint32_t* box, const char* what) {
  return make_map_any(m, is_bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2,
                      CU_TENSOR_MAP_SWIZZLE_128B, rank, ptr, dims, box, what);
}

// bytes (the e4m3 planes), with the 128-byte swizzle (operand tiles of 128-byte
// rows) or none (the input projection's 64-byte staged rows)
trimul_status make_map_u8(CUtensorMap* m, bool swizzle128, int rank, const void* ptr, const uint64_t* dims,
                          const uint32_t* box, const char* what) {
  return make_map_any(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1,
                      swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE, rank, ptr, dims, box, what);
}

float bf16_to_float(uint16_t v) {
  uint32_t u = static_cast<uint32_t>(v) << 16;
  float f;
  std::memcpy(&f, &u, 4);
  return f;
}

uint16_t float_to_half_bits(float f) {
  __half h = __float2half_rn(f);
  uint16_t u;
  std::memcpy(&u, &h, 2);
  return u;
}

uint16_t float_to_bf16_bits(float f) {
  __nv_bfloat16 h = __float2bfloat16_rn(f);
  uint16_t u;
  std::memcpy(&u, &h, 2);
  return u;
}

float half_bits_to_float(uint16_t v) {
  __half h;
  std::memcpy(&h, &v, 2);
  return __half2float(h);
}

constexpr float kHalfMax = 65504.0f;
// The host-buffer path splits calls whose z exceeds kHostChunkMin bytes into
// kHostChunks tile ranges, so each range's copy overlaps another's compute.
constexpr int kHostChunks = 8;
constexpr size_t kHostChunkMin = 256ull << 20;
constexpr unsigned long long kDefaultTimeoutNs = 4000000000ull;  // 4 s per wait
constexpr unsigned long long kStallTimeoutNs = 200000000ull;     // 0.2 s under TRIMUL_FLAG_INJECT_STALL

}  // namespace

struct trimul_handle_s {
  int device = 0;
  int D = 0, C = 0;
  float eps = 1e-5f;
  int num_sms = 0;
  int max_smem = 0;
  int tri_pairs = 0;       // co-resident CTA pairs of the triangle kernel
  int in_pairs = 0;        // co-resident CTA pairs of the input projection
  int gg_pairs = 0;        // co-resident CTA pairs of the backward's gate-gradient kernel
  int in_w_stages = 0;     // weight-ring depth of the input projection
  int in_z_bufs = 0;       // z buffers of the input projection
  int in_w_resident = 0;   // input-projection weights loaded once (they fit the ring)
  int n_chunks = 0;        // stage-1 weight chunks of 256 rows
  uint16_t* w_in = nullptr;  // fp16 [n_chunks * 256][D]
  uint16_t* w_in_bf = nullptr;  // the same rows in bf16 (after w_in in its allocation): the gate gradients' operand
  uint16_t* w_o = nullptr;   // fp16 [D][C]: W_o diag(gamma_out)
  uint16_t* w_g = nullptr;   // bf16 [D][D]: W_g diag(gamma_in)
  float* ln = nullptr;       // f32 gamma_in[D] beta_in[D] gamma_out[C] beta_out[C] (each 16-byte aligned)
  float* in_bias = nullptr;  // per input-weight row: W beta_in / 2 (same layout as w_in's rows)
  float4* colc = nullptr;    // per output feature d: (s_g, t_g / 2, s_o, t_o / 2), see trimul_create
  double ab_bound = 0;       // bound on |a| and |b| (value projection, |mask| <= 1)
  float *g_in = nullptr, *b_in = nullptr, *g_out = nullptr, *b_out = nullptr;
  // device words, cleared at the start of every call: [0] the site code of a
  // kernel wait that timed out, [1] set when a mask value lies outside [0, 1],
  // [2] the bits of max |a|, |b| of a forward (its x scale derives from it)
  int* status = nullptr;
  // workspace: a, b (fp16) and x (fp16 holding x * 2^-s), each [B][C][N][N],
  // then the LN_in statistics (float2 [B][N][N]) that stage 1 hands to stage 3
  uint16_t* ws = nullptr;
  size_t ws_bytes = 0;
  // trimul_forward_host: two staging slots (each z | out | mask), used by
  // alternate calls so that a call's input copy can run while the previous
  // call computes; copy streams and the events that order them
  uint16_t* stage = nullptr;
  size_t stage_bytes = 0;  // bytes of one slot
  unsigned long long host_calls = 0;
  cudaStream_t s_in = nullptr, s_out = nullptr;
  cudaEvent_t ev_in[kHostChunks] = {}, ev_out[kHostChunks] = {}, ev_zfree[2] = {}, ev_dfree[2] = {}, ev_done = nullptr;
  // optional per-stage timing events (trimul_set_stage_events)
  cudaEvent_t ev[4] = {nullptr, nullptr, nullptr, nullptr};
  bool timing = false;
  // backward: bf16 weights (raw, and with the LayerNorm gamma folded in), the
  // folded LayerNorm betas t = W beta (fp32), raw W_o in fp32, and a workspace
  int gemm_pairs = 0;            // co-resident CTA pairs of the backward GEMM
  uint16_t* bw = nullptr;        // one allocation holding the bf16 matrices below
  uint16_t* bw_in = nullptr;  // [4C][D]: W_a, W_ga, W_b, W_gb stacked (raw)
  uint16_t *bw_g = nullptr, *bw_o = nullptr;      // raw W_g [D][D], W_o [D][C]
  uint16_t* bw_o_t = nullptr;                     // W_o diag(gamma_out) [D][C]
  float* bf = nullptr;                            // fp32: t_g [D], t_o [D], W_o [D][C]
  float *bt_g = nullptr, *bt_o = nullptr, *bw_o_f32 = nullptr;
  char* bws = nullptr;           // backward workspace
  size_t bws_bytes = 0;
  bool log = false;              // TRIMUL_LOG set (not "0") at create: one stderr line per launch
};

namespace {

// One line on stderr, when the handle was created with TRIMUL_LOG set.
void tlog(trimul_handle h, const char* fmt, ...) {
  if (!h->log) return;
  char buf[320];
  va_list ap;
  va_start(ap, fmt);
  std::vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  std::fprintf(stderr, "trimul: %s\n", buf);
}

const char* out_kind_name(int k) {
  return k == INPROJ_OUT_BF16 ? "bf16" : k == INPROJ_OUT_E4M3 ? "e4m3" : "f16";
}

trimul_status check_handle(trimul_handle h) {
  if (!h) return fail(TRIMUL_ERR_INVALID_ARG, "null handle");
  return TRIMUL_OK;
}

trimul_status check_sizes(trimul_handle h, int B, int N) {
  if (B < 1 || N < 1) return fail(TRIMUL_ERR_SHAPE, "B (%d) and N (%d) must be >= 1", B, N);
  if (N % 8 != 0) return fail(TRIMUL_ERR_SHAPE, "N (%d) must be a multiple of 8", N);
  const long long NN = static_cast<long long>(N) * N;
  if (NN > (1ll << 31) || static_cast<long long>(B) * h->C > (1 << 30))
    return fail(TRIMUL_ERR_SHAPE, "B=%d N=%d is too large", B, N);
  return TRIMUL_OK;
}

trimul_status use_device(trimul_handle h) {
  TRY_CUDA(cudaSetDevice(h->device), "cudaSetDevice");
  return TRIMUL_OK;
}

// Bytes of workspace one forward of B x N needs: a, b, x and the LN_in statistics.
size_t workspace_bytes(trimul_handle h, int B, int N) {
  const size_t nn = static_cast<size_t>(N) * N;
  return 3 * static_cast<size_t>(B) * h->C * nn * sizeof(uint16_t) + static_cast<size_t>(B) * nn * sizeof(float2);
}

trimul_status ensure_workspace(trimul_handle h, int B, int N) {
  const size_t need = workspace_bytes(h, B, N);
  if (need <= h->ws_bytes) return TRIMUL_OK;
  uint16_t* p = nullptr;
  cudaError_t e = cudaMalloc(&p, need);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return cuda_fail(e, "workspace allocation");
  }
  if (h->ws) {
    cudaDeviceSynchronize();
    cudaFree(h->ws);
  }
  h->ws = p;
  h->ws_bytes = need;
  return TRIMUL_OK;
}

// The scale of the stage-2 entry point, whose a and b come from the caller: x
// is stored as fp16 scaled by 2^-s with |x| <= N * ab_bound^2 (a sum of N
// products of values bounded by the handle's bound), so 2^-s brings that bound
// under 32768.  The forward entry points instead derive s on the device from
// the call's own max |a|, |b| (x_scale_log2_from_max): the handle's bound can
// be loose by orders of magnitude, and a loose s pushes small x into the
// binary16 subnormals.
int x_scale_log2(trimul_handle h, int N) {
  const double bound = static_cast<double>(N) * h->ab_bound * h->ab_bound;
  int s = 0;
  while (s < 40 && bound * std::ldexp(1.0, -s) > 32768.0) ++s;
  return s;
}

unsigned long long timeout_for(unsigned flags) {
  return (flags & TRIMUL_FLAG_INJECT_STALL) ? kStallTimeoutNs : kDefaultTimeoutNs;
}

// Bytes of the status words cleared at the start of every call.
constexpr size_t kStatusBytes = 16;

trimul_status reset_status(trimul_handle h, cudaStream_t s) {
  TRY_CUDA(cudaMemsetAsync(h->status, 0, kStatusBytes, s), "status reset");
  return TRIMUL_OK;
}

trimul_status finish(trimul_handle h, cudaStream_t s, unsigned flags) {
  TRY_CUDA(cudaGetLastError(), "kernel launch");
  if (!(flags & TRIMUL_FLAG_CHECK)) return TRIMUL_OK;
  TRY_CUDA(cudaStreamSynchronize(s), "stream synchronize");
  int word[2] = {0, 0};
  TRY_CUDA(cudaMemcpy(word, h->status, sizeof(word), cudaMemcpyDeviceToHost), "status read");
  if (word[0] != 0 || word[1] != 0) cudaMemset(h->status, 0, sizeof(word));
  if (word[0] != 0) return fail(TRIMUL_ERR_TIMEOUT, "a kernel gave up on a bounded wait (site 0x%x)", word[0]);
  if (word[1] != 0)
    return fail(TRIMUL_ERR_INVALID_ARG, "a mask value lies outside [0, 1] (or is NaN): the result is undefined");
  return TRIMUL_OK;
}

unsigned* ab_max_word(trimul_handle h) { return reinterpret_cast<unsigned*>(h->status + 2); }

// ------------------------------------------------------------------ stage launches
// Stage launchers.  tile_begin / tile_end (end -1: all tiles) restrict a launch
// to a range of its tiles (INPROJ_TILE_PAIRS pairs for the input projection,
// 128 for the output projection), for the host-buffer path that overlaps
// copies with compute chunk by chunk.
// data_scale: record max |a|, |b| for the triangle GEMM's per-call x scale.
// out_kind: how a and b are stored (INPROJ_OUT_F16; INPROJ_OUT_BF16 for the
// backward's planes; INPROJ_OUT_E4M3 for the 8-bit triangle path, bytes).
// The 8-bit path's scale of a and b: the largest power of two that keeps the
// layer's bound on |a|, |b| (from the weights, computed at create) within
// e4m3's largest finite value, 448.
double fp8_scale_of(trimul_handle h) {
  if (!(h->ab_bound > 0.0)) return 1.0;
  return std::ldexp(1.0, static_cast<int>(std::floor(std::log2(448.0 / h->ab_bound))));
}

trimul_status run_inproj(trimul_handle h, const uint16_t* z, const uint16_t* mask, int B, int N, uint16_t* a,
                         uint16_t* b, float2* zstats, bool data_scale, cudaStream_t s, unsigned flags,
                         int tile_begin = 0, int tile_end = -1, int out_kind = INPROJ_OUT_F16,
                         uint16_t* zhat = nullptr) {
  InprojArgs p{};
  p.B = B;
  p.N = N;
  p.D = h->D;
  p.C = h->C;
  p.NN = static_cast<long long>(N) * N;
  p.k_slabs = (h->D + 63) / 64;
  p.n_chunks = h->n_chunks;
  p.tiles_per_batch = static_cast<int>((p.NN + INPROJ_TILE_PAIRS - 1) / INPROJ_TILE_PAIRS);
  p.tile_begin = tile_begin;
  p.tile_end = tile_end < 0 ? p.tiles_per_batch * B : tile_end;
  p.w_stages = h->in_w_stages;
  p.z_bufs = h->in_z_bufs;
  p.w_resident = h->in_w_resident;
  p.inject_stall = (flags & TRIMUL_FLAG_INJECT_STALL) ? 1 : 0;
  p.out_kind = out_kind;
  p.fp8_scale = static_cast<float>(fp8_scale_of(h));
  p.mask = reinterpret_cast<const __nv_bfloat16*>(mask);
  p.bias = h->in_bias;
  p.eps = h->eps;
  p.a = reinterpret_cast<__half*>(a);
  p.b = reinterpret_cast<__half*>(b);
  p.zstats = zstats;
  p.ab_max = data_scale ? ab_max_word(h) : nullptr;
  p.mask_flag = h->status + 1;
  p.status = h->status;
  p.timeout_ns = timeout_for(flags);
  if (p.w_stages < (p.w_resident ? 1 : 2) || p.z_bufs < 2)
    return fail(TRIMUL_ERR_SHAPE, "not enough shared memory for the input projection");

  CUtensorMap tz, tw;
  const uint64_t zd[3] = {static_cast<uint64_t>(h->D), static_cast<uint64_t>(p.NN), static_cast<uint64_t>(B)};
  const uint32_t zb[3] = {64, INPROJ_HALF_PAIRS, 1};  // one CTA's half tile: 128 pairs x 64 channels
  trimul_status st = make_map(&tz, true, 3, z, zd, zb, "z");
  if (st != TRIMUL_OK) return st;
  const uint64_t wd[2] = {static_cast<uint64_t>(h->D), static_cast<uint64_t>(h->n_chunks) * 256};
  const uint32_t wb[2] = {64, 128};  // one CTA's 128 rows of a chunk
  // bf16 weights with bf16 LayerNorm output for the backward's recompute, fp16 otherwise
  if (out_kind == INPROJ_OUT_BF16) {
    if ((st = make_map(&tw, true, 2, h->w_in_bf, wd, wb, "input weights (bf16)")) != TRIMUL_OK) return st;
  } else if ((st = make_map(&tw, false, 2, h->w_in, wd, wb, "input weights")) != TRIMUL_OK) {
    return st;
  }
  // zh = (z - mean) rstd (bf16, z's layout), stored from the LayerNorm's buffer
  CUtensorMap tzh = tz;
  p.write_zhat = (zhat && out_kind == INPROJ_OUT_BF16) ? 1 : 0;
  if (p.write_zhat && (st = make_map(&tzh, true, 3, zhat, zd, zb, "zh")) != TRIMUL_OK) return st;
  // channel-major outputs, stored as 16-channel (or, at the a / b boundary,
  // 8-channel) x 64-pair boxes
  CUtensorMap ta, tb, ta8, tb8;
  const uint64_t od[3] = {static_cast<uint64_t>(p.NN), static_cast<uint64_t>(h->C), static_cast<uint64_t>(B)};
  const uint32_t ob[3] = {64, 16, 1}, ob8[3] = {64, 8, 1};
  if (out_kind == INPROJ_OUT_E4M3) {
    if ((st = make_map_u8(&ta, false, 3, a, od, ob, "a")) != TRIMUL_OK) return st;
    if ((st = make_map_u8(&tb, false, 3, b, od, ob, "b")) != TRIMUL_OK) return st;
    if ((st = make_map_u8(&ta8, false, 3, a, od, ob8, "a")) != TRIMUL_OK) return st;
    if ((st = make_map_u8(&tb8, false, 3, b, od, ob8, "b")) != TRIMUL_OK) return st;
  } else {
    const bool bf = out_kind == INPROJ_OUT_BF16;
    if ((st = make_map(&ta, bf, 3, a, od, ob, "a")) != TRIMUL_OK) return st;
    if ((st = make_map(&tb, bf, 3, b, od, ob, "b")) != TRIMUL_OK) return st;
    if ((st = make_map(&ta8, bf, 3, a, od, ob8, "a")) != TRIMUL_OK) return st;
    if ((st = make_map(&tb8, bf, 3, b, od, ob8, "b")) != TRIMUL_OK) return st;
  }
  const int grid = 2 * static_cast<int>(std::min<long long>(p.tile_end - p.tile_begin, h->in_pairs));
  tlog(h, "k1_inproj B=%d N=%d tiles [%d, %d) of %d pairs, grid %d (pairs of 2), weight stages %d%s, z buffers %d, "
          "out %s%s",
       B, N, p.tile_begin, p.tile_end, INPROJ_TILE_PAIRS, grid, p.w_stages, p.w_resident ? " (resident)" : "",
       p.z_bufs, out_kind_name(out_kind), p.write_zhat ? " + zh" : "");
  TRY_CUDA(launch_inproj(p, tz, tw, ta, tb, ta8, tb8, tzh, grid, s), "input projection launch");
  return TRIMUL_OK;
}

// The backward of the gated input projections from the normalised z (zh) and
// the gradients of a and b: dP (bf16 [B][4C][NN]) and the per-tile row sums.
trimul_status run_gate_grad(trimul_handle h, const uint16_t* zh, const uint16_t* mask, const uint16_t* da,
                            const uint16_t* db, int B, int N, uint16_t* dp, float* rowpart, cudaStream_t s,
                            unsigned flags) {
  GateGradArgs p{};
  p.B = B;
  p.N = N;
  p.D = h->D;
  p.C = h->C;
  p.NN = static_cast<long long>(N) * N;
  p.k_slabs = (h->D + 63) / 64;
  p.n_chunks = h->n_chunks;
  p.tiles_per_batch = static_cast<int>((p.NN + INPROJ_TILE_PAIRS - 1) / INPROJ_TILE_PAIRS);
  p.tile_begin = 0;
  p.tile_end = p.tiles_per_batch * B;
  p.w_stages = h->in_w_stages;
  p.z_bufs = h->in_z_bufs;
  p.w_resident = h->in_w_resident;
  p.mask = reinterpret_cast<const __nv_bfloat16*>(mask);
  p.bias = h->in_bias;
  p.da = reinterpret_cast<const __nv_bfloat16*>(da);
  p.db = reinterpret_cast<const __nv_bfloat16*>(db);
  p.rowpart = rowpart;
  p.status = h->status;
  p.timeout_ns = timeout_for(flags);
  if (p.w_stages < (p.w_resident ? 1 : 2) || p.z_bufs < 2)
    return fail(TRIMUL_ERR_SHAPE, "not enough shared memory for the gate gradients");
  CUtensorMap tz, tw, tp8;
  const uint64_t zd[3] = {static_cast<uint64_t>(h->D), static_cast<uint64_t>(p.NN), static_cast<uint64_t>(B)};
  const uint32_t zb[3] = {64, INPROJ_HALF_PAIRS, 1};
  trimul_status st = make_map(&tz, true, 3, zh, zd, zb, "zh");
  if (st != TRIMUL_OK) return st;
  const uint64_t wd[2] = {static_cast<uint64_t>(h->D), static_cast<uint64_t>(h->n_chunks) * 256};
  const uint32_t wb[2] = {64, 128};
  if ((st = make_map(&tw, true, 2, h->w_in_bf, wd, wb, "input weights (bf16)")) != TRIMUL_OK) return st;
  const uint64_t pd[3] = {static_cast<uint64_t>(p.NN), static_cast<uint64_t>(4 * h->C), static_cast<uint64_t>(B)};
  const uint32_t pb8[3] = {64, 8, 1};  // 8 rows (channels) x 64 pairs
  if ((st = make_map(&tp8, true, 3, dp, pd, pb8, "dP")) != TRIMUL_OK) return st;
  const int grid = 2 * static_cast<int>(std::min<long long>(p.tile_end, h->gg_pairs));
  tlog(h, "k6_gate_grad B=%d N=%d tiles %d, grid %d (pairs of 2)", B, N, p.tile_end, grid);
  TRY_CUDA(launch_gate_grad(p, tz, tw, tp8, grid, s), "gate gradient launch");
  return TRIMUL_OK;
}

// The triangle GEMM runs as several launches over consecutive groups of
// planes, about kTriTilesPerPair tiles per CTA pair each.  Within one long
// launch the CTA pairs drift apart, the tiles in flight spread over several
// planes, and their a and b panels no longer fit in L2 together (at N = 4096,
// C = 256 one launch re-read the operands 3.5-4.6 times; launches of ~30
// planes read them 1.7 times and ran 6% faster).  Each launch starts its pairs
// together.  (Tiles handed out from a global counter kept the pairs on one
// plane and the reads at 1.05-1.07 times the operands, but cost 2-20% of the
// kernel's time in the queue that publishes them.)
constexpr long long kTriTilesPerPair = 100;

// Planes per triangle launch, and the number of launches, for B x N.
void triangle_groups(trimul_handle h, int B, int N, int* planes_per_launch, int* launches) {
  const int planes = B * h->C;
  const long long per_plane = static_cast<long long>((N + 255) / 256) * ((N + 255) / 256);
  const long long want = std::max<long long>(1, (h->tri_pairs * kTriTilesPerPair) / per_plane);
  const int n = static_cast<int>((planes + want - 1) / want);
  *planes_per_launch = (planes + n - 1) / n;
  *launches = (planes + *planes_per_launch - 1) / *planes_per_launch;
}

// data_scale: x is stored with the scale derived from this call's max |a|, |b|
// (recorded by run_inproj), else with the handle's bound (trimul_x_scale_log2).
// bf16: a and b are bf16 planes (the backward's), else fp16.
// The triangle kernel for either direction (dir) or, with explicit majors
// (a_mn / b_mn >= 0), for any operand-major pair (the backward's gradients).
trimul_status run_triangle(trimul_handle h, const uint16_t* a, const uint16_t* b, int B, int N,
                           trimul_direction dir, uint16_t* x, bool data_scale, cudaStream_t s, unsigned flags,
                           bool bf16 = false, bool fp8 = false, bool out_bf16 = false, int a_mn = -1,
                           int b_mn = -1) {
  TriangleArgs p{};
  p.N = N;
  p.planes = B * h->C;
  p.tiles_m = (N + 255) / 256;
  p.tiles_n = (N + 255) / 256;
  const int bk = fp8 ? 2 * TRI_BK : TRI_BK;  // K elements per stage
  p.k_iters = (N + bk - 1) / bk;
  p.fp8 = fp8 ? 1 : 0;
  p.a_mn = a_mn >= 0 ? a_mn : (dir == TRIMUL_INCOMING ? 1 : 0);
  p.b_mn = b_mn >= 0 ? b_mn : (dir == TRIMUL_INCOMING ? 1 : 0);
  if (fp8) {
    if (p.a_mn || p.b_mn) return fail(TRIMUL_ERR_INVALID_ARG, "the 8-bit triangle path is outgoing only");
    const double s8 = fp8_scale_of(h);
    p.fp8_descale = static_cast<float>(1.0 / (s8 * s8));
  }
  p.inject_stall = (flags & TRIMUL_FLAG_INJECT_STALL) ? 1 : 0;
  p.bf16 = bf16 ? 1 : 0;
  p.out_bf16 = out_bf16 ? 1 : 0;
  p.x = reinterpret_cast<__half*>(x);
  p.x_scale = static_cast<float>(std::ldexp(1.0, -x_scale_log2(h, N)));
  p.ab_max = data_scale ? ab_max_word(h) : nullptr;
  p.status = h->status;
  p.timeout_ns = timeout_for(flags);
  CUtensorMap ta, tb;
  const uint64_t d[3] = {static_cast<uint64_t>(N), static_cast<uint64_t>(N), static_cast<uint64_t>(p.planes)};
  // per CTA and K block: TRI_ROWS rows of A and of B; a K-major operand is
  // one TMA box of TRI_ROWS x TRI_BK, an MN-major one TRI_ROWS / 64 boxes of 64 x TRI_BK
  const uint32_t box_k[3] = {static_cast<uint32_t>(TRI_BK), static_cast<uint32_t>(TRI_ROWS), 1};
  const uint32_t box_mn[3] = {64, static_cast<uint32_t>(TRI_BK), 1};
  if (2u * box_k[0] * box_k[1] * 2u != TRI_STAGE_BYTES ||
      2u * (TRI_ROWS / 64) * box_mn[0] * box_mn[1] * 2u != TRI_STAGE_BYTES)
    return fail(TRIMUL_ERR_INVALID_ARG, "internal: triangle TMA boxes do not match the stage size");
  const uint32_t* boxa = p.a_mn ? box_mn : box_k;
  const uint32_t* boxb = p.b_mn ? box_mn : box_k;
  trimul_status st;
  if (fp8) {  // one box of 128 rows x 128 bytes (= 128 K elements) per operand, CTA and stage
    const uint32_t box8[3] = {static_cast<uint32_t>(2 * TRI_BK), static_cast<uint32_t>(TRI_ROWS), 1};
    if (2u * box8[0] * box8[1] != TRI_STAGE_BYTES)
      return fail(TRIMUL_ERR_INVALID_ARG, "internal: 8-bit triangle TMA boxes do not match the stage size");
    if ((st = make_map_u8(&ta, true, 3, a, d, box8, "a (e4m3)")) != TRIMUL_OK) return st;
    if ((st = make_map_u8(&tb, true, 3, b, d, box8, "b (e4m3)")) != TRIMUL_OK) return st;
  } else {
    if ((st = make_map(&ta, bf16, 3, a, d, boxa, "a")) != TRIMUL_OK) return st;
    if ((st = make_map(&tb, bf16, 3, b, d, boxb, "b")) != TRIMUL_OK) return st;
  }
  const int per_plane = p.tiles_m * p.tiles_n;
  int group = 0, launches = 0;
  triangle_groups(h, B, N, &group, &launches);
  for (int p0 = 0; p0 < p.planes; p0 += group) {
    const int p1 = std::min(p.planes, p0 + group);
    p.tile_begin = p0 * per_plane;
    p.tile_end = p1 * per_plane;
    const long long n = static_cast<long long>(p.tile_end - p.tile_begin);
    const int grid = 2 * static_cast<int>(std::min<long long>(n, h->tri_pairs));
    tlog(h,
         "k2_triangle N=%d planes [%d, %d) tiles [%d, %d) of 256x256, grid %d (pairs of 2), k blocks %d, "
         "majors a=%s b=%s, %s operands, %s out",
         N, p0, p1, p.tile_begin, p.tile_end, grid, p.k_iters, p.a_mn ? "mn" : "k", p.b_mn ? "mn" : "k",
         fp8 ? "e4m3" : bf16 ? "bf16" : "f16", out_bf16 ? "bf16" : "f16 scaled");
    TRY_CUDA(launch_triangle(p, ta, tb, grid, s), "triangle launch");
  }
  return TRIMUL_OK;
}

trimul_status run_outproj(trimul_handle h, const uint16_t* x, const uint16_t* z, const float2* zstats, int B, int N,
                          uint16_t* out, bool data_scale, cudaStream_t s, unsigned flags, int tile_begin = 0,
                          int tile_end = -1) {
  OutprojArgs p{};
  p.B = B;
  p.N = N;
  p.D = h->D;
  p.C = h->C;
  p.NN = static_cast<long long>(N) * N;
  p.x_slabs = (h->C + 63) / 64;
  p.z_slabs = (h->D + 63) / 64;
  p.tiles_per_batch = static_cast<int>((p.NN + 127) / 128);
  p.tile_begin = tile_begin;
  p.tile_end = tile_end < 0 ? p.tiles_per_batch * B : tile_end;
  // Weight ring: about 96 KB (3 slabs at D = 256); the activation ring takes
  // what is left, up to 8 slabs of 16 KB.
  const size_t wsb = outproj_w_stage_bytes(h->D);
  p.w_stages = static_cast<int>(std::min<size_t>(MAX_OUTPROJ_W_STAGES, std::max<size_t>(2, 98304 / wsb)));
  const size_t fixed = outproj_smem_bytes(0, p.w_stages, h->D);
  p.a_stages = static_cast<int>(std::min<size_t>(
      MAX_OUTPROJ_A_STAGES, static_cast<size_t>(h->max_smem) > fixed ? (h->max_smem - fixed) / (128 * 128) : 0));
  p.inject_stall = (flags & TRIMUL_FLAG_INJECT_STALL) ? 1 : 0;
  p.eps = h->eps;
  p.out = reinterpret_cast<__nv_bfloat16*>(out);
  p.zstats = zstats;
  p.colc = h->colc;
  {
    const double xs = std::ldexp(1.0, -x_scale_log2(h, N));
    p.eps_x = static_cast<float>(h->eps * xs * xs);  // LN of x * 2^-s with eps * 4^-s equals LN of x with eps
  }
  p.ab_max = data_scale ? ab_max_word(h) : nullptr;
  p.status = h->status;
  p.timeout_ns = timeout_for(flags);
  if (p.a_stages < 2) return fail(TRIMUL_ERR_SHAPE, "not enough shared memory for the output projection");
  CUtensorMap tx, tz, twg, two;
  const uint64_t xd[3] = {static_cast<uint64_t>(p.NN), static_cast<uint64_t>(h->C), static_cast<uint64_t>(B)};
  const uint32_t xb[3] = {64, 64, 1};
  trimul_status st = make_map(&tx, false, 3, x, xd, xb, "x");
  if (st != TRIMUL_OK) return st;
  const uint64_t zd[3] = {static_cast<uint64_t>(h->D), static_cast<uint64_t>(p.NN), static_cast<uint64_t>(B)};
  const uint32_t zb[3] = {64, 128, 1};
  if ((st = make_map(&tz, true, 3, z, zd, zb, "z")) != TRIMUL_OK) return st;
  const uint64_t gd[2] = {static_cast<uint64_t>(h->D), static_cast<uint64_t>(h->D)};
  const uint64_t od[2] = {static_cast<uint64_t>(h->C), static_cast<uint64_t>(h->D)};
  const uint32_t wb[2] = {64, static_cast<uint32_t>((h->D + 15) / 16 * 16)};  // one weight slab: all D rows x 64 K
  if ((st = make_map(&twg, true, 2, h->w_g, gd, wb, "gate weights")) != TRIMUL_OK) return st;
  if ((st = make_map(&two, false, 2, h->w_o, od, wb, "output weights")) != TRIMUL_OK) return st;
  CUtensorMap tout;
  const uint32_t ob[3] = {32, 32, 1};  // one epilogue store: 32 pair rows x 32 features, 64-byte swizzle
  if ((st = make_map_any(&tout, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, CU_TENSOR_MAP_SWIZZLE_64B, 3, out, zd, ob, "out")) !=
      TRIMUL_OK)
    return st;
  const int grid = std::min(p.tile_end - p.tile_begin, h->num_sms);
  tlog(h, "k3_outproj B=%d N=%d tiles [%d, %d) of 128 pairs, grid %d, activation stages %d, weight stages %d", B, N,
       p.tile_begin, p.tile_end, grid, p.a_stages, p.w_stages);
  TRY_CUDA(launch_outproj(p, tx, tz, twg, two, tout, grid, s), "output projection launch");
  return TRIMUL_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// ------------------------------------------------------------------ backward GEMMs
// One bf16 operand of k4_gemm: a matrix of `rows` (the M or N extent) by `k`,
// K-major ([rows][k]) or MN-major ([k][rows]), per batch (dense, `batches`
// of them) or one matrix for all.
struct Operand {
  const void* ptr;
  bool mn;
  bool batched;
  long long rows, k;
};

trimul_status operand_map(CUtensorMap* m, const Operand& o, int batches, const char* what) {
  const uint64_t r = static_cast<uint64_t>(o.rows), k = static_cast<uint64_t>(o.k);
  const uint64_t dims_k[3] = {k, r, static_cast<uint64_t>(batches)};
  const uint64_t dims_mn[3] = {r, k, static_cast<uint64_t>(batches)};
  const uint32_t box_k[3] = {64, 128, 1}, box_mn[3] = {64, 64, 1};
  return make_map(m, true, o.batched ? 3 : 2, o.ptr, o.mn ? dims_mn : dims_k, o.mn ? box_mn : box_k, what);
}

// K-split slices of a split-K GEMM of M x N over batches * ceil(K / 64) blocks:
// about one tile per co-resident CTA pair.
int gemm_split_slices(trimul_handle h, int M, int N, long long K, int batches, long long* kb_per_z) {
  const long long tiles_mn = static_cast<long long>((M + 255) / 256) * ((N + 255) / 256);
  const long long kb_total = static_cast<long long>(batches) * ((K + 63) / 64);
  const long long want = std::max<long long>(1, std::min<long long>(kb_total, h->gemm_pairs / tiles_mn));
  *kb_per_z = (kb_total + want - 1) / want;
  return static_cast<int>((kb_total + *kb_per_z - 1) / *kb_per_z);
}

// C = sum_k A(m, k) B(n, k): per batch (split = false: slice z = batch z, c
// holds `batches` outputs c_zstride apart) or split over batches and K
// (split = true: c holds gemm_split_slices(...) fp32 partials of M x N).
trimul_status run_gemm(trimul_handle h, const Operand& A, const Operand& Bop, int M, int N, long long K, int batches,
                       bool split, int out_mode, void* c, long long ldc, long long c_zstride, cudaStream_t s,
                       unsigned flags) {
  GemmArgs p{};
  p.M = M;
  p.N = N;
  p.kpb = static_cast<int>((K + 63) / 64);
  p.batches = batches;
  if (split) {
    p.n_z = gemm_split_slices(h, M, N, K, batches, &p.kb_per_z);
  } else {
    p.n_z = batches;
    p.kb_per_z = p.kpb;
  }
  p.tiles_m = (M + 255) / 256;
  p.tiles_n = (N + 255) / 256;
  p.a_mn = A.mn;
  p.b_mn = Bop.mn;
  p.a_batched = A.batched;
  p.b_batched = Bop.batched;
  p.bf16 = 1;
  p.out_mode = out_mode;
  p.m_fastest = (p.tiles_m > 1 && p.tiles_n > 4 * p.tiles_m) ? 1 : 0;
  p.c = c;
  p.ldc = ldc;
  p.c_zstride = c_zstride;
  p.status = h->status;
  p.timeout_ns = timeout_for(flags);
  if (M % 8 || N % 8 || K % 8) return fail(TRIMUL_ERR_SHAPE, "internal: GEMM extents must be multiples of 8");
  CUtensorMap ta, tb;
  trimul_status st = operand_map(&ta, A, batches, "GEMM operand A");
  if (st != TRIMUL_OK) return st;
  if ((st = operand_map(&tb, Bop, batches, "GEMM operand B")) != TRIMUL_OK) return st;
  // Launches of about kTriTilesPerPair tiles per CTA pair, in whole slices
  // where a slice is smaller: the pairs of a launch start together and work
  // on nearby slices, whose operands then share L2 (as for the triangle GEMM).
  const long long per_z = static_cast<long long>(p.tiles_m) * p.tiles_n;
  const long long total = per_z * p.n_z;
  long long group = std::max<long long>(1, static_cast<long long>(h->gemm_pairs) * kTriTilesPerPair);
  if (per_z < group) group = (group / per_z) * per_z;
  for (long long t0 = 0; t0 < total; t0 += group) {
    p.tile_begin = static_cast<int>(t0);
    p.tile_end = static_cast<int>(std::min(total, t0 + group));
    const int grid = 2 * static_cast<int>(std::min<long long>(p.tile_end - p.tile_begin, h->gemm_pairs));
    tlog(h, "k4_gemm M=%d N=%d K=%lld x%d%s tiles [%d, %d), grid %d (pairs of 2), majors a=%s b=%s, out mode %d", M, N,
         K, batches, split ? " split" : "", p.tile_begin, p.tile_end, grid, A.mn ? "mn" : "k", Bop.mn ? "mn" : "k",
         out_mode);
    TRY_CUDA(launch_gemm(p, ta, tb, grid, s), "backward GEMM launch");
  }
  return TRIMUL_OK;
}

// The backward workspace: byte offsets of every plane for B x N.  Regions are
// reused once their first tenant is dead (see trimul_backward).
struct BwdPlan {
  size_t ab, x, zstats, zh, xh, xstats, g, v, dyt, dzp, dzin, dvg, dv, dg, da, db, pt;
  size_t part_dout, part_gate, part_lnin, part_mo, part_mg, part_min, mo, mg, min_, cs, lnin, rowpart, rowtmp, total;
  int nz_o, nz_g, nz_in, dout_blk, nseg, lnin_blk, nslice;
};

BwdPlan backward_plan(trimul_handle h, int B, int N) {
  BwdPlan L{};
  const size_t P = static_cast<size_t>(N) * N, D = h->D, C = h->C, BP = static_cast<size_t>(B) * P;
  size_t o = 0;
  auto take = [&](size_t bytes) {
    const size_t at = o;
    o += (bytes + 255) / 256 * 256;
    return at;
  };
  L.ab = take(2 * B * C * P * 2);                       // a, b (bf16); later PT's first part is not here
  L.x = take(B * C * P * 2);                            // x (fp16, scaled)
  L.zstats = take(BP * 8);
  L.zh = take(BP * D * 2);
  L.xh = take(B * C * P * 2);                           // xh, then dx
  L.xstats = take(BP * 8);
  // two fp32-sized slots: gacc | vacc (fp16 [BP][D] each), then dy^T (bf16 [B][C][P]) | dz'
  // of the gate path ([BP][D]), then dz' of the input projections | (dz')
  const size_t slot = std::max(BP * D, static_cast<size_t>(B) * C * P) * 4;
  const size_t greg = take(2 * slot);
  L.g = greg;
  L.v = greg + slot;
  L.dyt = greg;
  L.dzp = greg + slot;
  L.dzin = greg;  // dy^T is dead once LN_out's backward has run
  // dv | dg (bf16 [BP][D] each), then da | db (bf16 [B][C][P] each)
  const size_t vsz = 2 * BP * std::max(C, D) * 2;
  L.dvg = take(vsz);
  L.dv = L.dvg;
  L.dg = L.dvg + BP * D * 2;
  L.da = L.dvg;
  L.db = L.dvg + B * C * P * 2;
  L.pt = take(B * 4 * C * P * 2);                       // gradients of the pre-activations
  long long kbz;
  L.nz_o = gemm_split_slices(h, h->D, h->C, static_cast<long long>(P), B, &kbz);
  L.nz_g = gemm_split_slices(h, h->D, h->D, static_cast<long long>(P), B, &kbz);
  L.nz_in = gemm_split_slices(h, 4 * h->C, h->D, static_cast<long long>(P), B, &kbz);
  L.dout_blk = dout_blocks(static_cast<long long>(BP), h->D, h->num_sms);
  L.nseg = 1;  // the gate-gradient row sums arrive reduced
  const int tpb = static_cast<int>((P + INPROJ_TILE_PAIRS - 1) / INPROJ_TILE_PAIRS);
  L.nslice = std::min(tpb, 256);
  L.lnin_blk = lnin_blocks(static_cast<long long>(BP), h->num_sms);
  L.part_dout = take(static_cast<size_t>(L.dout_blk) * 2 * D * 4);
  L.part_gate = take(static_cast<size_t>(B) * C * L.nseg * 4 * 4);
  L.rowpart = take(static_cast<size_t>(B) * tpb * h->n_chunks * 1024 * 4);
  L.rowtmp = take(static_cast<size_t>(B) * L.nslice * h->n_chunks * 1024 * 4);
  L.part_lnin = take(static_cast<size_t>(L.lnin_blk) * 2 * D * 4);
  L.part_mo = take(static_cast<size_t>(L.nz_o) * D * C * 4);
  L.part_mg = take(static_cast<size_t>(L.nz_g) * D * D * 4);
  L.part_min = take(static_cast<size_t>(L.nz_in) * 4 * C * D * 4);
  L.mo = take(D * C * 4);
  L.mg = take(D * D * 4);
  L.min_ = take(4 * C * D * 4);
  L.cs = take(2 * D * 4);
  L.lnin = take(2 * D * 4);
  L.total = o;
  return L;
}

trimul_status ensure_backward_workspace(trimul_handle h, size_t need) {
  if (need <= h->bws_bytes) return TRIMUL_OK;
  char* p = nullptr;
  cudaError_t e = cudaMalloc(&p, need);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return cuda_fail(e, "backward workspace allocation");
  }
  if (h->bws) {
    cudaDeviceSynchronize();
    cudaFree(h->bws);
  }
  h->bws = p;
  h->bws_bytes = need;
  return TRIMUL_OK;
}

}  // namespace

// ==================================================================== C ABI

// ------------------------------------------------------------------ fixed scratch
// Scratch for trimul_forward_noalloc: the a, b and x planes of one call live
// here instead of in a workspace allocated by the handle.  The array is part
// of this library's device image, so every GPU that loads the library holds
// kNoAllocScratchBytes of it until the process exits.
namespace {
constexpr size_t kNoAllocScratchBytes = size_t(64) << 20;  // 64 MiB
}
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

namespace {
constexpr int kMaxDevices = 64;
std::mutex g_noalloc_mu;
void* g_noalloc_dev_ptr[kMaxDevices] = {};

// Device address of g_noalloc_scratch on `device`, which must be current.  In
// host code the array's name only stands in for the symbol; the address the
// kernels need comes from cudaGetSymbolAddress, looked up once per device.
trimul_status noalloc_scratch(int device, uint16_t** out) {
  if (device < 0 || device >= kMaxDevices)
    return fail(TRIMUL_ERR_INVALID_ARG, "device %d is outside the fixed-scratch table", device);
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  if (!g_noalloc_dev_ptr[device]) {
    void* ptr = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&ptr, g_noalloc_scratch);
    if (e != cudaSuccess || !ptr) {
      cudaGetLastError();
      return fail(TRIMUL_ERR_CUDA, "cudaGetSymbolAddress of the fixed scratch failed: %s",
                  cudaGetErrorString(e == cudaSuccess ? cudaErrorInvalidSymbol : e));
    }
    g_noalloc_dev_ptr[device] = ptr;
  }
  *out = static_cast<uint16_t*>(g_noalloc_dev_ptr[device]);
  return TRIMUL_OK;
}
}  // namespace

extern "C" {

const char* trimul_last_error(void) { return g_err; }

int trimul_kernels_per_forward(trimul_handle h, int B, int N) {
  if (!h || B < 1 || N < 1) {
    fail(TRIMUL_ERR_INVALID_ARG, "null handle or empty shape");
    return -1;
  }
  int group = 0, launches = 0;
  triangle_groups(h, B, N, &group, &launches);
  return 2 + launches;
}

int trimul_kernels_per_forward_host(trimul_handle h, int B, int N) {
  if (!h || B < 1 || N < 1) {
    fail(TRIMUL_ERR_INVALID_ARG, "null handle or empty shape");
    return -1;
  }
  const long long NN = static_cast<long long>(N) * N;
  const long long total = ((NN + INPROJ_TILE_PAIRS - 1) / INPROJ_TILE_PAIRS) * B;
  const size_t zbytes = static_cast<size_t>(B) * NN * h->D * 2;
  const long long chunks = zbytes >= kHostChunkMin ? std::min<long long>(kHostChunks, total) : 1;
  int group = 0, launches = 0;
  triangle_groups(h, B, N, &group, &launches);
  return static_cast<int>(2 * chunks + launches);
}

trimul_status trimul_create(trimul_handle* out, const trimul_params* p, int device) {
  if (!out) return fail(TRIMUL_ERR_INVALID_ARG, "out is null");
  *out = nullptr;
  if (!p) return fail(TRIMUL_ERR_INVALID_ARG, "params is null");
  if (p->D < 8 || p->D > 256 || p->D % 8 != 0)
    return fail(TRIMUL_ERR_SHAPE, "D (%d) must be a multiple of 8 in [8, 256]", p->D);
  if (p->C < 8 || p->C > 256 || p->C % 8 != 0)
    return fail(TRIMUL_ERR_SHAPE, "C (%d) must be a multiple of 8 in [8, 256]", p->C);
  if (!(p->eps > 0.0f) || !std::isfinite(p->eps)) return fail(TRIMUL_ERR_INVALID_ARG, "eps must be finite and > 0");
  const void* ptrs[] = {p->W_a, p->W_ga, p->W_b, p->W_gb, p->W_o, p->W_g,
                        p->ln_in_gamma, p->ln_in_beta, p->ln_out_gamma, p->ln_out_beta};
  for (const void* q : ptrs)
    if (!q) return fail(TRIMUL_ERR_INVALID_ARG, "a weight pointer is null");

  int ndev = 0;
  TRY_CUDA(cudaGetDeviceCount(&ndev), "cudaGetDeviceCount");
  if (device < 0 || device >= ndev) return fail(TRIMUL_ERR_INVALID_ARG, "device %d out of range (%d devices)", device, ndev);
  TRY_CUDA(cudaSetDevice(device), "cudaSetDevice");
  cudaDeviceProp prop;
  TRY_CUDA(cudaGetDeviceProperties(&prop, device), "cudaGetDeviceProperties");
  if (!(prop.major == 10 && prop.minor == 3))
    return fail(TRIMUL_ERR_UNSUPPORTED_ARCH, "TriMul kernels are built for sm_103 (GB300); got sm_%d%d", prop.major,
                prop.minor);

  const int D = p->D, C = p->C;
  // ---- fetch the caller's weights (device) to the host
  auto fetch16 = [&](const uint16_t* src, size_t n, std::vector<uint16_t>& dst) -> cudaError_t {
    dst.resize(n);
    return cudaMemcpy(dst.data(), src, n * 2, cudaMemcpyDeviceToHost);
  };
  auto fetch32 = [&](const float* src, size_t n, std::vector<float>& dst) -> cudaError_t {
    dst.resize(n);
    return cudaMemcpy(dst.data(), src, n * 4, cudaMemcpyDeviceToHost);
  };
  std::vector<uint16_t> Wa, Wga, Wb, Wgb, Wo, Wg;
  std::vector<float> gi, bi, go, bo;
  TRY_CUDA(fetch16(p->W_a, (size_t)C * D, Wa), "copy W_a");
  TRY_CUDA(fetch16(p->W_ga, (size_t)C * D, Wga), "copy W_ga");
  TRY_CUDA(fetch16(p->W_b, (size_t)C * D, Wb), "copy W_b");
  TRY_CUDA(fetch16(p->W_gb, (size_t)C * D, Wgb), "copy W_gb");
  TRY_CUDA(fetch16(p->W_o, (size_t)D * C, Wo), "copy W_o");
  TRY_CUDA(fetch16(p->W_g, (size_t)D * D, Wg), "copy W_g");
  TRY_CUDA(fetch32(p->ln_in_gamma, D, gi), "copy ln_in_gamma");
  TRY_CUDA(fetch32(p->ln_in_beta, D, bi), "copy ln_in_beta");
  TRY_CUDA(fetch32(p->ln_out_gamma, C, go), "copy ln_out_gamma");
  TRY_CUDA(fetch32(p->ln_out_beta, C, bo), "copy ln_out_beta");

  // ---- range checks for the binary16 operands
  for (const auto* w : {&Wa, &Wga, &Wb, &Wgb, &Wo, &Wg})
    for (uint16_t v : *w) {
      const float f = bf16_to_float(v);
      if (!std::isfinite(f) || std::fabs(f) > kHalfMax)
        return fail(TRIMUL_ERR_INVALID_ARG, "weight value %g is outside the binary16 range", f);
    }
  for (const auto* v : {&gi, &bi, &go, &bo})
    for (float f : *v)
      if (!std::isfinite(f)) return fail(TRIMUL_ERR_INVALID_ARG, "LayerNorm parameters must be finite");
  double gmax_in = 0, bnorm_in = 0, bmax_in = 0, gmax_out = 0, bmax_out = 0;
  for (int d = 0; d < D; ++d) {
    gmax_in = std::max(gmax_in, (double)std::fabs(gi[d]));
    bnorm_in += (double)bi[d] * bi[d];
    bmax_in = std::max(bmax_in, (double)std::fabs(bi[d]));
  }
  for (int c = 0; c < C; ++c) {
    gmax_out = std::max(gmax_out, (double)std::fabs(go[c]));
    bmax_out = std::max(bmax_out, (double)std::fabs(bo[c]));
  }
  bnorm_in = std::sqrt(bnorm_in);
  if (std::sqrt((double)D) * gmax_in + bmax_in > kHalfMax || std::sqrt((double)C) * gmax_out + bmax_out > kHalfMax)
    return fail(TRIMUL_ERR_INVALID_ARG, "LayerNorm outputs could exceed the binary16 range");
  double wrow = 0;
  for (const auto* w : {&Wa, &Wb})
    for (int c = 0; c < C; ++c) {
      double s = 0;
      for (int d = 0; d < D; ++d) {
        const double f = bf16_to_float((*w)[(size_t)c * D + d]);
        s += f * f;
      }
      wrow = std::max(wrow, std::sqrt(s));
    }
  if ((std::sqrt((double)D) * gmax_in + bnorm_in) * wrow > kHalfMax)
    return fail(TRIMUL_ERR_INVALID_ARG, "input-projection values could exceed the binary16 range");

  // ---- re-layout
  const int n_chunks = (2 * C + 127) / 128;
  std::vector<uint16_t> w_in((size_t)n_chunks * 256 * D, 0), w_in_bf((size_t)n_chunks * 256 * D, 0);
  // Output channel o (a channels, then b channels) has its value row at
  // (o / 8) * 16 + o % 8 and its gate row 8 further: every 16 rows hold the
  // value rows of 8 channels then their gate rows, so a chunk of 256 rows
  // covers 128 channels (64 per CTA of a pair, 128 rows each).  LN_in's
  // affine is folded in: the input projection
  // multiplies the bare normalised row zh = (z - mean) rstd by
  //   W~ = W diag(gamma_in) / 2   (fp16)
  // and adds the bias  W beta_in / 2  (fp32, per output row) in its epilogue,
  // so its accumulators hold v/2 and g/2:  sigmoid(g) v m = (v/2) m (1 + tanh(g/2)).
  std::vector<float> in_bias((size_t)n_chunks * 256, 0.f);
  for (int o = 0; o < 2 * C; ++o) {
    const size_t rv = (size_t)(o / 8) * 16 + o % 8, rg = rv + 8;
    const std::vector<uint16_t>& V = o < C ? Wa : Wb;
    const std::vector<uint16_t>& G = o < C ? Wga : Wgb;
    const int c = o < C ? o : o - C;
    double tv = 0, tgs = 0;
    for (int d = 0; d < D; ++d) {
      const float wv = bf16_to_float(V[(size_t)c * D + d]), wg = bf16_to_float(G[(size_t)c * D + d]);
      const float sv = 0.5f * wv * gi[d], sg = 0.5f * wg * gi[d];
      if (!std::isfinite(sv) || !std::isfinite(sg) || std::fabs(sv) > kHalfMax || std::fabs(sg) > kHalfMax)
        return fail(TRIMUL_ERR_INVALID_ARG, "input weights * gamma_in are outside the binary16 range");
      w_in[rv * D + d] = float_to_half_bits(sv);
      w_in[rg * D + d] = float_to_half_bits(sg);
      w_in_bf[rv * D + d] = float_to_bf16_bits(sv);
      w_in_bf[rg * D + d] = float_to_bf16_bits(sg);
      tv += (double)wv * bi[d];
      tgs += (double)wg * bi[d];
    }
    in_bias[rv] = (float)(0.5 * tv);
    in_bias[rg] = (float)(0.5 * tgs);
  }
  // Output stage: the LayerNorm affine parameters are folded into the weights,
  //   LN(v) W^T = rstd (v W~^T - mean s) + t,  W~ = W diag(gamma), s = W~ 1, t = W beta,
  // so the raw x and z tiles feed the MMAs and the epilogue applies rstd, mean,
  // s and t.  W~_g is bf16 (z is bf16), W~_o fp16 (x is stored as fp16); s is
  // summed from the rounded W~ so that the mean term cancels exactly as in the MMA.
  std::vector<uint16_t> w_o((size_t)D * C), w_g((size_t)D * D);
  std::vector<float> colc((size_t)4 * D);
  for (int d = 0; d < D; ++d) {
    double sg = 0, tg = 0, so = 0, to = 0;
    for (int e = 0; e < D; ++e) {
      const float w = bf16_to_float(Wg[(size_t)d * D + e]);
      const uint16_t wt = float_to_bf16_bits(w * gi[e]);
      w_g[(size_t)d * D + e] = wt;
      sg += bf16_to_float(wt);
      tg += (double)w * bi[e];
    }
    for (int c = 0; c < C; ++c) {
      const float w = bf16_to_float(Wo[(size_t)d * C + c]);
      const float wt = w * go[c];
      if (!std::isfinite(wt) || std::fabs(wt) > kHalfMax)
        return fail(TRIMUL_ERR_INVALID_ARG, "W_o * gamma_out is outside the binary16 range");
      const uint16_t wh = float_to_half_bits(wt);
      w_o[(size_t)d * C + c] = wh;
      so += half_bits_to_float(wh);
      to += (double)w * bo[c];
    }
    colc[4 * d + 0] = (float)sg;
    colc[4 * d + 1] = (float)(0.5 * tg);  // halved: the epilogue evaluates gate/2 and value/2
    colc[4 * d + 2] = (float)so;
    colc[4 * d + 3] = (float)(0.5 * to);
  }
  const int Dr = (D + 3) / 4 * 4, Cr = (C + 3) / 4 * 4;
  std::vector<float> ln((size_t)2 * Dr + 2 * Cr, 0.f);
  std::copy(gi.begin(), gi.end(), ln.begin());
  std::copy(bi.begin(), bi.end(), ln.begin() + Dr);
  std::copy(go.begin(), go.end(), ln.begin() + 2 * Dr);
  std::copy(bo.begin(), bo.end(), ln.begin() + 2 * Dr + Cr);

  trimul_handle h = new trimul_handle_s();
  h->device = device;
  h->D = D;
  h->C = C;
  h->eps = p->eps;
  h->num_sms = prop.multiProcessorCount;
  h->n_chunks = n_chunks;
  int smem_optin = 0;
  cudaDeviceGetAttribute(&smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, device);
  h->max_smem = smem_optin;
  h->tri_pairs = triangle_max_pairs(h->num_sms);
  {
    const int k_slabs = (D + 63) / 64;
    // Rings of the input projection.  When all of a CTA's weight slabs
    // (n_chunks * k_slabs) fit beside two z buffers, they are loaded once and
    // kept, and the rest of shared memory goes to z buffers (the deeper the
    // ring, the more of z is in flight from HBM).  Otherwise three z buffers
    // when a weight ring of four stages still fits beside them, else two.
    const size_t w_stage = 128 * 128;
    const int w_slabs = n_chunks * k_slabs;
    auto stages_for = [&](int zbufs) {
      const size_t fixed = inproj_smem_bytes(k_slabs, 0, zbufs);
      return static_cast<int>(std::min<size_t>(
          INPROJ_MAX_W_STAGES,
          static_cast<size_t>(smem_optin) > fixed ? (static_cast<size_t>(smem_optin) - fixed) / w_stage : 0));
    };
    h->in_z_bufs = 0;
    if (stages_for(2) >= w_slabs) {
      const size_t fixed = inproj_smem_bytes(k_slabs, w_slabs, 0);
      const size_t zbuf = static_cast<size_t>(k_slabs) * INPROJ_HALF_PAIRS * 128;
      h->in_z_bufs = static_cast<int>(
          std::min<size_t>(INPROJ_MAX_Z_BUFS, (static_cast<size_t>(smem_optin) - fixed) / zbuf));
      h->in_w_stages = w_slabs;
      h->in_w_resident = 1;
    }
    for (int zbufs = 3; zbufs >= 2 && !h->in_z_bufs; --zbufs)
      if (stages_for(zbufs) >= 4 || zbufs == 2) {
        h->in_z_bufs = zbufs;
        h->in_w_stages = stages_for(zbufs);
        h->in_w_resident = 0;
      }
    const bool in_fits = h->in_z_bufs >= 2 && h->in_w_stages >= (h->in_w_resident ? 1 : 2);
    h->in_pairs = in_fits ? inproj_max_pairs(h->num_sms, k_slabs, h->in_w_stages, h->in_z_bufs) : 1;
    // the gate-gradient kernel has the input projection's tiles, rings and layout
    h->gg_pairs = in_fits ? gategrad_max_pairs(h->num_sms, k_slabs, h->in_w_stages, h->in_z_bufs) : 1;
  }
  h->ab_bound = (std::sqrt((double)D) * gmax_in + bnorm_in) * wrow;
  h->gemm_pairs = gemm_max_pairs(h->num_sms);
  {
    const char* e = std::getenv("TRIMUL_LOG");
    h->log = e && *e && std::strcmp(e, "0") != 0;
  }
  tlog(h,
       "create device %d (%d SMs, %d B shared memory per block) D=%d C=%d: input projection %d pairs, %d weight "
       "stages%s, %d z buffers; triangle %d pairs; backward GEMM %d pairs; |a|,|b| bound %.4g",
       device, h->num_sms, h->max_smem, D, C, h->in_pairs, h->in_w_stages, h->in_w_resident ? " (resident)" : "",
       h->in_z_bufs, h->tri_pairs, h->gemm_pairs, h->ab_bound);

  // Backward weights (bf16): the stacked input projections [W_a; W_ga; W_b;
  // W_gb], raw and with gamma_in folded in; raw W_g and W_o; W_o with
  // gamma_out folded in.  The folded betas t = W beta and raw W_o in fp32.
  const size_t n_in = (size_t)4 * C * D, n_g = (size_t)D * D, n_o = (size_t)D * C;
  std::vector<uint16_t> bw(n_in + n_g + 2 * n_o);
  std::vector<float> bf((size_t)2 * D + n_o);
  {
    uint16_t* const in_raw = bw.data();
    uint16_t* const g_raw = in_raw + n_in;
    uint16_t* const o_raw = g_raw + n_g;
    uint16_t* const o_t = o_raw + n_o;
    float* const t_g = bf.data();
    float* const t_o = t_g + D;
    float* const o_f32 = t_o + D;
    const std::vector<uint16_t>* ws[4] = {&Wa, &Wga, &Wb, &Wgb};
    for (int k = 0; k < 4; ++k)
      for (int c = 0; c < C; ++c)
        for (int d = 0; d < D; ++d) in_raw[((size_t)k * C + c) * D + d] = (*ws[k])[(size_t)c * D + d];
    for (int d = 0; d < D; ++d) {
      double tg = 0, to = 0;
      for (int e = 0; e < D; ++e) {
        g_raw[(size_t)d * D + e] = Wg[(size_t)d * D + e];
        tg += (double)bf16_to_float(Wg[(size_t)d * D + e]) * bi[e];
      }
      for (int c = 0; c < C; ++c) {
        const uint16_t w = Wo[(size_t)d * C + c];
        o_raw[(size_t)d * C + c] = w;
        o_t[(size_t)d * C + c] = float_to_bf16_bits(bf16_to_float(w) * go[c]);
        o_f32[(size_t)d * C + c] = bf16_to_float(w);
        to += (double)bf16_to_float(w) * bo[c];
      }
      t_g[d] = (float)tg;
      t_o[d] = (float)to;
    }
  }
  cudaError_t e = cudaSuccess;
  if (e == cudaSuccess) e = cudaMalloc(&h->bw, bw.size() * 2);
  if (e == cudaSuccess) e = cudaMalloc(&h->bf, bf.size() * 4);
  if (e == cudaSuccess) e = cudaMemcpy(h->bw, bw.data(), bw.size() * 2, cudaMemcpyHostToDevice);
  if (e == cudaSuccess) e = cudaMemcpy(h->bf, bf.data(), bf.size() * 4, cudaMemcpyHostToDevice);
  if (e == cudaSuccess) {
    h->bw_in = h->bw;
    h->bw_g = h->bw_in + n_in;
    h->bw_o = h->bw_g + n_g;
    h->bw_o_t = h->bw_o + n_o;
    h->bt_g = h->bf;
    h->bt_o = h->bt_g + D;
    h->bw_o_f32 = h->bt_o + D;
  }
  if (e == cudaSuccess) e = cudaMalloc(&h->w_in, 2 * w_in.size() * 2);
  if (e == cudaSuccess) e = cudaMalloc(&h->w_o, w_o.size() * 2);
  if (e == cudaSuccess) e = cudaMalloc(&h->w_g, w_g.size() * 2);
  if (e == cudaSuccess) e = cudaMalloc(&h->ln, ln.size() * 4);
  if (e == cudaSuccess) e = cudaMalloc(&h->colc, colc.size() * 4);
  if (e == cudaSuccess) e = cudaMalloc(&h->in_bias, in_bias.size() * 4);
  if (e == cudaSuccess) e = cudaMalloc(&h->status, 16);
  if (e == cudaSuccess) e = cudaMemcpy(h->w_in, w_in.data(), w_in.size() * 2, cudaMemcpyHostToDevice);
  if (e == cudaSuccess) {
    h->w_in_bf = h->w_in + w_in.size();
    e = cudaMemcpy(h->w_in_bf, w_in_bf.data(), w_in_bf.size() * 2, cudaMemcpyHostToDevice);
  }
  if (e == cudaSuccess) e = cudaMemcpy(h->w_o, w_o.data(), w_o.size() * 2, cudaMemcpyHostToDevice);
  if (e == cudaSuccess) e = cudaMemcpy(h->w_g, w_g.data(), w_g.size() * 2, cudaMemcpyHostToDevice);
  if (e == cudaSuccess) e = cudaMemcpy(h->ln, ln.data(), ln.size() * 4, cudaMemcpyHostToDevice);
  if (e == cudaSuccess) e = cudaMemcpy(h->colc, colc.data(), colc.size() * 4, cudaMemcpyHostToDevice);
  if (e == cudaSuccess) e = cudaMemcpy(h->in_bias, in_bias.data(), in_bias.size() * 4, cudaMemcpyHostToDevice);
  if (e == cudaSuccess) e = cudaMemset(h->status, 0, 16);
  if (e != cudaSuccess) {
    trimul_destroy(h);
    return cuda_fail(e, "handle allocation");
  }
  h->g_in = h->ln;
  h->b_in = h->ln + Dr;
  h->g_out = h->ln + 2 * Dr;
  h->b_out = h->ln + 2 * Dr + Cr;
  *out = h;
  return TRIMUL_OK;
}

trimul_status trimul_prepare(trimul_handle h, int B, int N, int masked) {
  (void)masked;
  trimul_status st = check_handle(h);
  if (st != TRIMUL_OK) return st;
  if ((st = check_sizes(h, B, N)) != TRIMUL_OK) return st;
  if ((st = use_device(h)) != TRIMUL_OK) return st;
  return ensure_workspace(h, B, N);
}

trimul_status trimul_inproj(trimul_handle h, const uint16_t* z, const uint16_t* mask, int B, int N,
                            uint16_t* a_out, uint16_t* b_out, void* stream, unsigned flags) {
  trimul_status st = check_handle(h);
  if (st != TRIMUL_OK) return st;
  if (flags & TRIMUL_FLAG_FP8) return fail(TRIMUL_ERR_INVALID_ARG, "TRIMUL_FLAG_FP8 is for trimul_forward only");
  if ((st = check_sizes(h, B, N)) != TRIMUL_OK) return st;
  if (!z || !a_out || !b_out) return fail(TRIMUL_ERR_INVALID_ARG, "null tensor pointer");
  if (!aligned16(z) || !aligned16(a_out) || !aligned16(b_out) || (mask && !aligned16(mask)))
    return fail(TRIMUL_ERR_INVALID_ARG, "tensor base addresses must be 16-byte aligned");
  if ((st = use_device(h)) != TRIMUL_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if ((st = reset_status(h, s)) != TRIMUL_OK) return st;
  if ((st = run_inproj(h, z, mask, B, N, a_out, b_out, nullptr, false, s, flags)) != TRIMUL_OK) return st;
  return finish(h, s, flags);
}

trimul_status trimul_triangle(trimul_handle h, const uint16_t* a, const uint16_t* b, int B, int N,
                              trimul_direction dir, uint16_t* x_out, void* stream, unsigned flags) {
  trimul_status st = check_handle(h);
  if (st != TRIMUL_OK) return st;
  if (flags & TRIMUL_FLAG_FP8) return fail(TRIMUL_ERR_INVALID_ARG, "TRIMUL_FLAG_FP8 is for trimul_forward only");
  if ((st = check_sizes(h, B, N)) != TRIMUL_OK) return st;
  if (dir != TRIMUL_OUTGOING && dir != TRIMUL_INCOMING) return fail(TRIMUL_ERR_INVALID_ARG, "bad direction %d", (int)dir);
  if (!a || !b || !x_out) return fail(TRIMUL_ERR_INVALID_ARG, "null tensor pointer");
  if (!aligned16(a) || !aligned16(b) || !aligned16(x_out))
    return fail(TRIMUL_ERR_INVALID_ARG, "tensor base addresses must be 16-byte aligned");
  if ((st = use_device(h)) != TRIMUL_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if ((st = reset_status(h, s)) != TRIMUL_OK) return st;
  if ((st = run_triangle(h, a, b, B, N, dir, x_out, false, s, flags)) != TRIMUL_OK) return st;
  return finish(h, s, flags);
}

trimul_status trimul_outproj(trimul_handle h, const uint16_t* x, const uint16_t* z, int B, int N, uint16_t* out,
                             void* stream, unsigned flags) {
  trimul_status st = check_handle(h);
  if (st != TRIMUL_OK) return st;
  if (flags & TRIMUL_FLAG_FP8) return fail(TRIMUL_ERR_INVALID_ARG, "TRIMUL_FLAG_FP8 is for trimul_forward only");
  if ((st = check_sizes(h, B, N)) != TRIMUL_OK) return st;
  if (!x || !z || !out) return fail(TRIMUL_ERR_INVALID_ARG, "null tensor pointer");
  if (!aligned16(x) || !aligned16(z) || !aligned16(out))
    return fail(TRIMUL_ERR_INVALID_ARG, "tensor base addresses must be 16-byte aligned");
  if ((st = use_device(h)) != TRIMUL_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if ((st = reset_status(h, s)) != TRIMUL_OK) return st;
  if ((st = run_outproj(h, x, z, nullptr, B, N, out, false, s, flags)) != TRIMUL_OK) return st;
  return finish(h, s, flags);
}

trimul_status trimul_forward(trimul_handle h, const uint16_t* z, const uint16_t* mask, int B, int N,
                             trimul_direction dir, uint16_t* out, void* stream, unsigned flags) {
  trimul_status st = check_handle(h);
  if (st != TRIMUL_OK) return st;
  if ((st = check_sizes(h, B, N)) != TRIMUL_OK) return st;
  if (dir != TRIMUL_OUTGOING && dir != TRIMUL_INCOMING) return fail(TRIMUL_ERR_INVALID_ARG, "bad direction %d", (int)dir);
  if (!z || !out) return fail(TRIMUL_ERR_INVALID_ARG, "null tensor pointer");
  if (!aligned16(z) || !aligned16(out) || (mask && !aligned16(mask)))
    return fail(TRIMUL_ERR_INVALID_ARG, "tensor base addresses must be 16-byte aligned");
  const size_t zbytes = (size_t)B * N * N * h->D * 2;
  const char* zc = reinterpret_cast<const char*>(z);
  const char* oc = reinterpret_cast<const char*>(out);
  if (oc < zc + zbytes && zc < oc + zbytes) return fail(TRIMUL_ERR_INVALID_ARG, "out must not overlap z");
  const bool fp8 = (flags & TRIMUL_FLAG_FP8) != 0;
  if (fp8 && dir != TRIMUL_OUTGOING) return fail(TRIMUL_ERR_INVALID_ARG, "TRIMUL_FLAG_FP8 supports the outgoing direction only");
  // an e4m3 plane row is N bytes; TMA wants row strides in multiples of 16 bytes
  if (fp8 && N % 16 != 0) return fail(TRIMUL_ERR_SHAPE, "TRIMUL_FLAG_FP8 needs N %% 16 == 0 (N = %d)", N);
  if ((st = use_device(h)) != TRIMUL_OK) return st;
  if ((st = ensure_workspace(h, B, N)) != TRIMUL_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const size_t plane = (size_t)B * h->C * N * N;
  uint16_t* a = h->ws;
  uint16_t* b = h->ws + plane;
  uint16_t* x = h->ws + 2 * plane;
  float2* zstats = reinterpret_cast<float2*>(h->ws + 3 * plane);
  if ((st = reset_status(h, s)) != TRIMUL_OK) return st;
  if (h->timing) TRY_CUDA(cudaEventRecord(h->ev[0], s), "event record");
  if ((st = run_inproj(h, z, mask, B, N, a, b, zstats, true, s, flags, 0, -1, fp8 ? INPROJ_OUT_E4M3 : INPROJ_OUT_F16)) !=
      TRIMUL_OK)
    return st;
  if (h->timing) TRY_CUDA(cudaEventRecord(h->ev[1], s), "event record");
  if ((st = run_triangle(h, a, b, B, N, dir, x, true, s, flags, false, fp8)) != TRIMUL_OK) return st;
  if (h->timing) TRY_CUDA(cudaEventRecord(h->ev[2], s), "event record");
  if ((st = run_outproj(h, x, z, zstats, B, N, out, true, s, flags)) != TRIMUL_OK) return st;
  if (h->timing) TRY_CUDA(cudaEventRecord(h->ev[3], s), "event record");
  return finish(h, s, flags);
}

trimul_status trimul_forward_host(trimul_handle h, const uint16_t* z_host, const uint16_t* mask_host, int B, int N,
                                  trimul_direction dir, uint16_t* out_host, void* stream, unsigned flags) {
  trimul_status st = check_handle(h);
  if (st != TRIMUL_OK) return st;
  if (flags & TRIMUL_FLAG_FP8) return fail(TRIMUL_ERR_INVALID_ARG, "TRIMUL_FLAG_FP8 is for trimul_forward only");
  if ((st = check_sizes(h, B, N)) != TRIMUL_OK) return st;
  if (dir != TRIMUL_OUTGOING && dir != TRIMUL_INCOMING) return fail(TRIMUL_ERR_INVALID_ARG, "bad direction %d", (int)dir);
  if (!z_host || !out_host) return fail(TRIMUL_ERR_INVALID_ARG, "null tensor pointer");
  if ((st = use_device(h)) != TRIMUL_OK) return st;
  const long long NN = static_cast<long long>(N) * N;
  const size_t zelems = (size_t)B * NN * h->D;
  const size_t melems = mask_host ? (size_t)B * NN : 0;
  // one staging slot: z | out | mask, each rounded up to 256 bytes
  auto up = [](size_t bytes) { return (bytes + 255) / 256 * 256; };
  const size_t slot_bytes = 2 * up(zelems * 2) + up(melems * 2);
  if (slot_bytes > h->stage_bytes) {
    uint16_t* p = nullptr;
    if (h->stage) {
      cudaDeviceSynchronize();
      cudaFree(h->stage);
      h->stage = nullptr;
      h->stage_bytes = 0;
    }
    cudaError_t e = cudaMalloc(&p, 2 * slot_bytes);
    if (e != cudaSuccess) {
      cudaGetLastError();
      return cuda_fail(e, "staging allocation");
    }
    h->stage = p;
    h->stage_bytes = slot_bytes;
  }
  if (!h->s_in) {
    cudaError_t e = cudaStreamCreateWithFlags(&h->s_in, cudaStreamNonBlocking);
    if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&h->s_out, cudaStreamNonBlocking);
    for (int i = 0; i < kHostChunks && e == cudaSuccess; ++i) {
      e = cudaEventCreateWithFlags(&h->ev_in[i], cudaEventDisableTiming);
      if (e == cudaSuccess) e = cudaEventCreateWithFlags(&h->ev_out[i], cudaEventDisableTiming);
    }
    for (int i = 0; i < 2 && e == cudaSuccess; ++i) {
      e = cudaEventCreateWithFlags(&h->ev_zfree[i], cudaEventDisableTiming);
      if (e == cudaSuccess) e = cudaEventCreateWithFlags(&h->ev_dfree[i], cudaEventDisableTiming);
    }
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&h->ev_done, cudaEventDisableTiming);
    if (e != cudaSuccess) return cuda_fail(e, "copy streams / events");
  }
  if ((st = ensure_workspace(h, B, N)) != TRIMUL_OK) return st;
  const int slot = static_cast<int>(h->host_calls++ & 1);
  char* const sb = reinterpret_cast<char*>(h->stage) + slot * h->stage_bytes;
  uint16_t* const dz = reinterpret_cast<uint16_t*>(sb);
  uint16_t* const dout = reinterpret_cast<uint16_t*>(sb + up(zelems * 2));
  uint16_t* const dmask = mask_host ? reinterpret_cast<uint16_t*>(sb + 2 * up(zelems * 2)) : nullptr;
  const size_t plane = (size_t)B * h->C * NN;
  uint16_t* const a = h->ws;
  uint16_t* const b = h->ws + plane;
  uint16_t* const x = h->ws + 2 * plane;
  float2* const zstats = reinterpret_cast<float2*>(h->ws + 3 * plane);
  cudaStream_t s = static_cast<cudaStream_t>(stream);

  // Chunks are ranges of input-projection tiles: tile t covers the pairs of
  // batch t / tpb from (t % tpb) * INPROJ_TILE_PAIRS, so a range of tiles is
  // one contiguous range of global pairs of z, mask and out.  The output
  // projection's 128-pair tiles split each of them in two (the second may lie
  // past N*N, i.e. not exist): out_tile maps a tile boundary to its index.
  const int tpb = static_cast<int>((NN + INPROJ_TILE_PAIRS - 1) / INPROJ_TILE_PAIRS), total = tpb * B;
  const int tpb3 = static_cast<int>((NN + 127) / 128);
  const int chunks = zelems * 2 >= kHostChunkMin ? std::min(kHostChunks, total) : 1;
  auto tile_pair = [&](int t) -> size_t {  // global pair index where tile t starts (t == total: the end)
    const int bb = t / tpb;
    return static_cast<size_t>(bb) * NN +
           std::min<long long>(static_cast<long long>(t - bb * tpb) * INPROJ_TILE_PAIRS, NN);
  };
  auto chunk_tile = [&](int c) { return static_cast<int>((static_cast<long long>(total) * c) / chunks); };
  auto out_tile = [&](int t) {
    const int bb = t / tpb;
    return bb * tpb3 + (t - bb * tpb) * (INPROJ_TILE_PAIRS / 128);
  };

  // inputs: wait until the call two back (same slot) no longer reads this slot
  TRY_CUDA(cudaStreamWaitEvent(h->s_in, h->ev_zfree[slot], 0), "copy stream wait");
  if (mask_host)
    TRY_CUDA(cudaMemcpyAsync(dmask, mask_host, melems * 2, cudaMemcpyHostToDevice, h->s_in), "mask host-to-device copy");
  for (int c = 0; c < chunks; ++c) {
    const size_t p0 = tile_pair(chunk_tile(c)), p1 = tile_pair(chunk_tile(c + 1));
    const size_t off = p0 * h->D, len = (p1 - p0) * h->D * 2;
    TRY_CUDA(cudaMemcpyAsync(dz + off, z_host + off, len, cudaMemcpyHostToDevice, h->s_in), "z host-to-device copy");
    TRY_CUDA(cudaEventRecord(h->ev_in[c], h->s_in), "event record");
  }
  // compute on the caller's stream; stage 1 follows the input copies chunk by chunk
  if ((st = reset_status(h, s)) != TRIMUL_OK) return st;
  if (h->timing) TRY_CUDA(cudaEventRecord(h->ev[0], s), "event record");
  for (int c = 0; c < chunks; ++c) {
    TRY_CUDA(cudaStreamWaitEvent(s, h->ev_in[c], 0), "stream wait");
    if ((st = run_inproj(h, dz, dmask, B, N, a, b, zstats, true, s, flags, chunk_tile(c), chunk_tile(c + 1))) !=
        TRIMUL_OK)
      return st;
  }
  if (h->timing) TRY_CUDA(cudaEventRecord(h->ev[1], s), "event record");
  if ((st = run_triangle(h, a, b, B, N, dir, x, true, s, flags)) != TRIMUL_OK) return st;
  if (h->timing) TRY_CUDA(cudaEventRecord(h->ev[2], s), "event record");
  // stage 3 chunk by chunk; each chunk's output is copied back while the next
  // computes.  This slot's out buffer is free once the copies of the call two
  // back (same slot) have completed.
  TRY_CUDA(cudaStreamWaitEvent(s, h->ev_dfree[slot], 0), "stream wait");
  for (int c = 0; c < chunks; ++c) {
    if ((st = run_outproj(h, x, dz, zstats, B, N, dout, true, s, flags, out_tile(chunk_tile(c)),
                          out_tile(chunk_tile(c + 1)))) !=
        TRIMUL_OK)
      return st;
    TRY_CUDA(cudaEventRecord(h->ev_out[c], s), "event record");
    TRY_CUDA(cudaStreamWaitEvent(h->s_out, h->ev_out[c], 0), "copy stream wait");
    const size_t p0 = tile_pair(chunk_tile(c)), p1 = tile_pair(chunk_tile(c + 1));
    const size_t off = p0 * h->D, len = (p1 - p0) * h->D * 2;
    TRY_CUDA(cudaMemcpyAsync(out_host + off, dout + off, len, cudaMemcpyDeviceToHost, h->s_out), "out device-to-host copy");
  }
  if (h->timing) TRY_CUDA(cudaEventRecord(h->ev[3], s), "event record");
  TRY_CUDA(cudaEventRecord(h->ev_zfree[slot], s), "event record");  // this call's last read of dz / dmask
  TRY_CUDA(cudaEventRecord(h->ev_dfree[slot], h->s_out), "event record");  // ... and of dout
  // Unless deferred, the caller's stream completes only once out_host holds the result.
  if (!(flags & TRIMUL_FLAG_DEFER_OUTPUT)) {
    TRY_CUDA(cudaEventRecord(h->ev_done, h->s_out), "event record");
    TRY_CUDA(cudaStreamWaitEvent(s, h->ev_done, 0), "stream wait");
  }
  return finish(h, s, flags);
}

trimul_status trimul_host_join(trimul_handle h, void* stream) {
  trimul_status st = check_handle(h);
  if (st != TRIMUL_OK) return st;
  if (!h->s_out) return TRIMUL_OK;  // no host-buffer call yet
  if ((st = use_device(h)) != TRIMUL_OK) return st;
  TRY_CUDA(cudaEventRecord(h->ev_done, h->s_out), "event record");
  TRY_CUDA(cudaStreamWaitEvent(static_cast<cudaStream_t>(stream), h->ev_done, 0), "stream wait");
  return TRIMUL_OK;
}

trimul_status trimul_set_stage_events(trimul_handle h, void* const* events) {
  trimul_status st = check_handle(h);
  if (st != TRIMUL_OK) return st;
  if (!events) {
    h->timing = false;
    return TRIMUL_OK;
  }
  for (int i = 0; i < 4; ++i)
    if (!events[i]) return fail(TRIMUL_ERR_INVALID_ARG, "event %d is null", i);
  for (int i = 0; i < 4; ++i) h->ev[i] = static_cast<cudaEvent_t>(events[i]);
  h->timing = true;
  return TRIMUL_OK;
}

trimul_status trimul_forward_noalloc(trimul_handle h, const uint16_t* z, const uint16_t* mask, int B, int N,
                                     trimul_direction dir, uint16_t* out, void* stream, unsigned flags) {
  trimul_status st = check_handle(h);
  if (st != TRIMUL_OK) return st;
  if (flags & TRIMUL_FLAG_FP8) return fail(TRIMUL_ERR_INVALID_ARG, "TRIMUL_FLAG_FP8 is for trimul_forward only");
  if ((st = check_sizes(h, B, N)) != TRIMUL_OK) return st;
  if (dir != TRIMUL_OUTGOING && dir != TRIMUL_INCOMING) return fail(TRIMUL_ERR_INVALID_ARG, "bad direction %d", (int)dir);
  if (!z || !out) return fail(TRIMUL_ERR_INVALID_ARG, "null tensor pointer");
  if (!aligned16(z) || !aligned16(out) || (mask && !aligned16(mask)))
    return fail(TRIMUL_ERR_INVALID_ARG, "tensor base addresses must be 16-byte aligned");
  const size_t zbytes = (size_t)B * N * N * h->D * 2;
  const char* zc = reinterpret_cast<const char*>(z);
  const char* oc = reinterpret_cast<const char*>(out);
  if (oc < zc + zbytes && zc < oc + zbytes) return fail(TRIMUL_ERR_INVALID_ARG, "out must not overlap z");
  // a, b (fp16) and x (fp16 holding x * 2^-s): three planes of B*C*N*N
  // 16-bit values, then the LN_in statistics (B*N*N float2)
  const size_t plane = (size_t)B * h->C * N * N;
  const size_t need = workspace_bytes(h, B, N);
  if (need > kNoAllocScratchBytes)
    return fail(TRIMUL_ERR_SHAPE,
                "trimul_forward_noalloc needs %zu bytes of scratch for B=%d C=%d N=%d, but its fixed scratch holds "
                "%zu bytes; use trimul_forward for this size",
                need, B, h->C, N, kNoAllocScratchBytes);
  if ((st = use_device(h)) != TRIMUL_OK) return st;
  uint16_t* scratch = nullptr;
  if ((st = noalloc_scratch(h->device, &scratch)) != TRIMUL_OK) return st;
  // Every byte of a, b and x that a later kernel reads is written earlier in
  // this same call, so the scratch needs no clearing between calls.
  uint16_t* a = scratch;
  uint16_t* b = scratch + plane;
  uint16_t* x = scratch + 2 * plane;
  float2* zstats = reinterpret_cast<float2*>(scratch + 3 * plane);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if ((st = reset_status(h, s)) != TRIMUL_OK) return st;
  if ((st = run_inproj(h, z, mask, B, N, a, b, zstats, true, s, flags)) != TRIMUL_OK) return st;
  if ((st = run_triangle(h, a, b, B, N, dir, x, true, s, flags)) != TRIMUL_OK) return st;
  if ((st = run_outproj(h, x, z, zstats, B, N, out, true, s, flags)) != TRIMUL_OK) return st;
  return finish(h, s, flags);
}

size_t trimul_noalloc_scratch_bytes(void) { return kNoAllocScratchBytes; }

size_t trimul_backward_workspace_bytes(trimul_handle h, int B, int N) {
  if (!h || B < 1 || N < 1) {
    fail(TRIMUL_ERR_INVALID_ARG, "null handle or empty shape");
    return 0;
  }
  return backward_plan(h, B, N).total;
}

trimul_status trimul_backward(trimul_handle h, const uint16_t* z, const uint16_t* mask, const uint16_t* dout, int B,
                              int N, trimul_direction dir, uint16_t* dz, const trimul_grads* grads, void* stream,
                              unsigned flags) {
  trimul_status st = check_handle(h);
  if (st != TRIMUL_OK) return st;
  if (flags & TRIMUL_FLAG_FP8) return fail(TRIMUL_ERR_INVALID_ARG, "TRIMUL_FLAG_FP8 is for trimul_forward only");
  if ((st = check_sizes(h, B, N)) != TRIMUL_OK) return st;
  if (dir != TRIMUL_OUTGOING && dir != TRIMUL_INCOMING) return fail(TRIMUL_ERR_INVALID_ARG, "bad direction %d", (int)dir);
  if (!z || !dout || !dz || !grads) return fail(TRIMUL_ERR_INVALID_ARG, "null tensor pointer");
  const float* gptr[] = {grads->dW_a, grads->dW_ga, grads->dW_b, grads->dW_gb, grads->dW_o,
                         grads->dW_g, grads->d_ln_in_gamma, grads->d_ln_in_beta, grads->d_ln_out_gamma,
                         grads->d_ln_out_beta};
  for (const float* q : gptr)
    if (!q) return fail(TRIMUL_ERR_INVALID_ARG, "null gradient pointer");
  if (!aligned16(z) || !aligned16(dout) || !aligned16(dz) || (mask && !aligned16(mask)))
    return fail(TRIMUL_ERR_INVALID_ARG, "tensor base addresses must be 16-byte aligned");
  const size_t zbytes = (size_t)B * N * N * h->D * 2;
  auto overlaps = [&](const void* u, const void* v) {
    const char* a = static_cast<const char*>(u);
    const char* b = static_cast<const char*>(v);
    return a < b + zbytes && b < a + zbytes;
  };
  if (overlaps(dz, z) || overlaps(dz, dout)) return fail(TRIMUL_ERR_INVALID_ARG, "dz must not overlap z or dout");
  if ((st = use_device(h)) != TRIMUL_OK) return st;
  const BwdPlan L = backward_plan(h, B, N);
  if ((st = ensure_backward_workspace(h, L.total)) != TRIMUL_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  char* const w = h->bws;
  const long long P = static_cast<long long>(N) * N, BP = B * P;
  const int D = h->D, C = h->C;
  uint16_t* const a = reinterpret_cast<uint16_t*>(w + L.ab);
  uint16_t* const b = a + static_cast<size_t>(B) * C * P;
  uint16_t* const x = reinterpret_cast<uint16_t*>(w + L.x);
  float2* const zstats = reinterpret_cast<float2*>(w + L.zstats);
  uint16_t* const zh = reinterpret_cast<uint16_t*>(w + L.zh);
  uint16_t* const xh = reinterpret_cast<uint16_t*>(w + L.xh);
  uint16_t* const dx = xh;  // xh is dead once the dv^T xh GEMM has run
  float2* const xstats = reinterpret_cast<float2*>(w + L.xstats);
  __half* const gacc = reinterpret_cast<__half*>(w + L.g);  // fp16 [BP][D]: recomputed activations
  __half* const vacc = reinterpret_cast<__half*>(w + L.v);
  uint16_t* const dyt = reinterpret_cast<uint16_t*>(w + L.dyt);  // bf16
  uint16_t* const dzp = reinterpret_cast<uint16_t*>(w + L.dzp);    // bf16
  uint16_t* const dzin = reinterpret_cast<uint16_t*>(w + L.dzin);  // bf16
  uint16_t* const dv = reinterpret_cast<uint16_t*>(w + L.dv);
  uint16_t* const dg = reinterpret_cast<uint16_t*>(w + L.dg);
  uint16_t* const da = reinterpret_cast<uint16_t*>(w + L.da);
  uint16_t* const db = reinterpret_cast<uint16_t*>(w + L.db);
  uint16_t* const pt = reinterpret_cast<uint16_t*>(w + L.pt);
  auto f32 = [&](size_t off) { return reinterpret_cast<float*>(w + off); };
  const unsigned* const abm = ab_max_word(h);
  const bool out = dir == TRIMUL_OUTGOING;
  auto bf = [](const void* q) { return reinterpret_cast<const __nv_bfloat16*>(q); };
  auto bfm = [](void* q) { return reinterpret_cast<__nv_bfloat16*>(q); };

  if ((st = reset_status(h, s)) != TRIMUL_OK) return st;
  // 1-2. forward recompute: a, b (bf16) with the LN_in statistics, then x
  if ((st = run_inproj(h, z, mask, B, N, a, b, zstats, true, s, flags, 0, -1, INPROJ_OUT_BF16, zh)) != TRIMUL_OK)
    return st;
  if ((st = run_triangle(h, a, b, B, N, dir, x, true, s, flags, true)) != TRIMUL_OK) return st;
  // 3-4. normalised planes: zh [BP][D] came from the recompute above (the
  // input projection stores its LayerNorm output); xh [B][C][P]
  TRY_CUDA(launch_xhat(reinterpret_cast<const __half*>(x), bfm(xh), xstats, abm, B, N, C, h->eps, h->num_sms, s),
           "xh launch");
  // 5-6. gate and value projections (fp16: recomputed activations, O(1)), then
  // dv and dg with their column sums
  if ((st = run_gemm(h, {zh, false, true, P, D}, {h->w_g, false, false, D, D}, static_cast<int>(P), D, D, B, false,
                     GEMM_OUT_F16, gacc, D, P * D, s, flags)) != TRIMUL_OK)
    return st;
  if ((st = run_gemm(h, {xh, true, true, P, C}, {h->bw_o_t, false, false, D, C}, static_cast<int>(P), D, C, B, false,
                     GEMM_OUT_F16, vacc, D, P * D, s, flags)) != TRIMUL_OK)
    return st;
  TRY_CUDA(launch_dout(bf(dout), gacc, vacc, h->bt_g, h->bt_o, bfm(dv), bfm(dg), f32(L.part_dout), BP, D, h->num_sms,
                       s),
           "output-gate backward launch");
  // 7-8. dy^T = W_o^T dv^T (bf16 [B][C][P]) and dz' = dg W_g (bf16 [BP][D])
  if ((st = run_gemm(h, {h->bw_o, true, false, C, D}, {dv, false, true, P, D}, C, static_cast<int>(P), D, B, false,
                     GEMM_OUT_BF16, dyt, P, C * P, s, flags)) != TRIMUL_OK)
    return st;
  if ((st = run_gemm(h, {dg, false, true, P, D}, {h->bw_g, true, false, D, D}, static_cast<int>(P), D, D, B, false,
                     GEMM_OUT_BF16, dzp, D, P * D, s, flags)) != TRIMUL_OK)
    return st;
  // 9-10. dv^T xh [D][C] and dg^T zh [D][D], split over all pairs
  if ((st = run_gemm(h, {dv, true, true, D, P}, {xh, false, true, C, P}, D, C, P, B, true, GEMM_OUT_F32,
                     f32(L.part_mo), C, static_cast<long long>(D) * C, s, flags)) != TRIMUL_OK)
    return st;
  if ((st = run_gemm(h, {dg, true, true, D, P}, {zh, true, true, D, P}, D, D, P, B, true, GEMM_OUT_F32,
                     f32(L.part_mg), D, static_cast<long long>(D) * D, s, flags)) != TRIMUL_OK)
    return st;
  // 11. LN_out backward -> dx (bf16, channel-major; over xh)
  TRY_CUDA(launch_lnout_bwd(bf(dyt), reinterpret_cast<const __half*>(x), xstats, h->g_out, bfm(dx), abm, B, N, C,
                            h->num_sms, s),
           "LN_out backward launch");
  // 12. triangle gradients (per plane of the B * C channel planes), on the
  // triangle kernel with the operand majors each product needs (bf16 out,
  // unscaled).  As C = A B^T over (rows of A, rows of B) with K shared:
  //   outgoing  dA[i][k] = sum_j dX[i][j] b[j][k]    A = dX K-major, B = b MN-major
  //             dB[j][k] = sum_i dX[i][j] a[i][k]    A = dX MN-major, B = a MN-major
  //   incoming  dA[k][i] = sum_j b[k][j] dX[i][j]    A = b K-major, B = dX K-major
  //             dB[k][j] = sum_i a[k][i] dX[i][j]    A = a K-major, B = dX MN-major
  if (out) {
    if ((st = run_triangle(h, dx, b, B, N, dir, da, false, s, flags, true, false, true, 0, 1)) != TRIMUL_OK) return st;
    if ((st = run_triangle(h, dx, a, B, N, dir, db, false, s, flags, true, false, true, 1, 1)) != TRIMUL_OK) return st;
  } else {
    if ((st = run_triangle(h, b, dx, B, N, dir, da, false, s, flags, true, false, true, 0, 0)) != TRIMUL_OK) return st;
    if ((st = run_triangle(h, a, dx, B, N, dir, db, false, s, flags, true, false, true, 0, 1)) != TRIMUL_OK) return st;
  }
  // 13-14. gradients of the gated input projections' pre-activations, dP
  // (bf16 [B][4C][P]), recomputing the pre-activations on the tensor cores,
  // then the row sums of dP for the bias part of the weight gradients
  if ((st = run_gate_grad(h, zh, mask, da, db, B, N, pt, f32(L.rowpart), s, flags)) != TRIMUL_OK) return st;
  TRY_CUDA(launch_gate_rowsums(f32(L.rowpart), f32(L.rowtmp), f32(L.part_gate), B,
                               static_cast<int>((P + INPROJ_TILE_PAIRS - 1) / INPROJ_TILE_PAIRS), h->n_chunks, C,
                               L.nslice, s),
           "gate row-sum launch");
  // 15. dP W_in, the input projections' part of dz' (its own buffer: a
  // read-modify-write epilogue would wait on DRAM reads tile by tile)
  if ((st = run_gemm(h, {pt, true, true, P, 4 * C}, {h->bw_in, true, false, D, 4 * C}, static_cast<int>(P), D, 4 * C,
                     B, false, GEMM_OUT_BF16, dzin, D, P * D, s, flags)) != TRIMUL_OK)
    return st;
  // 16. dP^T zh [4C][D], split over all pairs
  if ((st = run_gemm(h, {pt, false, true, 4 * C, P}, {zh, true, true, D, P}, 4 * C, D, P, B, true, GEMM_OUT_F32,
                     f32(L.part_min), D, 4ll * C * D, s, flags)) != TRIMUL_OK)
    return st;
  // 17. LN_in backward of dz' = both parts -> dz, with the sums for d gamma_in, d beta_in
  TRY_CUDA(launch_lnin_bwd(bf(dzp), bf(dzin), bf(z), zstats, h->g_in, bfm(dz), f32(L.part_lnin), BP, D, h->num_sms, s),
           "LN_in backward launch");
  // 18. reductions and the parameter gradients
  TRY_CUDA(launch_sum(f32(L.part_mo), f32(L.mo), static_cast<long long>(D) * C, L.nz_o, h->num_sms, s), "sum launch");
  TRY_CUDA(launch_sum(f32(L.part_mg), f32(L.mg), static_cast<long long>(D) * D, L.nz_g, h->num_sms, s), "sum launch");
  TRY_CUDA(launch_sum(f32(L.part_min), f32(L.min_), 4ll * C * D, L.nz_in, h->num_sms, s), "sum launch");
  TRY_CUDA(launch_sum(f32(L.part_dout), f32(L.cs), 2ll * D, L.dout_blk, h->num_sms, s), "sum launch");
  TRY_CUDA(launch_sum(f32(L.part_lnin), f32(L.lnin), 2ll * D, L.lnin_blk, h->num_sms, s), "sum launch");
  TrimulGradPtrs gp{grads->dW_a,          grads->dW_ga,        grads->dW_b,           grads->dW_gb,
                    grads->dW_o,          grads->dW_g,         grads->d_ln_in_gamma,  grads->d_ln_in_beta,
                    grads->d_ln_out_gamma, grads->d_ln_out_beta};
  TRY_CUDA(launch_assemble(f32(L.mo), f32(L.mg), f32(L.min_), f32(L.cs), f32(L.part_gate), L.nseg, f32(L.lnin),
                           h->bw_o_f32, h->g_in, h->b_in, h->g_out, h->b_out, gp, B, D, C, h->num_sms, s),
           "gradient assembly launch");
  return finish(h, s, flags);
}

int trimul_kernels_per_backward(trimul_handle h, int B, int N) {
  if (!h || B < 1 || N < 1) {
    fail(TRIMUL_ERR_INVALID_ARG, "null handle or empty shape");
    return -1;
  }
  int group = 0, launches = 0;
  triangle_groups(h, B, N, &group, &launches);
  const long long P = static_cast<long long>(N) * N;
  auto gemm_launches = [&](int M, int Nn, long long K, int batches, bool split) {
    long long n_z = batches, kbz;
    if (split) n_z = gemm_split_slices(h, M, Nn, K, batches, &kbz);
    const long long per_z = static_cast<long long>((M + 255) / 256) * ((Nn + 255) / 256);
    long long g = std::max<long long>(1, static_cast<long long>(h->gemm_pairs) * kTriTilesPerPair);
    if (per_z < g) g = (g / per_z) * per_z;
    return static_cast<int>((per_z * n_z + g - 1) / g);
  };
  const int D = h->D, C = h->C, Pi = static_cast<int>(P);
  int n = 1 + launches;                                        // input projection, triangle
  n += 1;                                                      // xh (zh comes from the recompute)
  n += gemm_launches(Pi, D, D, B, false) + gemm_launches(Pi, D, C, B, false) + 1;   // gate, value, dout
  n += gemm_launches(C, Pi, D, B, false) + gemm_launches(Pi, D, D, B, false);       // dy^T, dz'
  n += gemm_launches(D, C, P, B, true) + gemm_launches(D, D, P, B, true);           // dv^T xh, dg^T zh
  n += 1 + 2 * launches;                                                            // LN_out, triangle gradients
  n += 1 + 2;                                                                       // gate gradients, row sums
  n += gemm_launches(Pi, D, 4 * C, B, false) + gemm_launches(4 * C, D, P, B, true); // dz' += .., dP^T zh
  n += 1 + 5 + 1;                                              // LN_in, sums, assembly
  return n;
}

int trimul_x_scale_log2(trimul_handle h, int N) {
  if (!h || N < 1) {
    fail(TRIMUL_ERR_INVALID_ARG, "null handle or N < 1");
    return -1;
  }
  return x_scale_log2(h, N);
}

trimul_status trimul_destroy(trimul_handle h) {
  if (!h) return TRIMUL_OK;
  cudaSetDevice(h->device);
  cudaDeviceSynchronize();
  cudaFree(h->w_in);
  cudaFree(h->w_o);
  cudaFree(h->w_g);
  cudaFree(h->colc);
  cudaFree(h->in_bias);
  cudaFree(h->ln);
  cudaFree(h->status);
  cudaFree(h->ws);
  cudaFree(h->stage);
  cudaFree(h->bw);
  cudaFree(h->bf);
  cudaFree(h->bws);
  for (int i = 0; i < kHostChunks; ++i) {
    if (h->ev_in[i]) cudaEventDestroy(h->ev_in[i]);
    if (h->ev_out[i]) cudaEventDestroy(h->ev_out[i]);
  }
  for (int i = 0; i < 2; ++i) {
    if (h->ev_zfree[i]) cudaEventDestroy(h->ev_zfree[i]);
    if (h->ev_dfree[i]) cudaEventDestroy(h->ev_dfree[i]);
  }
  if (h->ev_done) cudaEventDestroy(h->ev_done);
  if (h->s_in) cudaStreamDestroy(h->s_in);
  if (h->s_out) cudaStreamDestroy(h->s_out);
  delete h;
  return TRIMUL_OK;
}

}  // extern "C"
