// api.cu -- the extern "C" boundary: argument validation, schedule plans,
// per-device state (SM count, device error word), tensor-map encoding.
// Nothing here allocates device memory or synchronizes, except
// r4_device_error(), which is documented as synchronous.

#include <cudaTypedefs.h>

#include <cstdio>
#include <mutex>
#include <map>
#include <set>
#include <utility>

#include "r4_internal.h"

namespace r4 {

__device__ int g_device_error;  // first error code any kernel recorded (0 = none)

namespace {
constexpr int kMaxDevices = 64;
int g_sms[kMaxDevices];
int *g_err_ptr[kMaxDevices];
std::mutex g_mu;
thread_local const char *t_last_kernel = "";
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

int current_device() {
  int d = 0;
  if (cudaGetDevice(&d) != cudaSuccess || d < 0 || d >= kMaxDevices) return 0;
  return d;
}

bool aligned(const void *p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }
}  // namespace

Options &options() {
  static Options o;
  return o;
}

int device_sm_count() {
  const int d = current_device();
  if (g_sms[d] == 0) {
    int v = 0;
    cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, d);
    g_sms[d] = v > 0 ? v : 1;
  }
  return g_sms[d];
}

int row_split(int64_t M, int64_t K, RowKind kind) {
  if (options().row_split > 0) return options().row_split;
  // Fitted on GB300 (graph-timed launches, M 1..256): a cluster costs about
  // 0.4 us more to launch and synchronise, so a row is split only when its
  // work is well above that (per-token quant K >= 10240, the norm producer
  // K >= 5120, the SiLU producer N >= 3072), and into no more CTAs than
  // still gain: up to one CTA per SM for the quantizer (half that for the
  // norm producer, whose CTAs synchronise twice), four per SM for the
  // SiLU producer, whose exponential and two divisions per element make it
  // issue-bound. Each CTA keeps at least 1024 elements.
  const int sms = device_sm_count();
  const int64_t min_k = kind == RowKind::kQuant ? 10240 : kind == RowKind::kNorm ? 5120 : 3072;
  const int64_t cap = kind == RowKind::kQuant ? sms : kind == RowKind::kNorm ? sms / 2 : 4 * sms;
  if (K < min_k || (kind == RowKind::kSilu && M >= sms)) return 1;
  int c = 1;
  while (c < 8 && M * 2 * c <= cap && K >= 1024 * 2 * c) c *= 2;
  return c;
}

int row_threads(RowKind kind, int64_t M, int64_t vecs) {
  if (options().row_threads > 0) return options().row_threads;
  // Fitted on GB300 (graph-timed launches): for rows of up to 768 vectors
  // of 8 (K <= 6144) a 128-thread block with more vectors per thread keeps
  // more rows resident per SM -- per-token quant M=8192, K=5120: 30.9 ->
  // 24.3 us; the norm producer gains only with many rows (M=8192: 67.6 ->
  // 63.1 us; M=64: 3.8 -> 4.6 us, so it keeps 256 below 2 rows per SM); the
  // SiLU producer is issue-bound and loses (M=2048: 72.5 -> 86.1 us); its
  // long rows at many tokens take 512 threads instead (fewer vectors per
  // thread, more warps per SM).
  if (kind == RowKind::kSilu) return (vecs > 1536 && M >= device_sm_count()) ? 512 : 256;
  if (vecs > 768) return 256;
  if (kind == RowKind::kNorm && M < 2 * static_cast<int64_t>(device_sm_count())) return 256;
  return 128;
}

int *device_error_word() {
  const int d = current_device();
  if (g_err_ptr[d] == nullptr) {
    std::lock_guard<std::mutex> lk(g_mu);
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_device_error) == cudaSuccess) g_err_ptr[d] = static_cast<int *>(p);
  }
  return g_err_ptr[d];
}

void set_last_kernel(const char *name) { t_last_kernel = name; }

cudaError_t ensure_smem_attr(const void *func, int bytes) {
  // largest size set so far per (device, kernel): a later launch of the same
  // kernel with more dynamic shared memory raises the attribute again
  static std::map<std::pair<int, const void *>, int> done;
  const int d = current_device();
  std::lock_guard<std::mutex> lk(g_mu);
  const auto it = done.find({d, func});
  if (it != done.end() && it->second >= bytes) return cudaSuccess;
  cudaError_t e = cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess) done[{d, func}] = bytes;
  return e;
}

CUresult encode_tiled(CUtensorMap *map, CUtensorMapDataType dtype, uint32_t rank, void *gaddr, const uint64_t *dims,
                      const uint64_t *strides_bytes, const uint32_t *box, CUtensorMapSwizzle swizzle) {
  if (g_encode == nullptr) {
    std::lock_guard<std::mutex> lk(g_mu);
    if (g_encode == nullptr) {
      void *fn = nullptr;
      cudaDriverEntryPointQueryResult q;
      if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) !=
              cudaSuccess ||
          q != cudaDriverEntryPointSuccess || fn == nullptr)
        return CUDA_ERROR_NOT_FOUND;
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    }
  }
  cuuint64_t d[5];
  cuuint64_t s[4];
  cuuint32_t b[5], e[5];
  for (uint32_t i = 0; i < rank; ++i) {
    d[i] = dims[i];
    b[i] = box[i];
    e[i] = 1;
    if (i + 1 < rank) s[i] = strides_bytes[i];
  }
  return g_encode(map, dtype, rank, gaddr, d, s, b, e, CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
}

}  // namespace r4

using namespace r4;


extern "C" {

// 0.3: W4A4 (MXFP4 activations, kind::mxf4), option 14, r4_mma_peak;
// 0.4: r4_plan_gemm, option 8 (block-FP8 weight rows per tile), option 9 unassigned
int r4_version(void) { return (0 << 16) | 4; }

const char *r4_status_string(int status) {
  switch (status) {
    case R4_OK: return "ok";
    case R4_ERR_INVALID_ARG: return "invalid argument (null pointer or bad size)";
    case R4_ERR_UNSUPPORTED_SHAPE: return "unsupported shape";
    case R4_ERR_MISALIGNED: return "misaligned pointer or stride";
    case R4_ERR_WORKSPACE: return "workspace or prepack buffer too small";
    case R4_ERR_CUDA: return "CUDA error";
    case R4_ERR_DEVICE_TIMEOUT: return "device-side wait timed out";
    default: return "unknown status";
  }
}

const char *r4_last_kernel_name(void) { return t_last_kernel; }

int r4_device_error(int *error_out, int clear) {
  if (error_out == nullptr) return R4_ERR_INVALID_ARG;
  int v = 0;
  if (cudaMemcpyFromSymbol(&v, g_device_error, sizeof(int)) != cudaSuccess) return R4_ERR_CUDA;
  *error_out = v;
  if (clear && v != 0) {
    const int zero = 0;
    if (cudaMemcpyToSymbol(g_device_error, &zero, sizeof(int)) != cudaSuccess) return R4_ERR_CUDA;
  }
  return v != 0 ? R4_ERR_DEVICE_TIMEOUT : R4_OK;
}

int r4_set_option(int key, int64_t value) {
  switch (key) {
    case 1: options().w4a8_splits = static_cast<int>(value); return R4_OK;
    case 2:
      if (value != 0 && value != 16 && value != 32 && value != 64 && value != 128 && value != 192 && value != 256)
        return R4_ERR_INVALID_ARG;
      options().w4a8_token_tile = static_cast<int>(value);
      return R4_OK;
    case 3: options().fp8_splits = static_cast<int>(value); return R4_OK;
    case 8:
      if (value != 0 && value != 128 && value != 256) return R4_ERR_INVALID_ARG;
      options().fp8_n_tile = static_cast<int>(value);
      return R4_OK;
    case 4: options().pdl = value ? 1 : 0; return R4_OK;
    case 14: options().early_weights = value ? 1 : 0; return R4_OK;
    case 15:
      if (value < 0 || value > 4) return R4_ERR_INVALID_ARG;
      options().skinny_groups = static_cast<int>(value);
      return R4_OK;
    case 16:
      if (value < 0 || value > 2) return R4_ERR_INVALID_ARG;
      options().stream_k = static_cast<int>(value);
      return R4_OK;
    case 5:
      if (value < 0 || value > 2) return R4_ERR_INVALID_ARG;
      options().l2_prefetch = static_cast<int>(value);
      return R4_OK;
    case 6: options().cluster_split = value ? 1 : 0; return R4_OK;
    case 10: options().inject_stall = value ? 1 : 0; return R4_OK;
    case 13:
      if (value != 0 && value != 64 && value != 128 && value != 256) return R4_ERR_INVALID_ARG;
      options().row_threads = static_cast<int>(value);
      return R4_OK;
    case 11:
      if (value != 0 && value != 1 && value != 2 && value != 4 && value != 8) return R4_ERR_INVALID_ARG;
      options().row_split = static_cast<int>(value);
      return R4_OK;
    case 7:
      if (value != 0 && value != 16 && value != 32 && value != 64 && value != 128) return R4_ERR_INVALID_ARG;
      options().fp8_token_tile = static_cast<int>(value);
      return R4_OK;
    default: return R4_ERR_INVALID_ARG;
  }
}

int r4_quant_fp8_per_token(const uint16_t *x, int64_t M, int64_t K, int64_t ldx, int64_t group, uint8_t *q, float *s,
                           r4_stream_t stream) {
  if (!x || !q || !s) return R4_ERR_INVALID_ARG;
  if (M < 1 || K < 8 || ldx < K || M > 0x7fffffff || K > 0x7fffffff) return R4_ERR_INVALID_ARG;
  if (K % 8 || ldx % 8) return R4_ERR_UNSUPPORTED_SHAPE;
  if (!(group == K || (group == 128 && K % 128 == 0))) return R4_ERR_UNSUPPORTED_SHAPE;
  if (!aligned(x, 16) || !aligned(q, 16) || !aligned(s, 4)) return R4_ERR_MISALIGNED;
  return launch_quant_act(x, M, K, ldx, group, q, s, reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess
             ? R4_OK
             : R4_ERR_CUDA;
}

int r4_mma_peak(int kind, int n, int blocks, int iters, r4_stream_t stream) {
  if (kind < 1 || kind > 3 || (n != 128 && n != 256) || blocks < 1 || blocks > 65535 || iters < 1)
    return R4_ERR_INVALID_ARG;
  if (device_error_word() == nullptr) return R4_ERR_CUDA;
  return launch_mma_peak(kind, n, blocks, iters, reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess ? R4_OK
                                                                                                      : R4_ERR_CUDA;
}

int r4_check_quotients(unsigned long long *count, float *example, r4_stream_t stream) {
  if (!count || !example) return R4_ERR_INVALID_ARG;
  if (!aligned(count, 8) || !aligned(example, 4)) return R4_ERR_MISALIGNED;
  return launch_check_quotients(count, example, reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess ? R4_OK
                                                                                                        : R4_ERR_CUDA;
}

int r4_add_rmsnorm_quant_fp8(const uint16_t *y, const uint16_t *residual, const uint16_t *weight, float eps,
                             int64_t M, int64_t K, uint16_t *residual_out, uint8_t *q, float *s, r4_stream_t stream) {
  if (!y || !residual || !weight || !residual_out || !q || !s) return R4_ERR_INVALID_ARG;
  if (M < 1 || K < 8 || M > (1 << 30) || !(eps >= 0.f) || eps > 3.0e38f) return R4_ERR_INVALID_ARG;
  if (K % 8 || K > 24576) return R4_ERR_UNSUPPORTED_SHAPE;
  if (!aligned(y, 16) || !aligned(residual, 16) || !aligned(weight, 16) || !aligned(residual_out, 16) ||
      !aligned(q, 8) || !aligned(s, 4))
    return R4_ERR_MISALIGNED;
  return launch_add_rmsnorm_quant(y, residual, weight, eps, M, K, residual_out, q, s,
                                  reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess
             ? R4_OK
             : R4_ERR_CUDA;
}

int r4_silu_mul_quant_fp8(const uint16_t *gu, int64_t M, int64_t N, uint8_t *q, float *s, r4_stream_t stream) {
  if (!gu || !q || !s) return R4_ERR_INVALID_ARG;
  if (M < 1 || N < 8 || M > (1 << 30)) return R4_ERR_INVALID_ARG;
  if (N % 8 || N > 24576) return R4_ERR_UNSUPPORTED_SHAPE;
  if (!aligned(gu, 16) || !aligned(q, 8) || !aligned(s, 4)) return R4_ERR_MISALIGNED;
  return launch_silu_mul_quant(gu, M, N, q, s, reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess ? R4_OK
                                                                                                    : R4_ERR_CUDA;
}

int r4_quantize_mxfp4_weight(const float *w, int64_t N, int64_t K, uint8_t *packed, uint8_t *scale,
                             r4_stream_t stream) {
  if (!w || !packed || !scale || N < 1 || K < 32) return R4_ERR_INVALID_ARG;
  if (K % 32) return R4_ERR_UNSUPPORTED_SHAPE;
  if (!aligned(w, 16) || !aligned(packed, 16)) return R4_ERR_MISALIGNED;
  return launch_quant_mxfp4_weight(w, N, K, packed, scale, reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess
             ? R4_OK
             : R4_ERR_CUDA;
}

int r4_quantize_blockfp8_weight(const float *w, int64_t N, int64_t K, uint8_t *q, float *s, r4_stream_t stream) {
  if (!w || !q || !s || N < 1 || K < 1) return R4_ERR_INVALID_ARG;
  if (N % 128 || K % 128) return R4_ERR_UNSUPPORTED_SHAPE;
  if (!aligned(w, 16) || !aligned(q, 4) || !aligned(s, 4)) return R4_ERR_MISALIGNED;
  return launch_quant_blockfp8_weight(w, N, K, q, s, reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess
             ? R4_OK
             : R4_ERR_CUDA;
}

size_t r4_quant_mxfp4_act_scale_bytes(int64_t M, int64_t K) {
  if (M < 1 || K < 32 || K % 32) return 0;
  return mx_act_scale_bytes(M, K);
}

int r4_quant_mxfp4_act(const uint16_t *x, int64_t M, int64_t K, int64_t ldx, uint8_t *q, uint8_t *scale,
                       size_t scale_bytes, r4_stream_t stream) {
  if (!x || !q || !scale) return R4_ERR_INVALID_ARG;
  if (M < 1 || K < 32 || ldx < K || M > (1 << 30) || K > (1 << 30)) return R4_ERR_INVALID_ARG;
  if (K % 32 || ldx % 8) return R4_ERR_UNSUPPORTED_SHAPE;
  // one warp per 256 columns of a token: the grid must fit a launch
  if (ceil_div(M * ceil_div(K, 256), 8) + ceil_div(K, 128) + 1 > 0x7fffffff) return R4_ERR_UNSUPPORTED_SHAPE;
  if (!aligned(x, 16) || !aligned(q, 16) || !aligned(scale, 16)) return R4_ERR_MISALIGNED;
  if (scale_bytes < mx_act_scale_bytes(M, K)) return R4_ERR_WORKSPACE;
  return launch_quant_mxfp4_act(x, M, K, ldx, q, scale, reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess
             ? R4_OK
             : R4_ERR_CUDA;
}

size_t r4_prepack_mxfp4_bytes(int64_t N, int64_t K) {
  if (N < 1 || K < 32 || K % 32) return 0;
  return mx_packed_bytes(N, K);
}

int r4_prepack_mxfp4(const uint8_t *w, const uint8_t *w_scale, int64_t N, int64_t K, void *packed,
                     size_t packed_bytes, r4_stream_t stream) {
  if (!w || !w_scale || !packed || N < 1 || K < 32) return R4_ERR_INVALID_ARG;
  if (K % 32) return R4_ERR_UNSUPPORTED_SHAPE;
  if (!aligned(w, 16) || !aligned(packed, 256)) return R4_ERR_MISALIGNED;
  if (packed_bytes < mx_packed_bytes(N, K)) return R4_ERR_WORKSPACE;
  return launch_prepack_mxfp4(w, w_scale, N, K, static_cast<uint8_t *>(packed),
                              reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess
             ? R4_OK
             : R4_ERR_CUDA;
}

size_t r4_prepack_blockfp8_bytes(int64_t N, int64_t K) {
  if (N < 128 || K < 128 || N % 128 || K % 128) return 0;
  return fp8_packed_bytes(N, K);
}

int r4_prepack_blockfp8(const uint8_t *w, const float *w_scale, int64_t N, int64_t K, void *packed,
                        size_t packed_bytes, r4_stream_t stream) {
  if (!w || !w_scale || !packed || N < 1 || K < 1) return R4_ERR_INVALID_ARG;
  if (N % 128 || K % 128) return R4_ERR_UNSUPPORTED_SHAPE;
  if (!aligned(w, 16) || !aligned(packed, 256) || !aligned(w_scale, 4)) return R4_ERR_MISALIGNED;
  if (packed_bytes < fp8_packed_bytes(N, K)) return R4_ERR_WORKSPACE;
  return launch_prepack_blockfp8(w, w_scale, N, K, static_cast<uint8_t *>(packed),
                                 reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess
             ? R4_OK
             : R4_ERR_CUDA;
}

size_t r4_gemm_workspace_bytes(int op, int64_t M, int64_t N, int64_t K) {
  if (M < 1 || N < 1 || K < 1) return 0;
  switch (op) {
    case R4_OP_W4A8_MXFP4:
      if (K % 32 || K < 128) return 0;
      return plan_w4a8(M, N, K, device_sm_count()).ws_bytes;
    case R4_OP_BLOCKFP8:
      if (N % 128 || K % 128) return 0;
      return plan_blockfp8(M, N, K, device_sm_count()).ws_bytes;
    case R4_OP_W4A4_MXFP4:
      if (K % 32 || K < 128) return 0;
      return plan_w4a4(M, N, K, device_sm_count()).ws_bytes;
    case R4_OP_LINEAR_W4A8_MXFP4:
      if (K % 32 || K < 128) return 0;
      return linear_gemm_part_bytes(plan_w4a8(M, N, K, device_sm_count()).ws_bytes) + linear_scratch_bytes(M, K);
    default: return 0;
  }
}

int r4_plan_gemm(int op, int64_t M, int64_t N, int64_t K, int sms, int32_t *out) {
  if (!out || M < 1 || N < 1 || K < 1 || sms < 1 || M > 0x7fffffff || N > 0x7fffffff || K > 0x7fffffff)
    return R4_ERR_INVALID_ARG;
  GemmPlan pl;
  switch (op) {
    case R4_OP_W4A8_MXFP4:
    case R4_OP_LINEAR_W4A8_MXFP4:
      if (K % 32 || K < 128) return R4_ERR_UNSUPPORTED_SHAPE;
      pl = plan_w4a8(M, N, K, sms);
      break;
    case R4_OP_W4A4_MXFP4:
      if (K % 32 || K < 128) return R4_ERR_UNSUPPORTED_SHAPE;
      pl = plan_w4a4(M, N, K, sms);
      break;
    case R4_OP_BLOCKFP8:
      if (N % 128 || K % 128) return R4_ERR_UNSUPPORTED_SHAPE;
      pl = plan_blockfp8(M, N, K, sms);
      break;
    default: return R4_ERR_INVALID_ARG;
  }
  const int32_t v[10] = {pl.BT, pl.BN, pl.n_tiles, pl.t_tiles, pl.splits, pl.kb_per_split, pl.units, pl.grid,
                         pl.cluster, pl.sk};
  for (int i = 0; i < 10; ++i) out[i] = v[i];
  return R4_OK;
}

int r4_gemm_w4a8_mxfp4(const uint8_t *q, const float *s, const void *packed, int64_t M, int64_t N, int64_t K,
                       uint16_t *c, int64_t ldc, void *workspace, size_t workspace_bytes, r4_stream_t stream) {
  if (!q || !s || !packed || !c) return R4_ERR_INVALID_ARG;
  if (M < 1 || N < 1 || K < 1 || ldc < N || M > (1 << 30) || N > (1 << 30)) return R4_ERR_INVALID_ARG;
  if (K % 32 || K < 128) return R4_ERR_UNSUPPORTED_SHAPE;
  if (!aligned(q, 16) || !aligned(packed, 256) || !aligned(s, 4) || !aligned(c, 2)) return R4_ERR_MISALIGNED;
  const GemmPlan pl = plan_w4a8(M, N, K, device_sm_count());
  if (pl.ws_bytes > 0) {
    if (!workspace || workspace_bytes < pl.ws_bytes) return R4_ERR_WORKSPACE;
    if (!aligned(workspace, 256)) return R4_ERR_MISALIGNED;
  }
  if (device_error_word() == nullptr) return R4_ERR_CUDA;
  return launch_gemm_w4a8(q, s, static_cast<const uint8_t *>(packed), M, N, K, c, ldc,
                          pl.ws_bytes ? workspace : nullptr, pl, reinterpret_cast<cudaStream_t>(stream));
}

int r4_linear_w4a8_mxfp4(const uint16_t *x, int64_t ldx, const void *packed, int64_t M, int64_t N, int64_t K,
                         uint16_t *c, int64_t ldc, void *workspace, size_t workspace_bytes, r4_stream_t stream) {
  if (!x || !packed || !c) return R4_ERR_INVALID_ARG;
  if (M < 1 || N < 1 || K < 1 || ldc < N || ldx < K || M > (1 << 30) || N > (1 << 30)) return R4_ERR_INVALID_ARG;
  if (K % 32 || K < 128 || ldx % 8) return R4_ERR_UNSUPPORTED_SHAPE;
  if (!aligned(packed, 256) || !aligned(c, 2) || !aligned(x, 16)) return R4_ERR_MISALIGNED;
  const GemmPlan pl = plan_w4a8(M, N, K, device_sm_count());
  // [the GEMM's workspace, counters first, at least the counter region][q][s]
  const size_t gpart = linear_gemm_part_bytes(pl.ws_bytes);
  if (!workspace || workspace_bytes < gpart + linear_scratch_bytes(M, K)) return R4_ERR_WORKSPACE;
  if (!aligned(workspace, 256)) return R4_ERR_MISALIGNED;
  if (device_error_word() == nullptr) return R4_ERR_CUDA;
  const cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  void *gws = pl.ws_bytes ? workspace : nullptr;
  uint8_t *q = static_cast<uint8_t *>(workspace) + gpart;
  float *s = reinterpret_cast<float *>(q + round_up(static_cast<size_t>(M) * K, 256));
  if (launch_quant_act(x, M, K, ldx, K, q, s, st) != cudaSuccess) return R4_ERR_CUDA;
  return launch_gemm_w4a8(q, s, static_cast<const uint8_t *>(packed), M, N, K, c, ldc, gws, pl, st);
}

int r4_gemm_w4a4_mxfp4(const uint8_t *q, const uint8_t *q_scale, const void *packed, int64_t M, int64_t N, int64_t K,
                       uint16_t *c, int64_t ldc, void *workspace, size_t workspace_bytes, r4_stream_t stream) {
  if (!q || !q_scale || !packed || !c) return R4_ERR_INVALID_ARG;
  if (M < 1 || N < 1 || K < 1 || ldc < N || M > (1 << 30) || N > (1 << 30)) return R4_ERR_INVALID_ARG;
  if (K % 32 || K < 128) return R4_ERR_UNSUPPORTED_SHAPE;
  if (!aligned(q, 16) || !aligned(q_scale, 16) || !aligned(packed, 256) || !aligned(c, 2)) return R4_ERR_MISALIGNED;
  const GemmPlan pl = plan_w4a4(M, N, K, device_sm_count());
  if (pl.ws_bytes > 0) {
    if (!workspace || workspace_bytes < pl.ws_bytes) return R4_ERR_WORKSPACE;
    if (!aligned(workspace, 256)) return R4_ERR_MISALIGNED;
  }
  if (device_error_word() == nullptr) return R4_ERR_CUDA;
  return launch_gemm_w4a4(q, q_scale, static_cast<const uint8_t *>(packed), M, N, K, c, ldc,
                          pl.ws_bytes ? workspace : nullptr, pl, reinterpret_cast<cudaStream_t>(stream));
}

int r4_gemm_blockfp8(const uint8_t *q, const float *As, const void *packed, int64_t M, int64_t N, int64_t K,
                     uint16_t *c, int64_t ldc, void *workspace, size_t workspace_bytes, r4_stream_t stream) {
  if (!q || !As || !packed || !c) return R4_ERR_INVALID_ARG;
  if (M < 1 || N < 1 || K < 1 || ldc < N || M > (1 << 30) || N > (1 << 30)) return R4_ERR_INVALID_ARG;
  if (N % 128 || K % 128) return R4_ERR_UNSUPPORTED_SHAPE;
  if (!aligned(q, 16) || !aligned(packed, 256) || !aligned(As, 4) || !aligned(c, 2)) return R4_ERR_MISALIGNED;
  const GemmPlan pl = plan_blockfp8(M, N, K, device_sm_count());
  if (pl.ws_bytes > 0) {
    if (!workspace || workspace_bytes < pl.ws_bytes) return R4_ERR_WORKSPACE;
    if (!aligned(workspace, 256)) return R4_ERR_MISALIGNED;
  }
  if (device_error_word() == nullptr) return R4_ERR_CUDA;
  return launch_gemm_blockfp8(q, As, static_cast<const uint8_t *>(packed), M, N, K, c, ldc,
                              pl.ws_bytes ? workspace : nullptr, pl, reinterpret_cast<cudaStream_t>(stream));
}

int r4_gemm_bf16_nt_skinny(const uint16_t *x, const uint16_t *w, int64_t M, int64_t N, int64_t K, uint16_t *c,
                           int64_t ldc, void *workspace, size_t workspace_bytes, r4_stream_t stream) {
  (void)workspace;
  (void)workspace_bytes;
  if (!x || !w || !c) return R4_ERR_INVALID_ARG;
  if (M < 1 || N < 1 || K < 1 || ldc < N || N > (1 << 30) || K > (1 << 30)) return R4_ERR_INVALID_ARG;
  if (M > 64 || K % 256) return R4_ERR_UNSUPPORTED_SHAPE;
  if (!aligned(x, 16) || !aligned(w, 16) || !aligned(c, 2)) return R4_ERR_MISALIGNED;
  return launch_gemm_skinny(x, w, M, N, K, c, ldc, reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess
             ? R4_OK
             : R4_ERR_CUDA;
}

}  // extern "C"
