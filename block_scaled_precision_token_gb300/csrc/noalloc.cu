// noalloc.cu -- r4_gemm_w4a8_mxfp4_noalloc: the W4A8 MXFP4 GEMM for callers
// that cannot allocate device memory.
//
// Who needs it: code that runs while a CUDA graph is being captured (a
// cudaMalloc there is illegal and aborts the capture), and hosts that hand a
// kernel library only the input/output pointers and a stream (custom-op and
// plugin interfaces of inference runtimes, fixed-pool embedded deployments).
// Such callers cannot provide the split-K workspace that r4_gemm_w4a8_mxfp4
// asks for.
//
// How: the split-K arrival counters and fp32 partials live in one file-scope
// static device array of kNoallocScratchBytes (16 MiB). Every GPU that loads
// the library holds it until the process exits. Host code may not use the
// array's name as a device address (it is a host-side stand-in), so the
// first call on each device looks the address up with cudaGetSymbolAddress,
// with that device current, and caches it. That first call should therefore
// come before any stream capture. Every call clears the counters (a
// cudaMemsetAsync on the caller's stream) before the GEMM, which then runs
// exactly as r4_gemm_w4a8_mxfp4 does with this array as its workspace.
// All calls share the array: two calls whose kernels can overlap on the GPU
// (different streams, or different host threads) race on it.

#include <mutex>

#include "r4_internal.h"

namespace r4 {
namespace {

constexpr size_t kNoallocScratchBytes = size_t(16) << 20;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoallocScratchBytes];

constexpr int kMaxDev = 64;
void *g_scratch_ptr[kMaxDev];
std::mutex g_scratch_mu;

// Device address of the static scratch on the current device (set up once).
void *scratch_address() {
  int d = 0;
  if (cudaGetDevice(&d) != cudaSuccess || d < 0 || d >= kMaxDev) return nullptr;
  std::lock_guard<std::mutex> lk(g_scratch_mu);
  if (g_scratch_ptr[d] == nullptr) {
    void *ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess) return nullptr;
    g_scratch_ptr[d] = ptr;
  }
  return g_scratch_ptr[d];
}

}  // namespace
}  // namespace r4

extern "C" int r4_gemm_w4a8_mxfp4_noalloc(const uint8_t *q, const float *s, const void *packed, int64_t M, int64_t N,
                                          int64_t K, uint16_t *c, int64_t ldc, r4_stream_t stream) {
  using namespace r4;
  if (!q || !s || !packed || !c) return R4_ERR_INVALID_ARG;
  if (M < 1 || N < 1 || K < 1 || ldc < N || M > (1 << 30) || N > (1 << 30)) return R4_ERR_INVALID_ARG;
  if (K % 32 || K < 128) return R4_ERR_UNSUPPORTED_SHAPE;
  // the same alignment rules as r4_gemm_w4a8_mxfp4, checked before any device query
  if (reinterpret_cast<uintptr_t>(q) % 16 || reinterpret_cast<uintptr_t>(packed) % 256 ||
      reinterpret_cast<uintptr_t>(s) % 4 || reinterpret_cast<uintptr_t>(c) % 2)
    return R4_ERR_MISALIGNED;
  const GemmPlan pl = plan_w4a8(M, N, K, device_sm_count());
  if (pl.ws_bytes > kNoallocScratchBytes) return R4_ERR_WORKSPACE;   // beyond the static maximum
  void *ws = nullptr;
  if (pl.ws_bytes > 0) {
    ws = scratch_address();
    if (ws == nullptr) return R4_ERR_CUDA;
    if (cudaMemsetAsync(ws, 0, pl.counters_bytes, reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
      return R4_ERR_CUDA;
  }
  return r4_gemm_w4a8_mxfp4(q, s, packed, M, N, K, c, ldc, ws, pl.ws_bytes, stream);
}
