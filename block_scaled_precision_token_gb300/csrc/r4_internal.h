// r4_internal.h -- host-side declarations shared by the library's translation
// units: schedule plans, tensor-map encoding, kernel launchers.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include <utility>

#include "../../include/r4q.h"

namespace r4 {

// ------------------------------------------------------------------ device info
int device_sm_count();           // SM count of the current device (cached per device)
int *device_error_word();        // device address of the error word (current device)
void set_last_kernel(const char *name);
// cudaFuncSetAttribute(MaxDynamicSharedMemorySize) once per (device, kernel).
cudaError_t ensure_smem_attr(const void *func, int bytes);

// Encode a tiled tensor map through the driver entry point (no libcuda link).
CUresult encode_tiled(CUtensorMap *map, CUtensorMapDataType dtype, uint32_t rank, void *gaddr,
                      const uint64_t *dims, const uint64_t *strides_bytes, const uint32_t *box,
                      CUtensorMapSwizzle swizzle);

// ------------------------------------------------------------------ options
struct Options {
  int w4a8_splits = 0;      // 0 = automatic
  int w4a8_token_tile = 0;  // 0 = automatic
  int fp8_splits = 0;       // 0 = automatic
  int fp8_token_tile = 0;   // 0 = automatic, else 16/32/64/128
  int fp8_n_tile = 0;       // block-FP8 128-token tiles: weight rows per tile, 0 = automatic, else 128/256
  int inject_stall = 0;     // tests only: the next W4A8/W4A4, block-FP8 and staged producer launches withhold one
                            // copy (bounded-wait test)
  int pdl = 1;              // launch with programmatic stream serialization
  int early_weights = 1;    // GEMMs read their weight operand before waiting for the preceding kernel
  int l2_prefetch = 2;      // W4A8/W4A4 decode tiles: 2 rolling L2 prefetch ahead of the ring, 1 whole range at
                            // kernel start, 0 none
  int cluster_split = 1;    // W4A8 decode tiles: split-K across a thread-block cluster when possible
  int row_split = 0;        // row-wise quantizers: CTAs per row (0 = automatic, else 1/2/4/8)
  int row_threads = 0;      // row-wise quantizers: threads per CTA at most (0 = automatic, else 64/128/256)
  int skinny_groups = 0;    // skinny GEMM: 16-token groups per CTA (0 = automatic, else 1..4)
  int stream_k = 0;         // W4A8/W4A4 decode tiles: stream-K schedule 0 never (default), 1 when the model gains, 2 always
};
Options &options();

// CTAs that share one row of a row-wise quantization kernel (1, 2, 4 or 8):
// short batches spread each row over a thread-block cluster so that more
// than M SMs take part.
enum class RowKind { kQuant, kNorm, kSilu };   // per-token quant, add+RMS norm+quant, SiLU-and-mul+quant
int row_split(int64_t M, int64_t K, RowKind kind);
// Threads per CTA at most for a row slice of `vecs` 16-byte vectors.
int row_threads(RowKind kind, int64_t M, int64_t vecs);

// Launch `kernel` on `st`; with options().pdl the launch allows programmatic
// dependent launch (the kernel may start before its predecessor in the
// stream finishes; it orders its dependent accesses with griddepcontrol.wait).
template <typename Kern, typename... Args>
cudaError_t launch_pdl(Kern kernel, dim3 grid, dim3 block, size_t smem, cudaStream_t st, Args &&...args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = options().pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// launch_pdl with a 1-D thread-block cluster of `cluster_x` CTAs.
template <typename Kern, typename... Args>
cudaError_t launch_pdl_cluster(Kern kernel, dim3 grid, dim3 block, size_t smem, cudaStream_t st, int cluster_x,
                               Args &&...args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = static_cast<unsigned>(cluster_x);
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = options().pdl ? 2 : 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// ------------------------------------------------------------------ plans
// One output tile = BN weight rows (n) x BT tokens (t). A work unit is a
// tile and a contiguous range of 128-K blocks (its split).
struct GemmPlan {
  int BT = 0;            // token tile
  int BN = 128;          // weight rows per tile (block-FP8 token-major tiles: 128 or 256)
  int n_tiles = 0, t_tiles = 0;
  int KB = 0;            // number of 128-K blocks (K padded to 128)
  int splits = 1, kb_per_split = 0;
  int units = 0, grid = 0;
  int cluster = 0;       // 1: split-K across a cluster of `splits` CTAs (partials in DSMEM, no workspace)
  int sk = 0;            // 1: stream-K (grid CTAs share the tile-major K blocks equally; units = grid x sk_segs)
  int sk_total = 0;      // stream-K: tiles x KB
  size_t counters_bytes = 0;  // arrival counters (one int per tile): kCounterBytes when used
  size_t ws_bytes = 0;        // total workspace (0 when splits == 1)
};

GemmPlan plan_w4a8(int64_t M, int64_t N, int64_t K, int sms);
GemmPlan plan_w4a4(int64_t M, int64_t N, int64_t K, int sms);
GemmPlan plan_blockfp8(int64_t M, int64_t N, int64_t K, int sms);

// ------------------------------------------------------------------ prepack layout
inline int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }
inline size_t round_up(size_t a, size_t b) { return (a + b - 1) / b * b; }
// Split-K / stream-K workspaces of every GEMM start with the same fixed
// region of arrival counters (one int per output tile), then the fp32
// partials. A fixed region keeps the counters where another shape's call on
// the same workspace left them zero: no call's partials ever overlap it.
// Schedules with more output tiles than the region holds run unsplit.
constexpr size_t kCounterBytes = 16384;
constexpr int64_t kMaxCounterTiles = static_cast<int64_t>(kCounterBytes / 4);
// r4_linear_w4a8_mxfp4's own part of its workspace: the e4m3 codes [M][K]
// and the token scales [M]. It follows the GEMM's part, which always
// reserves the counter region (so that this transient scratch never lands
// on another call's counters).
inline size_t linear_scratch_bytes(int64_t M, int64_t K) {
  return round_up(static_cast<size_t>(M) * static_cast<size_t>(K), 256) + round_up(static_cast<size_t>(M) * 4, 256);
}
inline size_t linear_gemm_part_bytes(size_t gemm_ws_bytes) {
  return gemm_ws_bytes > kCounterBytes ? gemm_ws_bytes : kCounterBytes;
}

constexpr int64_t kMxTileCodeBytes = 128 * 64;   // 128 rows x 128 K packed e2m1
constexpr int64_t kMxTileSfBytes = 512;          // 128 rows x 4 ue8m0, copy order
constexpr int64_t kFp8TileBytes = 128 * 128;     // 128 rows x 128 K e4m3

inline size_t mx_packed_codes_bytes(int64_t N, int64_t K) {
  return static_cast<size_t>(ceil_div(N, 128) * ceil_div(K, 128) * kMxTileCodeBytes);
}
inline size_t mx_packed_bytes(int64_t N, int64_t K) {
  return mx_packed_codes_bytes(N, K) + static_cast<size_t>(ceil_div(N, 128) * ceil_div(K, 128) * kMxTileSfBytes);
}
inline size_t fp8_packed_codes_bytes(int64_t N, int64_t K) { return static_cast<size_t>(N * K); }
// MXFP4 activation scales (W4A4): 512-byte atoms of 128 tokens x 128 K, for
// the token count rounded up to a multiple of 256 (so a 256-token tile
// always has both of its atoms).
inline int64_t mx_act_tokens_padded(int64_t M) { return ceil_div(M, 256) * 256; }
inline size_t mx_act_scale_bytes(int64_t M, int64_t K) {
  return static_cast<size_t>(mx_act_tokens_padded(M) / 128 * ceil_div(K, 128) * 512);
}
inline size_t fp8_packed_bytes(int64_t N, int64_t K) {
  return round_up(fp8_packed_codes_bytes(N, K) + static_cast<size_t>((N / 128) * (K / 128) * 4), 256);
}

// ------------------------------------------------------------------ launchers
// All return cudaSuccess or the launch error; arguments are already validated.
cudaError_t launch_add_rmsnorm_quant(const uint16_t *y, const uint16_t *res, const uint16_t *w, float eps, int64_t M,
                                     int64_t K, uint16_t *ro, uint8_t *q, float *s, cudaStream_t st);
cudaError_t launch_silu_mul_quant(const uint16_t *gu, int64_t M, int64_t N, uint8_t *q, float *s, cudaStream_t st);
cudaError_t launch_check_quotients(unsigned long long *count, float *example, cudaStream_t st);
cudaError_t launch_quant_act(const uint16_t *x, int64_t M, int64_t K, int64_t ldx, int64_t group, uint8_t *q,
                             float *s, cudaStream_t st);
cudaError_t launch_quant_mxfp4_act(const uint16_t *x, int64_t M, int64_t K, int64_t ldx, uint8_t *q, uint8_t *sf,
                                   cudaStream_t st);
cudaError_t launch_quant_mxfp4_weight(const float *w, int64_t N, int64_t K, uint8_t *packed, uint8_t *scale,
                                      cudaStream_t st);
cudaError_t launch_quant_blockfp8_weight(const float *w, int64_t N, int64_t K, uint8_t *q, float *s,
                                         cudaStream_t st);
cudaError_t launch_prepack_mxfp4(const uint8_t *w, const uint8_t *ws, int64_t N, int64_t K, uint8_t *packed,
                                 cudaStream_t st);
cudaError_t launch_prepack_blockfp8(const uint8_t *w, const float *ws, int64_t N, int64_t K, uint8_t *packed,
                                   cudaStream_t st);
// Returns an r4_status (tensor-map encoding can fail with R4_ERR_CUDA).
int launch_gemm_w4a8(const uint8_t *q, const float *s, const uint8_t *packed, int64_t M, int64_t N, int64_t K,
                     uint16_t *c, int64_t ldc, void *ws, const GemmPlan &plan, cudaStream_t st);
int launch_gemm_w4a4(const uint8_t *q, const uint8_t *q_scale, const uint8_t *packed, int64_t M, int64_t N,
                     int64_t K, uint16_t *c, int64_t ldc, void *ws, const GemmPlan &plan, cudaStream_t st);
int launch_gemm_blockfp8(const uint8_t *q, const float *As, const uint8_t *packed, int64_t M, int64_t N,
                         int64_t K, uint16_t *c, int64_t ldc, void *ws, const GemmPlan &plan, cudaStream_t st);
// Tensor-core issue-rate probe (kind 1 mxf8f6f4, 2 f8f6f4, 3 mxf4; n = 128 or 256).
cudaError_t launch_mma_peak(int kind, int n, int blocks, int iters, cudaStream_t st);
cudaError_t launch_gemm_skinny(const uint16_t *x, const uint16_t *w, int64_t M, int64_t N, int64_t K, uint16_t *c,
                               int64_t ldc, cudaStream_t st);

}  // namespace r4
