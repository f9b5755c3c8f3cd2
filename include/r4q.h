/*
 * r4q.h -- C ABI of the GB300 (sm_103a) block-scaled quantized linear library.
 *
 * The library computes the quantized linear-layer hot path described on the
 * pages "radiance_mxfp4.py" (W4A8 MXFP4 linear with per-token e4m3
 * activations), "radiance_kernels.py" (block-FP8 W8A8 GEMM, block_scaled_mm)
 * and "radiance_gemm.py" (skinny bf16 NT GEMM), re-designed for tcgen05
 * tensor cores, TMA and HBM3e.
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - Every pointer argument is a DEVICE pointer unless stated otherwise. All
 *    buffers are allocated and owned by the caller; the library never
 *    allocates device memory, never synchronizes the device or a stream, and
 *    never throws. This keeps every call legal inside CUDA-graph capture.
 *  - Every kernel is launched on `stream` (a cudaStream_t; 0 = legacy default
 *    stream). Results are ready when the stream reaches that point.
 *  - bf16 tensors are passed as uint16_t bit patterns, e4m3 / e2m1 / ue8m0
 *    codes as uint8_t. Matrices are row-major; "ld" arguments are row strides
 *    in elements.
 *  - Every call returns an R4_* status. On an error nothing is launched, except
 *    R4_ERR_CUDA, which reports a failure of the launch itself.
 *  - A device-side wait that runs out (a TMA or tensor-core completion that
 *    never arrives) makes the kernel stop early and set a device error word;
 *    r4_device_error() reads and clears it.
 *  - The per-token path (quantization and the three GEMMs) is launched with
 *    programmatic dependent launch: a kernel may start while its predecessor
 *    in the stream is still running. Activations, scales, outputs and the
 *    workspace are touched only after the kernel's dependency wait, which
 *    returns once every preceding kernel has completed and its writes are
 *    visible. The GEMMs read their WEIGHT operand (the prepacked buffer; the
 *    bf16 matrix w of the skinny GEMM) BEFORE that wait, so that the weight
 *    stream overlaps the tail of the preceding kernel. Rule for whoever writes
 *    a weight:
 *      * r4_prepack_mxfp4 / r4_prepack_blockfp8 may be followed by a GEMM
 *        directly: their kernels are launched without programmatic
 *        dependence and make every write visible device-wide before they
 *        exit.
 *      * A weight written by anything else (a kernel of another library, a
 *        copy) must be separated from the GEMM by a full stream
 *        serialization point: a cudaMemcpy*Async, an event wait, a host
 *        synchronization, or a kernel launched without programmatic
 *        dependence. This library's own per-token kernels are NOT such a
 *        point (they are launched with programmatic dependence).
 *      * Callers that cannot guarantee this turn the early weight read off
 *        with r4_set_option(14, 0) (the GEMMs then wait first and read
 *        after), or turn programmatic dependent launch off altogether with
 *        r4_set_option(4, 0).
 */
#ifndef R4Q_H
#define R4Q_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st *r4_stream_t; /* == cudaStream_t */

enum r4_status {
  R4_OK = 0,
  R4_ERR_INVALID_ARG = 1,       /* null pointer, non-positive or inconsistent size */
  R4_ERR_UNSUPPORTED_SHAPE = 2, /* shape outside the supported set (see each call) */
  R4_ERR_MISALIGNED = 3,        /* pointer or stride alignment rule broken */
  R4_ERR_WORKSPACE = 4,         /* workspace or prepack buffer too small */
  R4_ERR_CUDA = 5,              /* a CUDA runtime/driver call failed */
  R4_ERR_DEVICE_TIMEOUT = 6     /* a kernel's bounded device-side wait ran out */
};

/* GEMM identifiers for r4_gemm_workspace_bytes(). */
enum r4_gemm_op {
  R4_OP_W4A8_MXFP4 = 1,
  R4_OP_BLOCKFP8 = 2,
  R4_OP_BF16_SKINNY = 3,
  R4_OP_W4A4_MXFP4 = 4,
  R4_OP_LINEAR_W4A8_MXFP4 = 5 /* r4_linear_w4a8_mxfp4 */
};

int r4_version(void);                 /* (major << 16) | minor */
const char *r4_status_string(int status);
/* Name of the kernel the last successful launch on this host thread used. */
const char *r4_last_kernel_name(void);

/*
 * r4_device_error -- read (and with clear != 0, reset) the device error word
 * of the current device. 0 means no kernel has reported a timed-out wait.
 * Synchronous (it copies one word from the device): not for use in capture.
 */
int r4_device_error(int *error_out, int clear);

/*
 * r4_quant_fp8_per_token -- dynamic e4m3 activation quantization.
 * Source: "radiance_mxfp4.py", _traced_quant and the comment above it:
 *   s = max(amax(|x|) / 448, 1/(448*512))   (fp32, correctly rounded division)
 *   q = e4m3_rne(x / s), finite values saturate at +-448.
 * With group == K there is one scale per row (token); with group == 128 there
 * is one scale per token per 128 K, the activation side of block-FP8
 * ("radiance_kernels.py", block_scaled_mm).
 *   x     bf16 [M, ldx], row-major, first K columns used.  16-byte aligned.
 *   q     e4m3 [M, K] row-major (row stride K).            16-byte aligned.
 *   s     fp32 [M, K/group] row-major.
 * Requirements: M >= 1, K >= 8, K % 8 == 0, ldx >= K, ldx % 8 == 0,
 * group == K or (group == 128 and K % 128 == 0).
 * Non-finite input gives unspecified codes for that row (NaN poisons the scale).
 */
int r4_quant_fp8_per_token(const uint16_t *x, int64_t M, int64_t K, int64_t ldx,
                           int64_t group, uint8_t *q, float *s, r4_stream_t stream);

/*
 * r4_check_quotients -- device self-check of the quotient x / s that the
 * activation quantizers compute (a reciprocal and one FMA correction instead
 * of a full division): over every finite bf16 amax, the scale
 * s = max(amax/448, 1/(448*512)) the rule derives from it, and every bf16 x
 * with |x| <= amax (both signs), compares the quotient with a correctly
 * rounded fp32 division.
 *   count    device, 4 x uint64, zeroed by the call (stream-ordered), 8-byte
 *            aligned: [0] = pairs whose e4m3 codes differ (must be 0);
 *            [1] = internal; [2] = pairs whose fp32 quotients differ in any
 *            bit; [3] = fp32 bit pattern of the largest |x/s| among those.
 *   example  device, 2 x fp32: (x, s) of one pair with differing codes, if any.
 * Asynchronous on `stream`; ~1.07e9 pairs, about a millisecond on GB300.
 */
int r4_check_quotients(unsigned long long *count, float *example, r4_stream_t stream);

/*
 * r4_mma_peak -- tensor-core issue-rate probe, the denominator of the GEMMs'
 * roofline fractions. The pages measured their own matrix-instruction peak
 * the same way: a register-resident loop that touches no memory
 * ("radiance_mxfp4.py", module docstring, fp8 WMMA throughput). Launches
 * `blocks` CTAs (one per SM when blocks = the SM count); each zero-fills its
 * operand tiles in shared memory and one thread issues iters x 4 MMAs,
 * M = 128, N = n, into one tensor-memory accumulator:
 *   kind 1: kind::mxf8f6f4, e2m1 x e4m3, ue8m0 scales, K = 32 (the W4A8 GEMM);
 *   kind 2: kind::f8f6f4, e4m3 x e4m3, K = 32 (the block-FP8 GEMM);
 *   kind 3: kind::mxf4, e2m1 x e2m1, ue8m0 scales, K = 64.
 * Flops per launch = blocks * iters * 4 * 2 * 128 * n * K. Time it with
 * events on `stream`. Requirements: n = 128 or 256, 1 <= blocks <= 65535,
 * iters >= 1. No memory argument: nothing is read or written outside the
 * kernel's own shared and tensor memory.
 */
int r4_mma_peak(int kind, int n, int blocks, int iters, r4_stream_t stream);

/*
 * r4_add_rmsnorm_quant_fp8 -- residual add + Gemma RMS norm + per-token e4m3
 * quantization in one launch: the single-rank epilogue of
 * "radiance_arnq.py" (module docstring; ar_add_rms_quant):
 *   r[m,k]  = bf16(y[m,k] + residual[m,k])                    (fp32 add)
 *   h[m,k]  = bf16(r[m,k] / sqrt(mean_k(r^2) + eps) * (1 + w[k]))
 *   (q, s)  = the r4_quant_fp8_per_token rule on h (one scale per row)
 * The norm is formed in fp32 (correctly rounded division and reciprocal
 * square root); r is written to residual_out, which may be the residual
 * buffer itself (in-place update).
 *   y, residual, residual_out  bf16 [M, K] row-major (row stride K), 16-byte aligned.
 *   weight                     bf16 [K], 16-byte aligned.
 *   q  e4m3 [M, K] (8-byte aligned);  s  fp32 [M].
 * Requirements: M >= 1, K % 8 == 0, 8 <= K <= 24576, eps finite and >= 0.
 */
int r4_add_rmsnorm_quant_fp8(const uint16_t *y, const uint16_t *residual, const uint16_t *weight,
                             float eps, int64_t M, int64_t K, uint16_t *residual_out,
                             uint8_t *q, float *s, r4_stream_t stream);

/*
 * r4_silu_mul_quant_fp8 -- SiluAndMul + per-token e4m3 quantization in one
 * launch ("radiance_arnq.py", silu_mul_quant and the _SiluMulQuant
 * docstring). For each row of gu = [g | u] (N columns each):
 *   a = bf16(g / (1 + exp(-g))),  h = bf16(a * u),  (q, s) = per-token rule on h.
 *   gu  bf16 [M, 2N] row-major, 16-byte aligned;  q  e4m3 [M, N] (8-byte aligned);
 *   s   fp32 [M].
 * Requirements: M >= 1, N % 8 == 0, 8 <= N <= 24576.
 */
int r4_silu_mul_quant_fp8(const uint16_t *gu, int64_t M, int64_t N, uint8_t *q, float *s,
                          r4_stream_t stream);

/*
 * r4_quantize_mxfp4_weight -- OCP MX FP4 quantization of a float32 weight
 * (a load-time utility, not on the per-token path): per 32-element block of a
 * row, X = floor(log2(amax)) - 2 (all-zero block: X = 0), scale code X + 127
 * clamped to [0, 254], element = e2m1_rne_sat(w / 2^X).
 *   w       fp32 [N, K] row-major.
 *   packed  uint8 [N, K/2]: element 2j in the low nibble of byte j
 *           ("radiance_mxfp4.py", _exact_ref).
 *   scale   uint8 [N, K/32] ue8m0 (value 2^(code-127)).
 * Requirements: N >= 1, K % 32 == 0.
 */
int r4_quantize_mxfp4_weight(const float *w, int64_t N, int64_t K, uint8_t *packed,
                             uint8_t *scale, r4_stream_t stream);

/*
 * r4_quantize_blockfp8_weight -- 128x128 block e4m3 weight quantization
 * (load-time utility): s = amax/448 in fp32 (1 for an all-zero block),
 * q = e4m3_rne_sat(w / s).
 *   w      fp32 [N, K];  q  uint8 [N, K];  s  fp32 [N/128, K/128] (multiplier).
 * Requirements: N % 128 == 0, K % 128 == 0.
 */
int r4_quantize_blockfp8_weight(const float *w, int64_t N, int64_t K, uint8_t *q,
                                float *s, r4_stream_t stream);

/*
 * r4_quant_mxfp4_act -- MXFP4 activation quantization for the W4A4 GEMM.
 * Source: "radiance_mxfp4.py", module docstring and _debug_compare: the W4A4
 * path that the page's W4A8 kernel replaces quantizes the activations to
 * MXFP4 (the page measures its error against the exact product: relative
 * Frobenius 0.1119, against 0.0265 for W4A8). The page does not print that
 * quantizer's rule; this library reads it as the OCP MX v1.0 rule of the
 * weights (r4_quantize_mxfp4_weight), per 32 K of each token:
 *   X = floor(log2(amax)) - 2 (all-zero block: X = 0), scale code X + 127
 *   clamped to [0, 254], element = e2m1_rne_sat(x / 2^X).
 *   x      bf16 [M, ldx] row-major, first K columns used; 16-byte aligned.
 *   q      uint8 [M, K/2] packed e2m1, element 2j in the low nibble of byte j
 *          (the checkpoint order of the weights); 16-byte aligned.
 *   scale  the ue8m0 scale codes in the GEMM's scale-atom layout, 16-byte
 *          aligned, at least r4_quant_mxfp4_act_scale_bytes(M, K) bytes:
 *          atoms of 512 bytes, K-block-major: atom (a, kb) at byte offset
 *          (kb * A + a) * 512, A = ceil(M/256) * 2, for tokens
 *          [128 a, 128 a + 128) and K block [128 kb, 128 kb + 128) (the two
 *          atoms of a 256-token tile are adjacent); inside it, byte 16 r0 + 4 r1 + j
 *          is the scale of token 128 a + 32 r1 + r0, 32-K block 4 kb + j --
 *          the order in which tcgen05.cp 32x128b.warpx4 lays a scale block
 *          across tensor memory, the same as the weight's prepacked atoms.
 *          Tokens are padded to a multiple of 256 and K to a multiple of
 *          128; the padding holds code 127 (x1).
 * Requirements: M >= 1, K >= 32, K % 32 == 0, ldx >= K, ldx % 8 == 0.
 * Non-finite input gives unspecified codes for its 32-element block.
 */
size_t r4_quant_mxfp4_act_scale_bytes(int64_t M, int64_t K);
int r4_quant_mxfp4_act(const uint16_t *x, int64_t M, int64_t K, int64_t ldx, uint8_t *q,
                       uint8_t *scale, size_t scale_bytes, r4_stream_t stream);

/*
 * r4_prepack_mxfp4 -- one-time permutation of a checkpoint-order MXFP4 weight
 * into the GEMM-native layout (no re-quantization). Source of the idea:
 * "radiance_mxfp4.py", permute_w (a byte permutation done once at load so the
 * kernel's weight reads are contiguous). The layout here is the TMA/tcgen05
 * one: 128-row x 128-K tiles of packed codes (8 KiB each, tile-major along K)
 * followed by one 512-byte scale atom per tile in tensor-memory copy order.
 * Rows beyond N and K beyond the true K are padded with code 0 / scale 127.
 *   w        uint8 [N, K/2] packed e2m1, checkpoint order.
 *   w_scale  uint8 [N, K/32] ue8m0, checkpoint order [N, K/32].
 *   packed   output buffer of at least r4_prepack_mxfp4_bytes(N, K) bytes,
 *            256-byte aligned. Opaque: only r4_gemm_w4a8_mxfp4 reads it.
 * Requirements: N >= 1, K >= 32, K % 32 == 0.
 */
size_t r4_prepack_mxfp4_bytes(int64_t N, int64_t K);
int r4_prepack_mxfp4(const uint8_t *w, const uint8_t *w_scale, int64_t N, int64_t K,
                     void *packed, size_t packed_bytes, r4_stream_t stream);

/*
 * r4_prepack_blockfp8 -- one-time permutation of an e4m3 [N, K] weight into
 * 128x128 K-major tiles (16 KiB each, tile-major along K), followed by a copy
 * of the fp32 block scales. Source: "radiance_kernels.py", the preshuffle load
 * hook (only genuine 128-block weights: N % 128 == 0, K % 128 == 0, scale
 * [N/128, K/128]).
 *   w        uint8 [N, K] e4m3.   w_scale  fp32 [N/128, K/128].
 *   packed   >= r4_prepack_blockfp8_bytes(N, K) bytes, 256-byte aligned.
 */
size_t r4_prepack_blockfp8_bytes(int64_t N, int64_t K);
int r4_prepack_blockfp8(const uint8_t *w, const float *w_scale, int64_t N, int64_t K,
                        void *packed, size_t packed_bytes, r4_stream_t stream);

/*
 * r4_gemm_workspace_bytes -- device workspace a GEMM call needs for (M, N, K):
 * a fixed 16 KiB region of int32 arrival counters (one per output tile) at
 * the start, then the split-K fp32 partials. 0 when the chosen schedule needs
 * none (schedules with more than 4096 output tiles never split). Because the
 * counters are always at the start and no call writes anything else there,
 * one workspace may serve calls of different ops and shapes one after
 * another (sized for the largest). The counters must be zero when the
 * workspace is first used (e.g. cudaMemsetAsync once after allocation); every
 * call leaves them zero again, including a call whose kernel stopped early
 * because a bounded device wait expired (r4_device_error reports it): such a
 * launch still arrives, marked incomplete, at every counter it owed, and the
 * last arrival at a tile resets the counter without summing (that tile's
 * output is then unspecified, like the rest of that call's output). One
 * workspace must not serve two calls that can run at the same time (two
 * streams).
 */
size_t r4_gemm_workspace_bytes(int op, int64_t M, int64_t N, int64_t K);

/*
 * r4_plan_gemm -- the schedule a GEMM call of `op` (R4_OP_W4A8_MXFP4,
 * R4_OP_BLOCKFP8, R4_OP_W4A4_MXFP4, R4_OP_LINEAR_W4A8_MXFP4: its GEMM) would
 * launch for (M, N, K) on a GPU with `sms` streaming multiprocessors, under
 * the current r4_set_option overrides. Host arithmetic: the block-FP8
 * planner touches no device; the W4A8/W4A4 planners ask the current device
 * how many thread-block clusters of a split fit, and without one take no
 * cluster split. out: int32[10], host memory, written on R4_OK:
 *   [0] token tile  [1] weight rows per tile  [2] weight-row tiles
 *   [3] token tiles  [4] K splits  [5] 128-K blocks per split
 *   [6] work units  [7] grid (CTAs)  [8] split across a cluster (0/1)
 *   [9] stream-K schedule (0/1; then [6] counts stream-K segments)
 * R4_ERR_INVALID_ARG for a null out, non-positive sizes or another op;
 * R4_ERR_UNSUPPORTED_SHAPE where the GEMM call would refuse the shape.
 */
int r4_plan_gemm(int op, int64_t M, int64_t N, int64_t K, int sms, int32_t *out);

/*
 * r4_gemm_w4a8_mxfp4 -- C = bf16( s[m] * sum_k e4m3(q[m,k]) * e2m1(w[n,k]) * 2^(e[n,k/32]-127) ).
 * Source: "radiance_mxfp4.py", module docstring and _exact_ref.
 * Runs on tcgen05 block-scaled MMA (kind::mxf8f6f4, ue8m0 scale per 32 K) with
 * the weight as the 128-row MMA operand; token tiles of 16..256; split-K with
 * a last-arriving-CTA reduction when there are too few output tiles to fill
 * the GPU. Decode (M <= 64) and prefill use the same kernel.
 *   q       e4m3 [M, K] row-major (from r4_quant_fp8_per_token), 16-B aligned.
 *   s       fp32 [M] per-token scale.
 *   packed  prepacked weight from r4_prepack_mxfp4(N, K).
 *   c       bf16 [M, ldc] row-major; columns [0, N) are written, nothing else.
 * Requirements: M >= 1, N >= 1, K % 32 == 0, ldc >= N.
 */
int r4_gemm_w4a8_mxfp4(const uint8_t *q, const float *s, const void *packed, int64_t M,
                       int64_t N, int64_t K, uint16_t *c, int64_t ldc, void *workspace,
                       size_t workspace_bytes, r4_stream_t stream);

/*
 * r4_linear_w4a8_mxfp4 -- the W4A8 linear layer from bf16 activations:
 * r4_quant_fp8_per_token(x, group = K) followed by r4_gemm_w4a8_mxfp4, with
 * the same result bit for bit.
 * Source: "radiance_mxfp4.py", module docstring (per-token FP8 activations
 * feeding the W4A8 GEMM) and _traced_quant (the quantization rule).
 * It runs the quantization kernel into the workspace and then the GEMM (two
 * launches, the second under programmatic dependent launch).
 *   x        bf16 [M, ldx] row-major, ldx >= K, ldx % 8 == 0, 16-byte aligned.
 *   packed   prepacked weight from r4_prepack_mxfp4(N, K).
 *   c        bf16 [M, ldc] row-major; columns [0, N) are written, nothing else.
 *   workspace  r4_gemm_workspace_bytes(R4_OP_LINEAR_W4A8_MXFP4, M, N, K)
 *            bytes, 256-byte aligned, counters zeroed once: the GEMM's
 *            workspace (counter region always reserved), then room for the
 *            quantized activations and their scales.
 * Requirements: M >= 1, N >= 1, K % 32 == 0, K >= 128, ldc >= N. Errors as
 * r4_gemm_w4a8_mxfp4 (R4_ERR_WORKSPACE for a missing or short workspace).
 */
int r4_linear_w4a8_mxfp4(const uint16_t *x, int64_t ldx, const void *packed, int64_t M, int64_t N,
                         int64_t K, uint16_t *c, int64_t ldc, void *workspace, size_t workspace_bytes,
                         r4_stream_t stream);

/*
 * r4_gemm_w4a4_mxfp4 -- the W4A4 variant, MXFP4 activations x MXFP4 weights:
 *   C = bf16( sum_k e2m1(q[m,k]) 2^(a[m,k/32]-127) * e2m1(w[n,k]) 2^(e[n,k/32]-127) ).
 * Source: "radiance_mxfp4.py", module docstring and _debug_compare (the W4A4
 * path). tcgen05 kind::mxf4 (twice the f8 rate): both operands packed e2m1
 * in shared memory, both ue8m0 scales in tensor memory, so there is no
 * per-token epilogue scale. Same kernel structure, schedules and split-K as
 * r4_gemm_w4a8_mxfp4 (workspace: r4_gemm_workspace_bytes(R4_OP_W4A4_MXFP4, ...)),
 * with token tiles of 128 or 256, or one tile of up to 64 tokens.
 *   q        packed e2m1 [M, K/2] from r4_quant_mxfp4_act, 16-byte aligned.
 *   q_scale  its scale atoms (r4_quant_mxfp4_act), 16-byte aligned.
 *   packed   prepacked weight from r4_prepack_mxfp4(N, K) (the W4A8 weight).
 *   c        bf16 [M, ldc]; columns [0, N) are written, nothing else.
 * Requirements: M >= 1, N >= 1, K % 32 == 0, K >= 128, ldc >= N.
 */
int r4_gemm_w4a4_mxfp4(const uint8_t *q, const uint8_t *q_scale, const void *packed, int64_t M,
                       int64_t N, int64_t K, uint16_t *c, int64_t ldc, void *workspace,
                       size_t workspace_bytes, r4_stream_t stream);

/*
 * r4_gemm_blockfp8 -- C = bf16( sum_kb As[m,kb] * Ws[n/128,kb] * sum_{k in kb} e4m3(q[m,k]) e4m3(w[n,k]) ).
 * Source: "radiance_kernels.py", block_scaled_mm.
 * tcgen05 kind::f8f6f4 MMA per 128-K block into a fresh tensor-memory
 * accumulator, promoted into fp32 registers with the scale product by the
 * epilogue warps (double-buffered so promotion overlaps the next block's MMA).
 *   q   e4m3 [M, K];  As fp32 [M, K/128] row-major (from group-128 quant);
 *   packed from r4_prepack_blockfp8(N, K);  c bf16 [M, ldc].
 * Requirements: N % 128 == 0, K % 128 == 0, M >= 1, ldc >= N.
 */
int r4_gemm_blockfp8(const uint8_t *q, const float *As, const void *packed, int64_t M,
                     int64_t N, int64_t K, uint16_t *c, int64_t ldc, void *workspace,
                     size_t workspace_bytes, r4_stream_t stream);

/*
 * r4_gemm_bf16_nt_skinny -- C = bf16( x W^T ) with fp32 accumulation, for tiny
 * projections. Source: "radiance_gemm.py", module docstring (C[M,N] =
 * x[M,K] @ W[N,K]^T, split-K because a sub-megabyte weight otherwise leaves the
 * GPU idle). Split-K across a thread-block cluster, reduced through
 * distributed shared memory: needs no workspace (pass NULL, 0).
 *   x  bf16 [M, K] row-major (row stride K);  w  bf16 [N, K] row-major;
 *   c  bf16 [M, ldc].  x and w 16-byte aligned.
 * Requirements: 1 <= M <= 64, N >= 1, K % 256 == 0, ldc >= N.
 */
int r4_gemm_bf16_nt_skinny(const uint16_t *x, const uint16_t *w, int64_t M, int64_t N,
                           int64_t K, uint16_t *c, int64_t ldc, void *workspace,
                           size_t workspace_bytes, r4_stream_t stream);

/*
 * r4_gemm_w4a8_mxfp4_noalloc -- r4_gemm_w4a8_mxfp4 for callers that cannot
 * allocate device memory. (No counterpart on the pages: it is a convenience of
 * this library.) Code that runs during CUDA-graph capture may not call
 * cudaMalloc, and inference-runtime plugin or custom-op interfaces often hand
 * a kernel only its input/output pointers and a stream; neither can supply
 * the split-K workspace. This variant takes the same arguments and returns
 * the same result minus the workspace: its split-K counters and partials live
 * in a library-owned static device buffer of 16 MiB, which every GPU that
 * loads the library holds until the process exits. It allocates nothing.
 *  - The first call on a device looks up that buffer's device address (with
 *    the device current) and caches it: make that first call before any
 *    stream capture.
 *  - Each call clears the buffer's counters on `stream` before the GEMM.
 *  - All calls share the buffer: calls whose kernels can overlap on the GPU
 *    (other streams, other host threads) race on it and must be serialized by
 *    the caller.
 *  - A shape whose split-K schedule needs more than 16 MiB returns
 *    R4_ERR_WORKSPACE without launching anything.
 */
int r4_gemm_w4a8_mxfp4_noalloc(const uint8_t *q, const float *s, const void *packed, int64_t M, int64_t N,
                               int64_t K, uint16_t *c, int64_t ldc, r4_stream_t stream);

/*
 * r4_set_option -- benchmarking overrides of the host-side schedule choice
 * (process-wide, not thread-safe). key 1: force the W4A8 split-K factor
 * (0 = automatic); key 2: force the W4A8/W4A4 token tile (0 = automatic,
 * else 16/32/64/128/192/256; 192 is a W4A8 tile, W4A4 then chooses its
 * own); key 3: force the block-FP8 split-K factor; key 4:
 * programmatic dependent launch on (1, default) or off (0); key 5: L2
 * prefetch of the weight stream of the W4A8/W4A4 GEMMs: 2 (default) a
 * rolling window of 8 K blocks beyond each decode CTA's pipeline ring, 1
 * each CTA's whole weight range at kernel start, 0 none;
 * key 6: W4A8 decode split-K across a thread-block cluster with the partial
 * sums exchanged in distributed shared memory (1, default) or through the
 * caller's workspace (0); key 7: force the block-FP8 token tile (0 =
 * automatic, else 16/32/64/128); key 8: weight rows per block-FP8 128-token
 * tile, 0 (default) 256 when N is a multiple of 256 and the 256-row tiles
 * occupy at least half of the SMs, else 128; 128 or 256 forces it (256 only
 * applies where N is a multiple of 256);
 * key 10 (tests of failure detection only):
 * 1 makes the next W4A8, W4A4 and block-FP8 launches, and the fused
 * producers' one-CTA-per-row launches, withhold one activation copy in
 * their first CTA, so a pipeline wait never completes, expires after
 * ~2 s and is reported by r4_device_error (the launch itself returns R4_OK,
 * the output is unspecified, the workspace counters end at zero and the
 * context stays usable); 0 (default) turns it off;
 * key 11: CTAs that share one row in the row-wise activation quantizers
 * (per-token, group-128 and the two fused producers): 0 (default) chooses
 * automatically (short batches spread each row over a cluster of up to 8
 * CTAs), 1/2/4/8 force it; other values return R4_ERR_INVALID_ARG;
 * key 13: threads per CTA at most in the same quantizers: 0 (default)
 * chooses (128 for slices of up to 6144 columns where that gains, 512 for
 * the SiLU producer's rows over 12288 columns at many tokens, else 256),
 * 64/128/256 cap it (a row that would need more than 12 vectors of 8
 * per thread widens the block again); other values return
 * R4_ERR_INVALID_ARG;
 * key 14: the GEMMs request their weight operand before waiting for the
 * preceding kernel (1, default) or only after it (0); see the weight-writer
 * rule at the top of this header;
 * key 15: skinny bf16 GEMM, 16-token groups per CTA: 0 (default) chooses,
 * 1..4 force it (the tokens are split over that many more CTAs); other
 * values return R4_ERR_INVALID_ARG;
 * key 16: stream-K schedule of the W4A8/W4A4 decode tiles (M <= 64): every
 * CTA streams an equal share of all tiles' K blocks, and a tile shared by
 * several CTAs is summed through the workspace by its last arrival, in K
 * order: 0 (default) never, 1 when the schedule model expects a gain, 2
 * always (unless key 1 forces a split factor); other values return
 * R4_ERR_INVALID_ARG. It changes r4_gemm_workspace_bytes: query it after
 * setting the option. (Measured on GB300 it is slower than the default
 * schedule on the decode shapes; it is an option for other shapes and
 * GPUs.)
 */
int r4_set_option(int key, int64_t value);

#ifdef __cplusplus
}
#endif
#endif /* R4Q_H */
