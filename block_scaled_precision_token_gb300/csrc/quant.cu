// quant.cu -- e4m3 activation quantization (per token / per token per 128 K)
// and the load-time weight quantizers (OCP MX FP4, 128x128 block e4m3).
//
// Activation rule ("radiance_mxfp4.py", _traced_quant and the comment above
// it): s = max(amax/448, 1/(448*512)) in fp32, q = e4m3_rne_sat(x / s). Both
// divisions are correctly rounded (the scale by __fdiv_rn, the quotients by
// div_by_scale, proved equal to __fdiv_rn on the quantizers' domain), so the
// codes are bit-exact against any other correctly rounded fp32
// implementation.
//
// HBM-bound: 2 bytes read, 1 byte (+ scales) written per element. The CTAs
// of a row keep it in registers (read once), with 16-byte vector loads; a
// short batch spreads each row over a thread-block cluster whose CTAs agree
// on the row maximum through distributed shared memory.

#include <algorithm>

#include <cuda_bf16.h>
#include <cuda_fp4.h>
#include <cuda_fp8.h>

#include "quant_common.cuh"
#include "r4_device.cuh"
#include "r4_internal.h"

namespace r4 {
namespace {

using namespace qc;

// C CTAs per row (C = 1, or a thread-block cluster of C when the row's scale
// needs the whole row); CTA `part` owns columns [part * cols, part * cols +
// cols) and keeps them in registers, VPT 16-byte vectors per thread.
template <int VPT>
__global__ void __launch_bounds__(256) quant_act_kernel(const uint16_t *__restrict__ x, int K, int64_t ldx,
                                                        int group, int cols, int C, uint8_t *__restrict__ q,
                                                        float *__restrict__ s) {
  if (threadIdx.x == 0) pdl_launch_dependents();   // the next kernel may start its weight stream
  pdl_wait();                                       // x (and the q, s buffers) follow the stream order
  const int row = blockIdx.x / C;
  const int part = blockIdx.x - row * C;
  const int c0 = part * cols;
  const int c1 = min(K, c0 + cols);
  const int tid = threadIdx.x;
  const int nt = blockDim.x;
  const uint16_t *xr = x + static_cast<size_t>(row) * ldx;
  uint8_t *qr = q + static_cast<size_t>(row) * K;
  uint4 v[VPT];
#pragma unroll
  for (int i = 0; i < VPT; ++i) {
    const int k = c0 + (i * nt + tid) * 8;
    v[i] = (k < c1) ? __ldg(reinterpret_cast<const uint4 *>(xr + k)) : make_uint4(0, 0, 0, 0);
  }
  if (group == K) {
    __shared__ float red[8];
    __shared__ float slot;
    float a = 0.f;
#pragma unroll
    for (int i = 0; i < VPT; ++i) a = fmaxf(a, absmax8(v[i]));
    a = warp_max(a);
    if ((tid & 31) == 0) red[tid >> 5] = a;
    __syncthreads();
    a = red[0];
    for (int w = 1; w < (nt >> 5); ++w) a = fmaxf(a, red[w]);
    if (C > 1) {
      a = cluster_combine<true>(a, &slot, C);
      cluster_arrive();
    }
    const float sc = fmaxf(__fdiv_rn(a, kFp8Max), kMinScale);
    const float rc = __frcp_rn(sc);
    if (part == 0 && tid == 0) s[row] = sc;
#pragma unroll
    for (int i = 0; i < VPT; ++i) {
      const int k = c0 + (i * nt + tid) * 8;
      if (k < c1) *reinterpret_cast<uint2 *>(qr + k) = quant8(v[i], sc, rc);
    }
    if (C > 1) cluster_wait();   // peers may still read `slot` until they arrive
  } else {
    // group of 128 = 16 lanes x 8 elements; nt is a multiple of 32 and c0 of 128
    const int groups = K / 128;
#pragma unroll
    for (int i = 0; i < VPT; ++i) {
      const int k = c0 + (i * nt + tid) * 8;
      float a = absmax8(v[i]);
#pragma unroll
      for (int o = 8; o > 0; o >>= 1) a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, o));
      const float sc = fmaxf(__fdiv_rn(a, kFp8Max), kMinScale);
      if (k < c1) {
        if ((tid & 15) == 0) s[static_cast<size_t>(row) * groups + (k >> 7)] = sc;
        *reinterpret_cast<uint2 *>(qr + k) = quant8(v[i], sc, __frcp_rn(sc));
      }
    }
  }
}

// Two-pass variant for rows too long to hold in registers (re-reads x).
__global__ void __launch_bounds__(256) quant_act_long_kernel(const uint16_t *__restrict__ x, int K, int64_t ldx,
                                                             int group, uint8_t *__restrict__ q,
                                                             float *__restrict__ s) {
  if (threadIdx.x == 0) pdl_launch_dependents();   // the next kernel may start its weight stream
  pdl_wait();                                       // x (and the q, s buffers) follow the stream order
  const int row = blockIdx.x;
  const int tid = threadIdx.x;
  const int nt = blockDim.x;
  const uint16_t *xr = x + static_cast<size_t>(row) * ldx;
  uint8_t *qr = q + static_cast<size_t>(row) * K;
  if (group == K) {
    __shared__ float red[8];
    float a = 0.f;
    for (int k = tid * 8; k < K; k += nt * 8) a = fmaxf(a, absmax8(__ldg(reinterpret_cast<const uint4 *>(xr + k))));
    a = warp_max(a);
    if ((tid & 31) == 0) red[tid >> 5] = a;
    __syncthreads();
    a = red[0];
    for (int w = 1; w < (nt >> 5); ++w) a = fmaxf(a, red[w]);
    const float sc = fmaxf(__fdiv_rn(a, kFp8Max), kMinScale);
    const float rc = __frcp_rn(sc);
    if (tid == 0) s[row] = sc;
    for (int k = tid * 8; k < K; k += nt * 8)
      *reinterpret_cast<uint2 *>(qr + k) = quant8(__ldg(reinterpret_cast<const uint4 *>(xr + k)), sc, rc);
  } else {
    const int groups = K / 128;
    for (int base = 0; base < K; base += nt * 8) {
      const int k = base + tid * 8;
      const uint4 v = (k < K) ? __ldg(reinterpret_cast<const uint4 *>(xr + k)) : make_uint4(0, 0, 0, 0);
      float a = absmax8(v);
#pragma unroll
      for (int o = 8; o > 0; o >>= 1) a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, o));
      const float sc = fmaxf(__fdiv_rn(a, kFp8Max), kMinScale);
      if (k < K) {
        if ((tid & 15) == 0) s[static_cast<size_t>(row) * groups + (k >> 7)] = sc;
        *reinterpret_cast<uint2 *>(qr + k) = quant8(v, sc, __frcp_rn(sc));
      }
    }
  }
}

// OCP MX FP4: one thread per 32-element block.
__global__ void quant_mxfp4_weight_kernel(const float *__restrict__ w, int64_t N, int64_t K,
                                          uint8_t *__restrict__ packed, uint8_t *__restrict__ scale) {
  const int64_t nblk = K / 32;
  const int64_t b = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (b >= N * nblk) return;
  const int64_t row = b / nblk, kb = b % nblk;
  const float4 *src = reinterpret_cast<const float4 *>(w + row * K + kb * 32);
  float v[32];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const float4 f = __ldg(src + i);
    v[4 * i] = f.x; v[4 * i + 1] = f.y; v[4 * i + 2] = f.z; v[4 * i + 3] = f.w;
  }
  float amax = 0.f;
#pragma unroll
  for (int i = 0; i < 32; ++i) amax = fmaxf(amax, fabsf(v[i]));
  int X = 0;
  if (amax > 0.f) {
    int e;
    frexpf(amax, &e);        // amax = m 2^e, 0.5 <= m < 1
    X = (e - 1) - 2;         // floor(log2 amax) - emax(e2m1)
  }
  int code = X + 127;
  code = code < 0 ? 0 : (code > 254 ? 254 : code);
  X = code - 127;
  uint32_t out[4] = {0, 0, 0, 0};
#pragma unroll
  for (int i = 0; i < 32; ++i) {
    const uint32_t c =
        static_cast<uint32_t>(__nv_cvt_float_to_fp4(ldexpf(v[i], -X), __NV_E2M1, cudaRoundNearest)) & 0xFu;
    out[i / 8] |= c << (4 * (i % 8));
  }
  *reinterpret_cast<uint4 *>(packed + row * (K / 2) + kb * 16) = make_uint4(out[0], out[1], out[2], out[3]);
  scale[row * nblk + kb] = static_cast<uint8_t>(code);
}

// MXFP4 activations for the W4A4 GEMM: the OCP MX rule of the weights, per
// 32 K of each token. A warp quantizes SEGW segments of 256 consecutive
// columns of one token; all of its loads are issued before any arithmetic,
// so each lane keeps SEGW 16-byte loads in flight. Measured on GB300
// (graph-timed): with one segment per warp the kernel was latency-bound at
// ~2.9 TB/s (M=8192, K=5120: 36.6 us); four per warp: 25.0 us (4.2 TB/s).
// Short batches keep one segment per warp (more warps, a shorter serial
// path: M=8, K=5120 1.5 vs 2.2 us). In a segment lane l holds
// columns [8l, 8l + 8), lanes 4j .. 4j + 3 form 32-element block j (their
// maximum by two shuffles), and each lane packs its 8 codes into one
// 32-bit store (column 2i in the low nibble of byte i). The four scale codes
// of a 128-K block are one 32-bit word of the token's scale atom row (byte
// j = 32-K block j), OR-combined over the 16 lanes by shuffles and stored
// by one lane:
//   scale atom (a, kb) at (kb * A + a) * 512 (A = atoms per K block, the
//   token count padded to 256, / 128): 512 bytes, byte 16 r0 + 4 r1 + j =
//   token 128 a + 32 r1 + r0, 32-K block 4 kb + j. K-block-major, so the two
//   atoms of a 256-token tile are one contiguous 1 KB copy.
// Blocks past K and padding tokens (M .. the atoms' end) get code 127 (x1).
// Blocks of the grid past `real_blocks` write those padding tokens' words.
// Two fp32 -> two e2m1 codes in one instruction (round to nearest even,
// saturating to +-6): lo in bits 0-3, hi in bits 4-7.
__device__ __forceinline__ uint32_t e2m1x2_of(float lo, float hi) {
  uint32_t r;
  asm("{\n\t.reg .b8 t;\n\tcvt.rn.satfinite.e2m1x2.f32 t, %1, %2;\n\tcvt.u32.u8 %0, t;\n\t}"
      : "=r"(r)
      : "f"(hi), "f"(lo));
  return r;
}

template <int SEGW>
__global__ void __launch_bounds__(256) quant_mxfp4_act_kernel(const uint16_t *__restrict__ x, int M, int K,
                                                              int64_t ldx, int segs, int KB, int A, int real_blocks,
                                                              int pad_tokens, uint8_t *__restrict__ q,
                                                              uint8_t *__restrict__ sf) {
  if (threadIdx.x == 0) pdl_launch_dependents();   // the next kernel may start its weight stream
  pdl_wait();                                       // x (and the q, sf buffers) follow the stream order
  const int lane = threadIdx.x & 31;
  if (static_cast<int>(blockIdx.x) >= real_blocks) {
    // padding tokens M .. M + pad_tokens: every word of their atom rows is 0x7F7F7F7F
    const int64_t i = static_cast<int64_t>(blockIdx.x - real_blocks) * blockDim.x + threadIdx.x;
    if (i >= static_cast<int64_t>(pad_tokens) * KB) return;
    const int t = M + static_cast<int>(i / KB), kb = static_cast<int>(i % KB);
    const int r = t & 127;
    *reinterpret_cast<uint32_t *>(sf + (static_cast<size_t>(kb) * A + (t >> 7)) * 512 + 16 * (r & 31) + 4 * (r >> 5)) =
        0x7F7F7F7Fu;
    return;
  }
  const int wpr = (segs + SEGW - 1) / SEGW;     // warps per row
  const int64_t wg = static_cast<int64_t>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (wg >= static_cast<int64_t>(M) * wpr) return;   // whole warps only
  const int row = static_cast<int>(wg / wpr), seg0 = static_cast<int>(wg % wpr) * SEGW;
  const uint16_t *xr = x + static_cast<size_t>(row) * ldx;
  uint4 v[SEGW];
#pragma unroll
  for (int g = 0; g < SEGW; ++g) {
    const int k = (seg0 + g) * 256 + lane * 8;
    v[g] = k < K ? __ldg(reinterpret_cast<const uint4 *>(xr + k)) : make_uint4(0, 0, 0, 0);
  }
#pragma unroll
  for (int g = 0; g < SEGW; ++g) {
    const int seg = seg0 + g;
    if (seg >= segs) break;   // warp-uniform
    const int k = seg * 256 + lane * 8;
    float a = absmax8(v[g]);
    a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 1));
    a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 2));
    int X = 0;
    if (a > 0.f) {
      int e;
      frexpf(a, &e);           // a = m 2^e, 0.5 <= m < 1
      X = (e - 1) - 2;         // floor(log2 amax) - emax(e2m1)
    }
    int code = X + 127;
    code = code < 0 ? 0 : (code > 254 ? 254 : code);
    X = code - 127;
    if (k < K) {
      // x / 2^X as one multiply by the exact power of two (2^-X, -X in
      // [-127, 127]: 2^-127 is the subnormal 0x00400000), rounded once like
      // the exact scaling it stands for
      const float p = -X >= -126 ? __uint_as_float(static_cast<uint32_t>(127 - X) << 23) : __uint_as_float(0x00400000u);
      const uint32_t w[4] = {v[g].x, v[g].y, v[g].z, v[g].w};
      uint32_t out = 0;   // element i in nibble i, two per conversion
#pragma unroll
      for (int i = 0; i < 4; ++i)
        out |= e2m1x2_of(__fmul_rn(bf16lo(w[i]), p), __fmul_rn(bf16hi(w[i]), p)) << (8 * i);
      *reinterpret_cast<uint32_t *>(q + static_cast<size_t>(row) * (K / 2) + k / 2) = out;
    }
    uint32_t word = static_cast<uint32_t>(code) << (8 * ((lane >> 2) & 3));
    word |= __shfl_xor_sync(0xffffffffu, word, 4);
    word |= __shfl_xor_sync(0xffffffffu, word, 8);
    const int kb = seg * 2 + (lane >> 4);
    if ((lane & 15) == 0 && kb < KB) {
      const int r = row & 127;
      *reinterpret_cast<uint32_t *>(sf + (static_cast<size_t>(kb) * A + (row >> 7)) * 512 + 16 * (r & 31) +
                                    4 * (r >> 5)) = word;
    }
  }
}

// 128x128 block e4m3: one CTA (256 threads) per block.
__global__ void __launch_bounds__(256) quant_blockfp8_weight_kernel(const float *__restrict__ w, int64_t N,
                                                                    int64_t K, uint8_t *__restrict__ q,
                                                                    float *__restrict__ s) {
  const int64_t nb = blockIdx.y, kb = blockIdx.x;
  const int tid = threadIdx.x;
  __shared__ float red[8];
  float a = 0.f;
  for (int i = tid; i < 128 * 32; i += 256) {   // 128 rows x 32 float4
    const int r = i / 32, c4 = i % 32;
    const float4 f = __ldg(reinterpret_cast<const float4 *>(w + (nb * 128 + r) * K + kb * 128) + c4);
    a = fmaxf(a, fmaxf(fmaxf(fabsf(f.x), fabsf(f.y)), fmaxf(fabsf(f.z), fabsf(f.w))));
  }
  a = warp_max(a);
  if ((tid & 31) == 0) red[tid >> 5] = a;
  __syncthreads();
  a = red[0];
  for (int i = 1; i < 8; ++i) a = fmaxf(a, red[i]);
  float sc = __fdiv_rn(a, kFp8Max);
  if (sc == 0.f) sc = 1.f;
  if (tid == 0) s[nb * (K / 128) + kb] = sc;
  for (int i = tid; i < 128 * 32; i += 256) {
    const int r = i / 32, c4 = i % 32;
    const float4 f = __ldg(reinterpret_cast<const float4 *>(w + (nb * 128 + r) * K + kb * 128) + c4);
    const uint32_t b = e4m3_of(__fdiv_rn(f.x, sc)) | (e4m3_of(__fdiv_rn(f.y, sc)) << 8) |
                       (e4m3_of(__fdiv_rn(f.z, sc)) << 16) | (e4m3_of(__fdiv_rn(f.w, sc)) << 24);
    *reinterpret_cast<uint32_t *>(q + (nb * 128 + r) * K + kb * 128 + c4 * 4) = b;
  }
}

// Self-check of div_by_scale on the quantizers' whole domain: block b takes
// the bf16 amax with bit pattern b (0 .. 0x7F7F, every finite non-negative
// value), forms the scale the per-token rule derives from it, and compares
// div_by_scale with a correctly rounded division for every bf16 x with
// |x| <= amax, both signs. count[0]: pairs whose e4m3 codes differ (the
// first one's (x, s) lands in example[0..1]); count[2]: pairs whose fp32
// quotients differ at all; count[3]: the largest |x/s| (fp32 bits) among
// those. (Quotients of x within a few ulps of the fp32 normal range leave a
// remainder that underflows; they are far below the smallest e4m3 code.)
__global__ void __launch_bounds__(256) check_quotients_kernel(unsigned long long *count, float *example) {
  const uint32_t vb = blockIdx.x;
  const float sc = fmaxf(__fdiv_rn(__uint_as_float(vb << 16), kFp8Max), kMinScale);
  const float rc = __frcp_rn(sc);
  unsigned int bad_code = 0, bad_bits = 0, worst = 0;
  for (uint32_t m = threadIdx.x; m <= vb; m += blockDim.x) {
#pragma unroll
    for (uint32_t sgn = 0; sgn < 2; ++sgn) {
      const float x = __uint_as_float((m | (sgn << 15)) << 16);
      const float exact = __fdiv_rn(x, sc), fast = div_by_scale(x, sc, rc);
      if (__float_as_uint(exact) != __float_as_uint(fast)) {
        ++bad_bits;
        worst = max(worst, __float_as_uint(fabsf(exact)));
        if (e4m3_of(exact) != e4m3_of(fast)) {
          ++bad_code;
          if (atomicAdd(count + 1, 1ull) == 0) {
            example[0] = x;
            example[1] = sc;
          }
        }
      }
    }
  }
  if (bad_code) atomicAdd(count, static_cast<unsigned long long>(bad_code));
  if (bad_bits) {
    atomicAdd(count + 2, static_cast<unsigned long long>(bad_bits));
    atomicMax(count + 3, static_cast<unsigned long long>(worst));
  }
}

}  // namespace

cudaError_t launch_check_quotients(unsigned long long *count, float *example, cudaStream_t st) {
  cudaError_t e = cudaMemsetAsync(count, 0, 4 * sizeof(unsigned long long), st);
  if (e != cudaSuccess) return e;
  check_quotients_kernel<<<0x7F80, 256, 0, st>>>(count, example);
  set_last_kernel("check_quotients_kernel");
  return cudaGetLastError();
}

cudaError_t launch_quant_act(const uint16_t *x, int64_t M, int64_t K, int64_t ldx, int64_t group, uint8_t *q,
                             float *s, cudaStream_t st) {
  const bool per_token = group == K;
  int C = row_split(M, K, RowKind::kQuant);
  if (M * C > (int64_t{1} << 30)) C = 1;
  const int64_t align = per_token ? 8 : 128;
  int64_t cols = ceil_div(ceil_div(K, static_cast<int64_t>(C)), align) * align;
  int64_t vecs = cols / 8;
  const int cap = row_threads(RowKind::kQuant, M, vecs);
  int threads = static_cast<int>(vecs < cap ? ((vecs + 31) / 32) * 32 : cap);
  if (threads < 32) threads = 32;
  int64_t per = ceil_div(vecs, threads);
  if (per > 12 && threads < 256) {   // a capped block too small for the row: widen it first
    threads = static_cast<int>(std::min<int64_t>(256, ceil_div(ceil_div(vecs, int64_t{12}), int64_t{32}) * 32));
    per = ceil_div(vecs, threads);
  }
  if (per > 12 && C > 1) {   // the row does not fit in registers even when split: two-pass kernel
    C = 1;
    cols = K;
    threads = 256;
    per = 13;
  }
  const dim3 grid(static_cast<unsigned>(M * C));
  const int g = static_cast<int>(group), k = static_cast<int>(K), cl = static_cast<int>(cols);
#define R4_QA(V)                                                                                             \
  {                                                                                                          \
    const cudaError_t e =                                                                                    \
        (per_token && C > 1)                                                                                 \
            ? launch_pdl_cluster(quant_act_kernel<V>, grid, dim3(threads), 0, st, C, x, k, ldx, g, cl, C, q, s) \
            : launch_pdl(quant_act_kernel<V>, grid, dim3(threads), 0, st, x, k, ldx, g, cl, C, q, s);         \
    if (e != cudaSuccess) return e;                                                                          \
    set_last_kernel("quant_act_kernel<" #V ">");                                                             \
  }
  if (per <= 1) R4_QA(1) else if (per <= 2) R4_QA(2) else if (per <= 4) R4_QA(4) else if (per <= 6) R4_QA(6)
  else if (per <= 9) R4_QA(9) else if (per <= 12) R4_QA(12)
  else {
    const cudaError_t e = launch_pdl(quant_act_long_kernel, grid, dim3(threads), 0, st, x, k, ldx, g, q, s);
    if (e != cudaSuccess) return e;
    set_last_kernel("quant_act_long_kernel");
  }
#undef R4_QA
  return cudaGetLastError();
}

cudaError_t launch_quant_mxfp4_weight(const float *w, int64_t N, int64_t K, uint8_t *packed, uint8_t *scale,
                                      cudaStream_t st) {
  const int64_t blocks = N * (K / 32);
  quant_mxfp4_weight_kernel<<<static_cast<unsigned>(ceil_div(blocks, 256)), 256, 0, st>>>(w, N, K, packed, scale);
  set_last_kernel("quant_mxfp4_weight_kernel");
  return cudaGetLastError();
}

cudaError_t launch_quant_mxfp4_act(const uint16_t *x, int64_t M, int64_t K, int64_t ldx, uint8_t *q, uint8_t *sf,
                                   cudaStream_t st) {
  const int segs = static_cast<int>(ceil_div(K, 256));
  const int KB = static_cast<int>(ceil_div(K, 128));
  // four segments per warp once the batch has enough warps to fill the GPU
  const int segw = M * segs >= 32 * 8 * static_cast<int64_t>(device_sm_count()) ? 4 : 1;
  const int64_t real_blocks = ceil_div(M * ceil_div(segs, segw), 8);
  const int64_t pad_tokens = mx_act_tokens_padded(M) - M;
  const int A = static_cast<int>(mx_act_tokens_padded(M) / 128);
  const int64_t pad_blocks = ceil_div(pad_tokens * KB, 256);
  const dim3 grid(static_cast<unsigned>(real_blocks + pad_blocks));
  const cudaError_t e =
      segw == 4 ? launch_pdl(quant_mxfp4_act_kernel<4>, grid, dim3(256), 0, st, x, static_cast<int>(M),
                             static_cast<int>(K), ldx, segs, KB, A, static_cast<int>(real_blocks),
                             static_cast<int>(pad_tokens), q, sf)
                : launch_pdl(quant_mxfp4_act_kernel<1>, grid, dim3(256), 0, st, x, static_cast<int>(M),
                             static_cast<int>(K), ldx, segs, KB, A, static_cast<int>(real_blocks),
                             static_cast<int>(pad_tokens), q, sf);
  if (e != cudaSuccess) return e;
  set_last_kernel("quant_mxfp4_act_kernel");
  return cudaGetLastError();
}

cudaError_t launch_quant_blockfp8_weight(const float *w, int64_t N, int64_t K, uint8_t *q, float *s,
                                         cudaStream_t st) {
  const dim3 grid(static_cast<unsigned>(K / 128), static_cast<unsigned>(N / 128));
  quant_blockfp8_weight_kernel<<<grid, 256, 0, st>>>(w, N, K, q, s);
  set_last_kernel("quant_blockfp8_weight_kernel");
  return cudaGetLastError();
}

}  // namespace r4
