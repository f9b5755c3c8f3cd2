// fused_quant.cu -- per-token e4m3 quantization fused with the epilogue that
// produces a W4A8 linear's input ("radiance_arnq.py": ar_add_rms_quant and
// silu_mul_quant; the module docstring's single-rank epilogue).
//
//  * add + Gemma RMS norm + quant: r = bf16(y + residual) (the new residual,
//    written out), h = bf16(r / sqrt(mean(r^2) + eps) * (1 + w)), then the
//    per-token rule on h.
//  * SiluAndMul + quant on [g | u]: h = bf16(bf16(silu(g)) * u), then the
//    per-token rule.
//
// Row kernels, one launch where the unfused chain takes two or three: the
// row is read once, reduced (sum of squares, then the maximum magnitude)
// and written as codes. Where one CTA holds a whole row, the row is staged
// in shared memory by bulk asynchronous copies (one mbarrier per pass of the
// block's threads) and each thread keeps its results in registers; a short
// batch instead spreads each row over a thread-block cluster whose CTAs load
// their columns into registers and combine partial sums and maxima through
// distributed shared memory. Pairs of bf16 values are added, multiplied and
// rounded with packed bf16x2 instructions where that rounds as the
// definition does. The norm is fp32 with correctly rounded division and
// reciprocal square root; SiLU uses CUDA's expf and an approximate
// reciprocal (a few ulps); the codes come from correctly rounded quotients
// (quant_common.cuh).

#include <cuda_bf16.h>
#include <cuda_fp8.h>

#include "quant_common.cuh"
#include "r4_device.cuh"
#include "r4_internal.h"

namespace r4 {
namespace {

using namespace qc;

constexpr int kThreads = 256;
constexpr int kSiluThreads = 512;   // the SiLU producer's long rows at many tokens (row_threads)

__device__ __forceinline__ uint32_t bf16_rn_bits(float v) {
  const __nv_bfloat16 h = __float2bfloat16_rn(v);
  return static_cast<uint32_t>(*reinterpret_cast<const uint16_t *>(&h));
}
__device__ __forceinline__ uint32_t pack2(float lo, float hi) { return bf16_rn_bits(lo) | (bf16_rn_bits(hi) << 16); }

// Two floats to a bf16x2 word in one instruction, each rounded to nearest
// even: lo in bits 0-15.
__device__ __forceinline__ uint32_t bf16x2_rn(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

// Elementwise product of two bf16x2 words, each the exact product rounded
// once to bf16 (nearest even) -- what rounding the exact fp32 product of two
// bf16 values to bf16 gives.
__device__ __forceinline__ uint32_t mul_bf16x2(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}

// Elementwise sum of two bf16x2 words, each the exact sum rounded once to
// bf16 (nearest even) -- what rounding their fp32 sum to bf16 gives: two
// bf16 values whose exponents differ by at most 16 add exactly in fp32, and
// a farther one lies below half a bf16 ulp of the larger either way.
__device__ __forceinline__ uint32_t add_bf16x2(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("add.rn.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}

// Largest magnitude among 8 bf16 values, as a bf16x2 word of two candidates:
// the magnitudes' bit patterns order as the values do (finite or infinite),
// so a packed 16-bit integer maximum finds it.
__device__ __forceinline__ uint32_t absmax8_bits(const uint4 &v) {
  const uint32_t m = 0x7FFF7FFFu;
  uint32_t a, b;
  asm("max.u16x2 %0, %1, %2;" : "=r"(a) : "r"(v.x & m), "r"(v.y & m));
  asm("max.u16x2 %0, %1, %2;" : "=r"(b) : "r"(v.z & m), "r"(v.w & m));
  asm("max.u16x2 %0, %1, %2;" : "=r"(a) : "r"(a), "r"(b));
  return a;
}

// Block-wide sum / max of one float per thread (fixed order: deterministic).
__device__ __forceinline__ float block_sum(float a, float *red) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) a += __shfl_xor_sync(0xffffffffu, a, o);
  const int nw = blockDim.x >> 5;
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = a;
  __syncthreads();
  float t = red[0];
  for (int w = 1; w < nw; ++w) t += red[w];
  __syncthreads();   // red is reused by the next reduction
  return t;
}
__device__ __forceinline__ float block_max(float a, float *red) {
  a = warp_max(a);
  const int nw = blockDim.x >> 5;
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = a;
  __syncthreads();
  float t = red[0];
  for (int w = 1; w < nw; ++w) t = fmaxf(t, red[w]);
  return t;
}

// Scale and codes for the columns [c0, c1) of one row, held as bf16 vectors
// h[VPT]; the row's C CTAs (a cluster when C > 1) agree on its maximum.
// Writes s[row] (CTA 0 of the row) and the codes. With C > 1 the kernel
// must call cluster_wait() before it exits.
template <int VPT>
__device__ __forceinline__ void quant_row(const uint4 (&h)[VPT], int c0, int c1, int C, bool first, uint8_t *qr,
                                          float *s_row, float *red, float *slot) {
  const int tid = threadIdx.x, nt = blockDim.x;
  uint32_t ab = 0;                     // padding vectors are zero
#pragma unroll
  for (int i = 0; i < VPT; ++i) asm("max.u16x2 %0, %1, %2;" : "=r"(ab) : "r"(ab), "r"(absmax8_bits(h[i])));
  float a = fmaxf(bf16lo(ab), bf16hi(ab));
  a = block_max(a, red);
  if (C > 1) {
    a = cluster_combine<true>(a, slot, C);
    cluster_arrive();
  }
  const float sc = fmaxf(__fdiv_rn(a, kFp8Max), kMinScale);
  const float rc = __frcp_rn(sc);
  if (first && tid == 0) *s_row = sc;
#pragma unroll
  for (int i = 0; i < VPT; ++i) {
    const int k = c0 + (i * nt + tid) * 8;
    if (k < c1) *reinterpret_cast<uint2 *>(qr + k) = quant8(h[i], sc, rc);
  }
}

// The norm's output for 8 columns: h = bf16(RN(RN(r * inv) * (1 + w))) each.
__device__ __forceinline__ uint4 norm8(const uint4 &r4, const uint4 &w4, float inv) {
  const uint32_t rv[4] = {r4.x, r4.y, r4.z, r4.w}, wv[4] = {w4.x, w4.y, w4.z, w4.w};
  uint32_t hv[4];
#pragma unroll
  for (int j = 0; j < 4; ++j)
    hv[j] = bf16x2_rn(__fmul_rn(__fmul_rn(bf16lo(rv[j]), inv), 1.f + bf16lo(wv[j])),
                      __fmul_rn(__fmul_rn(bf16hi(rv[j]), inv), 1.f + bf16hi(wv[j])));
  return make_uint4(hv[0], hv[1], hv[2], hv[3]);
}

// One row per CTA, y and the residual staged in shared memory by bulk
// asynchronous copies, one pair per pass of the block's threads on its own
// mbarrier (as in the staged SiLU producer). The residual row is read into
// shared memory before any of it is written back, so ro may alias res.
template <int VPT>
__global__ void __launch_bounds__(kThreads) add_rmsnorm_quant_staged_kernel(const uint16_t *__restrict__ y,
                                                                          const uint16_t *res,
                                                                          const uint16_t *__restrict__ w, float eps,
                                                                          int K, uint16_t *ro,
                                                                          uint8_t *__restrict__ q,
                                                                          float *__restrict__ s, int *err,
                                                                          int inject) {
  extern __shared__ __align__(16) uint8_t smem_rows[];   // y row, then residual row (bf16)
  __shared__ float red[kThreads / 32];
  __shared__ float slot;
  __shared__ __align__(8) uint64_t bar[VPT];
  __shared__ int abort_flag;
  const int row = blockIdx.x, tid = threadIdx.x, nt = blockDim.x;
  const int nvec = K >> 3;
  const size_t base = static_cast<size_t>(row) * K;
  uint16_t *ys = reinterpret_cast<uint16_t *>(smem_rows);
  uint16_t *rs = ys + K;
  if (tid == 0) {
#pragma unroll
    for (int i = 0; i < VPT; ++i) mbar_init(&bar[i], 1);
    abort_flag = 0;
    fence_mbar_init();
    pdl_launch_dependents();
  }
  __syncthreads();
  pdl_wait();   // y and the residual come from the preceding kernels
  if (tid == 0) {
    const uint64_t pol = policy_evict_first();
#pragma unroll
    for (int i = 0; i < VPT; ++i) {
      const int v0 = i * nt;
      if (v0 < nvec) {
        const uint32_t bytes = static_cast<uint32_t>(min(nt, nvec - v0)) * 16u;
        mbar_arrive_expect_tx(&bar[i], 2u * bytes);
        // (failure-detection test: CTA 0 withholds its first pass, so that
        // pass's wait and the final drain run out)
        if (inject && blockIdx.x == 0 && i == 0) continue;
        bulk_load(ys + v0 * 8, y + base + v0 * 8, bytes, &bar[i], pol);
        bulk_load(rs + v0 * 8, res + base + v0 * 8, bytes, &bar[i], pol);
      }
    }
  }
  uint4 r[VPT];
  float ss = 0.f;
#pragma unroll
  for (int i = 0; i < VPT; ++i) {
    const int v = i * nt + tid;
    r[i] = make_uint4(0, 0, 0, 0);
    if (v < nvec && mbar_wait(&bar[i], 0, &abort_flag, err, DEV_ERR_WAIT_FULL)) {
      const uint4 a = *reinterpret_cast<const uint4 *>(ys + v * 8);
      const uint4 b = *reinterpret_cast<const uint4 *>(rs + v * 8);
      r[i] = make_uint4(add_bf16x2(a.x, b.x), add_bf16x2(a.y, b.y), add_bf16x2(a.z, b.z), add_bf16x2(a.w, b.w));
      const uint32_t rv[4] = {r[i].x, r[i].y, r[i].z, r[i].w};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const float lo = bf16lo(rv[j]), hi = bf16hi(rv[j]);
        ss = fmaf(lo, lo, ss);
        ss = fmaf(hi, hi, ss);
      }
      *reinterpret_cast<uint4 *>(ro + base + v * 8) = r[i];
    }
  }
  ss = block_sum(ss, red);
  const float inv = __frsqrt_rn(__fadd_rn(__fdiv_rn(ss, static_cast<float>(K)), eps));
#pragma unroll
  for (int i = 0; i < VPT; ++i) {
    const int v = i * nt + tid;
    if (v < nvec) r[i] = norm8(r[i], __ldg(reinterpret_cast<const uint4 *>(w + v * 8)), inv);
  }
  quant_row<VPT>(r, 0, K, 1, true, q + base, s + row, red, &slot);
  // Never leave a copy in flight (returns at once unless a wait above gave up).
  if (tid == 0) {
    volatile int dummy = 0;
#pragma unroll
    for (int i = 0; i < VPT; ++i)
      if (i * nt < nvec) mbar_wait(&bar[i], 0, &dummy, err, DEV_ERR_WAIT_DRAIN);
  }
}

// Row `blockIdx.x / C`, columns [part * cols, part * cols + cols) of it.
template <int VPT>
__global__ void __launch_bounds__(kThreads) add_rmsnorm_quant_kernel(const uint16_t *__restrict__ y,
                                                                   const uint16_t *res, const uint16_t *__restrict__ w,
                                                                   float eps, int K, int cols, int C, uint16_t *ro,
                                                                   uint8_t *__restrict__ q, float *__restrict__ s) {
  if (threadIdx.x == 0) pdl_launch_dependents();
  pdl_wait();   // y and the residual come from the preceding kernels
  __shared__ float red[kThreads / 32];
  __shared__ float slot[2];
  const int row = blockIdx.x / C, part = blockIdx.x - row * C, tid = threadIdx.x, nt = blockDim.x;
  const int c0 = part * cols, c1 = min(K, c0 + cols);
  const size_t base = static_cast<size_t>(row) * K;
  uint4 r[VPT];
  float ss = 0.f;
#pragma unroll
  for (int i = 0; i < VPT; ++i) {
    const int k = c0 + (i * nt + tid) * 8;
    if (k < c1) {
      // res may alias ro (in-place residual update): each vector is read
      // before the same thread writes it.
      const uint4 a = __ldg(reinterpret_cast<const uint4 *>(y + base + k));
      const uint4 b = *reinterpret_cast<const uint4 *>(res + base + k);
      const uint32_t av[4] = {a.x, a.y, a.z, a.w}, bv[4] = {b.x, b.y, b.z, b.w};
      uint32_t rv[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        rv[j] = pack2(bf16lo(av[j]) + bf16lo(bv[j]), bf16hi(av[j]) + bf16hi(bv[j]));
        const float lo = bf16lo(rv[j]), hi = bf16hi(rv[j]);
        ss = fmaf(lo, lo, ss);
        ss = fmaf(hi, hi, ss);
      }
      r[i] = make_uint4(rv[0], rv[1], rv[2], rv[3]);
      *reinterpret_cast<uint4 *>(ro + base + k) = r[i];
    } else {
      r[i] = make_uint4(0, 0, 0, 0);
    }
  }
  ss = block_sum(ss, red);
  if (C > 1) ss = cluster_combine<false>(ss, &slot[0], C);
  const float inv = __frsqrt_rn(__fadd_rn(__fdiv_rn(ss, static_cast<float>(K)), eps));
#pragma unroll
  for (int i = 0; i < VPT; ++i) {
    const int k = c0 + (i * nt + tid) * 8;
    if (k < c1) {
      r[i] = norm8(r[i], __ldg(reinterpret_cast<const uint4 *>(w + k)), inv);
    }
  }
  quant_row<VPT>(r, c0, c1, C, part == 0, q + base, s + row, red, &slot[1]);
  if (C > 1) cluster_wait();
}

// g * sigmoid(g) to a few float32 ulps: CUDA's expf, then g times the
// approximate reciprocal of 1 + exp(-g) (rcp.approx without flush to zero:
// within an ulp, subnormal reciprocals of denominators from 2^126 included;
// exp(-g) = inf gives -0 as the exact value rounds to). No branch.
__device__ __forceinline__ float silu_f32(float g) {
  const float t = 1.f + expf(-g);
  float r;
  asm("rcp.approx.f32 %0, %1;" : "=f"(r) : "f"(t));
  return g * r;
}

// h = bf16(bf16(silu(g)) * u) for 8 columns: one rounding each.
__device__ __forceinline__ uint4 silu_mul8(const uint4 &g4, const uint4 &u4) {
  const uint32_t gv[4] = {g4.x, g4.y, g4.z, g4.w}, uv[4] = {u4.x, u4.y, u4.z, u4.w};
  uint32_t hv[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) hv[j] = mul_bf16x2(bf16x2_rn(silu_f32(bf16lo(gv[j])), silu_f32(bf16hi(gv[j]))), uv[j]);
  return make_uint4(hv[0], hv[1], hv[2], hv[3]);
}

// One row per CTA, [g | u] staged in shared memory by bulk asynchronous
// copies: one pair per pass of the block's threads (pass i holds vectors
// [i * nt, (i + 1) * nt) of g and of u), each pass on its own mbarrier, all
// issued at once by one thread. The whole row is in flight without holding
// registers, and a pass is promoted as soon as it lands. (Three CTAs per SM
// at up to six passes.)
template <int VPT>
__global__ void __launch_bounds__(kSiluThreads, VPT <= 6 ? 3 : 2)
    silu_mul_quant_staged_kernel(const uint16_t *__restrict__ gu, int N, uint8_t *__restrict__ q,
                                 float *__restrict__ s, int *err, int inject) {
  extern __shared__ __align__(16) uint8_t smem_rows[];   // g row, then u row (bf16)
  __shared__ float red[kSiluThreads / 32];
  __shared__ float slot;
  __shared__ __align__(8) uint64_t bar[VPT];
  __shared__ int abort_flag;
  const int row = blockIdx.x, tid = threadIdx.x, nt = blockDim.x;
  const int nvec = N >> 3;
  uint16_t *gs = reinterpret_cast<uint16_t *>(smem_rows);
  uint16_t *us = gs + N;
  if (tid == 0) {
#pragma unroll
    for (int i = 0; i < VPT; ++i) mbar_init(&bar[i], 1);
    abort_flag = 0;
    fence_mbar_init();
    pdl_launch_dependents();
  }
  __syncthreads();
  pdl_wait();   // gu comes from the preceding kernel
  if (tid == 0) {
    const uint16_t *gr = gu + static_cast<size_t>(row) * 2 * N;
    const uint64_t pol = policy_evict_first();
#pragma unroll
    for (int i = 0; i < VPT; ++i) {
      const int v0 = i * nt;
      if (v0 < nvec) {
        const uint32_t bytes = static_cast<uint32_t>(min(nt, nvec - v0)) * 16u;
        mbar_arrive_expect_tx(&bar[i], 2u * bytes);
        // (failure-detection test: CTA 0 withholds its first pass)
        if (inject && blockIdx.x == 0 && i == 0) continue;
        bulk_load(gs + v0 * 8, gr + v0 * 8, bytes, &bar[i], pol);
        bulk_load(us + v0 * 8, gr + N + v0 * 8, bytes, &bar[i], pol);
      }
    }
  }
  uint4 h[VPT];
#pragma unroll
  for (int i = 0; i < VPT; ++i) {
    const int v = i * nt + tid;
    h[i] = make_uint4(0, 0, 0, 0);
    if (v < nvec && mbar_wait(&bar[i], 0, &abort_flag, err, DEV_ERR_WAIT_FULL))
      h[i] = silu_mul8(*reinterpret_cast<const uint4 *>(gs + v * 8), *reinterpret_cast<const uint4 *>(us + v * 8));
  }
  quant_row<VPT>(h, 0, N, 1, true, q + static_cast<size_t>(row) * N, s + row, red, &slot);
  // Never leave a copy in flight (returns at once unless a wait above gave up).
  if (tid == 0) {
    volatile int dummy = 0;
#pragma unroll
    for (int i = 0; i < VPT; ++i)
      if (i * nt < nvec) mbar_wait(&bar[i], 0, &dummy, err, DEV_ERR_WAIT_DRAIN);
  }
}

template <int VPT>
__global__ void __launch_bounds__(kSiluThreads) silu_mul_quant_kernel(const uint16_t *__restrict__ gu, int N, int cols,
                                                                int C, uint8_t *__restrict__ q,
                                                                float *__restrict__ s) {
  if (threadIdx.x == 0) pdl_launch_dependents();
  pdl_wait();   // gu comes from the preceding kernel
  __shared__ float red[kSiluThreads / 32];
  __shared__ float slot;
  const int row = blockIdx.x / C, part = blockIdx.x - row * C, tid = threadIdx.x, nt = blockDim.x;
  const int c0 = part * cols, c1 = min(N, c0 + cols);
  const uint16_t *gr = gu + static_cast<size_t>(row) * 2 * N;
  uint4 h[VPT];
#pragma unroll
  for (int i = 0; i < VPT; ++i) {
    const int k = c0 + (i * nt + tid) * 8;
    if (k < c1) {
      h[i] = silu_mul8(__ldg(reinterpret_cast<const uint4 *>(gr + k)), __ldg(reinterpret_cast<const uint4 *>(gr + N + k)));
    } else {
      h[i] = make_uint4(0, 0, 0, 0);
    }
  }
  quant_row<VPT>(h, c0, c1, C, part == 0, q + static_cast<size_t>(row) * N, s + row, red, &slot);
  if (C > 1) cluster_wait();
}

int threads_for(int64_t K, RowKind kind, int64_t M) {
  const int64_t vecs = K / 8;
  const int cap = row_threads(kind, M, vecs);
  int t = static_cast<int>(vecs < cap ? ((vecs + 31) / 32) * 32 : cap);
  if (t < 32) t = 32;
  if (ceil_div(vecs, static_cast<int64_t>(t)) > 12)   // at most 12 vectors per thread: widen a capped block
    t = static_cast<int>(ceil_div(ceil_div(vecs, int64_t{12}), int64_t{32}) * 32);
  return t;
}

// Row split for a row of K columns: CTAs per row, columns per CTA, threads
// and 16-byte vectors per thread.
struct RowSplit {
  int C, cols, threads;
  int64_t per;
};
RowSplit split_row(int64_t M, int64_t K, RowKind kind) {
  int C = row_split(M, K, kind);
  if (M * C > (int64_t{1} << 30)) C = 1;
  const int64_t cols = ceil_div(ceil_div(K, static_cast<int64_t>(C)), int64_t{8}) * 8;
  const int t = threads_for(cols, kind, M);
  return {C, static_cast<int>(cols), t, ceil_div(cols / 8, static_cast<int64_t>(t))};
}

}  // namespace

// Rows of up to 24576 columns fit in registers (VPT <= 12 at 256 threads),
// so the split never has to fall back to a two-pass kernel.
cudaError_t launch_add_rmsnorm_quant(const uint16_t *y, const uint16_t *res, const uint16_t *w, float eps, int64_t M,
                                     int64_t K, uint16_t *ro, uint8_t *q, float *s, cudaStream_t st) {
  const RowSplit rs = split_row(M, K, RowKind::kNorm);
  const dim3 grid(static_cast<unsigned>(M * rs.C));
  const int k = static_cast<int>(K);
  if (rs.C == 1) {   // one CTA per row: y and the residual staged in shared memory
    const size_t smem = static_cast<size_t>(4) * K;
#define R4_ARQS(V)                                                                                           \
  {                                                                                                          \
    auto kern = add_rmsnorm_quant_staged_kernel<V>;                                                          \
    cudaError_t e = ensure_smem_attr(reinterpret_cast<const void *>(kern), smem);                            \
    if (e == cudaSuccess)                                                                                    \
      e = launch_pdl(kern, grid, dim3(rs.threads), smem, st, y, res, w, eps, k, ro, q, s, device_error_word(), \
                     options().inject_stall);                                                                \
    if (e != cudaSuccess) return e;                                                                          \
    set_last_kernel("add_rmsnorm_quant_staged_kernel<" #V ">");                                              \
  }
    const int64_t per = rs.per;
    if (per <= 1) R4_ARQS(1) else if (per <= 2) R4_ARQS(2) else if (per <= 4) R4_ARQS(4) else if (per <= 6) R4_ARQS(6)
    else if (per <= 9) R4_ARQS(9) else R4_ARQS(12)
#undef R4_ARQS
    return cudaGetLastError();
  }
#define R4_ARQ(V)                                                                                            \
  {                                                                                                          \
    const cudaError_t e =                                                                                    \
        rs.C > 1 ? launch_pdl_cluster(add_rmsnorm_quant_kernel<V>, grid, dim3(rs.threads), 0, st, rs.C, y, res, \
                                      w, eps, k, rs.cols, rs.C, ro, q, s)                                      \
                 : launch_pdl(add_rmsnorm_quant_kernel<V>, grid, dim3(rs.threads), 0, st, y, res, w, eps, k,    \
                              rs.cols, rs.C, ro, q, s);                                                        \
    if (e != cudaSuccess) return e;                                                                          \
    set_last_kernel("add_rmsnorm_quant_kernel<" #V ">");                                                     \
  }
  const int64_t per = rs.per;
  if (per <= 1) R4_ARQ(1) else if (per <= 2) R4_ARQ(2) else if (per <= 4) R4_ARQ(4) else if (per <= 6) R4_ARQ(6)
  else if (per <= 9) R4_ARQ(9) else R4_ARQ(12)
#undef R4_ARQ
  return cudaGetLastError();
}

cudaError_t launch_silu_mul_quant(const uint16_t *gu, int64_t M, int64_t N, uint8_t *q, float *s, cudaStream_t st) {
  const RowSplit rs = split_row(M, N, RowKind::kSilu);
  const dim3 grid(static_cast<unsigned>(M * rs.C));
  const int n = static_cast<int>(N);
  if (rs.C == 1) {   // one CTA per row: the row staged in shared memory
    const size_t smem = static_cast<size_t>(4) * N;
#define R4_SMQS(V)                                                                                           \
  {                                                                                                          \
    auto kern = silu_mul_quant_staged_kernel<V>;                                                             \
    cudaError_t e = ensure_smem_attr(reinterpret_cast<const void *>(kern), smem);                            \
    if (e == cudaSuccess)                                                                                    \
      e = launch_pdl(kern, grid, dim3(rs.threads), smem, st, gu, n, q, s, device_error_word(), options().inject_stall); \
    if (e != cudaSuccess) return e;                                                                          \
    set_last_kernel("silu_mul_quant_staged_kernel<" #V ">");                                                 \
  }
    const int64_t per = rs.per;
    if (per <= 1) R4_SMQS(1) else if (per <= 2) R4_SMQS(2) else if (per <= 4) R4_SMQS(4) else if (per <= 6) R4_SMQS(6)
    else if (per <= 9) R4_SMQS(9) else R4_SMQS(12)
#undef R4_SMQS
    return cudaGetLastError();
  }
#define R4_SMQ(V)                                                                                            \
  {                                                                                                          \
    const cudaError_t e =                                                                                    \
        rs.C > 1 ? launch_pdl_cluster(silu_mul_quant_kernel<V>, grid, dim3(rs.threads), 0, st, rs.C, gu, n,    \
                                      rs.cols, rs.C, q, s)                                                     \
                 : launch_pdl(silu_mul_quant_kernel<V>, grid, dim3(rs.threads), 0, st, gu, n, rs.cols, rs.C, q, s); \
    if (e != cudaSuccess) return e;                                                                          \
    set_last_kernel("silu_mul_quant_kernel<" #V ">");                                                        \
  }
  const int64_t per = rs.per;
  if (per <= 1) R4_SMQ(1) else if (per <= 2) R4_SMQ(2) else if (per <= 4) R4_SMQ(4) else if (per <= 6) R4_SMQ(6)
  else if (per <= 9) R4_SMQ(9) else R4_SMQ(12)
#undef R4_SMQ
  return cudaGetLastError();
}

}  // namespace r4
