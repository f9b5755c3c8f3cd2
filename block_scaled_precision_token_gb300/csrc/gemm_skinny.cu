// gemm_skinny.cu -- skinny bf16 NT GEMM, C = bf16(x W^T), fp32 accumulation,
// for tiny projections (M <= 64 tokens, N of a few hundred, K of a few
// thousand): "radiance_gemm.py", module docstring.
//
// The page's diagnosis: a sub-megabyte weight gives a library GEMM only a
// handful of CTAs, each walking all of K while the rest of the GPU idles; the
// cure is split-K. Here the split is across a thread-block cluster:
//  * grid = (KS, ceil(N/16), token slices), cluster = (KS, 1, 1): each CTA
//    owns 16 weight rows (the mma M dimension -- weight-stationary, tokens
//    are the mma N), a contiguous K range and one slice of up to 16 * NG2
//    tokens; KS <= 8 CTAs of a cluster share one row tile and token slice.
//    Splitting the tokens over more CTAs (each re-reads the sub-megabyte
//    weight from L2) keeps the per-CTA work, and so the latency, close to
//    that of a few tokens as M grows.
//  * operands are staged in shared memory with cp.async (16-byte chunks,
//    rows padded by 16 bytes so ldmatrix is conflict-free) and multiplied
//    with mma.sync m16n8k16 bf16 -> fp32. The problem is latency- and
//    HBM-bound (about 2 flops per weight byte at M = 8), not tensor-bound, so
//    the warp-level MMA is sufficient; tcgen05 setup (TMEM allocation,
//    descriptor pipeline) would only add latency here.
//  * reduction: 4 warps -> shared memory -> one CTA partial in the CTA's own
//    shared memory; after one cluster barrier every CTA sums a 1/KS share of
//    the tile's outputs over the cluster's partials, read in rank order
//    through distributed shared memory (deterministic), rounds to bf16 and
//    stores (a reduce-scatter). No global workspace, no atomics, no second
//    kernel.

#include <cuda_bf16.h>

#include <algorithm>

#include "r4_internal.h"

namespace r4 {
namespace skinny {

constexpr int kThreads = 128;
constexpr int kRows = 16;
constexpr int kIter = 256;              // K staged per iteration
constexpr int kStride = kIter + 8;      // padded row, in bf16 elements
constexpr int kMaxKS = 8;

// Shared memory sized for the token groups actually present: at 1 CTA per
// SM a cluster of 8 fits only 15 times on GB300 (measured: the 16th of a
// 256-row weight's clusters ran as a second wave); small CTAs pack 2-7 per SM.
template <int NG2, int NB>   // NB staging buffers: 2 when a CTA walks several K chunks
struct Smem {
  static constexpr int kMpad = 16 * NG2;
  static constexpr size_t kW = kRows * kStride * 2;    // one buffer
  static constexpr size_t kX = kMpad * kStride * 2;
  // partial tiles [16 rows][kMpad tokens], rows kMpad + 1 floats apart: the
  // reductions walk rows fastest, and an odd stride keeps them conflict-free
  static constexpr int kRS = kMpad + 1;
  static constexpr size_t kRed = 4 * kRows * kRS * 4;
  static constexpr size_t kCluster = kRows * kRS * 4;   // this CTA's partial, read by the cluster
  static constexpr size_t kBytes = NB * (kW + kX) + kRed + kCluster;
};

__device__ __forceinline__ uint32_t smem_addr(const void *p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void cp_async16(void *dst, const void *src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_addr(dst)), "l"(src) : "memory");
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2, uint32_t &r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

__device__ __forceinline__ void mma_bf16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

__device__ __forceinline__ uint32_t map_rank(uint32_t saddr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(saddr), "r"(rank));
  return r;
}

template <int NG2, int NB>  // token groups of 16 (Mpad = 16 * NG2); NB staging buffers
__global__ void __launch_bounds__(kThreads, 1)
    skinny_bf16_kernel(const uint16_t *__restrict__ x, const uint16_t *__restrict__ w, int M, int N, int K,
                       int chunks_per_cta, uint16_t *__restrict__ c, int ldc, int early_w) {
  using S = Smem<NG2, NB>;
  constexpr int kMpad = S::kMpad;
  constexpr int kRS = S::kRS;
  extern __shared__ __align__(16) uint8_t smem[];
  // NB staging buffers (double-buffered K loop when NB == 2), then the partial tiles
  uint16_t *sW0 = reinterpret_cast<uint16_t *>(smem);
  uint16_t *sX0 = reinterpret_cast<uint16_t *>(smem + S::kW);
  float *sRed = reinterpret_cast<float *>(smem + NB * (S::kW + S::kX));              // [4][16][kRS]
  float *sCl = reinterpret_cast<float *>(smem + NB * (S::kW + S::kX) + S::kRed);     // [16][kRS]

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t rank = cluster_rank();
  const int KS = gridDim.x;
  const int n0 = blockIdx.y * kRows;
  const int t_off = blockIdx.z * kMpad;           // this CTA's token slice
  const int kbeg = static_cast<int>(rank) * chunks_per_cta * 256;
  const int kend = min(K, kbeg + chunks_per_cta * 256);

  if (tid == 0) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  if (!early_w) asm volatile("griddepcontrol.wait;" ::: "memory");   // w may come from the preceding kernel

  // Warp roles: NGW token-group slots x KP k-phases (4 warps). Warp w
  // multiplies token group w % NGW over the k-steps of phase w / NGW, so with
  // 64 tokens each warp owns one group over all of K and no two warps add
  // into the same outputs.
  constexpr int NGW = NG2 == 3 ? 4 : NG2;   // with 3 groups the 4th warp only stages and reduces
  constexpr int KP = 4 / NGW;
  const int g2w = warp % NGW, kp = warp / NGW;
  float acc[2][4];
#pragma unroll
  for (int g = 0; g < 2; ++g) acc[g][0] = acc[g][1] = acc[g][2] = acc[g][3] = 0.f;

  // Stage chunk kk (kIter columns of the 16 weight rows and of the tokens)
  // into buffer b: one cp.async group.
  constexpr int cpr = kIter / 8;                // 16-byte chunks per row
  auto stage = [&](int kk, int b) {
    uint16_t *sW = sW0 + b * ((S::kW + S::kX) / 2);
    uint16_t *sX = sX0 + b * ((S::kW + S::kX) / 2);
    for (int i = tid; i < kRows * cpr; i += kThreads) {
      const int r = i / cpr, ch = i % cpr;
      uint16_t *dst = sW + r * kStride + ch * 8;
      if (n0 + r < N)
        cp_async16(dst, w + static_cast<size_t>(n0 + r) * K + kk + ch * 8);
      else
        *reinterpret_cast<uint4 *>(dst) = make_uint4(0, 0, 0, 0);
    }
    // The weight is independent of the preceding kernel; x is not.
    if (kk == kbeg) asm volatile("griddepcontrol.wait;" ::: "memory");
    for (int i = tid; i < kMpad * cpr; i += kThreads) {
      const int r = i / cpr, ch = i % cpr;
      uint16_t *dst = sX + r * kStride + ch * 8;
      if (t_off + r < M)
        cp_async16(dst, x + static_cast<size_t>(t_off + r) * K + kk + ch * 8);
      else
        *reinterpret_cast<uint4 *>(dst) = make_uint4(0, 0, 0, 0);
    }
    asm volatile("cp.async.commit_group;" ::: "memory");
  };

  if (kbeg < kend) stage(kbeg, 0);
  for (int kk = kbeg, it = 0; kk < kend; kk += kIter, ++it) {
    const int klen = kIter;                       // K is a multiple of 256
    // prefetch the next chunk into the other buffer, then wait for this one
    if (NB == 2 && kk + kIter < kend) {
      stage(kk + kIter, (it + 1) & 1);
      asm volatile("cp.async.wait_group 1;" ::: "memory");
    } else {
      asm volatile("cp.async.wait_group 0;" ::: "memory");
    }
    __syncthreads();
    const int cur = NB == 2 ? (it & 1) : 0;
    const uint16_t *sW = sW0 + cur * ((S::kW + S::kX) / 2);
    const uint16_t *sX = sX0 + cur * ((S::kW + S::kX) / 2);
    const int nsteps = klen / 16;
    if (g2w < NG2) {
      for (int ks = kp; ks < nsteps; ks += KP) {
        uint32_t a0, a1, a2, a3, b0, b1, b2, b3;
        ldsm_x4(smem_addr(sW + (lane & 15) * kStride + ks * 16 + (lane >> 4) * 8), a0, a1, a2, a3);
        const int tok = g2w * 16 + (lane >> 4) * 8 + (lane & 7);
        ldsm_x4(smem_addr(sX + tok * kStride + ks * 16 + ((lane >> 3) & 1) * 8), b0, b1, b2, b3);
        mma_bf16(acc[0], a0, a1, a2, a3, b0, b1);
        mma_bf16(acc[1], a0, a1, a2, a3, b2, b3);
      }
    }
    __syncthreads();
    if (NB == 1 && kk + kIter < kend) stage(kk + kIter, 0);   // single buffer: refill after use
  }

  // warp partials -> shared memory, one [16][kMpad] tile per k-phase (D
  // fragment: rows lane/4 and lane/4 + 8, token columns 16 g2w + 8g +
  // 2(lane%4) + {0,1})
  if (g2w < NG2) {
    float *red = sRed + kp * kRows * kRS;
#pragma unroll
    for (int g = 0; g < 2; ++g) {
      const int r = lane >> 2, t = 16 * g2w + 8 * g + 2 * (lane & 3);
      red[r * kRS + t] = acc[g][0];
      red[r * kRS + t + 1] = acc[g][1];
      red[(r + 8) * kRS + t] = acc[g][2];
      red[(r + 8) * kRS + t + 1] = acc[g][3];
    }
  }
  __syncthreads();

  // this CTA's partial (sum over the k-phases) in its own shared memory
  for (int i = tid; i < kRows * kMpad; i += kThreads) {
    const int r = i % kRows, t = i / kRows;
    float v = sRed[r * kRS + t];
#pragma unroll
    for (int p = 1; p < KP; ++p) v += sRed[p * kRows * kRS + r * kRS + t];
    sCl[r * kRS + t] = v;
  }
  // Every CTA of the cluster has written its partial (release / acquire).
  asm volatile("barrier.cluster.arrive.release.aligned;\nbarrier.cluster.wait.acquire.aligned;" ::: "memory");
  // Reduce-scatter: CTA `rank` owns outputs e in [rank * per, rank * per + per)
  // of the tile's 16 x kMpad (e = token * 16 + row: 16 consecutive outputs
  // are one token's 16 consecutive columns of c).
  const int total = kRows * kMpad;
  const int per = (total + KS - 1) / KS;
  const uint32_t my_part = smem_addr(sCl);
  for (int e = static_cast<int>(rank) * per + tid; e < min(total, static_cast<int>(rank + 1) * per); e += kThreads) {
    const int r = e % kRows, t = e / kRows;
    if (t_off + t >= M || n0 + r >= N) continue;   // padded token or row: no load without a consumer
    const uint32_t off = 4u * static_cast<uint32_t>(r * kRS + t);
    float pq[kMaxKS];   // all loads in flight before the (rank-ordered) sum
#pragma unroll
    for (int q = 0; q < kMaxKS; ++q)
      if (q < KS) asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(pq[q]) : "r"(map_rank(my_part + off, q)));
    float v = 0.f;
#pragma unroll
    for (int q = 0; q < kMaxKS; ++q)
      if (q < KS) v += pq[q];
    __nv_bfloat16 h = __float2bfloat16_rn(v);
    c[static_cast<size_t>(t_off + t) * ldc + n0 + r] = *reinterpret_cast<uint16_t *>(&h);
  }
  // No CTA leaves while another may still read its partial. The arrive must
  // be a release: it is what orders this CTA's remote loads before the peers
  // may exit (a relaxed arrive, tried when padded tokens were still loaded,
  // let a CTA leave under a peer's load still in flight).
  asm volatile("barrier.cluster.arrive.release.aligned;\nbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

template <int NG2, int NB>
cudaError_t launch_ng(const uint16_t *x, const uint16_t *w, int64_t M, int64_t N, int64_t K, uint16_t *c,
                      int64_t ldc, int slices, int ks, cudaStream_t st) {
  const int chunks = static_cast<int>(K / 256);
  const int cpc = (chunks + ks - 1) / ks;
  auto kern = skinny_bf16_kernel<NG2, NB>;
  constexpr size_t kSmemBytes = Smem<NG2, NB>::kBytes;
  cudaError_t e = ensure_smem_attr(reinterpret_cast<const void *>(kern), static_cast<int>(kSmemBytes));
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(ks), static_cast<unsigned>(ceil_div(N, kRows)), static_cast<unsigned>(slices));
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = kSmemBytes;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = static_cast<unsigned>(ks);
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = options().pdl ? 2 : 1;
  e = cudaLaunchKernelEx(&cfg, kern, x, w, static_cast<int>(M), static_cast<int>(N), static_cast<int>(K), cpc, c,
                         static_cast<int>(ldc), options().early_weights);
  set_last_kernel(NG2 == 1 ? "skinny_bf16_kernel<1>" : NG2 == 2 ? "skinny_bf16_kernel<2>"
                  : NG2 == 3 ? "skinny_bf16_kernel<3>" : "skinny_bf16_kernel<4>");
  return e;
}

}  // namespace skinny

cudaError_t launch_gemm_skinny(const uint16_t *x, const uint16_t *w, int64_t M, int64_t N, int64_t K, uint16_t *c,
                               int64_t ldc, cudaStream_t st) {
  // A CTA that walks several 256-wide K chunks double-buffers them. One that
  // owns a single chunk keeps the smaller single-buffer footprint, except at
  // 64 tokens, where the larger footprint spreads the CTAs over more SMs
  // (measured, [256, 2048], one chunk per CTA: M <= 16 3.0 vs 3.2 us and
  // M = 32 4.3 vs 4.6 us with one buffer; M = 64 5.9 vs 6.6 us with two).
  // Token groups of 16 per CTA: from 32 tokens on one group per CTA, the
  // tokens split over more CTAs (measured on GB300, graph-timed, M = 64:
  // [256,2048] 6.05 -> 5.45 us, [96,5120] 6.38 -> 5.53 us; M = 32 with the
  // split of 8: 4.17 -> 4.00 and 4.50 -> 4.06 us); option 15 forces a count.
  const int64_t groups = ceil_div(M, 16);
  int64_t ng2 = groups >= 2 ? 1 : groups;
  if (options().skinny_groups > 0) ng2 = std::min<int64_t>(groups, options().skinny_groups);
  const int slices = static_cast<int>(ceil_div(groups, ng2));
  // K split (cluster size): the largest power of two up to 8 (and up to the
  // 256-wide K chunks) that keeps the grid within one CTA per SM. Measured
  // on GB300 (graph-timed, µs), against a fixed split of 8: [256,2048]
  // M=32 4.12 -> 3.60 (split 4), M=64 5.24 -> 4.43 (split 2); [96,5120] M=64
  // 5.16 -> 5.09 (split 4; a split of 2 took 7.3); the other shapes keep 8.
  const int64_t chunks = K / 256;
  const int64_t per_split = ceil_div(N, static_cast<int64_t>(skinny::kRows)) * slices;
  const int64_t fit = std::max<int64_t>(1, device_sm_count() / std::max<int64_t>(1, per_split));
  int ks = 1;
  while (ks * 2 <= skinny::kMaxKS && ks * 2 <= chunks && ks * 2 <= fit) ks *= 2;
  const bool multi = ceil_div(chunks, static_cast<int64_t>(ks)) > 1 || ng2 == 4;
#define R4_SK(G)                                                                               \
  return multi ? skinny::launch_ng<G, 2>(x, w, M, N, K, c, ldc, slices, ks, st)               \
               : skinny::launch_ng<G, 1>(x, w, M, N, K, c, ldc, slices, ks, st);
  switch (ng2) {
    case 1: R4_SK(1)
    case 2: R4_SK(2)
    case 3: R4_SK(3)
    default: R4_SK(4)
  }
#undef R4_SK
}

}  // namespace r4
