// peak.cu -- tensor-core issue-rate probe: the dense rate of the MMA
// instructions the GEMMs use, measured on the GPU they run on.
//
// The pages measured their own matrix-instruction peak with a
// register-resident microbenchmark that touches no memory
// ("radiance_mxfp4.py", the fp8 WMMA throughput figures quoted in the module
// docstring). This is the GB300 counterpart: every CTA allocates tensor
// memory, zero-fills one A tile (128 rows) and one B tile (N rows) in shared
// memory, and one thread issues `iters` x 4 MMAs of K = 32 (kind::mxf8f6f4 or
// kind::f8f6f4) or K = 64 (kind::mxf4) into one tensor-memory accumulator,
// back to back. Nothing but the tensor pipe is busy, so launch time x the
// flops issued gives the sustained rate of that instruction shape; the host
// times it with events.

#include "r4_device.cuh"
#include "r4_internal.h"

namespace r4 {
namespace peak {

constexpr uint32_t kATile = 128 * 128;            // A: 128 rows x 128 bytes (one 128-byte swizzle row each)
constexpr uint32_t kSfCol = 256;                  // ue8m0 scale columns (after an N = 256 accumulator)

// Instruction descriptor, kind::mxf4 with ue8m0 block scales (scale_vec::2X):
// A = B = e2m1 (format 1 in this kind), K-major, M = 128.
__host__ __device__ constexpr uint32_t idesc_mxf4(int n, int a_sf_id, int b_sf_id) {
  return (static_cast<uint32_t>(b_sf_id & 3) << 4) | (1u << 7) | (1u << 10) | (static_cast<uint32_t>(n >> 3) << 17) |
         (1u << 23) | (static_cast<uint32_t>(128 >> 4) << 24) | (static_cast<uint32_t>(a_sf_id & 3) << 29);
}

template <int KIND, int N>   // KIND 1: mxf8f6f4 (e2m1 x e4m3), 2: f8f6f4 (e4m3 x e4m3), 3: mxf4 (e2m1 x e2m1)
__global__ void __launch_bounds__(128, 1) mma_peak_kernel(int iters, int *err) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t *a_tile = smem;
  uint8_t *b_tile = smem + kATile;
  uint8_t *sf = b_tile + N * 128;                  // 512 bytes of scale code 127 (x1)
  uint64_t *done = reinterpret_cast<uint64_t *>(sf + 512);
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(done + 1);

  const int warp = threadIdx.x >> 5;
  for (uint32_t i = threadIdx.x; i < (kATile + N * 128) / 16; i += blockDim.x)
    reinterpret_cast<uint4 *>(smem)[i] = make_uint4(0, 0, 0, 0);
  for (int i = threadIdx.x; i < 128; i += blockDim.x) reinterpret_cast<uint32_t *>(sf)[i] = 0x7F7F7F7Fu;
  if (threadIdx.x == 0) {
    mbar_init(done, 1);
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (threadIdx.x == 0) {
    const uint32_t a0 = smem_u32(a_tile), b0 = smem_u32(b_tile);
    if constexpr (KIND != 2) {
      const uint64_t sdesc = sdesc_sf_32x16(smem_u32(sf));
      tc_cp_32x128b_warpx4(tmem + kSfCol, sdesc);        // A scales
      tc_cp_32x128b_warpx4(tmem + kSfCol + 4, sdesc);    // B scales (N <= 128)
      tc_cp_32x128b_warpx4(tmem + kSfCol + 8, sdesc);    // B scales (N = 256: 8 columns)
    }
    for (int it = 0; it < iters; ++it) {
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) {
        const uint64_t ad = sdesc_sw128_kmajor(a0 + 32u * kk);
        const uint64_t bd = sdesc_sw128_kmajor(b0 + 32u * kk);
        const uint32_t acc = (it > 0 || kk > 0) ? 1u : 0u;
        if constexpr (KIND == 1) {
          tc_mma_mxf8f6f4(tmem, ad, bd, idesc_mxf8f6f4_e2m1_e4m3(N, kk, 0),
                          (tmem + kSfCol) | (static_cast<uint32_t>(kk) << 30), tmem + kSfCol + 4, acc);
        } else if constexpr (KIND == 2) {
          tc_mma_f8f6f4(tmem, ad, bd, idesc_f8f6f4_e4m3(N), acc);
        } else {
          const int id = (kk & 1) * 2;
          tc_mma_mxf4(tmem, ad, bd, idesc_mxf4(N, id, id), (tmem + kSfCol) | (static_cast<uint32_t>(id) << 30),
                      (tmem + kSfCol + 4) | (static_cast<uint32_t>(id) << 30), acc);
        }
      }
    }
    tc_commit(done);
    volatile int dummy = 0;
    mbar_wait(done, 0, &dummy, err, DEV_ERR_WAIT_DRAIN);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

template <int KIND, int N>
cudaError_t launch_kind(int blocks, int iters, cudaStream_t st) {
  constexpr int kSmem = 1024 + kATile + N * 128 + 512 + 64;
  auto kern = mma_peak_kernel<KIND, N>;
  cudaError_t e = ensure_smem_attr(reinterpret_cast<const void *>(kern), kSmem);
  if (e != cudaSuccess) return e;
  kern<<<static_cast<unsigned>(blocks), 128, kSmem, st>>>(iters, device_error_word());
  return cudaGetLastError();
}

}  // namespace peak

cudaError_t launch_mma_peak(int kind, int n, int blocks, int iters, cudaStream_t st) {
  if (kind == 1) return n == 128 ? peak::launch_kind<1, 128>(blocks, iters, st) : peak::launch_kind<1, 256>(blocks, iters, st);
  if (kind == 2) return n == 128 ? peak::launch_kind<2, 128>(blocks, iters, st) : peak::launch_kind<2, 256>(blocks, iters, st);
  return n == 128 ? peak::launch_kind<3, 128>(blocks, iters, st) : peak::launch_kind<3, 256>(blocks, iters, st);
}

}  // namespace r4
