// prepack.cu -- one-time weight permutations into the GEMM-native layouts.
//
// The idea is the one "radiance_mxfp4.py" applies in permute_w: reorder the
// weight bytes once at load so the GEMM's weight reads are long and
// contiguous; a permutation, never a re-quantization. The target layout here
// is the one the tcgen05/TMA kernels read, not a WMMA fragment order.
//
// MXFP4 packed buffer (N_t = ceil(N/128) row tiles, KB = ceil(K/128) K blocks):
//   codes: [N_t][KB][128 rows][64 bytes]   packed e2m1, low nibble = even k
//   scale: [N_t][KB][512 bytes]            byte 16*r0 + 4*r1 + j holds the
//          ue8m0 scale of row 32*r1 + r0, 32-K block j of the 128-K block --
//          the order in which tcgen05.cp 32x128b.warpx4 lays a 128-row x 4
//          scale block across the four 32-lane quarters of tensor memory.
//   Rows >= N and K >= true K: code 0, scale 127 (x1.0).
// Block-FP8 packed buffer:
//   codes: [N/128][K/128][128 rows][128 bytes]  e4m3
//   scale: [N/128][K/128] fp32 (copied unchanged)

#include "r4_internal.h"

namespace r4 {
namespace {

__global__ void __launch_bounds__(512) prepack_mxfp4_kernel(const uint8_t *__restrict__ w,
                                                            const uint8_t *__restrict__ wsc, int64_t N,
                                                            int64_t K, int KB, uint8_t *__restrict__ codes,
                                                            uint8_t *__restrict__ sf) {
  const int64_t tile = blockIdx.x;           // nt * KB + kb
  const int64_t nt = tile / KB, kb = tile % KB;
  const int tid = threadIdx.x;
  const int64_t halfK = K / 2, nblk = K / 32;
  {  // 128 rows x 64 bytes = 512 x 16-byte chunks
    const int r = tid >> 2, c = (tid & 3) * 16;
    const int64_t row = nt * 128 + r, col = kb * 64 + c;
    uint4 v = make_uint4(0, 0, 0, 0);
    if (row < N && col < halfK) v = __ldg(reinterpret_cast<const uint4 *>(w + row * halfK + col));
    *reinterpret_cast<uint4 *>(codes + tile * 8192 + r * 64 + c) = v;
  }
  if (tid < 128) {  // scale atom: 128 x 4 bytes
    const int r0 = tid >> 2, r1 = tid & 3;
    const int64_t row = nt * 128 + r0 + 32 * r1;
    uint32_t word = 0;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int64_t blk = kb * 4 + j;
      const uint32_t b = (row < N && blk < nblk) ? wsc[row * nblk + blk] : 127u;
      word |= b << (8 * j);
    }
    *reinterpret_cast<uint32_t *>(sf + tile * 512 + 4 * tid) = word;
  }
  // The GEMMs read the packed weight before their dependency wait (they may
  // start once this kernel's blocks have exited): make every write visible
  // device-wide before the block exits.
  __threadfence();
}

__global__ void __launch_bounds__(256) prepack_fp8_kernel(const uint8_t *__restrict__ w, int64_t K, int KB,
                                                          uint8_t *__restrict__ codes) {
  const int64_t tile = blockIdx.x;
  const int64_t nt = tile / KB, kb = tile % KB;
  for (int i = threadIdx.x; i < 1024; i += 256) {   // 128 rows x 8 chunks of 16 B
    const int r = i >> 3, c = (i & 7) * 16;
    const uint4 v = __ldg(reinterpret_cast<const uint4 *>(w + (nt * 128 + r) * K + kb * 128 + c));
    *reinterpret_cast<uint4 *>(codes + tile * 16384 + r * 128 + c) = v;
  }
  __threadfence();   // visible device-wide before the block exits (see prepack_mxfp4_kernel)
}

}  // namespace

cudaError_t launch_prepack_mxfp4(const uint8_t *w, const uint8_t *ws, int64_t N, int64_t K, uint8_t *packed,
                                 cudaStream_t st) {
  const int64_t NT = ceil_div(N, 128), KB = ceil_div(K, 128);
  uint8_t *codes = packed;
  uint8_t *sf = packed + mx_packed_codes_bytes(N, K);
  prepack_mxfp4_kernel<<<static_cast<unsigned>(NT * KB), 512, 0, st>>>(w, ws, N, K, static_cast<int>(KB), codes,
                                                                       sf);
  set_last_kernel("prepack_mxfp4_kernel");
  return cudaGetLastError();
}

cudaError_t launch_prepack_blockfp8(const uint8_t *w, const float *ws, int64_t N, int64_t K, uint8_t *packed,
                                   cudaStream_t st) {
  const int64_t NT = N / 128, KB = K / 128;
  prepack_fp8_kernel<<<static_cast<unsigned>(NT * KB), 256, 0, st>>>(w, K, static_cast<int>(KB), packed);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  set_last_kernel("prepack_fp8_kernel");
  return cudaMemcpyAsync(packed + fp8_packed_codes_bytes(N, K), ws, static_cast<size_t>(NT * KB) * 4,
                         cudaMemcpyDeviceToDevice, st);
}

}  // namespace r4
