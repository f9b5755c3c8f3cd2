// quant_common.cuh -- the per-token e4m3 quantization rule shared by the
// standalone quantization kernel and the fused producers.
//
// ("radiance_mxfp4.py", _traced_quant and the comment above it:
// s = max(amax/448, 1/(448*512)) in fp32, q = e4m3_rne_sat(x / s), both
// divisions correctly rounded.)

#pragma once

#include <cuda_bf16.h>
#include <cuda_fp8.h>

#include <cstdint>

#include "r4_device.cuh"

namespace r4 {
namespace qc {

constexpr float kFp8Max = 448.0f;
constexpr float kMinScale = 1.0f / 229376.0f;  // 1 / (448 * 512)

__device__ __forceinline__ float bf16lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16hi(uint32_t v) { return __uint_as_float(v & 0xFFFF0000u); }

// Largest magnitude among 8 bf16 values: the magnitudes' bit patterns order
// as the values do (finite or infinite), so packed 16-bit integer maxima
// find it without unpacking.
__device__ __forceinline__ float absmax8(const uint4 &v) {
  const uint32_t m = 0x7FFF7FFFu;
  uint32_t a, b;
  asm("max.u16x2 %0, %1, %2;" : "=r"(a) : "r"(v.x & m), "r"(v.y & m));
  asm("max.u16x2 %0, %1, %2;" : "=r"(b) : "r"(v.z & m), "r"(v.w & m));
  asm("max.u16x2 %0, %1, %2;" : "=r"(a) : "r"(a), "r"(b));
  return fmaxf(bf16lo(a), bf16hi(a));
}

__device__ __forceinline__ uint32_t e4m3_of(float v) {
  return static_cast<uint32_t>(__nv_cvt_float_to_fp8(v, __NV_SATFINITE, __NV_E4M3));
}

// x / s rounded once to fp32 -- the correctly rounded quotient -- from
// rc = RN(1/s), by Markstein's correction step (P. Markstein, "Computation of
// elementary functions on the IBM RISC System/6000 processor", IBM J. Res.
// Dev. 34(1), 1990): q = RN(x rc); the remainder e = x - s q is exact in one
// FMA; q' = RN(q + e rc). The sign is taken from x, so a quotient that
// underflows to zero keeps the sign of the exact one. The quantizers only
// divide a bf16 value x by a scale s = max(RN(amax/448), 1/(448*512)) with
// |x| <= amax; on that whole domain (every bf16 x, every bf16 amax) the
// result is bit-identical to a correctly rounded division, which
// r4_check_quotients verifies on the device.
__device__ __forceinline__ float div_by_scale(float x, float s, float rc) {
  const float q = __fmul_rn(x, rc);
  const float e = __fmaf_rn(-s, q, x);
  return copysignf(__fmaf_rn(e, rc, q), x);
}

// Two fp32 -> two e4m3 codes in one instruction (round to nearest even,
// saturating to +-448): lo in bits 0-7, hi in bits 8-15.
__device__ __forceinline__ uint32_t e4m3x2_of(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

// 8 bf16 -> 8 e4m3 codes (element i in byte i), each x/s correctly rounded;
// rc = __frcp_rn(sc).
__device__ __forceinline__ uint2 quant8(const uint4 &v, float sc, float rc) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
  uint32_t b[4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
    b[i] = e4m3x2_of(div_by_scale(bf16lo(w[i]), sc, rc), div_by_scale(bf16hi(w[i]), sc, rc));
  uint2 r;
  r.x = b[0] | (b[1] << 16);
  r.y = b[2] | (b[3] << 16);
  return r;
}

__device__ __forceinline__ float warp_max(float a) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, o));
  return a;
}

// A row split over the C CTAs (C <= 32) of a 1-D thread-block cluster:
// combines the CTAs' block-reduced values t (sum, or max of non-negative
// values), every thread of every CTA returning the same result. Each CTA
// publishes t in its own shared word `slot`; after a cluster barrier lane i
// of every warp reads CTA i's word and a butterfly shuffle combines the
// lanes, so every CTA forms the same sum in the same order. Each combine
// needs a slot of its own, and a CTA may not exit while a peer can still
// read its slot: after the last combine the kernel calls cluster_arrive()
// and, before it exits, cluster_wait().
template <bool kMax>
__device__ __forceinline__ float cluster_combine(float t, float *slot, int C) {
  if (threadIdx.x == 0) *slot = t;
  cluster_sync_all();
  const int lane = threadIdx.x & 31;
  float v = 0.f;
  if (lane < C) v = ld_dsmem_f32(mapa_shared(smem_u32(slot), static_cast<uint32_t>(lane)));
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float u = __shfl_xor_sync(0xffffffffu, v, o);
    v = kMax ? fmaxf(v, u) : v + u;
  }
  return v;
}

}  // namespace qc
}  // namespace r4
