// gemm_blockfp8.cu -- block-FP8 W8A8 GEMM on tcgen05 (kind::f8f6f4).
//
//   C[m, n] = bf16( sum_kb As[m,kb] * Ws[n/128,kb] * sum_{k in kb} e4m3(q[m,k]) e4m3(w[n,k]) )
//
// ("radiance_kernels.py", block_scaled_mm: e4m3 weights with one fp32 scale
// per 128x128 block, activations with one fp32 scale per token per 128 K.)
//
// The scales are arbitrary fp32, so the tensor core cannot apply them (its
// block-scale kinds take power-of-two ue8m0 scales only). Instead:
//  * weight-stationary orientation: a 128-row weight tile is exactly one
//    scale block along N, so Ws[n/128, kb] is one scalar per tile per K block;
//  * per 128-K block, 4 MMAs (K = 32 each) write a FRESH fp32 accumulator in
//    tensor memory; two accumulators alternate so the MMAs of block kb+1 run
//    while the epilogue promotes block kb;
//  * 8 epilogue warps (two per tensor-memory lane quarter, each owning half of
//    the token columns) load the block result and fold it into fp32 registers:
//    acc[t] += (As[t,kb] * Ws[nt,kb]) * D_kb[n,t]. The per-column scale
//    products are staged in shared memory once per block.
// Split-K and the last-arriving-CTA reduction are as in the W4A8 kernel.

#include <cuda_bf16.h>

#include <algorithm>
#include <cmath>

#include "r4_device.cuh"
#include "r4_internal.h"

namespace r4 {
namespace fp8 {

constexpr int kThreads = 320;   // warp 0 TMA, warp 1 MMA, warps 2..9 epilogue
constexpr int kEpiThreads = 256;
constexpr uint32_t kWSmem = 128 * 128;
constexpr int kMaxStages = 16;

struct Params {
  int M, KB;           // KB = K / 128 (blocks per row of As / Ws)
  int t_tiles, splits, kb_per_split, units;
  int ldc;
  const float *As;     // [M, KB]
  const float *Ws;     // [N/128, KB]
  uint16_t *c;
  float *partials;
  int *counters;
  int *err;
};

template <int BT>
struct Cfg {
  static constexpr uint32_t kXSmem = BT * 128;
  static constexpr uint32_t kStageBytes = ((kWSmem + kXSmem + 1023) / 1024) * 1024;
  static constexpr int kStagesRaw = static_cast<int>((220u * 1024u) / kStageBytes);
  static constexpr int kStages = kStagesRaw > kMaxStages ? kMaxStages : kStagesRaw;
  static constexpr uint32_t kTxBytes = kWSmem + kXSmem;
  static constexpr uint32_t kTmemCols = (2 * BT) < 32 ? 32 : 2 * BT;
  static constexpr uint32_t kMiscBytes = 2048;  // barriers + 2 x BT scale products
  static constexpr uint32_t kSmemBytes = kStages * kStageBytes + kMiscBytes + 1024;
  static constexpr int kHalf = BT / 2;          // columns per epilogue warp
  static constexpr int kCh = kHalf < 32 ? kHalf : 32;
};

__device__ __forceinline__ void decode_unit(const Params &p, int u, int &nt, int &tt, int &sp) {
  const int tile = u / p.splits;
  sp = u - tile * p.splits;
  nt = tile / p.t_tiles;
  tt = tile - nt * p.t_tiles;
}

template <int BT>
__global__ void __launch_bounds__(kThreads, 1)
    blockfp8_f8f6f4_kernel(const __grid_constant__ CUtensorMap tm_w, const __grid_constant__ CUtensorMap tm_x,
                           const Params p) {
  using C = Cfg<BT>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t *misc = smem + C::kStages * C::kStageBytes;
  float *sscale = reinterpret_cast<float *>(misc);                    // [2][BT]
  uint64_t *full_bar = reinterpret_cast<uint64_t *>(misc + 1024);     // [8]
  uint64_t *empty_bar = full_bar + kMaxStages;                        // [16]
  uint64_t *accf_bar = empty_bar + kMaxStages;                        // [2]
  uint64_t *acce_bar = accf_bar + 2;                                  // [2]
  uint64_t *drain_bar = acce_bar + 2;
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(drain_bar + 1);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
  volatile int *is_last = abort_flag + 1;
  volatile int *epi_abort = abort_flag + 2;   // set and read by epilogue threads only

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(&full_bar[s], 1);
      mbar_init(&empty_bar[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&accf_bar[a], 1);
      mbar_init(&acce_bar[a], kEpiThreads / 32);
    }
    mbar_init(drain_bar, 1);
    *abort_flag = 0;
    *is_last = 0;
    *epi_abort = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tm_w);
    tma_prefetch_desc(&tm_x);
    pdl_launch_dependents();
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, C::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    if (lane == 0) {
      const uint64_t pol_w = policy_evict_first();
      const uint64_t pol_x = policy_evict_last();
      int stage = 0;
      uint32_t phase = 0, issued_mask = 0, issued_phase = 0;
      bool ok = true;
      // Weights first (independent of the preceding kernel), then wait for
      // it before the first activation tile.
      int pre = 0;
      for (int u = blockIdx.x; u < p.units && pre < C::kStages; u += gridDim.x) {
        int nt, tt, sp;
        decode_unit(p, u, nt, tt, sp);
        const int kb0 = sp * p.kb_per_split, kb1 = min(p.KB, kb0 + p.kb_per_split);
        for (int kb = kb0; kb < kb1 && pre < C::kStages; ++kb, ++pre) {
          mbar_arrive_expect_tx(&full_bar[pre], C::kTxBytes);
          tma_load_3d(smem + pre * C::kStageBytes, &tm_w, &full_bar[pre], 0, 0, nt * p.KB + kb, pol_w);
        }
      }
      pdl_wait();
      int it = 0;
      for (int u = blockIdx.x; u < p.units && ok; u += gridDim.x) {
        int nt, tt, sp;
        decode_unit(p, u, nt, tt, sp);
        const int kb0 = sp * p.kb_per_split, kb1 = min(p.KB, kb0 + p.kb_per_split);
        for (int kb = kb0; kb < kb1; ++kb, ++it) {
          uint8_t *st = smem + stage * C::kStageBytes;
          if (it >= pre) {
            if (!mbar_wait(&empty_bar[stage], phase ^ 1u, abort_flag, p.err, DEV_ERR_WAIT_EMPTY)) {
              ok = false;
              break;
            }
            mbar_arrive_expect_tx(&full_bar[stage], C::kTxBytes);
            tma_load_3d(st, &tm_w, &full_bar[stage], 0, 0, nt * p.KB + kb, pol_w);
          }
          tma_load_2d(st + kWSmem, &tm_x, &full_bar[stage], kb * 128, tt * BT, pol_x);
          issued_mask |= 1u << stage;
          issued_phase = (issued_phase & ~(1u << stage)) | (phase << stage);
          if (++stage == C::kStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      for (int s = 0; s < C::kStages; ++s)
        if (issued_mask & (1u << s)) {
          volatile int dummy = 0;
          mbar_wait(&full_bar[s], (issued_phase >> s) & 1u, &dummy, p.err, DEV_ERR_WAIT_DRAIN);
        }
    }
    __syncwarp();
  } else if (warp == 1) {
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      uint32_t blk = 0;   // running count of 128-K blocks: accumulator = blk & 1
      bool ok = true;
      const uint32_t idesc = idesc_f8f6f4_e4m3(BT);
      for (int u = blockIdx.x; u < p.units && ok; u += gridDim.x) {
        int nt, tt, sp;
        decode_unit(p, u, nt, tt, sp);
        const int kb0 = sp * p.kb_per_split, kb1 = min(p.KB, kb0 + p.kb_per_split);
        for (int kb = kb0; kb < kb1; ++kb, ++blk) {
          const int acc = static_cast<int>(blk & 1u);
          const uint32_t acc_phase = (blk >> 1) & 1u;
          if (!mbar_wait(&acce_bar[acc], acc_phase ^ 1u, abort_flag, p.err, DEV_ERR_WAIT_ACC_EMPTY)) {
            ok = false;
            break;
          }
          if (!mbar_wait(&full_bar[stage], phase, abort_flag, p.err, DEV_ERR_WAIT_FULL)) {
            ok = false;
            break;
          }
          tc_fence_after();
          uint8_t *st = smem + stage * C::kStageBytes;
          const uint32_t a_base = smem_u32(st), b_base = smem_u32(st + kWSmem);
          const uint32_t d_tmem = tmem + static_cast<uint32_t>(acc * BT);
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            tc_mma_f8f6f4(d_tmem, sdesc_sw128_kmajor(a_base + 32u * kk), sdesc_sw128_kmajor(b_base + 32u * kk),
                          idesc, kk > 0 ? 1u : 0u);
          tc_commit(&empty_bar[stage]);
          tc_commit(&accf_bar[acc]);
          if (++stage == C::kStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      tc_commit(drain_bar);
      volatile int dummy = 0;
      mbar_wait(drain_bar, 0, &dummy, p.err, DEV_ERR_WAIT_DRAIN);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ promotion epilogue
    pdl_wait();                        // As, C and the workspace follow the stream order
    const int e = threadIdx.x - 64;    // 0..255
    const int ew = warp - 2;           // 0..7
    const int q = warp & 3;            // lane quarter
    const int h = ew >> 2;             // column half
    uint32_t blk = 0;
    bool ok = true;
    for (int u = blockIdx.x; u < p.units && ok; u += gridDim.x) {
      int nt, tt, sp;
      decode_unit(p, u, nt, tt, sp);
      const int kb0 = sp * p.kb_per_split, kb1 = min(p.KB, kb0 + p.kb_per_split);
      const int t0 = tt * BT;
      const int n = nt * 128 + q * 32 + lane;
      const int tile = nt * p.t_tiles + tt;
      float accv[C::kHalf];
#pragma unroll
      for (int j = 0; j < C::kHalf; ++j) accv[j] = 0.f;
      for (int kb = kb0; kb < kb1; ++kb, ++blk) {
        const int acc = static_cast<int>(blk & 1u);
        const uint32_t acc_phase = (blk >> 1) & 1u;
        float *ss = sscale + acc * BT;
        if (e < BT) {
          const int t = t0 + e;
          const float a = (t < p.M) ? __ldg(p.As + static_cast<size_t>(t) * p.KB + kb) : 0.f;
          ss[e] = a * __ldg(p.Ws + static_cast<size_t>(nt) * p.KB + kb);
        }
        // One barrier both publishes the scale products and makes the stop
        // decision uniform across the 256 epilogue threads.
        if (!mbar_wait(&accf_bar[acc], acc_phase, abort_flag, p.err, DEV_ERR_WAIT_ACC_FULL)) *epi_abort = 1;
        named_bar_sync(1, kEpiThreads);
        if (*epi_abort) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t taddr =
            tmem + (static_cast<uint32_t>(q * 32) << 16) + static_cast<uint32_t>(acc * BT + h * C::kHalf);
        uint32_t r[C::kHalf];
#pragma unroll
        for (int c0 = 0; c0 < C::kHalf; c0 += C::kCh) {
          uint32_t tmp[32];
          if constexpr (C::kCh == 32) {
            tc_ld_32x32b_x32(taddr + c0, tmp);
          } else {
            tc_ld_32x32b_x16(taddr + c0, tmp);
          }
#pragma unroll
          for (int j = 0; j < C::kCh; ++j) r[c0 + j] = tmp[j];
        }
        tc_wait_ld();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&acce_bar[acc]);
        const float4 *s4 = reinterpret_cast<const float4 *>(ss + h * C::kHalf);
#pragma unroll
        for (int j4 = 0; j4 < C::kHalf / 4; ++j4) {
          const float4 f = s4[j4];
          accv[4 * j4 + 0] = fmaf(f.x, __uint_as_float(r[4 * j4 + 0]), accv[4 * j4 + 0]);
          accv[4 * j4 + 1] = fmaf(f.y, __uint_as_float(r[4 * j4 + 1]), accv[4 * j4 + 1]);
          accv[4 * j4 + 2] = fmaf(f.z, __uint_as_float(r[4 * j4 + 2]), accv[4 * j4 + 2]);
          accv[4 * j4 + 3] = fmaf(f.w, __uint_as_float(r[4 * j4 + 3]), accv[4 * j4 + 3]);
        }
      }
      if (!ok) break;
      const int tc0 = t0 + h * C::kHalf;
      if (p.splits == 1) {
#pragma unroll
        for (int j = 0; j < C::kHalf; ++j)
          if (tc0 + j < p.M) p.c[static_cast<size_t>(tc0 + j) * p.ldc + n] = f32_to_bf16_rn(accv[j]);
      } else {
        float *part = p.partials + (static_cast<size_t>(tile) * p.splits + sp) * (128 * BT);
#pragma unroll
        for (int j = 0; j < C::kHalf; ++j) part[(h * C::kHalf + j) * 128 + q * 32 + lane] = accv[j];
        __threadfence();
        named_bar_sync(2, kEpiThreads);
        if (e == 0) {
          const int prev = atomicAdd(p.counters + tile, 1);
          *is_last = (prev == p.splits - 1) ? 1 : 0;
        }
        named_bar_sync(2, kEpiThreads);
        if (*is_last) {
          __threadfence();
          const float *base = p.partials + static_cast<size_t>(tile) * p.splits * (128 * BT);
          reduce_partials_store<BT>(base, p.splits, min(BT, p.M - t0), nt * 128, nt * 128 + 128, nullptr, t0, p.c,
                                    p.ldc, e, kEpiThreads);
          if (e == 0) p.counters[tile] = 0;
        }
        named_bar_sync(2, kEpiThreads);
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
}

template <int BT>
int launch_bt(const uint8_t *q, const float *As, const uint8_t *packed, int64_t M, int64_t N, int64_t K,
              uint16_t *c, int64_t ldc, void *ws, const GemmPlan &pl, cudaStream_t st) {
  using C = Cfg<BT>;
  CUtensorMap tm_w, tm_x;
  {
    const uint64_t dims[3] = {128, 128, static_cast<uint64_t>((N / 128) * (K / 128))};
    const uint64_t strides[2] = {128, 16384};
    const uint32_t box[3] = {128, 128, 1};
    if (encode_tiled(&tm_w, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<uint8_t *>(packed), dims, strides, box,
                     CU_TENSOR_MAP_SWIZZLE_128B) != CUDA_SUCCESS)
      return R4_ERR_CUDA;
  }
  {
    const uint64_t dims[2] = {static_cast<uint64_t>(K), static_cast<uint64_t>(M)};
    const uint64_t strides[1] = {static_cast<uint64_t>(K)};
    const uint32_t box[2] = {128, static_cast<uint32_t>(BT)};
    if (encode_tiled(&tm_x, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t *>(q), dims, strides, box,
                     CU_TENSOR_MAP_SWIZZLE_128B) != CUDA_SUCCESS)
      return R4_ERR_CUDA;
  }
  Params p;
  p.M = static_cast<int>(M);
  p.KB = pl.KB;
  p.t_tiles = pl.t_tiles;
  p.splits = pl.splits;
  p.kb_per_split = pl.kb_per_split;
  p.units = pl.units;
  p.ldc = static_cast<int>(ldc);
  p.As = As;
  p.Ws = reinterpret_cast<const float *>(packed + fp8_packed_codes_bytes(N, K));
  p.c = c;
  p.counters = reinterpret_cast<int *>(ws);
  p.partials = ws ? reinterpret_cast<float *>(reinterpret_cast<uint8_t *>(ws) + pl.counters_bytes) : nullptr;
  p.err = device_error_word();
  auto kern = blockfp8_f8f6f4_kernel<BT>;
  if (ensure_smem_attr(reinterpret_cast<const void *>(kern), C::kSmemBytes) != cudaSuccess) return R4_ERR_CUDA;
  if (launch_pdl(kern, dim3(pl.grid), dim3(kThreads), C::kSmemBytes, st, tm_w, tm_x, p) != cudaSuccess)
    return R4_ERR_CUDA;
  set_last_kernel(BT == 32 ? "blockfp8_f8f6f4_kernel<32>"
                  : BT == 64 ? "blockfp8_f8f6f4_kernel<64>"
                             : "blockfp8_f8f6f4_kernel<128>");
  return cudaGetLastError() == cudaSuccess ? R4_OK : R4_ERR_CUDA;
}

}  // namespace fp8

GemmPlan plan_blockfp8(int64_t M, int64_t N, int64_t K, int sms) {
  GemmPlan pl;
  const int bt = M <= 32 ? 32 : M <= 64 ? 64 : 128;
  pl.BT = bt;
  pl.n_tiles = static_cast<int>(N / 128);
  pl.t_tiles = static_cast<int>(ceil_div(M, bt));
  pl.KB = static_cast<int>(K / 128);
  const int64_t tiles = static_cast<int64_t>(pl.n_tiles) * pl.t_tiles;
  // per-SM streaming rate is capped (bytes in flight / latency), not hbm/active
  const double hbm = 6.5e12, sm_bw = 60e9, sm_flops = 4.5e15 / 152.0, sm_l2 = 150e9;
  const double kb_bytes = 128.0 * 128 + 128.0 * bt;
  const double kb_flops = 2.0 * 128 * bt * 128;
  int best_s = 1;
  double best_t = 1e30;
  const int forced = options().fp8_splits;
  for (int s = 1; s <= std::min(pl.KB, 64); ++s) {
    const int kbps = static_cast<int>(ceil_div(pl.KB, s));
    if (static_cast<int64_t>(s - 1) * kbps >= pl.KB) continue;
    const int64_t units = tiles * s;
    const int64_t active = std::min<int64_t>(units, sms);
    const double waves = std::ceil(static_cast<double>(units) / sms);
    const double t_unit = std::max(kbps * kb_bytes / std::min(hbm / active, sm_bw), kbps * kb_flops / sm_flops);
    double t = waves * t_unit;
    if (s > 1) {
      const double pbytes = static_cast<double>(units) * 128 * bt * 4;
      t += 2 * pbytes / hbm + s * 128.0 * bt * 4 / sm_l2;
    }
    if (forced ? (s == forced) : (t < best_t * 0.97)) {
      best_t = t;
      best_s = s;
    }
  }
  if (forced && forced <= pl.KB) best_s = forced;
  pl.kb_per_split = static_cast<int>(ceil_div(pl.KB, best_s));
  pl.splits = static_cast<int>(ceil_div(pl.KB, pl.kb_per_split));
  pl.units = static_cast<int>(tiles * pl.splits);
  pl.grid = std::min(pl.units, sms);
  if (pl.splits > 1) {
    pl.counters_bytes = round_up(static_cast<size_t>(tiles) * 4, 256);
    pl.ws_bytes = pl.counters_bytes + static_cast<size_t>(pl.units) * 128 * bt * 4;
  }
  return pl;
}

int launch_gemm_blockfp8(const uint8_t *q, const float *As, const uint8_t *packed, int64_t M, int64_t N,
                         int64_t K, uint16_t *c, int64_t ldc, void *ws, const GemmPlan &pl, cudaStream_t st) {
  switch (pl.BT) {
    case 32: return fp8::launch_bt<32>(q, As, packed, M, N, K, c, ldc, ws, pl, st);
    case 64: return fp8::launch_bt<64>(q, As, packed, M, N, K, c, ldc, ws, pl, st);
    case 128: return fp8::launch_bt<128>(q, As, packed, M, N, K, c, ldc, ws, pl, st);
    default: return R4_ERR_INVALID_ARG;
  }
}

}  // namespace r4
