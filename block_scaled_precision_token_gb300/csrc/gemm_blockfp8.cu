// gemm_blockfp8.cu -- block-FP8 W8A8 GEMM on tcgen05 (kind::f8f6f4).
//
//   C[m, n] = bf16( sum_kb As[m,kb] * Ws[n/128,kb] * sum_{k in kb} e4m3(q[m,k]) e4m3(w[n,k]) )
//
// ("radiance_kernels.py", block_scaled_mm: e4m3 weights with one fp32 scale
// per 128x128 block, activations with one fp32 scale per token per 128 K.)
//
// The scales are arbitrary fp32, so the tensor core cannot apply them (its
// block-scale kinds take power-of-two ue8m0 scales only). Instead:
//  * a 128-row weight block is exactly one scale block along N, so
//    Ws[n/128, kb] is one scalar per 128 rows per K block (the 128-token
//    tile takes two such blocks, 256 rows, when N allows);
//  * every 128-K block is its own "slot": 4 MMAs (K = 32 each) write a FRESH
//    fp32 accumulator in tensor memory. Slot g uses accumulator buffer
//    g % kNumBuf; with 512 columns there are 2 (256 weight rows) to 16
//    buffers, so the MMAs run ahead of the promotion epilogue;
//  * 4 x kH epilogue warps (one per tensor-memory lane quarter and column
//    group) load each block result and fold it into fp32 registers. Tiles of
//    up to 64 tokens keep the weights on the lanes, 32 (or 16) token columns
//    per warp: acc[t] += As[t,kb] * (Ws[nt,kb] * D_kb[n,t]), the scaling and
//    the accumulation each one packed f32x2 instruction per two columns. The
//    128-token tile puts the tokens on the lanes (see Cfg::kTokMajor), eight
//    warps of 128 (or 64) n columns: acc[n] += (As[t,kb] * Ws[n/128,kb]) *
//    D_kb[t,n];
//  * the scales reach the epilogue without a handshake per K block: the
//    epilogue threads themselves copy As and Ws for a chunk of 16 K blocks
//    of their tile into shared memory (As transposed, [kb][token], so a
//    warp's 32 token columns of one K block are 128 contiguous bytes read
//    as broadcasts), one chunk ahead: the global loads of chunk c + 1 are in
//    flight while chunk c is promoted, and one barrier of the epilogue
//    threads per chunk publishes them. (Measured on GB300 against a scale
//    warp publishing As * Ws in a ring with ready / empty barriers per K
//    block: that handshake alone held the pipeline -- no MMA, no promotion
//    -- at 50 us for M=2048, N=6144, K=2048, 37 us without it.)
//  * decode tiles (BT <= 64) run two TMA producer warps: one thread issuing
//    every weight and activation copy caps the weight stream (each TMA issue
//    holds its thread for a few hundred cycles on GB300);
//  * the per-K-block handshakes (block result ready, accumulator free, stage
//    full) spin on a non-blocking mbarrier test, bounded like every wait;
//  * unsplit tiles of 32- and 64-column warps store through shared memory
//    and TMA tensor stores, so the next unit's promotion starts at once.
// Split-K and the last-arriving-CTA reduction follow the W4A8 kernel, with
// the partials staged for coalesced stores, one acq_rel fence per CTA
// around the arrival and a sum that stores four bf16 at a time.

#include <cuda_bf16.h>

#include <algorithm>
#include <cmath>

#include "r4_device.cuh"
#include "r4_internal.h"

namespace r4 {
namespace fp8 {

constexpr uint32_t kWSmem = 128 * 128;
constexpr int kMaxStages = 16;
constexpr int kMaxBuf = 16;
constexpr int kChunk = 16;          // K blocks of scales staged per epilogue chunk

struct Params {
  int M, KB;           // KB = K / 128 (blocks per row of As / Ws)
  int t_tiles, splits, kb_per_split, units;
  int ldc;
  int tma_store;       // 1: unsplit tiles leave through shared memory and TMA tensor stores
  int inject_stall;    // test of the bounded waits: CTA 0 withholds its first activation copy
  int early_w;         // 1: weight tiles are requested before waiting for the preceding kernel
  int c_vec4;          // 1: C rows start 8-byte aligned (4 bf16 per store in the split-K sum)
  const float *As;     // [M, KB]
  const float *Ws;     // [N/128, KB]
  uint16_t *c;
  float *partials;
  int *counters;
  int *err;
};

template <int BT, int BN = 128>
struct Cfg {
  static constexpr int kProd = BT <= 64 ? 2 : 1;           // TMA producer warps
  static constexpr int kMmaWarp = kProd;                   // first MMA-issuing warp
  static constexpr int kMma = 2;                           // MMA-issuing warps (slot g: warp g % kMma)
  static constexpr int kEpiWarp0 = kProd + kMma;
  // 128-token tiles accumulate token-major: the activation tile is the MMA's
  // A operand (tensor-memory lane = token) and the weight tile its B operand
  // (column = n), so each thread's scale for a K block is the single product
  // As[t,kb] * Ws[n/128,kb] -- one FMA per element -- and its outputs are
  // contiguous in a row of C. Narrower tiles keep the weights on the lanes
  // (the MMA needs 128 rows).
  static constexpr bool kTokMajor = BT == 128;
  // Weight rows per tile: 128, or 256 for the token-major tile (two 128-row
  // scale blocks side by side; one N = 256 MMA per K step).
  static constexpr int kNB = BN / 128;                     // 128-row weight blocks per tile
  static constexpr int kAccCols = kTokMajor ? BN : BT;     // accumulator columns (the MMA's N)
  // accumulator columns per epilogue warp: the token-major tile's n columns
  // in two groups (eight warps), else 32 (or BT) tokens. (Sixteen warps of
  // 64 columns for the 256-row tile, at 96 registers: 13 % slower.)
  static constexpr int kCW = kTokMajor ? kAccCols / 2 : (BT < 32 ? BT : 32);
  static constexpr int kH = kAccCols / kCW;                // column groups
  static constexpr int kEpiWarps = 4 * kH;
  static constexpr int kEpiThreads = 32 * kEpiWarps;
  static constexpr int kThreads = 32 * (kEpiWarp0 + kEpiWarps);
  // A scheduler's 16384 registers serve every warp placed on it (warps are
  // spread over the SM's four schedulers), in steps of 8 a thread.
  static constexpr int kWarpsPerSched = (kThreads / 32 + 3) / 4;
  static constexpr int kRegLimit = (16384 / (32 * kWarpsPerSched)) / 8 * 8;
  static constexpr int kMaxReg = kTokMajor ? (kRegLimit > 168 ? 168 : kRegLimit) : (kThreads > 576 ? 96 : 128);
  // Token-major promotion: all loads of a K block, then one wait, when the
  // registers hold a second copy of the accumulators; else 16-column loads,
  // each waited for (the registers hold the accumulators and one load).
  static constexpr bool kLdAll = kCW * 2 + 40 <= kMaxReg;
  static constexpr int kNumBufRaw = 512 / kAccCols;
  static constexpr int kNumBuf = kNumBufRaw > kMaxBuf ? kMaxBuf : kNumBufRaw;
  static constexpr uint32_t kTmemCols = static_cast<uint32_t>(kNumBuf * kAccCols);
  static constexpr uint32_t kWBytes = kNB * kWSmem;         // weight part of a stage
  static constexpr uint32_t kXSmem = BT * 128;
  static constexpr uint32_t kStageBytes = ((kWBytes + kXSmem + 1023) / 1024) * 1024;
  // scale chunks: 2 buffers of As [kChunk][BT] and Ws [kNB][kChunk]
  static constexpr uint32_t kScFloats = kChunk * BT + kChunk * kNB;
  static constexpr uint32_t kScBytes = 2 * kScFloats * 4;
  static constexpr int kScPer = (BT * kChunk + kEpiThreads - 1) / kEpiThreads;   // As values per thread
  static constexpr uint32_t kMiscBytes = 1024;             // barriers and flags
  // Unsplit tiles of 32-token warps store their output through shared
  // memory: one [32 tokens][32 n] bf16 buffer per epilogue warp, written by
  // the warp and handed to a TMA tensor store, so the next unit's promotion
  // starts without waiting for global stores.
  static constexpr bool kTmaOut = kCW >= 32;
  // Split-K reduction: 4 x 4 loads in flight; for the 128-token tile in a
  // separate (not inlined) function, whose registers then do not add to
  // the promotion loop's.
  static constexpr bool kRedCall = BT == 128;
  static constexpr uint32_t kOutBytes = kTmaOut ? static_cast<uint32_t>(kEpiWarps * kCW) * 64u : 0u;
  static constexpr int kStagesRaw =
      static_cast<int>((227u * 1024u - 1024u - kMiscBytes - kScBytes - kOutBytes) / kStageBytes);
  static constexpr int kStagesCap = kStagesRaw > kMaxStages ? kMaxStages : kStagesRaw;
  static constexpr int kStages = (kStagesCap / kProd) * kProd;   // each producer owns fixed stages
  // With at least as many stages as accumulator buffers, the stage's empty
  // barrier (the MMA commit after slot g) also tells the epilogue that slot
  // g's accumulator is complete, and the MMA thread commits once per slot:
  // the MMAs of slot g + kStages (the stage's next phase) need the buffer of
  // slot g + kStages - kNumBuf >= g back from the epilogue, so that barrier
  // cannot run a phase ahead of the epilogue's wait.
  static constexpr bool kFullIsEmpty = kStages >= kNumBuf;
  static constexpr uint32_t kTxBytes = kWBytes + kXSmem;
  static constexpr uint32_t kSmemBytes = kStages * kStageBytes + kOutBytes + kScBytes + kMiscBytes + 1024;
  static_assert(kTmemCols >= 32 && (kTmemCols & (kTmemCols - 1)) == 0, "tensor-memory allocation");
  static_assert(kThreads <= 1024, "block size");
  static_assert(kStages >= kProd, "stage count");
  static_assert(BN == 128 || (BN == 256 && kTokMajor), "256-row weight tiles only with the token-major tile");
  static_assert(!kTokMajor || kCW % 16 == 0, "epilogue columns");
  static_assert(kSmemBytes <= 227u * 1024u, "shared memory");
};

// Walks the K-block slots of this CTA's units in order.
struct SlotCursor {
  int u, kb, kb1, nt, tt, sp;
  __device__ __forceinline__ void decode(const Params &p) {
    const int tile = u / p.splits;
    sp = u - tile * p.splits;
    nt = tile / p.t_tiles;
    tt = tile - nt * p.t_tiles;
    kb = sp * p.kb_per_split;
    kb1 = min(p.KB, kb + p.kb_per_split);
  }
  __device__ __forceinline__ void start(const Params &p) {
    u = blockIdx.x;
    if (u < p.units) decode(p);
  }
  __device__ __forceinline__ bool valid(const Params &p) const { return u < p.units; }
  __device__ __forceinline__ void next(const Params &p) {
    if (++kb == kb1) {
      u += gridDim.x;
      if (u < p.units) decode(p);
    }
  }
};

// Walks this CTA's units in chunks of up to kChunk consecutive K blocks.
struct ChunkCursor {
  int u, kb, kb1, nt, tt;
  __device__ __forceinline__ void decode(const Params &p) {
    const int tile = u / p.splits;
    const int sp = u - tile * p.splits;
    nt = tile / p.t_tiles;
    tt = tile - nt * p.t_tiles;
    kb = sp * p.kb_per_split;
    kb1 = min(p.KB, kb + p.kb_per_split);
  }
  __device__ __forceinline__ void start(const Params &p) {
    u = blockIdx.x;
    if (u < p.units) decode(p);
  }
  __device__ __forceinline__ bool valid(const Params &p) const { return u < p.units; }
  __device__ __forceinline__ int len() const { return min(kChunk, kb1 - kb); }
  __device__ __forceinline__ void next(const Params &p) {
    kb += kChunk;
    if (kb >= kb1) {
      u += gridDim.x;
      if (u < p.units) decode(p);
    }
  }
};

// tcgen05.wait::ld that also names the loaded registers as its operands, so
// no use of them can be scheduled before the wait.
__device__ __forceinline__ void wait_ld_into(uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.wait::ld.sync.aligned;"
      : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]), "+r"(r[7]),
        "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]), "+r"(r[14]), "+r"(r[15])
      :
      : "memory");
}

// Sum of `splits` partial tiles [tokens][128] of one 128-row block, stored
// `stride` floats apart, to bf16 C rows t0 .. t0 + tmax - 1, columns n0 ..
// n0 + 127. A thread takes groups of four columns, 32 groups to a token row
// (coalesced loads), with up to 4 groups x 4 partials in flight; each sum
// runs in split order (deterministic) and its four bf16 leave in one 8-byte
// store when C's rows allow it (vec4), else one at a time.
__device__ __forceinline__ void reduce_block(const float *base, size_t stride, int splits, int tmax, int n0, int t0,
                                             uint16_t *c, int ldc, int vec4, int tid, int nthreads) {
  constexpr int U = 4, S = 4;
  const int total = tmax * 32;
  for (int g0 = tid; g0 < total; g0 += nthreads * U) {
    float4 acc[U];
#pragma unroll
    for (int k = 0; k < U; ++k) {
      const int idx = g0 + k * nthreads;
      acc[k] = idx < total ? __ldcg(reinterpret_cast<const float4 *>(base + (idx >> 5) * 128 + (idx & 31) * 4))
                           : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    for (int s0 = 1; s0 < splits; s0 += S) {
      float4 v[S][U];
#pragma unroll
      for (int ss = 0; ss < S; ++ss) {
        const float *sp = base + static_cast<size_t>(s0 + ss) * stride;
#pragma unroll
        for (int k = 0; k < U; ++k) {
          const int idx = g0 + k * nthreads;
          v[ss][k] = (s0 + ss < splits && idx < total)
                         ? __ldcg(reinterpret_cast<const float4 *>(sp + (idx >> 5) * 128 + (idx & 31) * 4))
                         : make_float4(0.f, 0.f, 0.f, 0.f);
        }
      }
#pragma unroll
      for (int ss = 0; ss < S; ++ss)
        if (s0 + ss < splits) {
#pragma unroll
          for (int k = 0; k < U; ++k) {
            acc[k].x += v[ss][k].x;
            acc[k].y += v[ss][k].y;
            acc[k].z += v[ss][k].z;
            acc[k].w += v[ss][k].w;
          }
        }
    }
#pragma unroll
    for (int k = 0; k < U; ++k) {
      const int idx = g0 + k * nthreads;
      if (idx >= total) continue;
      uint16_t *dst = c + static_cast<size_t>(t0 + (idx >> 5)) * ldc + n0 + (idx & 31) * 4;
      if (vec4) {
        *reinterpret_cast<uint2 *>(dst) = make_uint2(pack_bf16x2(acc[k].x, acc[k].y), pack_bf16x2(acc[k].z, acc[k].w));
      } else {
        dst[0] = f32_to_bf16_rn(acc[k].x);
        dst[1] = f32_to_bf16_rn(acc[k].y);
        dst[2] = f32_to_bf16_rn(acc[k].z);
        dst[3] = f32_to_bf16_rn(acc[k].w);
      }
    }
  }
}

// The same, not inlined: the 168-register 128-token kernel keeps its own
// register budget around the call.
__device__ __noinline__ void reduce_block_call(const float *base, size_t stride, int splits, int tmax, int n0, int t0,
                                               uint16_t *c, int ldc, int vec4, int tid, int nthreads) {
  reduce_block(base, stride, splits, tmax, n0, t0, c, ldc, vec4, tid, nthreads);
}

__device__ __forceinline__ void fence_acq_rel_gpu() { asm volatile("fence.acq_rel.gpu;" ::: "memory"); }

// 4-byte asynchronous copy global -> shared; src_bytes = 0 writes zero.
__device__ __forceinline__ void cp_async4(void *dst, const void *src, uint32_t src_bytes) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;" ::"r"(smem_u32(dst)), "l"(src), "r"(src_bytes)
               : "memory");
}

// Copies one scale chunk into `buf` with cp.async (no registers held while
// it is in flight): As transposed, buf[i * BT + t] = As[t0 + t, kb + i], then
// buf[kChunk * BT + h * kChunk + i] = Ws[nt * kNB + h, kb + i]; 0 past M or
// past the chunk. Element
// r of thread e is (t, i) = divmod(e + kEpiThreads * r, kChunk): consecutive
// threads walk a token's 16 consecutive K blocks (64 contiguous bytes).
template <int BT, int BN>
__device__ __forceinline__ void copy_scale_chunk(const Params &p, const ChunkCursor &ch, float *buf, int e) {
  using C = Cfg<BT, BN>;
  const int n = ch.len();
  const int t0 = ch.tt * BT;
#pragma unroll
  for (int r = 0; r < C::kScPer; ++r) {
    const int idx = e + C::kEpiThreads * r;
    const int t = idx / kChunk, i = idx - t * kChunk;
    if (t < BT) {
      const bool in = i < n && t0 + t < p.M;
      cp_async4(buf + i * BT + t, in ? p.As + static_cast<size_t>(t0 + t) * p.KB + ch.kb + i : p.As, in ? 4u : 0u);
    }
  }
  if (e < kChunk * C::kNB) {
    const int h = e / kChunk, i = e - h * kChunk;
    cp_async4(buf + kChunk * BT + e,
              i < n ? p.Ws + static_cast<size_t>(ch.nt * C::kNB + h) * p.KB + ch.kb + i : p.Ws, i < n ? 4u : 0u);
  }
  asm volatile("cp.async.commit_group;" ::: "memory");
}

template <int BT, int BN>
__global__ void __launch_bounds__(Cfg<BT, BN>::kThreads, 1) __maxnreg__((Cfg<BT, BN>::kMaxReg))
    blockfp8_f8f6f4_kernel(const __grid_constant__ CUtensorMap tm_w, const __grid_constant__ CUtensorMap tm_x,
                           const __grid_constant__ CUtensorMap tm_c, const Params p) {
  using C = Cfg<BT, BN>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t *outbuf = smem + C::kStages * C::kStageBytes;                         // [kEpiWarps][32][kCW] bf16
  float *scbuf = reinterpret_cast<float *>(outbuf + C::kOutBytes);              // [2][kScFloats]
  uint8_t *misc = reinterpret_cast<uint8_t *>(scbuf) + C::kScBytes;
  uint64_t *full_bar = reinterpret_cast<uint64_t *>(misc);   // [kMaxStages]
  uint64_t *empty_bar = full_bar + kMaxStages;               // [kMaxStages]
  uint64_t *accf_bar = empty_bar + kMaxStages;               // [kMaxBuf]
  uint64_t *acce_bar = accf_bar + kMaxBuf;                   // [kMaxBuf]
  uint64_t *drain_bar = acce_bar + kMaxBuf;
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(drain_bar + C::kMma);   // drain_bar: one per MMA warp
  volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
  volatile int *is_last = abort_flag + 1;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(&full_bar[s], 1);
      mbar_init(&empty_bar[s], 1);   // the MMA commit
    }
    for (int b = 0; b < C::kNumBuf; ++b) {
      mbar_init(&accf_bar[b], 1);
      mbar_init(&acce_bar[b], C::kEpiWarps);
    }
    for (int m = 0; m < C::kMma; ++m) mbar_init(&drain_bar[m], 1);
    *abort_flag = 0;
    *is_last = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tm_w);
    tma_prefetch_desc(&tm_x);
    pdl_launch_dependents();
  }
  if (warp == C::kMmaWarp) {
    tmem_alloc(tmem_slot, C::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp < C::kProd) {
    // ------------------------------------------------------------ TMA producers
    // Slot g belongs to producer g % kProd and lives in stage g % kStages.
    const int pw = warp;
    if (lane == 0) {
      const uint64_t pol_w = policy_evict_first();
      const uint64_t pol_x = policy_evict_last();
      uint32_t issued_mask = 0, issued_phase = 0;
      // Weights first (independent of the preceding kernel), then wait for
      // it before the first activation tile.
      if (!p.early_w) pdl_wait();
      {
        SlotCursor cu;
        cu.start(p);
        for (int g = 0; cu.valid(p) && g < C::kStages; ++g, cu.next(p))
          if (g % C::kProd == pw) {
            mbar_arrive_expect_tx(&full_bar[g], C::kTxBytes);
#pragma unroll
            for (int h = 0; h < C::kNB; ++h)
              tma_load_3d(smem + g * C::kStageBytes + h * kWSmem, &tm_w, &full_bar[g], 0, 0,
                          (cu.nt * C::kNB + h) * p.KB + cu.kb, pol_w);
          }
      }
      pdl_wait();
      SlotCursor cu;
      cu.start(p);
      for (int g = 0; cu.valid(p); ++g, cu.next(p)) {
        if (g % C::kProd != pw) continue;
        const int stage = g % C::kStages;
        const uint32_t phase = static_cast<uint32_t>(g / C::kStages) & 1u;
        uint8_t *st = smem + stage * C::kStageBytes;
        if (g >= C::kStages) {
          if (!mbar_wait(&empty_bar[stage], phase ^ 1u, abort_flag, p.err, DEV_ERR_WAIT_EMPTY)) break;
          mbar_arrive_expect_tx(&full_bar[stage], C::kTxBytes);
#pragma unroll
          for (int h = 0; h < C::kNB; ++h)
            tma_load_3d(st + h * kWSmem, &tm_w, &full_bar[stage], 0, 0, (cu.nt * C::kNB + h) * p.KB + cu.kb, pol_w);
        }
        // (Failure-detection test: with inject_stall, CTA 0 never issues its
        // first activation copy, so the stage's transaction never completes.)
        if (!(p.inject_stall && blockIdx.x == 0 && g == 0))
          tma_load_2d(st + C::kWBytes, &tm_x, &full_bar[stage], cu.kb * 128, cu.tt * BT, pol_x);
        // Record the newest phase of every stage: a parity wait cannot tell
        // phase k from k + 2, and a stage only advances once its earlier
        // phases completed.
        issued_mask |= 1u << stage;
        issued_phase = (issued_phase & ~(1u << stage)) | (phase << stage);
      }
      // Never leave a copy in flight: wait (bounded, even after an abort)
      // for the last load issued into each of this producer's stages.
      for (int s_ = 0; s_ < C::kStages; ++s_)
        if (issued_mask & (1u << s_)) {
          volatile int dummy = 0;
          mbar_wait(&full_bar[s_], (issued_phase >> s_) & 1u, &dummy, p.err, DEV_ERR_WAIT_DRAIN);
        }
    }
    __syncwarp();
  } else if (warp < C::kMmaWarp + C::kMma) {
    // ------------------------------------------------------------ MMA issuers
    // Every slot writes a fresh accumulator buffer, so the slots can be
    // issued by two threads independently (slot g by warp g % kMma): one
    // thread's barrier waits and commits overlap the other's MMAs in the
    // tensor pipe. (With one issuer, four N = 128 MMAs of ~80 cycles each
    // left the pipe idle during ~400-700 cycles of per-slot handshake.)
    const int mw = warp - C::kMmaWarp;
    if (lane == 0) {
      const uint32_t idesc = idesc_f8f6f4_e4m3(C::kAccCols);
      SlotCursor cu;
      cu.start(p);
      for (int g = 0; cu.valid(p); ++g, cu.next(p)) {
        if (g % C::kMma != mw) continue;
        const int stage = g % C::kStages;
        const uint32_t phase = static_cast<uint32_t>(g / C::kStages) & 1u;
        const int buf = g % C::kNumBuf;
        const uint32_t bphase = static_cast<uint32_t>(g / C::kNumBuf) & 1u;
        if (!mbar_spin_wait(&acce_bar[buf], bphase ^ 1u, abort_flag, p.err, DEV_ERR_WAIT_ACC_EMPTY)) break;
        if (!mbar_spin_wait(&full_bar[stage], phase, abort_flag, p.err, DEV_ERR_WAIT_FULL)) break;
        tc_fence_after();
        uint8_t *st = smem + stage * C::kStageBytes;
        const uint32_t w_base = smem_u32(st), x_base = smem_u32(st + C::kWBytes);
        const uint32_t a_base = C::kTokMajor ? x_base : w_base, b_base = C::kTokMajor ? w_base : x_base;
        const uint32_t d_tmem = tmem + static_cast<uint32_t>(buf * C::kAccCols);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          tc_mma_f8f6f4(d_tmem, sdesc_sw128_kmajor(a_base + 32u * kk), sdesc_sw128_kmajor(b_base + 32u * kk), idesc,
                        kk > 0 ? 1u : 0u);
        tc_commit(&empty_bar[stage]);
        if constexpr (!C::kFullIsEmpty) tc_commit(&accf_bar[buf]);
      }
      // All MMAs this thread issued must be complete before tensor memory is freed.
      tc_commit(&drain_bar[mw]);
      volatile int dummy = 0;
      mbar_wait(&drain_bar[mw], 0, &dummy, p.err, DEV_ERR_WAIT_DRAIN);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ promotion epilogue
    pdl_wait();                        // As, C and the workspace follow the stream order
    const int ew = warp - C::kEpiWarp0;
    const int e = ew * 32 + lane;      // 0 .. kEpiThreads-1
    const int q = warp & 3;            // tensor-memory lane quarter this warp may access
    const int h = ew >> 2;             // column group
    const int col0 = h * C::kCW;
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(q * 32) << 16) + static_cast<uint32_t>(col0);
    // Scale chunks: the first is staged before the loop; each chunk's
    // barrier makes the next one (stored at the end of the chunk) visible.
    {
      ChunkCursor c0;
      c0.start(p);
      if (c0.valid(p)) copy_scale_chunk<BT, BN>(p, c0, scbuf, e);
    }
    asm volatile("cp.async.wait_all;" ::: "memory");
    named_bar_sync(1, C::kEpiThreads);
    int cur = 0;                       // scale buffer of the chunk being promoted
    SlotCursor cu;
    cu.start(p);
    int g = 0;
    int abort_u = -1;                  // unit at which an expired wait stopped the epilogue
    while (cu.valid(p)) {
      const int nt = cu.nt, tt = cu.tt, sp = cu.sp, u = cu.u;
      const int t0 = tt * BT;
      const int n = nt * BN + q * 32 + lane;
      const int tile = nt * p.t_tiles + tt;
      float acc[C::kCW];
#pragma unroll
      for (int j = 0; j < C::kCW; ++j) acc[j] = 0.f;
      bool ok = true, stop = false;
      while (cu.valid(p) && cu.u == u) {
        // one chunk: up to kChunk K blocks of this unit
        const int kbc = cu.kb;
        const int nblk = min(kChunk, cu.kb1 - kbc);
        {                              // next chunk's scales, in flight during the promotion
          ChunkCursor cn;
          cn.u = u;
          cn.nt = nt;
          cn.tt = tt;
          cn.kb = kbc;
          cn.kb1 = cu.kb1;
          cn.next(p);
          if (cn.valid(p)) copy_scale_chunk<BT, BN>(p, cn, scbuf + (cur ^ 1) * C::kScFloats, e);
        }
        const float *sc = scbuf + cur * C::kScFloats;
        for (int i = 0; i < nblk; ++i, ++g, cu.next(p)) {
          if (!ok) continue;           // stopped: skip to the chunk barrier
          const int buf = g % C::kNumBuf;
          uint64_t *fbar = C::kFullIsEmpty ? &empty_bar[g % C::kStages] : &accf_bar[buf];
          const uint32_t fpar = static_cast<uint32_t>(C::kFullIsEmpty ? g / C::kStages : g / C::kNumBuf) & 1u;
          // Warp-uniform wait (tcgen05.ld needs the whole warp).
          if (!warp_spin_wait(fbar, fpar, abort_flag, p.err, DEV_ERR_WAIT_ACC_FULL)) {
            ok = false;
            continue;
          }
          tc_fence_after();
          const uint32_t ta = lane_base + static_cast<uint32_t>(buf * C::kAccCols);
          if constexpr (C::kTokMajor && !C::kLdAll) {
            // kCW columns in 16-column loads, each waited for; the buffer
            // is released after the last.
            // acc[n] += (As[t,kb] * Ws[n/128,kb]) * D[t,n]
            const float sa = sc[i * BT + q * 32 + lane] * sc[kChunk * BT + (col0 >> 7) * kChunk + i];
#pragma unroll
            for (int part = 0; part < C::kCW / 16; ++part) {
              uint32_t d[16];
              tc_ld_32x32b_x16h(ta + 16u * part, d);
              wait_ld_into(d);
              if (part == C::kCW / 16 - 1) {
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&acce_bar[buf]);
              }
#pragma unroll
              for (int j = 0; j < 16; j += 2)
                fma_f32x2(acc[16 * part + j], acc[16 * part + j + 1], sa, sa, __uint_as_float(d[j]),
                          __uint_as_float(d[j + 1]));
            }
            continue;
          }
          uint32_t d[C::kCW > 32 ? C::kCW : 32];
          if constexpr (C::kCW == 64) {
            tc_ld_32x32b_x32(ta, *reinterpret_cast<uint32_t(*)[32]>(&d[0]));
            tc_ld_32x32b_x32(ta + 32u,
                             *reinterpret_cast<uint32_t(*)[32]>(&d[32]));
          } else if constexpr (C::kCW == 32) {
            tc_ld_32x32b_x32(ta, *reinterpret_cast<uint32_t(*)[32]>(&d[0]));
          } else {
            tc_ld_32x32b_x16(ta, *reinterpret_cast<uint32_t(*)[32]>(&d[0]));
          }
          tc_wait_ld();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&acce_bar[buf]);
          const float ws = sc[kChunk * BT + (C::kTokMajor ? (col0 >> 7) * kChunk : 0) + i];
          if constexpr (C::kTokMajor) {
            // acc[n] += (As[t,kb] * Ws[kb]) * D[t,n]
            const float sa = sc[i * BT + q * 32 + lane] * ws;
#pragma unroll
            for (int j = 0; j < C::kCW; j += 2)
              fma_f32x2(acc[j], acc[j + 1], sa, sa, __uint_as_float(d[j]), __uint_as_float(d[j + 1]));
            continue;
          }
          const float4 *a4 = reinterpret_cast<const float4 *>(sc + i * BT + col0);
          // acc[t] += As[t,kb] * (Ws[kb] * D[n,t]): the weight scale is applied
          // to the block result in place (no extra registers), then the
          // activation scale in the accumulating FMA.
#pragma unroll
          for (int j4 = 0; j4 < C::kCW / 4; ++j4) {
            const float4 a = a4[j4];
            float d0 = __uint_as_float(d[4 * j4 + 0]), d1 = __uint_as_float(d[4 * j4 + 1]);
            float d2 = __uint_as_float(d[4 * j4 + 2]), d3 = __uint_as_float(d[4 * j4 + 3]);
            mul_f32x2(d0, d1, ws, ws);
            mul_f32x2(d2, d3, ws, ws);
            fma_f32x2(acc[4 * j4 + 0], acc[4 * j4 + 1], a.x, a.y, d0, d1);
            fma_f32x2(acc[4 * j4 + 2], acc[4 * j4 + 3], a.z, a.w, d2, d3);
          }
        }
        asm volatile("cp.async.wait_all;" ::: "memory");
        // Every epilogue thread reaches this barrier once per chunk, whether
        // or not its waits succeeded: the stop decision is the same
        // everywhere, and the next chunk's scales are visible after it.
        if (named_bar_any(1, C::kEpiThreads, !ok)) {
          stop = true;
          break;
        }
        cur ^= 1;
      }
      if (stop) {
        abort_u = u;
        break;
      }
      const int tcol = t0 + col0;
      if constexpr (C::kTokMajor) {
        // Thread = token t0 + 32q + lane, its kCW values = n nt*BN + col0 + j.
        const int t = t0 + q * 32 + lane;
        const int nc = nt * BN + col0;
        if (p.splits == 1 && p.tma_store) {
          // [32 tokens][32 n] in the 64-byte swizzle (row r's 16-byte unit u at
          // u ^ ((r >> 1) & 3): conflict-free rows); the store clips tokens past M.
          // one [32 tokens][32 n] box per 32 columns
          uint8_t *ob = outbuf + ew * (C::kCW * 64);
          if (lane == 0) bulk_wait_read0();   // this warp's previous stores have read the buffer
          __syncwarp();
#pragma unroll
          for (int hh = 0; hh < C::kCW / 32; ++hh)
#pragma unroll
            for (int u4 = 0; u4 < 4; ++u4) {
              const float *a = acc + 32 * hh + 8 * u4;
              uint4 v;
              v.x = pack_bf16x2(a[0], a[1]);
              v.y = pack_bf16x2(a[2], a[3]);
              v.z = pack_bf16x2(a[4], a[5]);
              v.w = pack_bf16x2(a[6], a[7]);
              *reinterpret_cast<uint4 *>(ob + hh * 2048 + lane * 64 + ((u4 ^ ((lane >> 1) & 3)) << 4)) = v;
            }
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
#pragma unroll
            for (int hh = 0; hh < C::kCW / 32; ++hh) tma_store_2d(&tm_c, ob + hh * 2048, nc + 32 * hh, t0 + q * 32);
            bulk_commit();
          }
        } else if (p.splits == 1) {
          if (t < p.M) {
            uint16_t *dst = p.c + static_cast<size_t>(t) * p.ldc + nc;
#pragma unroll
            for (int j = 0; j < C::kCW; ++j) dst[j] = f32_to_bf16_rn(acc[j]);
          }
        } else {
          // partial tile [n / 128][token][128 n], as the reduction reads it.
          // The warp's 32 tokens x kCW columns pass through its output
          // buffer in 16-column pieces ([32][20] floats: conflict-free
          // writes), so each global store covers 8 token rows x 64 bytes;
          // stored straight from the registers, one token row per thread,
          // every store touched 32 sectors and the load/store queue backed up.
          float *pw = p.partials + (static_cast<size_t>(tile) * p.splits + sp) * (BN * BT) +
                      (col0 >> 7) * (128 * BT) + (q * 32) * 128 + (col0 & 127);
          float *ob = reinterpret_cast<float *>(outbuf + ew * (C::kCW * 64));
#pragma unroll
          for (int c16 = 0; c16 < C::kCW / 16; ++c16) {
            __syncwarp();
#pragma unroll
            for (int k = 0; k < 4; ++k)
              *reinterpret_cast<float4 *>(ob + lane * 20 + 4 * k) =
                  make_float4(acc[16 * c16 + 4 * k], acc[16 * c16 + 4 * k + 1], acc[16 * c16 + 4 * k + 2],
                              acc[16 * c16 + 4 * k + 3]);
            __syncwarp();
#pragma unroll
            for (int r8 = 0; r8 < 4; ++r8) {
              const int row = r8 * 8 + (lane >> 2);
              *reinterpret_cast<float4 *>(pw + row * 128 + 16 * c16 + 4 * (lane & 3)) =
                  *reinterpret_cast<const float4 *>(ob + row * 20 + 4 * (lane & 3));
            }
          }
        }
      } else if (C::kTmaOut && p.splits == 1 && p.tma_store) {
        // [token][n] rows of 64 bytes; the store clips tokens past M.
        uint16_t *ob = reinterpret_cast<uint16_t *>(outbuf + ew * (C::kCW * 64));
        if (lane == 0) bulk_wait_read0();   // this warp's previous store has read the buffer
        __syncwarp();
#pragma unroll
        for (int j = 0; j < C::kCW; ++j) ob[j * 32 + lane] = f32_to_bf16_rn(acc[j]);
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          tma_store_2d(&tm_c, ob, nt * BN + q * 32, tcol);
          bulk_commit();
        }
      } else if (p.splits == 1) {
#pragma unroll
        for (int j = 0; j < C::kCW; ++j)
          if (tcol + j < p.M) p.c[static_cast<size_t>(tcol + j) * p.ldc + n] = f32_to_bf16_rn(acc[j]);
      } else {
        float *part = p.partials + (static_cast<size_t>(tile) * p.splits + sp) * (BN * BT);
#pragma unroll
        for (int j = 0; j < C::kCW; ++j) part[(col0 + j) * 128 + q * 32 + lane] = acc[j];
      }
      if (p.splits > 1) {
        // Arrival: the epilogue threads' partial stores reach thread 0
        // through the barrier, and its gpu-scope acq_rel fence before the
        // counter update releases them all (after the update, the same
        // fence acquires the other CTAs' partials for the last arrival,
        // whose threads read them after the next barrier). One fence for
        // the CTA instead of a __threadfence in every thread, before
        // arriving and again before summing (a timeline of M=256, N=6144,
        // K=2048 split 2 ways: stores + arrival 3.1 -> 3.3 us per unit, the
        // sum 2.5 -> 2.3; the launch 26.4 -> 25.9 us).
        named_bar_sync(2, C::kEpiThreads);
        if (e == 0) {
          fence_acq_rel_gpu();
          const int prev = atomicAdd(p.counters + tile, 1);
          fence_acq_rel_gpu();
          // 1: last arrival, sum; 2: last arrival after a poisoned one, no sum
          *is_last = ((prev & kArrivalMask) == p.splits - 1) ? ((prev >> kPoisonShift) ? 2 : 1) : 0;
        }
        named_bar_sync(2, C::kEpiThreads);
        if (*is_last == 1) {
          const float *base = p.partials + static_cast<size_t>(tile) * p.splits * (BN * BT);
#pragma unroll 1
          for (int h = 0; h < C::kNB; ++h) {
            if constexpr (C::kRedCall)
              reduce_block_call(base + h * (128 * BT), static_cast<size_t>(BN) * BT, p.splits, min(BT, p.M - t0),
                                nt * BN + h * 128, t0, p.c, p.ldc, p.c_vec4, e, C::kEpiThreads);
            else
              reduce_block(base + h * (128 * BT), static_cast<size_t>(BN) * BT, p.splits, min(BT, p.M - t0),
                           nt * BN + h * 128, t0, p.c, p.ldc, p.c_vec4, e, C::kEpiThreads);
          }
        }
        if (*is_last && e == 0) p.counters[tile] = 0;
        named_bar_sync(2, C::kEpiThreads);
      }
    }
    if (C::kTmaOut && lane == 0) bulk_wait_all();   // output stores complete before the CTA's smem goes away
    // An expired wait stopped this CTA: it still arrives, poisoned, at the
    // counter of every split-K tile it owed, so every counter ends at zero.
    if (abort_u >= 0 && p.splits > 1 && e == 0) {
      for (int u2 = abort_u; u2 < p.units; u2 += gridDim.x) {
        const int tile2 = u2 / p.splits;
        const int prev = atomicAdd(p.counters + tile2, 1 + kPoisonArrival);
        if ((prev & kArrivalMask) == p.splits - 1) atomicExch(p.counters + tile2, 0);
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == C::kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
}

template <int BT, int BN>
int launch_bt(const uint8_t *q, const float *As, const uint8_t *packed, int64_t M, int64_t N, int64_t K,
              uint16_t *c, int64_t ldc, void *ws, const GemmPlan &pl, cudaStream_t st) {
  using C = Cfg<BT, BN>;
  if (N % BN != 0) return R4_ERR_UNSUPPORTED_SHAPE;
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
  // Output through TMA tensor stores when C's base, row stride and row
  // length are 16-byte multiples (N is a multiple of 128 here).
  CUtensorMap tm_c;
  int use_tma_store = 0;
  if (C::kTmaOut && pl.splits == 1 && (reinterpret_cast<uintptr_t>(c) % 16) == 0 && (ldc * 2) % 16 == 0 &&
      (N * 2) % 16 == 0) {
    const uint64_t dims[2] = {static_cast<uint64_t>(N), static_cast<uint64_t>(M)};
    const uint64_t strides[1] = {static_cast<uint64_t>(ldc) * 2};
    const uint32_t box[2] = {32, 32};
    use_tma_store = encode_tiled(&tm_c, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, c, dims, strides, box,
                                 C::kTokMajor ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_NONE) == CUDA_SUCCESS;
  }
  if (!use_tma_store) tm_c = tm_x;   // not read by the kernel in that case
  Params p;
  p.M = static_cast<int>(M);
  p.KB = pl.KB;
  p.tma_store = use_tma_store;
  p.inject_stall = options().inject_stall;
  p.early_w = options().early_weights;
  p.c_vec4 = (reinterpret_cast<uintptr_t>(c) % 8) == 0 && ldc % 4 == 0;
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
  auto kern = blockfp8_f8f6f4_kernel<BT, BN>;
  if (ensure_smem_attr(reinterpret_cast<const void *>(kern), C::kSmemBytes) != cudaSuccess) return R4_ERR_CUDA;
  if (launch_pdl(kern, dim3(pl.grid), dim3(C::kThreads), C::kSmemBytes, st, tm_w, tm_x, tm_c, p) != cudaSuccess)
    return R4_ERR_CUDA;
  set_last_kernel(BT == 16   ? "blockfp8_f8f6f4_kernel<16>"
                  : BT == 32 ? "blockfp8_f8f6f4_kernel<32>"
                  : BT == 64 ? "blockfp8_f8f6f4_kernel<64>"
                  : BN == 256 ? "blockfp8_f8f6f4_kernel<128, 256>"
                             : "blockfp8_f8f6f4_kernel<128>");
  return cudaGetLastError() == cudaSuccess ? R4_OK : R4_ERR_CUDA;
}

}  // namespace fp8

// Token tile and split-K choice: the wave model of plan_w4a8 with the
// block-FP8 per-K-block bytes (16 KiB of e4m3 weights).
GemmPlan plan_blockfp8(int64_t M, int64_t N, int64_t K, int sms) {
  GemmPlan pl;
  int bt = options().fp8_token_tile;
  // 33..64 tokens run as two 32-token tiles: twice the weight reads from L2,
  // but half the promotion work per CTA (measured: M=64, 6144x2048 9.95 vs
  // 10.96 us; 4096x4096 14.0 vs 15.5 us).
  if (bt == 0) bt = M <= 16 ? 16 : M <= 64 ? 32 : 128;
  pl.BT = bt;
  // Token-major tiles take 256 weight rows when N allows and the 256-row
  // tiles still occupy half of the SMs: each per-K-block handshake
  // (accumulator ready, promoted, released) then covers twice the tensor
  // work. (Measured on GB300, 128 -> 256 rows: M=2048 6144x2048 44.9 ->
  // 33.6 us, 2048x6144 41.5 -> 30.3, 4096x4096 56.0 -> 40.8; at M=256,
  // 48 or fewer tiles, 9.6 -> 12.5 us.)
  int bn = options().fp8_n_tile;
  if (bn == 0) bn = (N / 256) * ceil_div(M, 128) * 2 >= sms ? 256 : 128;
  if (bt != 128 || N % 256 != 0) bn = 128;
  pl.BN = bn;
  pl.n_tiles = static_cast<int>(N / bn);
  pl.t_tiles = static_cast<int>(ceil_div(M, bt));
  pl.KB = static_cast<int>(K / 128);
  const int64_t tiles = static_cast<int64_t>(pl.n_tiles) * pl.t_tiles;
  const double hbm = 6.0e12, sm_bw = 70e9, sm_flops = 4.5e15 / 152.0, red_bw = 20e9;
  const double kb_bytes = 128.0 * bn + 128.0 * bt;
  const double kb_flops = 2.0 * bn * bt * 128;
  const double part_bytes = static_cast<double>(bn) * bt * 4;
  const int max_s = (bt >= 128 && tiles * 4 >= sms && !options().fp8_splits) ? 1 : std::min(pl.KB, 64);
  int best_s = 1;
  double best_t = 1e30;
  for (int s = 1; s <= max_s; ++s) {
    const int kbps = static_cast<int>(ceil_div(pl.KB, s));
    if (static_cast<int64_t>(s - 1) * kbps >= pl.KB) continue;   // would leave an empty split
    const int64_t units = tiles * s;
    const int64_t active = std::min<int64_t>(units, sms);
    const double waves = std::ceil(static_cast<double>(units) / sms);
    const double t_unit = std::max(kbps * kb_bytes / std::min(hbm / active, sm_bw), kbps * kb_flops / sm_flops);
    double t = waves * t_unit;
    if (s > 1) t += (waves + s) * part_bytes / red_bw;
    if (t < best_t) {
      best_t = t;
      best_s = s;
    }
  }
  // Decode tiles: as many splits as keep every unit in one wave. Measured
  // on GB300 against the wave model above (cold weights, M = 8 / 64):
  // 4096x4096 9.73 -> 9.06 / 15.89 -> 13.92 us, 2048x6144 9.03 -> 8.99 /
  // 15.71 -> 14.49 us, 6144x2048 8.13 -> 8.22 / 9.98 -> 9.97 us.
  if (bt <= 64) {
    best_s = static_cast<int>(std::max<int64_t>(1, std::min<int64_t>(sms / tiles, std::min(pl.KB, 64))));
  }
  const int forced = options().fp8_splits;
  if (forced && forced <= pl.KB) best_s = forced;
  if (tiles > kMaxCounterTiles) best_s = 1;   // the counter region holds at most this many tiles
  pl.kb_per_split = static_cast<int>(ceil_div(pl.KB, best_s));
  pl.splits = static_cast<int>(ceil_div(pl.KB, pl.kb_per_split));
  pl.units = static_cast<int>(tiles * pl.splits);
  pl.grid = std::min(pl.units, sms);
  if (pl.splits > 1) {
    pl.counters_bytes = kCounterBytes;
    pl.ws_bytes = pl.counters_bytes + static_cast<size_t>(pl.units) * bn * bt * 4;
  }
  return pl;
}

int launch_gemm_blockfp8(const uint8_t *q, const float *As, const uint8_t *packed, int64_t M, int64_t N,
                         int64_t K, uint16_t *c, int64_t ldc, void *ws, const GemmPlan &pl, cudaStream_t st) {
  switch (pl.BT) {
    case 16: return fp8::launch_bt<16, 128>(q, As, packed, M, N, K, c, ldc, ws, pl, st);
    case 32: return fp8::launch_bt<32, 128>(q, As, packed, M, N, K, c, ldc, ws, pl, st);
    case 64: return fp8::launch_bt<64, 128>(q, As, packed, M, N, K, c, ldc, ws, pl, st);
    case 128:
      return pl.BN == 256 ? fp8::launch_bt<128, 256>(q, As, packed, M, N, K, c, ldc, ws, pl, st)
                          : fp8::launch_bt<128, 128>(q, As, packed, M, N, K, c, ldc, ws, pl, st);
    default: return R4_ERR_INVALID_ARG;
  }
}

}  // namespace r4
