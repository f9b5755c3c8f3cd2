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
//  * every 128-K block is its own "slot": 4 MMAs (K = 32 each) write a FRESH
//    fp32 accumulator in tensor memory. Slot g uses accumulator buffer
//    g % kNumBuf; with 512 columns there are 4 (BT = 128) to 16 buffers, so
//    the MMAs run several K blocks ahead of the promotion epilogue;
//  * a scale warp turns As[t0.., kb] and Ws[nt, kb] into the per-token
//    products As * Ws of each K block and publishes them in a ring of shared
//    memory slots. With K/128 a multiple of 4 the scales arrive with the
//    pipeline stage (a TMA box of As and a 16-byte copy of Ws); otherwise the
//    warp loads As in coalesced row chunks, one chunk ahead in registers;
//  * 4 x kH epilogue warps (one per tensor-memory lane quarter and column
//    group of 32 tokens) load the block result and fold it into fp32
//    registers: acc[t] += (As[t,kb] * Ws[nt,kb]) * D_kb[n,t], two columns per
//    packed f32x2 FMA;
//  * decode tiles (BT <= 64) run two TMA producer warps: one thread issuing
//    every weight and activation copy caps the weight stream (each TMA issue
//    holds its thread for a few hundred cycles on GB300).
// Split-K and the last-arriving-CTA reduction are as in the W4A8 kernel.

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
constexpr int kMaxRing = 16;        // published scale slots (products As * Ws for one K block)
// K blocks of As staged per coalesced load (the scale warp holds one chunk
// in registers: BT * chunk / 32 values per lane).
constexpr int chunk_of(int bt) { return bt >= 128 ? 8 : 16; }

struct Params {
  int M, KB;           // KB = K / 128 (blocks per row of As / Ws)
  int t_tiles, splits, kb_per_split, units;
  int ldc;
  int as_tma;          // 1: As and Ws travel with each pipeline stage (TMA), needs KB % 4 == 0
  int inject_stall;    // test of the bounded waits: CTA 0 withholds its first activation copy
  int early_w;         // 1: weight tiles are requested before waiting for the preceding kernel
  const float *As;     // [M, KB]
  const float *Ws;     // [N/128, KB]
  uint16_t *c;
  float *partials;
  int *counters;
  int *err;
};

template <int BT>
struct Cfg {
  static constexpr int kProd = BT <= 64 ? 2 : 1;           // TMA producer warps
  static constexpr int kMmaWarp = kProd;
  static constexpr int kScaleWarp = kProd + 1;
  static constexpr int kEpiWarp0 = kProd + 2;
  static constexpr int kCW = BT < 32 ? BT : 32;            // token columns per epilogue warp
  static constexpr int kH = BT / kCW;                      // column groups
  static constexpr int kEpiWarps = 4 * kH;
  static constexpr int kEpiThreads = 32 * kEpiWarps;
  static constexpr int kThreads = 32 * (kEpiWarp0 + kEpiWarps);
  static constexpr int kNumBufRaw = 512 / BT;
  static constexpr int kNumBuf = kNumBufRaw > kMaxBuf ? kMaxBuf : kNumBufRaw;
  static constexpr uint32_t kTmemCols = static_cast<uint32_t>(kNumBuf * BT);
  static constexpr uint32_t kXSmem = BT * 128;
  // With KB % 4 == 0 each stage also carries As[t0.., kb & ~3 .. +4) as a
  // [BT][4] fp32 TMA box and Ws[nt, kb & ~3 .. +4) (16 bytes).
  static constexpr uint32_t kAsSmem = BT * 16;
  static constexpr uint32_t kAsTx = kAsSmem + 16;
  static constexpr uint32_t kStageBytes = ((kWSmem + kXSmem + kAsTx + 1023) / 1024) * 1024;
  static constexpr int kRing = BT >= 128 ? 8 : kMaxRing;
  static constexpr uint32_t kSlotFloats = BT + 4;          // BT products, then Ws (16-byte pitch)
  static constexpr uint32_t kRingBytes = kRing * kSlotFloats * 4;
  // As staging: 2 buffers of [BT rows][kChunk + 1] (+1: conflict-free column
  // reads) and the chunk's Ws values.
  static constexpr int kChunk = chunk_of(BT);
  static constexpr uint32_t kStageRow = kChunk + 1;
  static constexpr uint32_t kAsBufFloats = ((BT * kStageRow + kChunk + 3) / 4) * 4;
  static constexpr uint32_t kAsBytes = 2 * kAsBufFloats * 4;
  static constexpr uint32_t kMiscBytes = 1024;             // barriers and flags
  static constexpr int kStagesRaw =
      static_cast<int>((227u * 1024u - 1024u - kMiscBytes - kRingBytes - kAsBytes) / kStageBytes);
  static constexpr int kStagesCap = kStagesRaw > kMaxStages ? kMaxStages : kStagesRaw;
  static constexpr int kStages = (kStagesCap / kProd) * kProd;   // each producer owns fixed stages
  static constexpr uint32_t kTxBytes = kWSmem + kXSmem;
  static constexpr uint32_t kSmemBytes = kStages * kStageBytes + kRingBytes + kAsBytes + kMiscBytes + 1024;
  static_assert(kTmemCols >= 32 && (kTmemCols & (kTmemCols - 1)) == 0, "tensor-memory allocation");
  static_assert(kThreads <= 1024, "block size");
  static_assert(kStages >= kProd, "stage count");
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

// Walks this CTA's units in chunks of up to CH consecutive K blocks.
template <int CH>
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
  __device__ __forceinline__ int len() const { return min(CH, kb1 - kb); }
  __device__ __forceinline__ void next(const Params &p) {
    kb += CH;
    if (kb >= kb1) {
      u += gridDim.x;
      if (u < p.units) decode(p);
    }
  }
};

// One chunk of scales in registers: As[t0 + c, kb .. kb + n) for the tile's
// BT rows (0 past M) and Ws[nt, kb .. kb + n). Element e = lane + 32 i walks
// the [BT][n] block row-major, so a warp's load covers whole row segments.
template <int BT>
struct AsChunk {
  static constexpr int kChunk = chunk_of(BT);
  static constexpr int kPer = BT * kChunk / 32;   // elements per lane
  float v[kPer];
  float w;
  __device__ __forceinline__ void load(const Params &p, const ChunkCursor<kChunk> &ch, int lane) {
    const int n = ch.len();
    const int t0 = ch.tt * BT;
#pragma unroll
    for (int i = 0; i < kPer; ++i) {
      const int idx = lane + 32 * i;
      const int c = idx / n, j = idx - c * n;
      const int t = t0 + c;
      v[i] = (c < BT && t < p.M) ? __ldg(p.As + static_cast<size_t>(t) * p.KB + ch.kb + j) : 0.f;
    }
    w = lane < n ? __ldg(p.Ws + static_cast<size_t>(ch.nt) * p.KB + ch.kb + lane) : 0.f;
  }
  // Into buf[c * (kChunk + 1) + j], Ws after the BT rows.
  __device__ __forceinline__ void store(const ChunkCursor<kChunk> &ch, float *buf, int lane) const {
    const int n = ch.len();
#pragma unroll
    for (int i = 0; i < kPer; ++i) {
      const int idx = lane + 32 * i;
      const int c = idx / n, j = idx - c * n;
      if (c < BT) buf[c * (kChunk + 1) + j] = v[i];
    }
    if (lane < n) buf[BT * (kChunk + 1) + lane] = w;
  }
};

template <int BT>
__global__ void __launch_bounds__(Cfg<BT>::kThreads, 1)
    blockfp8_f8f6f4_kernel(const __grid_constant__ CUtensorMap tm_w, const __grid_constant__ CUtensorMap tm_x,
                           const __grid_constant__ CUtensorMap tm_as, const Params p) {
  using C = Cfg<BT>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  float *ring = reinterpret_cast<float *>(smem + C::kStages * C::kStageBytes);   // [kRing][kSlotFloats]
  float *as_stage = ring + C::kRing * C::kSlotFloats;                            // [2][kAsBufFloats]
  uint8_t *misc = reinterpret_cast<uint8_t *>(as_stage) + C::kAsBytes;
  uint64_t *full_bar = reinterpret_cast<uint64_t *>(misc);   // [kMaxStages]
  uint64_t *empty_bar = full_bar + kMaxStages;               // [kMaxStages]
  uint64_t *accf_bar = empty_bar + kMaxStages;               // [kMaxBuf]
  uint64_t *acce_bar = accf_bar + kMaxBuf;                   // [kMaxBuf]
  uint64_t *sready_bar = acce_bar + kMaxBuf;                 // [kRing] products published
  uint64_t *sempty_bar = sready_bar + kMaxRing;              // [kRing] read by every epilogue warp
  uint64_t *drain_bar = sempty_bar + kMaxRing;
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(drain_bar + 1);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
  volatile int *is_last = abort_flag + 1;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(&full_bar[s], 1);
      mbar_init(&empty_bar[s], p.as_tma ? 2 : 1);   // MMA commit (+ scale warp when As rides along)
    }
    for (int b = 0; b < C::kNumBuf; ++b) {
      mbar_init(&accf_bar[b], 1);
      mbar_init(&acce_bar[b], C::kEpiWarps);
    }
    for (int r = 0; r < C::kRing; ++r) {
      mbar_init(&sready_bar[r], 1);
      mbar_init(&sempty_bar[r], C::kEpiWarps);
    }
    mbar_init(drain_bar, 1);
    *abort_flag = 0;
    *is_last = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tm_w);
    tma_prefetch_desc(&tm_x);
    if (p.as_tma) tma_prefetch_desc(&tm_as);
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
      bool ok = true;
      const uint32_t tx = C::kTxBytes + (p.as_tma ? C::kAsTx : 0u);
      // Weights first (independent of the preceding kernel), then wait for
      // it before the first activation tile.
      if (!p.early_w) pdl_wait();
      {
        SlotCursor cu;
        cu.start(p);
        for (int g = 0; cu.valid(p) && g < C::kStages; ++g, cu.next(p))
          if (g % C::kProd == pw) {
            mbar_arrive_expect_tx(&full_bar[g], tx);
            tma_load_3d(smem + g * C::kStageBytes, &tm_w, &full_bar[g], 0, 0, cu.nt * p.KB + cu.kb, pol_w);
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
          if (!mbar_wait(&empty_bar[stage], phase ^ 1u, abort_flag, p.err, DEV_ERR_WAIT_EMPTY)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&full_bar[stage], tx);
          tma_load_3d(st, &tm_w, &full_bar[stage], 0, 0, cu.nt * p.KB + cu.kb, pol_w);
        }
        // (Failure-detection test: with inject_stall, CTA 0 never issues its
        // first activation copy, so the stage's transaction never completes.)
        if (!(p.inject_stall && blockIdx.x == 0 && g == 0))
          tma_load_2d(st + kWSmem, &tm_x, &full_bar[stage], cu.kb * 128, cu.tt * BT, pol_x);
        if (p.as_tma) {
          const int kb4 = cu.kb & ~3;
          tma_load_2d(st + kWSmem + C::kXSmem, &tm_as, &full_bar[stage], kb4, cu.tt * BT, pol_x);
          bulk_load(st + kWSmem + C::kXSmem + C::kAsSmem, p.Ws + static_cast<size_t>(cu.nt) * p.KB + kb4, 16,
                    &full_bar[stage], pol_w);
        }
        // Record the newest phase of every stage: a parity wait cannot tell
        // phase k from k + 2, and a stage only advances once its earlier
        // phases completed.
        issued_mask |= 1u << stage;
        issued_phase = (issued_phase & ~(1u << stage)) | (phase << stage);
      }
      (void)ok;
      // Never leave a copy in flight: wait (bounded, even after an abort)
      // for the last load issued into each of this producer's stages.
      for (int s_ = 0; s_ < C::kStages; ++s_)
        if (issued_mask & (1u << s_)) {
          volatile int dummy = 0;
          mbar_wait(&full_bar[s_], (issued_phase >> s_) & 1u, &dummy, p.err, DEV_ERR_WAIT_DRAIN);
        }
    }
    __syncwarp();
  } else if (warp == C::kMmaWarp) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t idesc = idesc_f8f6f4_e4m3(BT);
      SlotCursor cu;
      cu.start(p);
      for (int g = 0; cu.valid(p); ++g, cu.next(p)) {
        const int stage = g % C::kStages;
        const uint32_t phase = static_cast<uint32_t>(g / C::kStages) & 1u;
        const int buf = g % C::kNumBuf;
        const uint32_t bphase = static_cast<uint32_t>(g / C::kNumBuf) & 1u;
        if (!mbar_wait(&acce_bar[buf], bphase ^ 1u, abort_flag, p.err, DEV_ERR_WAIT_ACC_EMPTY)) break;
        if (!mbar_wait(&full_bar[stage], phase, abort_flag, p.err, DEV_ERR_WAIT_FULL)) break;
        tc_fence_after();
        uint8_t *st = smem + stage * C::kStageBytes;
        const uint32_t a_base = smem_u32(st), b_base = smem_u32(st + kWSmem);
        const uint32_t d_tmem = tmem + static_cast<uint32_t>(buf * BT);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          tc_mma_f8f6f4(d_tmem, sdesc_sw128_kmajor(a_base + 32u * kk), sdesc_sw128_kmajor(b_base + 32u * kk), idesc,
                        kk > 0 ? 1u : 0u);
        tc_commit(&empty_bar[stage]);
        tc_commit(&accf_bar[buf]);
      }
      // All MMAs this thread issued must be complete before tensor memory is freed.
      tc_commit(drain_bar);
      volatile int dummy = 0;
      mbar_wait(drain_bar, 0, &dummy, p.err, DEV_ERR_WAIT_DRAIN);
    }
    __syncwarp();
  } else if (warp == C::kScaleWarp) {
    // ------------------------------------------------------------ scale warp
    // Ring slot r = g % kRing holds the products As[t, kb] * Ws[nt, kb] of K
    // block g: empty -> written -> ready -> read by every epilogue warp ->
    // empty. With KB % 4 == 0 the scales arrive with the pipeline stage (the
    // warp is a second consumer of its full barrier and a second arrival on
    // its empty barrier); otherwise they are loaded in coalesced chunks.
    if (p.as_tma) {
      SlotCursor cu;
      cu.start(p);
      for (int g = 0; cu.valid(p); ++g, cu.next(p)) {
        const int stage = g % C::kStages;
        const uint32_t phase = static_cast<uint32_t>(g / C::kStages) & 1u;
        const int r = g % C::kRing;
        const uint32_t ph = static_cast<uint32_t>(g / C::kRing) & 1u;
        if (!warp_wait(&sempty_bar[r], ph ^ 1u, abort_flag, p.err, DEV_ERR_WAIT_EMPTY)) break;
        if (!warp_wait(&full_bar[stage], phase, abort_flag, p.err, DEV_ERR_WAIT_FULL)) break;
        const float *as_s = reinterpret_cast<const float *>(smem + stage * C::kStageBytes + kWSmem + C::kXSmem);
        const int j = cu.kb & 3;
        const float ws = as_s[BT * 4 + j];
        float *slot = ring + r * C::kSlotFloats;
        for (int c = lane; c < BT; c += 32) slot[c] = as_s[c * 4 + j] * ws;
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(&sready_bar[r]);
          mbar_arrive(&empty_bar[stage]);
        }
      }
    } else {
    pdl_wait();   // As comes from the preceding kernel
    ChunkCursor<C::kChunk> cl, cn;   // chunk being published, chunk being loaded
    cl.start(p);
    cn.start(p);
    AsChunk<BT> regs;
    if (cn.valid(p)) {
      regs.load(p, cn, lane);
      regs.store(cn, as_stage, lane);
      cn.next(p);
    }
    __syncwarp();
    bool ok = true;
    int g = 0;
    for (int ci = 0; cl.valid(p) && ok; ++ci, cl.next(p)) {
      const bool more = cn.valid(p);
      if (more) regs.load(p, cn, lane);   // in flight during the publishing below
      const float *buf = as_stage + (ci & 1) * C::kAsBufFloats;
      const int n = cl.len();
      for (int j = 0; j < n; ++j, ++g) {
        const int r = g % C::kRing;
        const uint32_t ph = static_cast<uint32_t>(g / C::kRing) & 1u;
        if (!warp_wait(&sempty_bar[r], ph ^ 1u, abort_flag, p.err, DEV_ERR_WAIT_EMPTY)) {
          ok = false;
          break;
        }
        float *slot = ring + r * C::kSlotFloats;
        const float ws = buf[BT * C::kStageRow + j];
        for (int c = lane; c < BT; c += 32) slot[c] = buf[c * C::kStageRow + j] * ws;
        __syncwarp();
        if (lane == 0) mbar_arrive(&sready_bar[r]);
      }
      if (more) {
        regs.store(cn, as_stage + ((ci + 1) & 1) * C::kAsBufFloats, lane);
        cn.next(p);
      }
      __syncwarp();
    }
    }
  } else {
    // ------------------------------------------------------------ promotion epilogue
    pdl_wait();                        // C and the workspace follow the stream order
    const int ew = warp - C::kEpiWarp0;
    const int e = ew * 32 + lane;      // 0 .. kEpiThreads-1
    const int q = warp & 3;            // tensor-memory lane quarter this warp may access
    const int h = ew >> 2;             // column group
    const int col0 = h * C::kCW;
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(q * 32) << 16) + static_cast<uint32_t>(col0);
    SlotCursor cu;
    cu.start(p);
    int g = 0;
    int abort_u = -1;                  // unit at which an expired wait stopped the epilogue
    while (cu.valid(p)) {
      const int nt = cu.nt, tt = cu.tt, sp = cu.sp, u = cu.u;
      const int t0 = tt * BT;
      const int n = nt * 128 + q * 32 + lane;
      const int tile = nt * p.t_tiles + tt;
      float acc[C::kCW];
#pragma unroll
      for (int j = 0; j < C::kCW; ++j) acc[j] = 0.f;
      bool ok = true;
      for (; cu.valid(p) && cu.u == u; ++g, cu.next(p)) {
        const int buf = g % C::kNumBuf;
        const uint32_t bphase = static_cast<uint32_t>(g / C::kNumBuf) & 1u;
        const int r = g % C::kRing;
        const uint32_t rphase = static_cast<uint32_t>(g / C::kRing) & 1u;
        // Warp-uniform waits (tcgen05.ld needs the whole warp).
        if (!warp_wait(&accf_bar[buf], bphase, abort_flag, p.err, DEV_ERR_WAIT_ACC_FULL)) {
          ok = false;
          break;
        }
        tc_fence_after();
        uint32_t d[32];
        if constexpr (C::kCW == 32) {
          tc_ld_32x32b_x32(lane_base + static_cast<uint32_t>(buf * BT), d);
        } else {
          tc_ld_32x32b_x16(lane_base + static_cast<uint32_t>(buf * BT), d);
        }
        tc_wait_ld();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&acce_bar[buf]);
        if (!warp_wait(&sready_bar[r], rphase, abort_flag, p.err, DEV_ERR_WAIT_FULL)) {
          ok = false;
          break;
        }
        const float4 *s4 = reinterpret_cast<const float4 *>(ring + r * C::kSlotFloats + col0);
#pragma unroll
        for (int j4 = 0; j4 < C::kCW / 4; ++j4) {
          const float4 f = s4[j4];
          fma_f32x2(acc[4 * j4 + 0], acc[4 * j4 + 1], f.x, f.y, __uint_as_float(d[4 * j4 + 0]),
                    __uint_as_float(d[4 * j4 + 1]));
          fma_f32x2(acc[4 * j4 + 2], acc[4 * j4 + 3], f.z, f.w, __uint_as_float(d[4 * j4 + 2]),
                    __uint_as_float(d[4 * j4 + 3]));
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&sempty_bar[r]);
      }
      // Every epilogue thread reaches this barrier once per unit, whether or
      // not its waits succeeded, so the stop decision is the same everywhere.
      if (named_bar_any(1, C::kEpiThreads, !ok)) {
        abort_u = u;
        break;
      }
      const int tcol = t0 + col0;
      if (p.splits == 1) {
#pragma unroll
        for (int j = 0; j < C::kCW; ++j)
          if (tcol + j < p.M) p.c[static_cast<size_t>(tcol + j) * p.ldc + n] = f32_to_bf16_rn(acc[j]);
      } else {
        float *part = p.partials + (static_cast<size_t>(tile) * p.splits + sp) * (128 * BT);
#pragma unroll
        for (int j = 0; j < C::kCW; ++j) part[(col0 + j) * 128 + q * 32 + lane] = acc[j];
        __threadfence();
        named_bar_sync(2, C::kEpiThreads);
        if (e == 0) {
          const int prev = atomicAdd(p.counters + tile, 1);
          // 1: last arrival, sum; 2: last arrival after a poisoned one, no sum
          *is_last = ((prev & kArrivalMask) == p.splits - 1) ? ((prev >> kPoisonShift) ? 2 : 1) : 0;
        }
        named_bar_sync(2, C::kEpiThreads);
        if (*is_last == 1) {
          __threadfence();
          const float *base = p.partials + static_cast<size_t>(tile) * p.splits * (128 * BT);
          reduce_partials_store<BT>(base, p.splits, min(BT, p.M - t0), nt * 128, nt * 128 + 128, nullptr, t0, p.c,
                                    p.ldc, e, C::kEpiThreads);
        }
        if (*is_last && e == 0) p.counters[tile] = 0;
        named_bar_sync(2, C::kEpiThreads);
      }
    }
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

template <int BT>
int launch_bt(const uint8_t *q, const float *As, const uint8_t *packed, int64_t M, int64_t N, int64_t K,
              uint16_t *c, int64_t ldc, void *ws, const GemmPlan &pl, cudaStream_t st) {
  using C = Cfg<BT>;
  CUtensorMap tm_w, tm_x, tm_as;
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
  // The activation scales ride along with each stage when their rows are
  // 16-byte multiples (TMA) and the pointers are 16-byte aligned.
  const float *Ws = reinterpret_cast<const float *>(packed + fp8_packed_codes_bytes(N, K));
  int as_tma = 0;
  if (options().fp8_stage_scales && pl.KB % 4 == 0 && reinterpret_cast<uintptr_t>(Ws) % 16 == 0) {
    const uint64_t dims[2] = {static_cast<uint64_t>(pl.KB), static_cast<uint64_t>(M)};
    const uint64_t strides[1] = {static_cast<uint64_t>(pl.KB) * 4};
    const uint32_t box[2] = {4, static_cast<uint32_t>(BT)};
    as_tma = encode_tiled(&tm_as, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float *>(As), dims, strides, box,
                          CU_TENSOR_MAP_SWIZZLE_NONE) == CUDA_SUCCESS;
  }
  if (!as_tma) tm_as = tm_x;   // not read by the kernel in that case
  Params p;
  p.M = static_cast<int>(M);
  p.KB = pl.KB;
  p.as_tma = as_tma;
  p.inject_stall = options().inject_stall;
  p.early_w = options().early_weights;
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
  if (launch_pdl(kern, dim3(pl.grid), dim3(C::kThreads), C::kSmemBytes, st, tm_w, tm_x, tm_as, p) != cudaSuccess)
    return R4_ERR_CUDA;
  set_last_kernel(BT == 16   ? "blockfp8_f8f6f4_kernel<16>"
                  : BT == 32 ? "blockfp8_f8f6f4_kernel<32>"
                  : BT == 64 ? "blockfp8_f8f6f4_kernel<64>"
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
  pl.n_tiles = static_cast<int>(N / 128);
  pl.t_tiles = static_cast<int>(ceil_div(M, bt));
  pl.KB = static_cast<int>(K / 128);
  const int64_t tiles = static_cast<int64_t>(pl.n_tiles) * pl.t_tiles;
  const double hbm = 6.0e12, sm_bw = 70e9, sm_flops = 4.5e15 / 152.0, red_bw = 20e9;
  const double kb_bytes = 128.0 * 128 + 128.0 * bt;
  const double kb_flops = 2.0 * 128 * bt * 128;
  const double part_bytes = 128.0 * bt * 4;
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
    case 16: return fp8::launch_bt<16>(q, As, packed, M, N, K, c, ldc, ws, pl, st);
    case 32: return fp8::launch_bt<32>(q, As, packed, M, N, K, c, ldc, ws, pl, st);
    case 64: return fp8::launch_bt<64>(q, As, packed, M, N, K, c, ldc, ws, pl, st);
    case 128: return fp8::launch_bt<128>(q, As, packed, M, N, K, c, ldc, ws, pl, st);
    default: return R4_ERR_INVALID_ARG;
  }
}

}  // namespace r4
