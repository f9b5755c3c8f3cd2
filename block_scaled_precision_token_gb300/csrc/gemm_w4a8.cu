// gemm_w4a8.cu -- W4A8 MXFP4 linear on tcgen05 block-scaled MMA.
//
//   C[m, n] = bf16( s[m] * sum_k e4m3(q[m,k]) * e2m1(w[n,k]) * 2^(e[n,k/32]-127) )
//
// ("radiance_mxfp4.py": module docstring -- fp8 activations against e2m1
// weights with a ue8m0 scale per 32 K -- and _exact_ref.)
//
// Design (GB300, sm_103a):
//  * Weight-stationary orientation ("swap AB"): the MMA's 128-row A operand is
//    128 weight rows, its N operand is a tile of BT tokens (16..256). One
//    kernel serves decode (M <= 64: BT = 16/32/64, the weight stream is the
//    whole cost) and prefill (BT = 128/256, tensor-bound).
//  * kind::mxf8f6f4 with .scale_vec::1X: A = e2m1 (weights) with its ue8m0
//    scale per 32 K, B = e4m3 (activations) with a constant scale 127 (x1).
//    The hardware applies the MX block scale exactly; the per-token fp32
//    scale s[m] is applied in the epilogue.
//  * TMA: the prepacked 8 KiB weight tile is loaded with the 16U4_ALIGN16B
//    data type, which expands 16 packed nibbles to the 16-byte smem slot the
//    MMA reads for 4-bit operands (HBM traffic stays 0.5 B per weight); the
//    activation tile is a 2-D e4m3 box; both in the 128-byte swizzle. The
//    512-byte scale atom of the tile is a plain bulk copy, then tcgen05.cp
//    places it in tensor memory (one 4-column slot per pipeline stage).
//  * Roles: TMA producer warps (1 for prefill tiles, 4 for decode tiles),
//    MMA-issuing warps (as many; one thread each, each with its own
//    tensor-memory accumulator -- see Cfg for why decode needs several), and
//    4 epilogue warps that sum the accumulators (tcgen05.ld), scale by s[m],
//    round to bf16 and stage [32 tokens x 128 n] chunks in smem that leave
//    through TMA tensor stores (ragged token edges clipped by the hardware;
//    plain stores when C's base, row stride or row length is not a 16-byte
//    multiple). A multi-stage smem
//    ring decouples TMA from MMA; double-buffered accumulators let the
//    epilogue of one unit overlap the MMAs of the next.
//  * Split-K when the output has too few tiles to fill 152 SMs, two ways:
//    - decode tiles of 32/64 tokens: the splits of a tile are the CTAs of one
//      thread-block cluster; each writes its fp32 partial [32 tokens][128 n]
//      into its own shared memory, and every CTA then sums its 1/splits share
//      of the n range over all the cluster's partials (distributed shared
//      memory, rank order: deterministic) and stores it. mbarrier arrivals
//      across the cluster sequence the exchange, with bounded waits;
//    - otherwise fp32 partials go to the caller's workspace and the last CTA
//      to arrive at a tile (one atomic counter per tile) sums them in split
//      order -- deterministic -- and resets the counter.
//  * Every mbarrier wait is bounded (see r4_device.cuh).

#include <cuda_bf16.h>

#include <algorithm>
#include <cmath>

#include "r4_device.cuh"
#include "r4_internal.h"

namespace r4 {
namespace w4a8 {

constexpr int kBK = 128;
constexpr uint32_t kWSmem = 128 * 128;  // expanded e2m1 tile: 128 rows x 128 one-byte slots
// The 16U4_ALIGN16B tile load completes the mbarrier transaction with the
// bytes it READS (8 KiB of packed nibbles), not the 16 KiB it writes to
// shared memory (measured on GB300: a 16 KiB expectation never completes).
constexpr uint32_t kWTxBytes = 8192;
constexpr uint32_t kSfBytes = 512;
constexpr uint32_t kTmemCols = 512;
// Tensor-memory columns: the accumulators first (kIss x kNumAcc x BT
// columns), then the scale columns from kSfaCol on -- 256, or 384 behind the
// two 192-column accumulators of the W4A8 192-token tile:
//   kSfaCol + 4 x stage          weight scales, 4 columns per stage (up to 16 stages)
//   kSfaCol + 64 + 16 x warp     W4A8: 16 columns of constant 127 per MMA warp (up to 4)
//   kSfaCol + 64 + 8 x stage     W4A4: activation scales, 8 columns per stage (up to 16)
constexpr int kMaxStages = 16;
constexpr int kMaxClusterSplit = 6;   // the planner splits K across a cluster of 2..6 CTAs

struct Params {
  int M, N, KB;
  const uint8_t *xsf;    // W4A4: activation scale atoms [KB][xatoms][512] (K-block-major)
  int xatoms;            // W4A4: 128-token scale atoms per K block
  int t_tiles, splits, kb_per_split, units;
  int sk;                // 1: stream-K -- CTA c of sk_grid owns the K blocks [c*T/G, (c+1)*T/G) of the
                         // tile-major sequence of all T = tiles x KB blocks; unit c + j*G is its j-th tile piece
  int sk_grid, sk_total; // G and T of the stream-K schedule
  int ldc;
  int tma_store;         // 1: bf16 output tiles leave through smem + TMA tensor stores
  int l2_prefetch;       // 1: producer 0 prefetches the CTA's whole weight range into L2 at start;
                         // 2: decode tiles prefetch a rolling window of kPfAhead K blocks beyond the ring
  int cluster;           // 1: the `splits` CTAs of a cluster split K and exchange partials in DSMEM
  int xchg_stage;        // 1 (cluster, one unit per CTA): exchange the whole tile from the pipeline stages
  int inject_stall;      // test of the bounded waits: CTA 0 withholds its first activation copy
  int early_w;           // 1: weight tiles are requested before waiting for the preceding kernel
  const uint8_t *w;      // packed weight codes [NT][KB][128][64]
  const float *s;
  const uint8_t *sf;     // scale atoms of the prepacked weight
  uint16_t *c;
  float *partials;
  int *counters;
  int *err;
};

// Decode tiles (BT <= 64) are bound by instruction issue, not by HBM or the
// tensor core (measured on GB300): issuing one TMA operation occupies the
// issuing thread for a few hundred cycles, and an M=128, N<=64, K=32 MMA
// occupies its issuing thread for ~53 cycles whatever N is, plus the per-stage
// scale copy, commit and barrier handshake. So decode tiles run kIss TMA
// producer warps and kIss MMA-issuing warps: slot g (one 128-K block) belongs
// to producer g % kIss and MMA warp g % kIss, lives in ring stage g % kStages,
// and is accumulated into MMA warp (g % kIss)'s own tensor-memory accumulator;
// the epilogue sums the kIss partial accumulators. Prefill tiles of the
// W4A4 mode run two producer warps to one MMA warp (kProd = 2): their
// kind::mxf4 slots take half the MMA time of the f8 ones, and one thread
// issuing the slot's five copies (weight, activations, three scale atoms)
// could not keep up (measured on GB300: dropping two of the five copies
// alone made M=2048 8-19 % faster). Slot g then belongs to producer
// g % kProd and MMA warp g % kIss; a unit's slots are padded to a multiple
// of kPad = max(kProd, kIss).
//
// A4 = true is the W4A4 variant (kind::mxf4): both operands are packed e2m1
// (two per byte, loaded as plain bytes in the 64-byte swizzle: 8 KiB of
// weight and BT x 64 bytes of activations per 128-K block), and each stage
// also carries the activation scale atom(s) of its K block; the MMA applies
// both operands' ue8m0 scales, so the epilogue has no per-token scale.
template <int BT, bool A4 = false>
struct Cfg {
  static constexpr int kIss = BT <= 64 ? 4 : 1;
  static constexpr int kProd = BT <= 64 ? 4 : (A4 ? 2 : 1);   // TMA producer warps
  static constexpr int kPad = kProd > kIss ? kProd : kIss;    // slot padding of a unit
  // Two accumulators (the epilogue drains one while the MMAs fill the
  // other) wherever they leave room for the scale columns.
  static constexpr int kNumAcc = (kIss * 2 * BT <= 256 || (!A4 && kIss * 2 * BT <= 384)) ? 2 : 1;
  static constexpr uint32_t kAccCols = static_cast<uint32_t>(kIss * kNumAcc * BT);
  static constexpr uint32_t kSfaCol = kAccCols <= 256 ? 256u : 384u;
  static constexpr uint32_t kSfbCol = kSfaCol + 64u;
  // 256-token tiles (one accumulator) drain it into registers with 8
  // epilogue warps, two per tensor-memory lane quarter, 128 columns each
  // (see the epilogue); other tiles use 4.
  static constexpr bool kRegDrain = BT == 256;
  static constexpr int kEpiWarps = kRegDrain ? 8 : 4;
  // W4A4 prefill tiles (one MMA warp) have a scale warp: it waits for each
  // stage, copies its three scale atoms into tensor memory and commits them
  // to the stage's "scales ready" barrier, which is what the MMA thread waits
  // on -- the copies leave the MMA thread's per-K-block handshake, the bound
  // of a kind::mxf4 slot (two MMAs). Measured on GB300 (graph-timed, cold
  // weights): W4A4 M=2048 18-27 % faster (34816x5120 184.5 -> 156.6 us,
  // 5120x17408 119.6 -> 93.9 us), M=256 5-15 %; W4A8 (one atom, four MMAs
  // per slot) 2-9 % slower, so it keeps the copy in the MMA thread.
  static constexpr int kScaleWarp = (kIss == 1 && A4) ? 1 : 0;
  static constexpr int kThreads = 32 * (kProd + kIss + kScaleWarp + kEpiWarps);
  static constexpr int kEpiWarp0 = kProd + kIss + kScaleWarp;
  // Registers per thread: with more than 8 warps three share one SMSP, whose
  // 16K registers then allow 170 each.
  static constexpr int kMaxReg = kThreads > 256 ? 168 : 255;
  static constexpr uint32_t kWBytes = A4 ? 8192u : kWSmem;      // weight tile in shared memory
  static constexpr uint32_t kXSmem = A4 ? BT * 64 : BT * 128;   // activation tile
  static constexpr int kXAtoms = A4 ? (BT > 128 ? 2 : 1) : 0;   // activation scale atoms per stage
  static constexpr uint32_t kSfOff = kWBytes + kXSmem;          // weight scale atom, then activation atoms
  static constexpr uint32_t kStageBytes = ((kSfOff + kSfBytes * (1 + kXAtoms) + 1023) / 1024) * 1024;
  static constexpr int kOutChunk = BT < 32 ? BT : 32;                // tokens per output chunk
  static constexpr uint32_t kOutBytes = 2u * kOutChunk * 128u * 2u;  // two bf16 [chunk][128] buffers
  static constexpr int kStagesRaw = static_cast<int>((208u * 1024u) / kStageBytes);
  static constexpr int kStagesCap = kStagesRaw > kMaxStages ? kMaxStages : kStagesRaw;
  static constexpr int kStages = (kStagesCap / kPad) * kPad;        // every warp owns fixed stages
  static constexpr uint32_t kTxBytes = kWTxBytes + kXSmem + kSfBytes * (1 + kXAtoms);
  static constexpr uint32_t kMiscBytes = 1024;
  static constexpr uint32_t kSmemBytes = kStages * kStageBytes + kMiscBytes + kOutBytes + 1024;  // + align slack
  static_assert(kAccCols <= kSfaCol, "accumulators overlap the scale columns");
  static_assert(kSfbCol + (A4 ? 8u * kMaxStages : 16u * kIss) <= kTmemCols, "scale columns past tensor memory");
  static_assert(kStages >= kPad && kStages % kPad == 0, "stage count");
};

// Stream-K: first K block (tile-major) of CTA c, and the CTA that owns
// block x (the largest c with c*T/G <= x).
// (The planner keeps sk_total x sk_grid below 2^31: 32-bit arithmetic.)
__device__ __forceinline__ int sk_begin(const Params &p, int c) {
  return static_cast<int>(static_cast<uint32_t>(c * p.sk_total) / static_cast<uint32_t>(p.sk_grid));
}
__device__ __forceinline__ int sk_cta(const Params &p, int x) {
  return static_cast<int>(static_cast<uint32_t>((x + 1) * p.sk_grid - 1) / static_cast<uint32_t>(p.sk_total));
}
// CTAs whose K ranges share `tile` (1: the tile is one CTA's alone).
__device__ __forceinline__ int sk_segments(const Params &p, int tile) {
  return sk_cta(p, tile * p.KB + p.KB - 1) - sk_cta(p, tile * p.KB) + 1;
}

// Unit u -> weight tile nt, token tile tt, piece sp and K blocks [kb0, kb1)
// of the tile. Under stream-K a unit past its CTA's range is empty
// (kb0 == kb1): every role skips it.
__device__ __forceinline__ void decode_unit(const Params &p, int u, int &nt, int &tt, int &sp, int &kb0, int &kb1) {
  int tile;
  if (p.sk) {
    const int c = u % p.sk_grid, j = u / p.sk_grid;
    const int a = sk_begin(p, c), b = sk_begin(p, c + 1);
    const int ntiles = p.sk_total / p.KB;
    tile = a / p.KB + j;
    const int lo = max(a, tile * p.KB), hi = min(b, (tile + 1) * p.KB);
    sp = j;
    if (hi <= lo || tile >= ntiles) {
      tile = min(tile, ntiles - 1);
      kb0 = kb1 = 0;
    } else {
      kb0 = lo - tile * p.KB;
      kb1 = hi - tile * p.KB;
    }
  } else {
    tile = u / p.splits;
    sp = u - tile * p.splits;
    kb0 = sp * p.kb_per_split;
    kb1 = min(p.KB, kb0 + p.kb_per_split);
  }
  nt = tile / p.t_tiles;
  tt = tile - nt * p.t_tiles;
}

// Rolling L2 prefetch of the decode weight stream: one CTA keeps only its
// ring's worth of weight bytes in flight (~70 KB; measured ~45-50 GB/s per
// CTA on GB300, latency-bound), so producer 0 asks L2 for the next
// kPfAhead K blocks beyond the ring as it goes (one bulk prefetch per
// contiguous run, no shared memory). Measured on GB300 (cold weights,
// graph-timed): decode 34816x5120 19.1 -> 18.1 us (M=6), 22.9 -> 21.5 us
// (M=64); 5120x17408 15.0 -> 13.6 us (M=6); larger windows (16, 32) were
// slower; the whole range at kernel start (option 5 = 1) helps 5120x17408
// and hurts 34816x5120.
constexpr int kPfAhead = 8;

// Prefetch cursor over this CTA's unit sequence: unit u, K block kb
// (relative to the unit's first block).
struct PfCursor {
  int u, kb;
  int nkb = 0;      // K blocks of unit u
  size_t blk = 0;   // tile-major index of unit u's first K block
};

// Decode the cursor's unit once (the rolling prefetch runs every slot).
__device__ __forceinline__ void pf_load(const Params &p, PfCursor &c) {
  if (c.u >= p.units) return;
  int nt, tt, sp, kb0, kb1;
  decode_unit(p, c.u, nt, tt, sp, kb0, kb1);
  c.nkb = kb1 - kb0;
  c.blk = static_cast<size_t>(nt) * p.KB + kb0;
}

// Bulk L2 prefetch of `count` K blocks (weight codes and scale atoms, both
// contiguous within a unit) from the cursor on, across unit boundaries.
__device__ __forceinline__ void prefetch_blocks_l2(const Params &p, PfCursor &c, int count) {
  while (count > 0 && c.u < p.units) {
    const int n = min(count, c.nkb - c.kb);
    if (n > 0) {
      const size_t blk = c.blk + c.kb;
      bulk_prefetch_l2(p.w + blk * 8192, static_cast<uint32_t>(n) * 8192u);
      bulk_prefetch_l2(p.sf + blk * kSfBytes, static_cast<uint32_t>(n) * kSfBytes);
      c.kb += n;
      count -= n;
    }
    if (c.kb >= c.nkb) {
      c.u += gridDim.x;
      c.kb = 0;
      pf_load(p, c);
    }
  }
}

// Bulk L2 prefetch of unit u's weight codes and scale atoms (both contiguous).
__device__ __forceinline__ void prefetch_unit_l2(const Params &p, int u) {
  if (u >= p.units) return;
  int nt, tt, sp, kb0, kb1;
  decode_unit(p, u, nt, tt, sp, kb0, kb1);
  const size_t blk = static_cast<size_t>(nt) * p.KB + kb0;
  const uint32_t nkb = static_cast<uint32_t>(kb1 - kb0);
  if (nkb == 0) return;
  bulk_prefetch_l2(p.w + blk * 8192, nkb * 8192u);
  bulk_prefetch_l2(p.sf + blk * kSfBytes, nkb * kSfBytes);
}

// Shared-memory descriptor of a K-major operand in the 64-byte swizzle
// (rows of 64 bytes, 8-row groups 512 bytes apart, tile base 512-byte
// aligned): the W4A4 tiles, 128 packed e2m1 per row.
__device__ __forceinline__ uint64_t sdesc_sw64_kmajor(uint32_t saddr) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr >> 4) & 0x3FFFu);
  d |= static_cast<uint64_t>(1u) << 16;                 // LBO (unused for swizzled K-major)
  d |= static_cast<uint64_t>(512u >> 4) << 32;          // SBO: 8 rows x 64 B
  d |= static_cast<uint64_t>(1u) << 46;                 // descriptor version (tcgen05)
  d |= static_cast<uint64_t>(4u) << 61;                 // 64-byte swizzle
  return d;
}

// Instruction descriptor, kind::mxf4 with ue8m0 block scales (scale_vec::2X):
// A = B = e2m1 (format 1 in this kind), K-major, M = 128.
__host__ __device__ constexpr uint32_t idesc_mxf4_e2m1(int n, int a_sf_id, int b_sf_id) {
  return (static_cast<uint32_t>(b_sf_id & 3) << 4) | (1u << 7) | (1u << 10) | (static_cast<uint32_t>(n >> 3) << 17) |
         (1u << 23) | (static_cast<uint32_t>(128 >> 4) << 24) | (static_cast<uint32_t>(a_sf_id & 3) << 29);
}

// Register drain of one warp's half of a 256-token accumulator (one
// tensor-memory lane quarter q, 128 token columns from abase): all four
// 32-token chunks leave tensor memory in the 16x256b shape at once (128
// registers), the accumulator is released (one arrival on `acce`), and only
// then are the chunks scaled, rounded, written by stmatrix.trans into the
// warp's own 2 KB region ([32 token][32 n], 64-byte rows, 64-byte swizzle)
// and stored with one TMA store each -- while the next unit's MMAs already
// run. t0 is the first token of the half; tokens >= M get scale 0 and the
// TMA store clips them.
template <bool A4>
__device__ __forceinline__ void drain_half_to_regs(const Params &p, const CUtensorMap *tm_c, uint32_t abase,
                                                   uint16_t *region, int t0, int nt, int q, int lane,
                                                   uint64_t *acce) {
  uint32_t r[4][32];
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    tc_ld_16x256b_x4(abase + static_cast<uint32_t>(32 * c), r[c]);
    tc_ld_16x256b_x4(abase + (16u << 16) + static_cast<uint32_t>(32 * c), r[c] + 16);
  }
  tc_wait_ld();
  tc_fence_before();   // every chunk is in registers: the accumulator is free
  __syncwarp();
  if (lane == 0) mbar_arrive(acce);
  const int tq = 2 * (lane & 3);
  const int mrow = lane & 7, mmat = lane >> 3;
  const uint32_t sbase = smem_u32(region) + static_cast<uint32_t>(mrow * 64 + ((mmat ^ ((mrow >> 1) & 3)) << 4));
  const bool q_store = nt * 128 + q * 32 < p.N;
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    float sc[8];
#pragma unroll
    for (int g = 0; g < 4; ++g) {
      const int t = t0 + 32 * c + 8 * g + tq;
      if constexpr (A4) {
        sc[2 * g] = sc[2 * g + 1] = 1.f;
      } else {
        sc[2 * g] = (t < p.M) ? __ldg(p.s + t) : 0.f;
        sc[2 * g + 1] = (t + 1 < p.M) ? __ldg(p.s + t + 1) : 0.f;
      }
    }
    if (lane == 0) bulk_wait_read0();   // the previous chunk's store has read the region
    __syncwarp();
#pragma unroll
    for (int g = 0; g < 4; ++g) {
      uint32_t w[4];   // matrix m: n = 8m + lane/4 of the quarter, tokens 8g + tq, +1
#pragma unroll
      for (int m = 0; m < 4; ++m) {
        const int b = 16 * (m >> 1) + 4 * g + 2 * (m & 1);
        w[m] = pack_bf16x2(__uint_as_float(r[c][b]) * sc[2 * g], __uint_as_float(r[c][b + 1]) * sc[2 * g + 1]);
      }
      stmatrix_x4_trans(sbase + static_cast<uint32_t>(g * 8 * 64), w[0], w[1], w[2], w[3]);
    }
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) {
      if (q_store) tma_store_2d(tm_c, region, nt * 128 + q * 32, t0 + 32 * c);
      bulk_commit();
    }
  }
}

template <int BT, bool A4>
__global__ void __launch_bounds__(Cfg<BT, A4>::kThreads, 1) __maxnreg__((Cfg<BT, A4>::kMaxReg))
    w4a8_mxf8f6f4_kernel(const __grid_constant__ CUtensorMap tm_w, const __grid_constant__ CUtensorMap tm_x,
                         const __grid_constant__ CUtensorMap tm_c, const Params p) {
  using C = Cfg<BT, A4>;
  constexpr int kXStep = A4 ? 64 : kBK;   // activation tile x coordinate per 128-K block (bytes)
  // per-token output scale: s[t] for W4A8; none for W4A4 (both scales are in the MMA)
  auto out_scale = [&](int t) -> float {
    if constexpr (A4) {
      return 1.f;
    } else {
      return __ldg(p.s + t);
    }
  };
  constexpr int ISS = C::kIss;    // MMA-issuing warps
  constexpr int PROD = C::kProd;  // TMA producer warps
  constexpr int PAD = C::kPad;    // a unit's slots are padded to a multiple of this
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t *misc = smem + C::kStages * C::kStageBytes;
  uint8_t *sfb_const = misc;                                         // 512 B of 0x7F
  uint64_t *full_bar = reinterpret_cast<uint64_t *>(misc + 512);     // [16]
  uint64_t *empty_bar = full_bar + kMaxStages;                       // [16]
  uint64_t *accf_bar = empty_bar + kMaxStages;                       // [2]
  uint64_t *acce_bar = accf_bar + 2;                                 // [2]
  uint64_t *drain_bar = acce_bar + 2;                                // [4], one per MMA warp
  uint64_t *red_full = drain_bar + 4;    // cluster split-K: all partials of a chunk written
  uint64_t *red_empty = red_full + 1;    // cluster split-K: all CTAs have read this CTA's partial
  uint64_t *sready_bar = red_empty + 1;   // [kMaxStages]: a stage's scale atoms are in tensor memory
  uint64_t *sdrain_bar = sready_bar + kMaxStages;
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(sdrain_bar + 1);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
  volatile int *is_last = abort_flag + 1;
  volatile int *epi_abort = abort_flag + 2;   // set and read by epilogue threads only
  uint16_t *staging = reinterpret_cast<uint16_t *>(misc + C::kMiscBytes);   // [2][kOutChunk][128] bf16

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  for (int i = threadIdx.x; i < 128; i += C::kThreads) reinterpret_cast<uint32_t *>(sfb_const)[i] = 0x7F7F7F7Fu;
  if (threadIdx.x == 0) {
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(&full_bar[s], 1);
      mbar_init(&empty_bar[s], 1);
      mbar_init(&sready_bar[s], 1);
    }
    mbar_init(sdrain_bar, 1);
    for (int a = 0; a < 2; ++a) {
      mbar_init(&accf_bar[a], ISS);   // one arrival per MMA warp per unit
      mbar_init(&acce_bar[a], C::kEpiWarps);   // one per epilogue warp
    }
    for (int w = 0; w < 4; ++w) mbar_init(&drain_bar[w], 1);
    mbar_init(red_full, p.splits);    // one arrival per CTA of the cluster
    mbar_init(red_empty, p.splits);
    *abort_flag = 0;
    *is_last = 0;
    *epi_abort = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tm_w);
    tma_prefetch_desc(&tm_x);
    pdl_launch_dependents();   // let the next kernel in the stream start its own prologue
  }
  if (warp == PROD) {          // first MMA warp owns the tensor-memory allocation
    tmem_alloc(tmem_slot, kTmemCols);
    tmem_relinquish();
  }
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // Every CTA of the cluster has initialised its barriers before any remote arrival.
  if (p.cluster) cluster_sync_all();

  if (warp < PROD) {
    // ------------------------------------------------------------ TMA producers (warps 0..PROD-1)
    // Slot sequence: every unit's k-blocks, padded to a multiple of PAD. A
    // padding slot carries no data: its full barrier gets a plain arrival.
    const int pw = warp;
    if (lane == 0) {
      const uint64_t pol_w = policy_evict_first();
      const uint64_t pol_x = policy_evict_last();
      uint32_t issued_mask = 0, issued_phase = 0;
      bool ok = true;
      // Weights do not depend on the preceding kernel: fill this producer's
      // stages with weight tiles (+ scale atoms) before waiting for it, so
      // under programmatic dependent launch the weight stream starts while
      // the previous kernel is still running.
      // Optionally ask L2 for this CTA's whole weight range up front: the
      // stream then runs at HBM rate while this kernel waits for its
      // predecessor, not only for the ring's depth.
      if (!p.early_w) pdl_wait();   // weights may come from the preceding kernel
      if (p.l2_prefetch == 1 && pw == 0)
        for (int u = blockIdx.x; u < p.units; u += gridDim.x) prefetch_unit_l2(p, u);
      // Rolling prefetch (decode tiles, producer 0): the cursor starts at the
      // first K block the ring's initial fill leaves out (the fill below
      // covers the first kStages slots, padding slots included).
      PfCursor pf{p.units, 0};
      const bool rolling = p.l2_prefetch == 2 && pw == 0 && BT <= 64;
      if (rolling) {
        int left = C::kStages;
        pf.u = blockIdx.x;
        while (pf.u < p.units) {
          int nt, tt, sp, kb0, kb1;
          decode_unit(p, pf.u, nt, tt, sp, kb0, kb1);
          const int nkb = kb1 - kb0, nslots = (nkb + PAD - 1) / PAD * PAD;
          if (left < nslots) {
            pf.kb = min(left, nkb);
            if (pf.kb == nkb) {
              pf.u += gridDim.x;
              pf.kb = 0;
            }
            break;
          }
          left -= nslots;
          pf.u += gridDim.x;
        }
        pf_load(p, pf);
        prefetch_blocks_l2(p, pf, kPfAhead);
      }
      {
        int g = 0;
        for (int u = blockIdx.x; u < p.units && g < C::kStages; u += gridDim.x) {
          int nt, tt, sp, kb0, kb1;
          decode_unit(p, u, nt, tt, sp, kb0, kb1);
          const int nkb = kb1 - kb0;
          const int nslots = (nkb + PAD - 1) / PAD * PAD;
          for (int i = pw; i < nslots && g + i < C::kStages; i += PROD) {
            const int s_ = g + i;
            if (i < nkb) {
              uint8_t *st = smem + s_ * C::kStageBytes;
              const int kb = kb0 + i;
              mbar_arrive_expect_tx(&full_bar[s_], C::kTxBytes);
              tma_load_3d(st, &tm_w, &full_bar[s_], 0, 0, nt * p.KB + kb, pol_w);
              bulk_load(st + C::kSfOff, p.sf + static_cast<size_t>(nt * p.KB + kb) * kSfBytes, kSfBytes,
                        &full_bar[s_], pol_w);
            } else {
              mbar_arrive(&full_bar[s_]);
            }
          }
          g += nslots;
        }
      }
      pdl_wait();   // activations come from the preceding kernel
      int stage = pw;
      uint32_t phase = 0;
      int gbase = 0;
      for (int u = blockIdx.x; u < p.units && ok; u += gridDim.x) {
        int nt, tt, sp, kb0, kb1;
        decode_unit(p, u, nt, tt, sp, kb0, kb1);
        const int nkb = kb1 - kb0;
        const int nslots = (nkb + PAD - 1) / PAD * PAD;
        for (int i = pw; i < nslots; i += PROD) {
          uint8_t *st = smem + stage * C::kStageBytes;
          const int kb = kb0 + i;
          if (rolling) prefetch_blocks_l2(p, pf, PROD);   // one block per slot, PROD slots per turn
          if (gbase + i >= C::kStages) {   // not pre-issued
            if (!mbar_wait(&empty_bar[stage], phase ^ 1u, abort_flag, p.err, DEV_ERR_WAIT_EMPTY)) {
              ok = false;
              break;
            }
            if (i < nkb) {
              mbar_arrive_expect_tx(&full_bar[stage], C::kTxBytes);
              tma_load_3d(st, &tm_w, &full_bar[stage], 0, 0, nt * p.KB + kb, pol_w);
              bulk_load(st + C::kSfOff, p.sf + static_cast<size_t>(nt * p.KB + kb) * kSfBytes, kSfBytes,
                        &full_bar[stage], pol_w);
            } else {
              mbar_arrive(&full_bar[stage]);
            }
          }
          // (Failure-detection test: with inject_stall, CTA 0 never issues its
          // first activation copy, so that stage's transaction never completes
          // and the consumer's bounded wait must expire and report.)
          const bool withhold = p.inject_stall && blockIdx.x == 0 && gbase + i == 0;
          if (i < nkb && !withhold) tma_load_2d(st + C::kWBytes, &tm_x, &full_bar[stage], kb * kXStep, tt * BT, pol_x);
          if constexpr (A4) {
            // the activation scale atom(s) of this token tile and K block:
            // adjacent in the K-block-major layout, one copy
            if (i < nkb)
              bulk_load(st + C::kSfOff + kSfBytes,
                        p.xsf + (static_cast<size_t>(kb) * p.xatoms + tt * BT / 128) * kSfBytes,
                        kSfBytes * C::kXAtoms, &full_bar[stage], pol_x);
          }
          // Record the newest phase of every stage, padding slots included: a
          // parity wait cannot tell phase k from k + 2, and a stage only
          // advances after its earlier phases completed.
          issued_mask |= 1u << stage;
          issued_phase = (issued_phase & ~(1u << stage)) | (phase << stage);
          stage += PROD;
          if (stage >= C::kStages) {
            stage -= C::kStages;
            phase ^= 1u;
          }
        }
        gbase += nslots;
      }
      // Never leave a copy in flight: wait (bounded, even after an abort) for
      // the last load issued into each of this producer's stages.
      for (int s_ = 0; s_ < C::kStages; ++s_)
        if (issued_mask & (1u << s_)) {
          volatile int dummy = 0;
          mbar_wait(&full_bar[s_], (issued_phase >> s_) & 1u, &dummy, p.err, DEV_ERR_WAIT_DRAIN);
        }
    }
    __syncwarp();
  } else if (warp < PROD + ISS) {
    // ------------------------------------------------------------ MMA issuers (warps PROD..PROD+ISS-1)
    const int mw = warp - PROD;
    if (lane == 0) {
      const uint32_t sfb = tmem + C::kSfbCol + 16u * static_cast<uint32_t>(mw);
      if constexpr (!A4) {
        const uint64_t sfb_desc = sdesc_sf_32x16(smem_u32(sfb_const));
#pragma unroll
        for (int j = 0; j < 4; ++j) tc_cp_32x128b_warpx4(sfb + 4 * j, sfb_desc);
      }
      int stage = mw;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      bool ok = true;
      for (int u = blockIdx.x; u < p.units && ok; u += gridDim.x) {
        int nt, tt, sp, kb0, kb1;
        decode_unit(p, u, nt, tt, sp, kb0, kb1);
        const int nkb = kb1 - kb0;
        if (nkb <= 0) continue;   // empty stream-K unit
        const int nslots = (nkb + PAD - 1) / PAD * PAD;
        if (!mbar_wait(&acce_bar[acc], acc_phase ^ 1u, abort_flag, p.err, DEV_ERR_WAIT_ACC_EMPTY)) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem + static_cast<uint32_t>((mw * C::kNumAcc + acc) * BT);
        bool first = true;
        for (int i = mw; i < nslots; i += ISS) {
          // with a scale warp, its "scales ready" barrier (which follows the
          // stage's full barrier) also stands for the stage's data
          if (!mbar_wait(C::kScaleWarp ? &sready_bar[stage] : &full_bar[stage], phase, abort_flag, p.err,
                         DEV_ERR_WAIT_FULL)) {
            ok = false;
            break;
          }
          if (i < nkb) {
            tc_fence_after();
            uint8_t *st = smem + stage * C::kStageBytes;
            const uint32_t sfa = tmem + C::kSfaCol + 4u * static_cast<uint32_t>(stage);
            if constexpr (!C::kScaleWarp) tc_cp_32x128b_warpx4(sfa, sdesc_sf_32x16(smem_u32(st + C::kSfOff)));
            const uint32_t a_base = smem_u32(st);
            const uint32_t b_base = smem_u32(st + C::kWBytes);
            if constexpr (A4) {
              // activation scales: column 4a + (token / 32) of this stage's slot holds
              // tokens 128a .. 128a + 127 of the tile, one byte per 32 K
              const uint32_t sfbs = tmem + C::kSfbCol + 8u * static_cast<uint32_t>(stage);
              if constexpr (!C::kScaleWarp) {
#pragma unroll
                for (int a = 0; a < C::kXAtoms; ++a)
                  tc_cp_32x128b_warpx4(sfbs + 4u * a,
                                       sdesc_sf_32x16(smem_u32(st + C::kSfOff + kSfBytes * (1 + a))));
              }
              // two MMAs of K = 64; scale id 0 / 2 picks the byte pair of 32-K blocks (0,1) / (2,3)
#pragma unroll
              for (int kk = 0; kk < 2; ++kk) {
                const uint32_t id = 2u * kk;
                tc_mma_mxf4(d_tmem, sdesc_sw64_kmajor(a_base + 32u * kk), sdesc_sw64_kmajor(b_base + 32u * kk),
                            idesc_mxf4_e2m1(BT, id, id), sfa | (id << 30), sfbs | (id << 30),
                            (!first || kk > 0) ? 1u : 0u);
              }
            } else {
#pragma unroll
              for (int kk = 0; kk < 4; ++kk) {
                const uint64_t ad = sdesc_sw128_kmajor(a_base + 32u * kk);
                const uint64_t bd = sdesc_sw128_kmajor(b_base + 32u * kk);
                const uint32_t idesc = idesc_mxf8f6f4_e2m1_e4m3(BT, kk, 0);
                tc_mma_mxf8f6f4(d_tmem, ad, bd, idesc, sfa | (static_cast<uint32_t>(kk) << 30), sfb,
                                (!first || kk > 0) ? 1u : 0u);
              }
            }
            first = false;
            tc_commit(&empty_bar[stage]);
          } else {
            mbar_arrive(&empty_bar[stage]);   // padding slot: nothing read it
          }
          stage += ISS;
          if (stage >= C::kStages) {
            stage -= C::kStages;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        if (first)
          mbar_arrive(&accf_bar[acc]);   // this warp owned no k-block of the unit
        else
          tc_commit(&accf_bar[acc]);
        if (++acc == C::kNumAcc) {
          acc = 0;
          acc_phase ^= 1u;
        }
      }
      // All MMAs this thread issued must be complete before tensor memory is freed.
      tc_commit(&drain_bar[mw]);
      volatile int dummy = 0;
      mbar_wait(&drain_bar[mw], 0, &dummy, p.err, DEV_ERR_WAIT_DRAIN);
    }
    __syncwarp();
  } else if (C::kScaleWarp && warp == PROD + ISS) {
    // ------------------------------------------------------------ scale warp (prefill tiles)
    // Walks the slots in the MMA thread's order: waits for a stage, copies
    // its weight scale atom (and, for W4A4, the activation atoms) into the
    // stage's tensor-memory columns and commits the copies to the stage's
    // "scales ready" barrier (a padding slot gets a plain arrival). A stage's
    // columns are overwritten only after its next full barrier, which needs
    // the MMAs of its previous use to have released the stage.
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      for (int u = blockIdx.x; u < p.units && ok; u += gridDim.x) {
        int nt, tt, sp, kb0, kb1;
        decode_unit(p, u, nt, tt, sp, kb0, kb1);
        const int nkb = kb1 - kb0;
        if (nkb <= 0) continue;   // empty stream-K unit
        const int nslots = (nkb + PAD - 1) / PAD * PAD;
        for (int i = 0; i < nslots; ++i) {
          if (!mbar_wait(&full_bar[stage], phase, abort_flag, p.err, DEV_ERR_WAIT_FULL)) {
            ok = false;
            break;
          }
          if (i < nkb) {
            tc_fence_after();
            uint8_t *st = smem + stage * C::kStageBytes;
            tc_cp_32x128b_warpx4(tmem + C::kSfaCol + 4u * static_cast<uint32_t>(stage),
                                 sdesc_sf_32x16(smem_u32(st + C::kSfOff)));
            if constexpr (A4) {
              const uint32_t sfbs = tmem + C::kSfbCol + 8u * static_cast<uint32_t>(stage);
#pragma unroll
              for (int a = 0; a < C::kXAtoms; ++a)
                tc_cp_32x128b_warpx4(sfbs + 4u * a, sdesc_sf_32x16(smem_u32(st + C::kSfOff + kSfBytes * (1 + a))));
            }
            tc_commit(&sready_bar[stage]);
          } else {
            mbar_arrive(&sready_bar[stage]);   // padding slot
          }
          if (++stage == C::kStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      // Every copy this thread issued completes before tensor memory is freed.
      tc_commit(sdrain_bar);
      volatile int dummy = 0;
      mbar_wait(sdrain_bar, 0, &dummy, p.err, DEV_ERR_WAIT_DRAIN);
    }
    __syncwarp();
  } else if (C::kRegDrain && warp >= C::kEpiWarp0 + 4) {
    // ------------------------------------------------------------ epilogue helpers (256-token tiles)
    // Columns 128-255 of the accumulator, lane quarter q: drained into
    // registers with the first four epilogue warps' halves, when the tile
    // is stored directly through TMA. On every other path (split-K, a C
    // that TMA cannot store) the first four warps read the whole tile, and
    // a helper only adds its arrival to the accumulator's release (the
    // release counts all eight warps, so it cannot complete before those
    // four have read it).
    pdl_wait();
    const int q = warp & 3;
    const int ew = warp - C::kEpiWarp0;
    int acc = 0;
    uint32_t acc_phase = 0;
    for (int u = blockIdx.x; u < p.units; u += gridDim.x) {
      int nt, tt, sp, kb0, kb1;
      decode_unit(p, u, nt, tt, sp, kb0, kb1);
      if (kb1 <= kb0) continue;   // empty stream-K unit
      const int tile = nt * p.t_tiles + tt;
      const int nseg = p.sk ? sk_segments(p, tile) : p.splits;
      if (!warp_wait(&accf_bar[acc], acc_phase, abort_flag, p.err, DEV_ERR_WAIT_ACC_FULL)) break;
      tc_fence_after();
      if (nseg == 1 && p.tma_store) {
        const uint32_t lane_base = tmem + (static_cast<uint32_t>(q * 32) << 16);
        drain_half_to_regs<A4>(p, &tm_c, lane_base + static_cast<uint32_t>(acc * BT + 128), staging + ew * 1024,
                               tt * BT + 128, nt, q, lane, &acce_bar[acc]);
      } else {
        __syncwarp();
        if (lane == 0) mbar_arrive(&acce_bar[acc]);
      }
      if (++acc == C::kNumAcc) {
        acc = 0;
        acc_phase ^= 1u;
      }
    }
    if (lane == 0) bulk_wait_all();   // output stores complete before the CTA's smem goes away
  } else {
    // ------------------------------------------------------------ epilogue (4 warps)
    pdl_wait();                     // s, C and the workspace belong to the kernel stream order
    const int q = warp & 3;         // tensor-memory lane quarter this warp may access
    const int ew = warp - C::kEpiWarp0;
    int acc = 0;
    uint32_t acc_phase = 0;
    constexpr int CH = BT < 32 ? BT : 32;
    const bool leader = (ew == 0 && lane == 0);
    uint32_t out_chunk = 0;   // running count of staged output chunks (selects the buffer)
    uint32_t xchg = 0;        // running count of cluster split-K exchanges
    bool stop = false;
    int abort_u = -1;         // unit at which an expired wait stopped the epilogue
    for (int u = blockIdx.x; u < p.units; u += gridDim.x) {
      int nt, tt, sp, kb0, kb1;
      decode_unit(p, u, nt, tt, sp, kb0, kb1);
      if (kb1 <= kb0) continue;                   // empty stream-K unit
      const int ncontrib = min(ISS, kb1 - kb0);   // MMA warps that accumulated something
      // The decision to stop must be the same in all 128 epilogue threads
      // (they meet at named barriers below): a failed wait is published
      // before the barrier and read after it.
      if (!mbar_wait(&accf_bar[acc], acc_phase, abort_flag, p.err, DEV_ERR_WAIT_ACC_FULL)) *epi_abort = 1;
      named_bar_sync(1, 128);
      if (*epi_abort) {
        abort_u = u;
        break;
      }
      tc_fence_after();
      const int n = nt * 128 + q * 32 + lane;
      const int t0 = tt * BT;
      const int tile = nt * p.t_tiles + tt;
      const uint32_t lane_base = tmem + (static_cast<uint32_t>(q * 32) << 16);
      // CTAs that share this tile's K range, and this unit's workspace slot
      const int nseg = p.sk ? sk_segments(p, tile) : p.splits;
      const size_t slot = p.sk ? static_cast<size_t>(u) : static_cast<size_t>(tile) * p.splits + sp;
      const bool ws_split = nseg > 1 && !p.cluster;
      float *part = ws_split ? p.partials + slot * (128 * BT) : nullptr;
      bool drained = false;
      if constexpr (ISS == 1 && CH == 32 && BT % 64 == 0) {
        if (nseg == 1 && p.tma_store) {
          // Prefill tile on one accumulator (the MMA waits for it: a second
          // 256-column accumulator would not leave room for the scale
          // columns). Every cycle spent here is tensor-pipe idle time, so
          // the drain is built for throughput:
          //  * 32-token chunks leave tensor memory in the 16x256b shape
          //    (two loads of 16 lanes), one chunk in flight while the
          //    previous one is stored;
          //  * each thread scales and rounds token PAIRS of one n into a
          //    bf16x2 word (the per-token scales of the next chunk are read
          //    one chunk ahead), and four stmatrix.trans per chunk write the
          //    8x8 blocks as [token][n] rows -- 4 shared stores per chunk
          //    instead of 32 two-byte ones;
          //  * each warp owns a [32 token][32 n] region per buffer (64-byte
          //    rows, 64-byte swizzle: the eight rows of a matrix land in
          //    eight different bank groups) and issues its own TMA store of
          //    it, so the four warps never wait for one another.
          // Measured on GB300 (graph-timed, cold weights), against one
          // thread storing a [32][128] buffer between two 128-thread
          // barriers, filled by 32 two-byte stores per thread: the drain of
          // a 256-token tile 5,500 -> 3,450 cycles (W4A4), M=2048 prefill
          // 5-7 % faster (W4A8 34816x5120 263 -> 247 us, W4A4 216 -> 201
          // us). Not kept: the same stmatrix stores into an unswizzled
          // [32][128] buffer (slower than the two-byte stores: eight rows of
          // a matrix share four banks); per-token scales staged for the
          // whole tile in shared memory (as fast here, but the cluster
          // split-K prefill of the same kernel lost 12 %); draining every
          // chunk into registers first (255 registers, spills); plain
          // coalesced global stores (M=2048, 34816x5120: 260 -> 345 us).
          if constexpr (C::kRegDrain) {
            // 256-token tile: this warp drains columns 0-127 of its quarter,
            // the matching helper warp (ew + 4) columns 128-255.
            drain_half_to_regs<A4>(p, &tm_c, lane_base + static_cast<uint32_t>(acc * BT), staging + ew * 1024, t0,
                                   nt, q, lane, &acce_bar[acc]);
          } else {
            uint32_t ra[32], rb[32];   // [0,16): lanes 0-15 of the quarter; [16,32): lanes 16-31
            const uint32_t abase = lane_base + static_cast<uint32_t>(acc * BT);
            auto load_chunk = [&](uint32_t (&r)[32], int c0) {
              tc_ld_16x256b_x4(abase + static_cast<uint32_t>(c0), r);
              tc_ld_16x256b_x4(abase + (16u << 16) + static_cast<uint32_t>(c0), r + 16);
            };
            const int tq = 2 * (lane & 3);                 // first of this thread's token pair in an 8-token group
            const int mrow = lane & 7, mmat = lane >> 3;   // stmatrix row (token) and matrix (8-n group) addressed
            const uint32_t st_off =
                static_cast<uint32_t>(q * 2048 + mrow * 64 + ((mmat ^ ((mrow >> 1) & 3)) << 4));
            const bool q_store = nt * 128 + q * 32 < p.N;  // this warp's 32 n hold at least one column
            float sc_cur[8], sc_nxt[8];                    // per-token scales of the token pairs, 4 groups
            auto load_scales = [&](float (&sc)[8], int c0) {
              if constexpr (!A4) {
  #pragma unroll
                for (int g = 0; g < 4; ++g) {
                  const int t = t0 + c0 + 8 * g + tq;
                  sc[2 * g] = (t < p.M) ? __ldg(p.s + t) : 0.f;
                  sc[2 * g + 1] = (t + 1 < p.M) ? __ldg(p.s + t + 1) : 0.f;
                }
              }
            };
            auto stage_and_store = [&](const uint32_t (&r)[32], int c0) {
              if (c0 + 32 < BT) load_scales(sc_nxt, c0 + 32);
              uint16_t *stg = staging + (out_chunk & 1u) * (CH * 128);
              const uint32_t sbase = smem_u32(stg) + st_off;
              if (lane == 0) bulk_wait_read1();   // this warp's store from two chunks ago has read its region
              __syncwarp();
  #pragma unroll
              for (int g = 0; g < 4; ++g) {
                uint32_t w[4];   // matrix m: n = 8m + lane/4 of the quarter, tokens 8g + tq, +1
  #pragma unroll
                for (int m = 0; m < 4; ++m) {
                  const int b = 16 * (m >> 1) + 4 * g + 2 * (m & 1);
                  float v0 = __uint_as_float(r[b]), v1 = __uint_as_float(r[b + 1]);
                  if constexpr (!A4) {
                    v0 *= sc_cur[2 * g];
                    v1 *= sc_cur[2 * g + 1];
                  }
                  w[m] = pack_bf16x2(v0, v1);
                }
                stmatrix_x4_trans(sbase + static_cast<uint32_t>(g * 8 * 64), w[0], w[1], w[2], w[3]);
              }
              fence_proxy_async_smem();
              __syncwarp();
              if (lane == 0) {
                if (q_store) tma_store_2d(&tm_c, stg + q * 1024, nt * 128 + q * 32, t0 + c0);
                bulk_commit();   // (an empty group when nothing was stored keeps the count per chunk)
              }
              ++out_chunk;
  #pragma unroll
              for (int i = 0; i < 8; ++i) sc_cur[i] = sc_nxt[i];
            };
            load_scales(sc_cur, 0);
            load_chunk(ra, 0);
  #pragma unroll 1
            for (int c0 = 0; c0 < BT; c0 += 64) {
              tc_wait_ld();              // chunk c0 in ra
              load_chunk(rb, c0 + 32);   // chunk c0 + 32 in flight
              stage_and_store(ra, c0);
              tc_wait_ld();              // chunk c0 + 32 in rb
              if (c0 + 64 < BT) {
                load_chunk(ra, c0 + 64);
              } else {
                tc_fence_before();   // every chunk is in registers: the accumulator is free
                __syncwarp();
                if (lane == 0) mbar_arrive(&acce_bar[acc]);
              }
              stage_and_store(rb, c0 + 32);
            }
          }
          drained = true;
        }
      }
#pragma unroll 1
      for (int c0 = 0; c0 < (drained ? 0 : BT); c0 += CH) {
        uint32_t r[32], r2[32];
        float v[32];
        // The MMA warps' accumulators are summed in warp order; the load of
        // accumulator w + 1 is in flight while accumulator w is added.
        auto ld_acc = [&](int w, uint32_t (&dst)[32]) {
          const uint32_t taddr = lane_base + static_cast<uint32_t>((w * C::kNumAcc + acc) * BT + c0);
          if constexpr (CH == 32) {
            tc_ld_32x32b_x32(taddr, dst);
          } else {
            tc_ld_32x32b_x16(taddr, dst);
          }
        };
        ld_acc(0, r);
        tc_wait_ld();
#pragma unroll
        for (int j = 0; j < CH; ++j) v[j] = __uint_as_float(r[j]);
#pragma unroll 1
        for (int w = 1; w < ncontrib; w += 2) {
          ld_acc(w, r2);
          tc_wait_ld();
          if (w + 1 < ncontrib) ld_acc(w + 1, r);
#pragma unroll
          for (int j = 0; j < CH; ++j) v[j] += __uint_as_float(r2[j]);
          if (w + 1 < ncontrib) {
            tc_wait_ld();
#pragma unroll
            for (int j = 0; j < CH; ++j) v[j] += __uint_as_float(r[j]);
          }
        }
        if (c0 + CH >= BT) {
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&acce_bar[acc]);
        }
        if (BT < 128 && nseg == 1 && p.tma_store) {
          // Stage [CH tokens][128 n] bf16 in smem, then one TMA tensor store;
          // the store clips rows >= M and columns >= N. (Prefill tiles with a
          // TMA-storable C took the per-warp drain above: their tensor map
          // has the per-warp box.)
          uint16_t *stg = staging + (out_chunk & 1u) * (CH * 128);
          if (leader) bulk_wait_read1();   // the store issued two chunks ago has read this buffer
          named_bar_sync(1, 128);
#pragma unroll
          for (int j = 0; j < CH; ++j) {
            const int t = t0 + c0 + j;
            const float sc = (t < p.M) ? out_scale(t) : 0.f;
            stg[j * 128 + q * 32 + lane] = f32_to_bf16_rn(v[j] * sc);
          }
          fence_proxy_async_smem();
          named_bar_sync(1, 128);
          if (leader) {
            tma_store_2d(&tm_c, stg, nt * 128, t0 + c0);
            bulk_commit();
          }
          ++out_chunk;
        } else if (nseg == 1) {
          if (n < p.N) {
#pragma unroll
            for (int j = 0; j < CH; ++j) {
              const int t = t0 + c0 + j;
              if (t < p.M) p.c[static_cast<size_t>(t) * p.ldc + n] = f32_to_bf16_rn(v[j] * out_scale(t));
            }
          }
        } else if (p.cluster) {
          // Split-K inside the cluster: this CTA's partial goes to its own
          // shared memory as fp32 [tokens][128]; then every CTA sums its
          // 1/splits share of the 128 n (in groups of 4) over all CTAs'
          // partials, in rank order (deterministic), and stores
          // bf16(s[t] * sum). With one unit per CTA (p.xchg_stage) the whole
          // tile goes into the drained pipeline stages -- every MMA of the
          // unit has completed (its accumulator barrier) and no load follows --
          // and one exchange round covers all BT tokens; otherwise the
          // staging buffer carries one 32-token chunk per round.
          const bool whole = p.xchg_stage != 0;
          float *red = whole ? reinterpret_cast<float *>(smem) : reinterpret_cast<float *>(staging);
          const int row0 = whole ? c0 : 0;        // this chunk's first token row in red
          const int rows = whole ? BT : CH;       // token rows of one exchange round
          const int tbase = whole ? t0 : t0 + c0;
          if (!whole) {
            if (xchg > 0 && leader &&
                !mbar_wait_cluster(red_empty, (xchg - 1u) & 1u, abort_flag, p.err, DEV_ERR_WAIT_PEER))
              *epi_abort = 1;
            named_bar_sync(1, 128);
            if (*epi_abort) {
              stop = true;
              break;
            }
          }
#pragma unroll
          for (int j = 0; j < CH; ++j) red[(row0 + j) * 128 + q * 32 + lane] = v[j];
          if (whole && c0 + CH < BT) continue;   // more chunks before the (single) round
          named_bar_sync(1, 128);
          if (leader) {
            fence_acq_rel_cluster();
            for (int pr = 0; pr < p.splits; ++pr) mbar_arrive_remote(mapa_shared(smem_u32(red_full), pr));
            if (!mbar_wait_cluster(red_full, xchg & 1u, abort_flag, p.err, DEV_ERR_WAIT_PEER)) *epi_abort = 1;
          }
          named_bar_sync(1, 128);
          if (*epi_abort) {
            stop = true;
            break;
          }
          const int rank = static_cast<int>(cluster_ctarank());
          const int qlo = rank * 32 / p.splits, nq = (rank + 1) * 32 / p.splits - qlo;
          const uint32_t red_base = smem_u32(red);
          // Only token rows that exist (t < M) are read from the peers: a
          // load whose value has no consumer is never issued.
          const int vrows = min(rows, p.M - tbase);
          for (int idx = ew * 32 + lane; idx < vrows * nq; idx += 128) {
            const int j = idx / nq, qd = qlo + (idx - j * nq);
            const uint32_t off = red_base + static_cast<uint32_t>((j * 128 + qd * 4) * 4);
            float4 a4;
            if constexpr (BT >= 128) {
              // Prefill tiles (one whole-tile round of up to 20 loads per
              // thread): all partials' loads in flight before the
              // rank-ordered sum (M=256, 5120x17408: 34.7 -> 33.0 us).
              // Decode tiles keep the short loop: the extra live registers
              // cost them more than the overlap gains.
              float4 b4[kMaxClusterSplit];
#pragma unroll
              for (int pr = 0; pr < kMaxClusterSplit; ++pr)
                if (pr < p.splits) b4[pr] = ld_dsmem_f32x4(mapa_shared(off, static_cast<uint32_t>(pr)));
              a4 = b4[0];
#pragma unroll
              for (int pr = 1; pr < kMaxClusterSplit; ++pr)
                if (pr < p.splits) {
                  a4.x += b4[pr].x;
                  a4.y += b4[pr].y;
                  a4.z += b4[pr].z;
                  a4.w += b4[pr].w;
                }
            } else {
              a4 = ld_dsmem_f32x4(mapa_shared(off, 0));
              for (int pr = 1; pr < p.splits; ++pr) {
                const float4 b4 = ld_dsmem_f32x4(mapa_shared(off, static_cast<uint32_t>(pr)));
                a4.x += b4.x;
                a4.y += b4.y;
                a4.z += b4.z;
                a4.w += b4.w;
              }
            }
            const int t = tbase + j;
            if (t < p.M) {
              const float sc = out_scale(t);
              const int n0 = nt * 128 + qd * 4;
              uint16_t *dst = p.c + static_cast<size_t>(t) * p.ldc + n0;
              const float o[4] = {a4.x * sc, a4.y * sc, a4.z * sc, a4.w * sc};
#pragma unroll
              for (int e = 0; e < 4; ++e)
                if (n0 + e < p.N) dst[e] = f32_to_bf16_rn(o[e]);
            }
          }
          named_bar_sync(1, 128);
          if (leader)
            for (int pr = 0; pr < p.splits; ++pr) mbar_arrive_remote(mapa_shared(smem_u32(red_empty), pr));
          ++xchg;
        } else {
#pragma unroll
          for (int j = 0; j < CH; ++j) part[(c0 + j) * 128 + q * 32 + lane] = v[j];
        }
      }
      if (stop) break;
      if (ws_split) {
        __threadfence();
        named_bar_sync(1, 128);
        if (ew == 0 && lane == 0) {
          const int prev = atomicAdd(p.counters + tile, 1);
          // 1: last arrival, sum; 2: last arrival after a poisoned one, no sum
          *is_last = ((prev & kArrivalMask) == nseg - 1) ? ((prev >> kPoisonShift) ? 2 : 1) : 0;
        }
        named_bar_sync(1, 128);
        if (*is_last == 1) {
          __threadfence();
          if (p.sk) {
            // the tile's pieces in K order: CTAs c0 .. c0 + nseg - 1, each
            // its piece j = tile - (first tile of the CTA)
            const int c0 = sk_cta(p, tile * p.KB);
            auto slot_ptr = [&](int s2) -> const float * {
              const int c = c0 + s2;
              const int j = tile - sk_begin(p, c) / p.KB;
              return p.partials + (static_cast<size_t>(c) + static_cast<size_t>(j) * p.sk_grid) * (128 * BT);
            };
            reduce_slots_store(slot_ptr, nseg, min(BT, p.M - t0), nt * 128, p.N, A4 ? nullptr : p.s, t0, p.c,
                               p.ldc, ew * 32 + lane, 128);
          } else {
            const float *base = p.partials + static_cast<size_t>(tile) * p.splits * (128 * BT);
            reduce_partials_store<BT>(base, p.splits, min(BT, p.M - t0), nt * 128, p.N, A4 ? nullptr : p.s, t0,
                                      p.c, p.ldc, ew * 32 + lane, 128);
          }
        }
        if (*is_last && ew == 0 && lane == 0) p.counters[tile] = 0;
        named_bar_sync(1, 128);
      }
      if (++acc == C::kNumAcc) {
        acc = 0;
        acc_phase ^= 1u;
      }
    }
    // An expired wait stopped this CTA: it still arrives, poisoned, at the
    // counter of every workspace split-K tile it owed (the one it stopped in
    // and all later ones), so that every counter ends the launch at zero.
    if (abort_u >= 0 && (p.splits > 1 || p.sk) && !p.cluster && leader) {
      for (int u2 = abort_u; u2 < p.units; u2 += gridDim.x) {
        int nt2, tt2, sp2, kb02, kb12;
        decode_unit(p, u2, nt2, tt2, sp2, kb02, kb12);
        if (kb12 <= kb02) continue;   // empty stream-K unit: owed nothing
        const int tile2 = nt2 * p.t_tiles + tt2;
        const int nseg2 = p.sk ? sk_segments(p, tile2) : p.splits;
        if (nseg2 <= 1) continue;     // stored directly, no counter
        const int prev = atomicAdd(p.counters + tile2, 1 + kPoisonArrival);
        if ((prev & kArrivalMask) == nseg2 - 1) atomicExch(p.counters + tile2, 0);
      }
    }
    if (lane == 0) bulk_wait_all();   // output stores complete before the CTA's smem goes away
  }

  tc_fence_before();
  __syncthreads();
  if (warp == PROD) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
  // No CTA leaves while another may still read its shared memory or arrive
  // on its barriers. Every role's waits are bounded, so all threads get here.
  if (p.cluster) cluster_sync_all();
}

template <int BT, bool A4>
int launch_bt(const uint8_t *q, const float *s, const uint8_t *xsf, const uint8_t *packed, int64_t M, int64_t N,
              int64_t K, uint16_t *c, int64_t ldc, void *ws, const GemmPlan &pl, cudaStream_t st) {
  using C = Cfg<BT, A4>;
  const int64_t NT = ceil_div(N, 128);
  CUtensorMap tm_w, tm_x, tm_c;
  if constexpr (A4) {
    // packed e2m1 bytes as they are: 128 rows x 64 bytes per tile, 64-byte swizzle
    {
      const uint64_t dims[3] = {64, 128, static_cast<uint64_t>(NT * pl.KB)};
      const uint64_t strides[2] = {64, 8192};
      const uint32_t box[3] = {64, 128, 1};
      if (encode_tiled(&tm_w, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<uint8_t *>(packed), dims, strides, box,
                       CU_TENSOR_MAP_SWIZZLE_64B) != CUDA_SUCCESS)
        return R4_ERR_CUDA;
    }
    {
      const uint64_t dims[2] = {static_cast<uint64_t>(K / 2), static_cast<uint64_t>(M)};
      const uint64_t strides[1] = {static_cast<uint64_t>(K / 2)};
      const uint32_t box[2] = {64, static_cast<uint32_t>(BT)};
      if (encode_tiled(&tm_x, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t *>(q), dims, strides, box,
                       CU_TENSOR_MAP_SWIZZLE_64B) != CUDA_SUCCESS)
        return R4_ERR_CUDA;
    }
  } else {
    {
      const uint64_t dims[3] = {128, 128, static_cast<uint64_t>(NT * pl.KB)};
      const uint64_t strides[2] = {64, 8192};
      const uint32_t box[3] = {128, 128, 1};
      if (encode_tiled(&tm_w, CU_TENSOR_MAP_DATA_TYPE_16U4_ALIGN16B, 3, const_cast<uint8_t *>(packed), dims, strides,
                       box, CU_TENSOR_MAP_SWIZZLE_128B) != CUDA_SUCCESS)
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
  }
  // Output through TMA tensor stores when C's base, row stride and row length
  // are 16-byte multiples. (Measured on GB300: a tensor store whose row ends
  // inside a 16-byte granule writes the whole granule, past column N.)
  int use_tma_store = 0;
  if ((reinterpret_cast<uintptr_t>(c) % 16) == 0 && (ldc * 2) % 16 == 0 && (N * 2) % 16 == 0) {
    const uint64_t dims[2] = {static_cast<uint64_t>(N), static_cast<uint64_t>(M)};
    const uint64_t strides[1] = {static_cast<uint64_t>(ldc) * 2};
    // Prefill tiles (BT >= 128) store per warp: [32 tokens][32 n] boxes in
    // the 64-byte swizzle; decode tiles store [chunk][128 n] unswizzled.
    const uint32_t box[2] = {BT >= 128 ? 32u : 128u, static_cast<uint32_t>(C::kOutChunk)};
    use_tma_store = encode_tiled(&tm_c, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, c, dims, strides, box,
                                 BT >= 128 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_NONE) == CUDA_SUCCESS;
  }
  if (!use_tma_store) tm_c = tm_x;   // not read by the kernel in that case
  Params p;
  p.M = static_cast<int>(M);
  p.N = static_cast<int>(N);
  p.KB = pl.KB;
  p.xsf = xsf;
  p.xatoms = static_cast<int>(mx_act_tokens_padded(M) / 128);
  p.t_tiles = pl.t_tiles;
  p.splits = pl.splits;
  p.kb_per_split = pl.kb_per_split;
  p.sk = pl.sk;
  p.sk_grid = pl.grid;
  p.sk_total = pl.sk_total;
  p.units = pl.units;
  p.ldc = static_cast<int>(ldc);
  p.tma_store = use_tma_store;
  p.l2_prefetch = options().l2_prefetch;
  p.cluster = pl.cluster;
  p.xchg_stage = (pl.cluster && pl.units <= pl.grid) ? 1 : 0;
  p.inject_stall = options().inject_stall;
  p.early_w = options().early_weights;
  p.w = packed;
  p.s = s;
  p.sf = packed + mx_packed_codes_bytes(N, K);
  p.c = c;
  p.counters = reinterpret_cast<int *>(ws);
  p.partials = ws ? reinterpret_cast<float *>(reinterpret_cast<uint8_t *>(ws) + pl.counters_bytes) : nullptr;
  p.err = device_error_word();
  auto kern = w4a8_mxf8f6f4_kernel<BT, A4>;
  if (ensure_smem_attr(reinterpret_cast<const void *>(kern), C::kSmemBytes) != cudaSuccess) return R4_ERR_CUDA;
  const cudaError_t le =
      pl.cluster ? launch_pdl_cluster(kern, dim3(pl.grid), dim3(C::kThreads), C::kSmemBytes, st, pl.splits, tm_w, tm_x,
                                      tm_c, p)
                 : launch_pdl(kern, dim3(pl.grid), dim3(C::kThreads), C::kSmemBytes, st, tm_w, tm_x, tm_c, p);
  if (le != cudaSuccess) return R4_ERR_CUDA;
  if constexpr (A4)
    set_last_kernel(BT == 16    ? "w4a8_mxf8f6f4_kernel<16,mxf4>"
                    : BT == 32  ? "w4a8_mxf8f6f4_kernel<32,mxf4>"
                    : BT == 64  ? "w4a8_mxf8f6f4_kernel<64,mxf4>"
                    : BT == 128 ? "w4a8_mxf8f6f4_kernel<128,mxf4>"
                                : "w4a8_mxf8f6f4_kernel<256,mxf4>");
  else
    set_last_kernel(BT == 16    ? "w4a8_mxf8f6f4_kernel<16>"
                    : BT == 32  ? "w4a8_mxf8f6f4_kernel<32>"
                    : BT == 64  ? "w4a8_mxf8f6f4_kernel<64>"
                    : BT == 128 ? "w4a8_mxf8f6f4_kernel<128>"
                    : BT == 192 ? "w4a8_mxf8f6f4_kernel<192>"
                                : "w4a8_mxf8f6f4_kernel<256>");
  return cudaGetLastError() == cudaSuccess ? R4_OK : R4_ERR_CUDA;
}

// Co-resident clusters of `s` CTAs (2..8) the BT kernel can have on this
// device (0: none / unsupported). Cached after the first query.
template <int BT, bool A4>
int max_clusters_bt(int s) {
  using C = Cfg<BT, A4>;
  static int cache[9] = {0, 0, 0, 0, 0, 0, 0, 0, 0};   // 0 unknown, -1 none
  if (s < 2 || s > 8) return 0;
  if (cache[s] != 0) return cache[s] > 0 ? cache[s] : 0;
  auto kern = w4a8_mxf8f6f4_kernel<BT, A4>;
  int n = 0;
  if (ensure_smem_attr(reinterpret_cast<const void *>(kern), C::kSmemBytes) == cudaSuccess) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(s * 16));
    cfg.blockDim = dim3(C::kThreads);
    cfg.dynamicSmemBytes = C::kSmemBytes;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = static_cast<unsigned>(s);
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess) n = 0;
  }
  (void)cudaGetLastError();   // a failed query leaves no sticky error
  cache[s] = n > 0 ? n : -1;
  return n > 0 ? n : 0;
}

int max_clusters(int bt, int s, bool a4) {
  switch (bt) {
    case 16: return a4 ? max_clusters_bt<16, true>(s) : max_clusters_bt<16, false>(s);
    case 32: return a4 ? max_clusters_bt<32, true>(s) : max_clusters_bt<32, false>(s);
    case 64: return a4 ? max_clusters_bt<64, true>(s) : max_clusters_bt<64, false>(s);
    case 128: return a4 ? max_clusters_bt<128, true>(s) : max_clusters_bt<128, false>(s);
    case 192: return a4 ? 0 : max_clusters_bt<192, false>(s);
    case 256: return a4 ? max_clusters_bt<256, true>(s) : max_clusters_bt<256, false>(s);
    default: return 0;
  }
}

}  // namespace w4a8

// Token tile and split-K choice. A small wave model: every SM streams its
// unit's weight bytes at an equal share of HBM bandwidth (capped by what one
// CTA keeps in flight) or runs its MMAs at the per-SM FP8 rate, whichever is
// slower. Split-K either exchanges partials inside a thread-block cluster of
// `splits` CTAs (decode tiles, 2..8 splits: a fixed cost per unit, no
// workspace) or writes them to the workspace, where the last-arriving CTA
// sums them at the few tens of GB/s one CTA's plain loads reach. The
// constants were fitted to a GB300 sweep of split factors on the decode and
// prefill shapes. Prefill tiles (BT >= 128) are never split once the tile
// count is a quarter of the SM count: there the partial tiles cost more than
// the idle SMs.
//
// The W4A4 variant (a4) uses the same model with its own bytes and rate per
// K block (packed e2m1 activations, two scale atoms, the mxf4 rate is twice
// the f8 one) and one more rule: a token tile starts on a 128-token scale
// atom (tiles of 128 or 256 tokens, or a single tile of up to 64 tokens
// starting at token 0), so that every activation scale of a tile sits at the
// start of the atom copied into tensor memory.
//
// Over 128 tokens W4A8 chooses between 256-token tiles (one accumulator: the
// tensor pipe waits while the epilogue drains it, ~2.5 us per unit) and
// 192-token tiles (two accumulators: the drain overlaps the next unit's
// MMAs, at a quarter less work per unit and up to 191 padding tokens) by
// the modeled time of each.
static GemmPlan plan_mx_bt(int64_t M, int64_t N, int64_t K, int sms, bool a4, int bt, double *t_model) {
  GemmPlan pl;
  pl.BT = bt;
  pl.n_tiles = static_cast<int>(ceil_div(N, 128));
  pl.t_tiles = static_cast<int>(ceil_div(M, bt));
  pl.KB = static_cast<int>(ceil_div(K, 128));
  const int64_t tiles = static_cast<int64_t>(pl.n_tiles) * pl.t_tiles;
  // 16-token partial tiles (8 KiB) sum faster per byte than larger ones
  // (fitted: 2048x5120 decode, 5 splits 6.1 us vs 4 splits 7.3 us).
  const double hbm = 6.0e12, sm_bw = 70e9, sm_flops = (a4 ? 9.0e15 : 4.5e15) / 152.0,
               red_bw = bt <= 16 ? 40e9 : 20e9;
  // weight + its scales + activations (+ their scale atoms for W4A4)
  const double kb_bytes = a4 ? 128.0 * 128 * 0.5 + 512 + 64.0 * bt + 512.0 * (bt > 128 ? 2 : 1)
                             : 128.0 * 128 * 0.5 + 512 + 128.0 * bt;
  const double kb_flops = 2.0 * 128 * bt * 128;
  const double part_bytes = 128.0 * bt * 4;
  // Prefill tiles (BT >= 128): the activation tile is read from L2 (every
  // weight tile re-reads it), so only the weight bytes share HBM, and every
  // K block's bytes pass through the CTA's shared-memory feed at ~110 GB/s
  // per SM. Fitted to GB300 timings of forced 192- and 256-token tiles
  // (interleaved, cold weights): 1024x34816x5120 predicted 121 / 133 us,
  // measured 122 / 133; 4096x10240x5120 136 / 145 vs 137 / 145;
  // 512x5120x17408 picks the 192-token tile (42.0 vs 48.1 us).
  const double w_bytes = 128.0 * 128 * 0.5 + 512, feed_bw = 110e9;
  auto unit_time = [&](int64_t kbps_, int64_t active) {
    if (bt < 128)
      return std::max(kbps_ * kb_bytes / std::min(hbm / active, sm_bw), kbps_ * kb_flops / sm_flops);
    return std::max({kbps_ * w_bytes / std::min(hbm / active, sm_bw), kbps_ * kb_flops / sm_flops,
                     kbps_ * kb_bytes / feed_bw});
  };
  const double xchg_s = (bt <= 64 ? 2.5e-6 : 1.0e-6) * ((bt + 31) / 32);   // one cluster exchange per 32 tokens
  // Epilogue drain of a prefill unit: at 256 tokens (one accumulator) the
  // tensor pipe waits ~0.3 us per unit while eight warps pull it into
  // registers; with two accumulators it costs once per CTA.
  const bool one_acc = bt == 256;
  const double drain = bt == 256 ? 0.3e-6 : bt >= 128 ? 1.0e-8 * bt : 0.0;
  const int forced = options().w4a8_splits;
  // Prefill tiles (BT >= 128) split through the workspace only while the
  // tile count is under a quarter of the SM count, and through a cluster
  // only while one wave of clusters covers every tile.
  const bool prefill_ws_ok = tiles * 4 < sms;
  const int max_s = std::min(pl.KB, 64);
  int best_s = 1, best_cl = 0;
  int64_t best_grid = std::min<int64_t>(tiles, sms);
  double best_t = 1e30;
  // A forced factor is rounded to the nearest schedule without an empty split.
  const int forced_s =
      forced > 0 ? static_cast<int>(ceil_div(pl.KB, ceil_div(pl.KB, std::min(forced, pl.KB)))) : 0;
  for (int s = 1; s <= max_s; ++s) {
    if (forced_s && s != forced_s) continue;
    const int kbps = static_cast<int>(ceil_div(pl.KB, s));
    if (static_cast<int64_t>(s - 1) * kbps >= pl.KB) continue;   // would leave an empty split
    const int64_t units = tiles * s;
    // Decode tiles split only while all units fit in one wave (measured: a
    // second wave of split units always loses to fewer splits).
    if (!forced_s && s > 1 && bt <= 64 && units > sms) continue;
    // The cluster exchange beats the workspace path from 32 tokens up
    // (measured); at 16 tokens the partial tiles are small enough that the
    // last-arriving CTA sums them faster than a cluster round trip.
    // Prefill tiles take the cluster path when one wave of clusters covers
    // every tile: each CTA then has one unit and exchanges its whole tile
    // from the drained pipeline stages in one round (per-32-token rounds ate
    // the gain at 256 tokens: M=256, 5120x17408, 3 splits 49.9 us vs 49.8 us
    // unsplit).
    int ncl = (options().cluster_split && bt >= 32 && s >= 2 && s <= 6) ? w4a8::max_clusters(bt, s, a4) : 0;
    if (bt >= 128 && !forced_s && tiles > ncl) ncl = 0;
    if (bt >= 128 && !forced_s && s > 1 && ncl == 0 && !prefill_ws_ok) continue;
    // Prefill tiles split only while every CTA holds at most one split unit
    // (forced factors included; otherwise the schedule stays unsplit). The
    // split paths with several split units per CTA are not run on prefill
    // tiles: a timing sweep of forced factors at M=256, 34816x5120 (272
    // tiles) ended in an illegal-address error whose cause was not found.
    if (bt >= 128 && s > 1 && units > (ncl > 0 ? std::min<int64_t>(tiles, ncl) * s : static_cast<int64_t>(sms)))
      continue;
    double t;
    int64_t grid;
    if (ncl > 0) {
      const int64_t nclust = std::min<int64_t>(tiles, ncl);
      const int64_t active = nclust * s;
      const double waves = std::ceil(static_cast<double>(tiles) / nclust);
      const double t_unit = unit_time(kbps, active);
      const double xchg = waves == 1 ? 3.0e-6 : xchg_s;   // one whole-tile round, or a round per 32 tokens
      t = waves * t_unit + xchg + 0.5e-6 * s + (one_acc ? waves : 1.0) * drain;
      grid = active;
    } else {
      const int64_t active = std::min<int64_t>(units, sms);
      const double waves = std::ceil(static_cast<double>(units) / sms);
      const double t_unit = unit_time(kbps, active);
      t = waves * t_unit + (one_acc ? waves : 1.0) * drain;
      if (s > 1) t += (waves + s) * part_bytes / red_bw;
      grid = active;
    }
    if (t < best_t) {
      best_t = t;
      best_s = s;
      best_cl = ncl > 0;
      best_grid = grid;
    }
  }
  pl.splits = best_s;
  pl.kb_per_split = static_cast<int>(ceil_div(pl.KB, best_s));
  pl.splits = static_cast<int>(ceil_div(pl.KB, pl.kb_per_split));  // no empty split
  if (pl.splits != best_s) best_cl = 0;                              // (cannot happen: empty splits skipped)
  pl.units = static_cast<int>(tiles * pl.splits);
  pl.cluster = best_cl;
  pl.grid = static_cast<int>(best_grid);
  if (pl.splits > 1 && !pl.cluster && tiles > kMaxCounterTiles) {   // (only a forced split gets here)
    pl.splits = 1;
    pl.kb_per_split = pl.KB;
    pl.units = static_cast<int>(tiles);
    pl.grid = static_cast<int>(std::min<int64_t>(tiles, sms));
  }
  if (pl.splits > 1 && !pl.cluster) {
    pl.counters_bytes = kCounterBytes;
    pl.ws_bytes = pl.counters_bytes + static_cast<size_t>(pl.units) * 128 * bt * 4;
  }
  // Stream-K for decode tiles. A decode CTA streams its weights at ~35 GB/s
  // whatever its share of HBM (latency-bound, measured on GB300), so what
  // counts is the longest K range one CTA streams: a uniform split leaves
  // SMs idle when tiles x splits is not a multiple of the SM count (5120 x
  // 17408: 40 tiles x 3 splits on 120 of 152 SMs) or runs a second partial
  // wave (34816 x 5120: 272 tiles, 80 K blocks on the busiest CTA against
  // 72 on average). Stream-K gives every CTA the same number of K blocks of
  // the tile-major sequence; a tile shared by several CTAs is summed through
  // the workspace by its last arrival, in K order.
  // Measured on GB300 (graph-timed, cold weights) it loses to the uniform
  // schedule on every decode shape -- 6x34816x5120 22.2 vs 19.1 us,
  // 6x5120x17408 15.9 vs 14.5 us, 64x5120x17408 26.9 vs 19.4 us: a shared
  // tile's partial write, fence and counter, and the last arrival's sum at
  // the end of its CTA's range, cost more than the balance gains. So it is
  // off by default (option 16 = 0) and kept as a tested option.
  const int sk_opt = options().stream_k;
  if (bt <= 64 && sk_opt != 0 && !forced_s && tiles <= kMaxCounterTiles &&
      tiles * pl.KB * std::min<int64_t>(sms, tiles * pl.KB) < (int64_t(1) << 31)) {
    const int64_t T = tiles * pl.KB;   // (T x G < 2^31: the kernel's stream-K arithmetic is 32-bit)
    const int G = static_cast<int>(std::min<int64_t>(sms, T));
    auto sk_cta = [&](int64_t x) { return static_cast<int>(((x + 1) * G - 1) / T); };
    int segs_cta = 1, segs_tile = 1;
    for (int c = 0; c < G; ++c) {
      const int64_t a = static_cast<int64_t>(c) * T / G, b = static_cast<int64_t>(c + 1) * T / G;
      if (b > a) segs_cta = std::max(segs_cta, static_cast<int>((b - 1) / pl.KB - a / pl.KB + 1));
    }
    for (int64_t t = 0; t < tiles; ++t)
      segs_tile = std::max(segs_tile, sk_cta(t * pl.KB + pl.KB - 1) - sk_cta(t * pl.KB) + 1);
    const double cta_bw = 35e9, hbm_eff = 6.0e12;
    auto rate = [&](int64_t active) { return std::min(cta_bw, hbm_eff / static_cast<double>(active)); };
    // the uniform plan in the same terms: the busiest CTA's K blocks, plus its exchange or sum
    const int64_t u_waves = pl.cluster ? ceil_div(tiles, std::max<int64_t>(1, pl.grid / pl.splits))
                                       : ceil_div(static_cast<int64_t>(pl.units), pl.grid);
    double t_u = u_waves * pl.kb_per_split * kb_bytes / rate(pl.grid);
    if (pl.splits > 1) t_u += pl.cluster ? 1.5e-6 : pl.splits * part_bytes / red_bw;
    double t_sk = static_cast<double>(ceil_div(T, G)) * kb_bytes / rate(G);
    if (segs_tile > 1) t_sk += 1.0e-6 + segs_tile * part_bytes / red_bw;
    if (sk_opt == 2 || t_sk < 0.95 * t_u) {
      pl.sk = 1;
      pl.sk_total = static_cast<int>(T);
      pl.splits = 1;
      pl.kb_per_split = pl.KB;
      pl.cluster = 0;
      pl.grid = G;
      pl.units = G * segs_cta;
      pl.counters_bytes = segs_tile > 1 ? kCounterBytes : 0;
      pl.ws_bytes = segs_tile > 1 ? pl.counters_bytes + static_cast<size_t>(pl.units) * 128 * bt * 4 : 0;
      best_t = t_sk;
    }
  }
  if (t_model) *t_model = best_t;
  return pl;
}

static GemmPlan plan_mx(int64_t M, int64_t N, int64_t K, int sms, bool a4) {
  int bt = options().w4a8_token_tile;
  if (a4 && bt != 0 && bt < 128 && M > bt) bt = 0;   // a forced small tile must hold every token
  if (a4 && bt == 192) bt = 0;                        // W4A4 tiles start on 128-token scale atoms
  if (bt != 0) return plan_mx_bt(M, N, K, sms, a4, bt, nullptr);
  // 33..64 tokens against a narrow weight (few 128-row tiles) run as two
  // 32-token tiles: twice the tiles to spread over the SMs (measured: M=64,
  // 2048x5120 9.2 vs 10.2 us; at 5120x17408 the 64-token tile wins, 19.4 vs
  // 25.3 us).
  if (M <= 128) {
    bt = M <= 16 ? 16 : M <= 32 ? 32 : M <= 64 ? ((!a4 && ceil_div(N, 128) <= 24) ? 32 : 64) : 128;
    return plan_mx_bt(M, N, K, sms, a4, bt, nullptr);
  }
  double t256 = 0.0, t192 = 0.0;
  const GemmPlan p256 = plan_mx_bt(M, N, K, sms, a4, 256, &t256);
  if (a4) return p256;
  const GemmPlan p192 = plan_mx_bt(M, N, K, sms, a4, 192, &t192);
  return t192 < t256 ? p192 : p256;
}

GemmPlan plan_w4a8(int64_t M, int64_t N, int64_t K, int sms) { return plan_mx(M, N, K, sms, false); }
GemmPlan plan_w4a4(int64_t M, int64_t N, int64_t K, int sms) { return plan_mx(M, N, K, sms, true); }

int launch_gemm_w4a8(const uint8_t *q, const float *s, const uint8_t *packed, int64_t M, int64_t N, int64_t K,
                     uint16_t *c, int64_t ldc, void *ws, const GemmPlan &pl, cudaStream_t st) {
  switch (pl.BT) {
    case 16: return w4a8::launch_bt<16, false>(q, s, nullptr, packed, M, N, K, c, ldc, ws, pl, st);
    case 32: return w4a8::launch_bt<32, false>(q, s, nullptr, packed, M, N, K, c, ldc, ws, pl, st);
    case 64: return w4a8::launch_bt<64, false>(q, s, nullptr, packed, M, N, K, c, ldc, ws, pl, st);
    case 128: return w4a8::launch_bt<128, false>(q, s, nullptr, packed, M, N, K, c, ldc, ws, pl, st);
    case 192: return w4a8::launch_bt<192, false>(q, s, nullptr, packed, M, N, K, c, ldc, ws, pl, st);
    case 256: return w4a8::launch_bt<256, false>(q, s, nullptr, packed, M, N, K, c, ldc, ws, pl, st);
    default: return R4_ERR_INVALID_ARG;
  }
}

int launch_gemm_w4a4(const uint8_t *q, const uint8_t *q_scale, const uint8_t *packed, int64_t M, int64_t N,
                     int64_t K, uint16_t *c, int64_t ldc, void *ws, const GemmPlan &pl, cudaStream_t st) {
  switch (pl.BT) {
    case 16: return w4a8::launch_bt<16, true>(q, nullptr, q_scale, packed, M, N, K, c, ldc, ws, pl, st);
    case 32: return w4a8::launch_bt<32, true>(q, nullptr, q_scale, packed, M, N, K, c, ldc, ws, pl, st);
    case 64: return w4a8::launch_bt<64, true>(q, nullptr, q_scale, packed, M, N, K, c, ldc, ws, pl, st);
    case 128: return w4a8::launch_bt<128, true>(q, nullptr, q_scale, packed, M, N, K, c, ldc, ws, pl, st);
    case 256: return w4a8::launch_bt<256, true>(q, nullptr, q_scale, packed, M, N, K, c, ldc, ws, pl, st);
    default: return R4_ERR_INVALID_ARG;
  }
}

}  // namespace r4
