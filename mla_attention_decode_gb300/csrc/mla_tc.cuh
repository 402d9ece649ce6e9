// mla_tc.cuh -- split-K MLA decode for e4m3 and e2m1 (MXFP4) KV on the
// 5th-generation tensor cores (tcgen05, accumulators in tensor memory), sm_103a.
//
// Same contract as the split kernel in mla_stage1.cuh (kernelindex
// "amd-mixed-mla" submission 593653, "Slow fallback" for the definition and
// "_flash_fp8_split_s1" for the split form; submission 754939 "Stage 1" for the
// MXFP4 layout): per work unit, softmax attention of the 16 query heads over a
// contiguous range of KV rows; final bf16 output and lse for unsplit
// sequences, fp32 partials and lse for split ones.
//
// Per 128-row tile t of a unit (one persistent CTA per SM: 8 warps for e4m3, 16 for MXFP4):
//   scores  S^T[128 rows x 32] = K_t[128 x 576] . [Q_hi | Q_lo]^T   (tcgen05 kind::f8f6f4,
//           18 k32 steps; K straight from the TMA stage, K-major, 64 B swizzle;
//           the query as two e4m3 terms x = hi + lo with a power-of-two scale
//           per head, 32 "columns" = 16 heads x 2 terms, in TMEM)
//   softmax one thread per row reads its 32 accumulators, builds the scores,
//           exponentials and row sums, and writes P^T[128 rows x 32] =
//           [P_hi | P_lo] (two e4m3 terms) as the MN-major B operand
//   P.V     O^T[512 features x 32] += V_t^T[512 x 128] . P^T   (4 blocks of 128
//           features x 4 k32 steps; V^T read MN-major from the same stage --
//           V is the first 512 columns of K -- so each KV byte is read from HBM
//           once per unit), O^T resident in TMEM across the unit's tiles
// The running max is applied lazily: P = 2^(s - m_ref) with m_ref raised (and
// O^T, l rescaled in place) only when some score of a head exceeds m_ref by more
// than 8 (log2 units), which keeps P <= 256 inside e4m3 range.  Deciding that
// takes one OR over the tile's rows; the tile max itself is reduced only for
// the heads that rise (always on a unit's first tile).  Scores are in log2
// units: s = (q . k) * sm_scale * log2(e) * kv_scale.
//
// Warp roles: 0 TMA producer (9 column boxes of 64 B x 128 rows per tile: the
// 8 V blocks in pairs into a ring of 11 pair slots, each released by the
// commit after its P.V block, the rope block into a ring of 2); 1 QK issuer and
// TMEM owner; 2 P.V issuer (two issuing threads: one thread cannot issue these
// small MMAs as fast as the tensor pipe retires them); 3 query loader (the
// query image prepared by mla_prep_q_kernel, two bulk copies per unit); 4-7
// softmax, O^T rescale and the unit epilogue (warp w reads TMEM lanes
// [32 (w mod 4), +32)).  Hand-offs are mbarriers (TMA transaction bytes,
// tcgen05.commit, thread arrivals).
//
// Two query tokens per unit (kTok = 2, e4m3; several tokens per sequence,
// the causal reading): each tile feeds two QKs and two P.V chains, one per
// token, into their own TMEM columns, and warps 8-11 form a second softmax
// group for token 1, so the cache rows are read once for both tokens.  Token
// 0 does not see its sequence's last row (token 1's own entry).
//
// MXFP4 KV (kMx): rows arrive packed (288 B of e2m1 pairs, element 2i in the low
// nibble of byte i) by 1-D bulk copies of 64-row halves into a staging ring,
// and eight converter warps (8-15, four per half tile) write them into the same e4m3 ring layout
// the tensor cores read (8 pair slots: two whole tiles, so that converting
// tile t only waits for the P.V of tile t-2).  Per row, with G = the largest of its 18 e8m0 bytes,
// element n * 2^(e-127) becomes the e4m3 value n * 2^(e-G) (exact while the
// row's block exponents lie within 8 of G; smaller ones round to e4m3's
// subnormal grid), through an 8-entry magnitude table per shift applied with
// prmt.  2^(G-127) goes into the row's score factor, and into P for P.V
// relative to a running per-unit reference Gv (raised lazily like the softmax
// reference, with O^T rescaled); the output is O^T 2^Gv / l.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>

#include "mla_common.cuh"

namespace mla {
namespace tcfp8 {

constexpr int kTileRows = 128;
constexpr int kChunkBytes = kTileRows * 64;  // one 64-byte feature column block of a tile
constexpr int kPairBytes = 2 * kChunkBytes;  // two column blocks = features [128 f, 128 f + 128)
// kTok: query tokens one work unit serves (2: the fused two-token e4m3 form,
// which holds a second query image and a second pair of P buffers in shared
// memory at the cost of two ring slots).  kPath: which instance -- the
// contiguous cache and pages of 64 rows or more (kPathRows), pages of fewer
// rows (kPathSmallPages), or MXFP4 scores from block-scaled MMAs on the e2m1
// tile itself (kPathBlockScaled; otherwise MXFP4 is converted to e4m3 from a
// staging ring for both MMAs).
constexpr int kPathRows = 0, kPathSmallPages = 1, kPathBlockScaled = 2;
template <bool kMx, int kTok = 1, int kPath = kPathRows>
struct Geo {
  static_assert(kTok == 1 || (kTok == 2 && !kMx), "two tokens per unit: e4m3 KV only");
  static_assert(kPath != kPathBlockScaled || (kMx && kTok == 1), "block-scaled scores: MXFP4, one token");
  static constexpr bool bs = kPath == kPathBlockScaled;
  static constexpr int pair_slots = kMx ? (bs ? 10 : 8) : (kTok == 1 ? 11 : 9);  // ring of column-block pairs (4 per tile)
  // e4m3, one token per unit: a separate epilogue group (warps 8-11) drains
  // each unit's O^T from its own TMEM buffer, two buffers in turn, so that the
  // softmax warps and the next unit's P.V do not wait for the epilogue
  static constexpr bool epi = !kMx && kTok == 1;
  // roles: 4 single-thread warps, 4 softmax warps per token, MXFP4: 8 converter
  // warps, e4m3 one token: 4 epilogue warps
  static constexpr int threads = kMx ? 512 : 384;
  static constexpr int max_units = kMx ? kMaxUnitsPerCtaMx : kMaxUnitsPerCta;  // work units one CTA may own
};
constexpr int kRopeSlots = 2;                // ring of the rope column block (features 512..575)
constexpr int kQsBytes = 9 * 32 * 64;        // two-term query: 32 rows x 576 B, K-major, 64 B swizzle
constexpr int kPBytes = kTileRows * 32;      // two-term P^T: 128 rows x 32 B, MN-major, 32 B swizzle
constexpr int kHalfRows = 64;                        // MXFP4 staging unit: 64 packed rows
constexpr int kPackedRowBytes = 288;
constexpr int kStageBytes = kHalfRows * kPackedRowBytes;  // 18 KB
constexpr int kStageSlots = 3;
// block-scaled MXFP4: the rope block's packed bytes (128 rows x 32 B) are staged
// for the converters, which lay them out as the tensor core's 4-bit operand;
// the tile's scale bytes go to shared memory as five 512-byte chunks of 4
// K-blocks (the 32 x 128-bit source of one tcgen05.cp each: chunk word
// (m mod 32) x 4 + m / 32 holds the scale bytes of row m)
constexpr int kRopeStageBytes = kTileRows * 32;
constexpr int kSfChunks = 5;
constexpr int kSfTileBytes = kSfChunks * 512;
// TMEM columns: the S^T double buffer [blk (t mod 2), +blk), then O^T, 4
// feature blocks of blk columns; token i of a unit owns columns [32 i, +32) of
// each buffer and block.  With a separate epilogue group (one token) there are
// two O^T buffers, obuf columns apart, used by a CTA's units in turn.
template <int kTok>
struct Tmem {
  static constexpr uint32_t blk = 32 * kTok;
  static constexpr uint32_t cols = 512;
  static constexpr uint32_t s = 0;
  static constexpr uint32_t o = 2 * blk;
  static constexpr uint32_t obuf = 4 * blk;
  static_assert(kTok == 2 || o + 2 * obuf <= cols, "two O^T buffers");
  // block-scaled MXFP4 (one O^T buffer): the A scale factors of tile t at
  // sfa + 32 (t mod 2), chunk g at +4 g (4 columns, replicated over the four
  // lane quarters), the B scale factors (all 2^0) at sfb
  static constexpr uint32_t sfa = 256;
  static constexpr uint32_t sfb = 320;
};
constexpr float kRescaleLog2 = 8.f;
constexpr uint32_t kBarSoftmax = 1;  // named barrier of softmax group 0 (128 threads); group 1: 2
constexpr uint32_t kIdescQK = tc::idesc_e4m3(128, 32, 0, 0);
constexpr uint32_t kIdescPV = tc::idesc_e4m3(128, 32, 1, 1);
// two tokens per unit: one MMA with N = 64 covers both tokens' columns
constexpr uint32_t kIdescQK2 = tc::idesc_e4m3(128, 64, 0, 0);
constexpr uint32_t kIdescPV2 = tc::idesc_e4m3(128, 64, 1, 1);


__host__ __device__ constexpr int round_up_1024(int v) { return (v + 1023) / 1024 * 1024; }
template <bool kMx, int kTok = 1, int kPath = kPathRows>
struct Layout {
  using G = Geo<kMx, kTok, kPath>;
  static constexpr int kPairSlots = G::pair_slots;
  static constexpr int pairs = 0;                             // 1024-aligned
  static constexpr int rope = pairs + kPairSlots * kPairBytes;
  // MXFP4: packed rows (staging ring), or the rope blocks (block-scaled)
  static constexpr int stage = rope + kRopeSlots * kChunkBytes;
  static constexpr int sf = stage + (kMx ? (G::bs ? kRopeSlots * kRopeStageBytes : kStageSlots * kStageBytes) : 0);
  static constexpr int sfb = sf + (G::bs ? 2 * kSfTileBytes : 0);  // block-scaled: [2 tiles] A chunks, then B
  static constexpr int qs = round_up_1024(sfb + (G::bs ? 512 : 0));
  static constexpr int pb = qs + kQsBytes * kTok;             // [2 tiles][kTok]
  static constexpr int rq = pb + 2 * kPBytes * kTok;          // float [kTok][16] score factor per head
  static constexpr int red = rq + 16 * 4 * kTok;              // float [2][4 warps][16 kTok]
  static constexpr int gred = red + 2 * 4 * 16 * 4 * kTok;    // int [2][4] tile max of the row exponents
  static constexpr int grow = gred + 2 * 4 * 4;               // int8 [2][128] row exponent G - 127 (MXFP4)
  static constexpr int lut = grow + (kMx ? 2 * 128 : 0);      // u8 [32][8] e2m1 magnitude -> e4m3 per shift
  static constexpr int hand = lut + (kMx ? 256 : 0);          // float [2][32] l, m handed to the epilogue group
  static constexpr int units = hand + (G::epi ? 256 : 0);
  static constexpr int bars = units + G::max_units * (int)sizeof(UnitDesc);
  // the epilogue group's four (e4m3, one token), then the two of block-scaled MXFP4
  static constexpr int nbars = G::bs ? 55 : (G::epi ? 53 : 49);
  static constexpr int misc = bars + nbars * 8;  // tmem slot, abort flag, unit count
  static constexpr int total = misc + 16;
};

// mbarrier slots
enum {
  kPairFull = 0,    // [<=11] TMA bytes of a V column-block pair (e4m3)
  kPairEmpty = 11,  // [<=11] commit after the P.V block that read it
  kRopeFull = 22,   // [2]  TMA bytes of a rope column block
  kRopeEmpty = 24,  // [2]  commit after the QK that read it
  kQFull = 26,      // query of the next unit copied in (transaction bytes)
  kQEmpty = 27,     // commit after the unit's last QK
  kSFull = 28,      // [2]  commit after QK
  kSEmpty = 30,     // [2]  softmax read S (4 warps)
  kPFull = 32,      // [2]  P written, O^T rescaled (4 warps)
  kODone = 34,      // commit after each tile's P.V
  kOFree = 35,      // unit epilogue read O^T (4 warps)
  kRFree = 36,      // softmax copied the unit's score factors (4 warps)
  kOLast = 37,      // commit after a unit's last P.V (once per unit with tiles)
  kFinal = 38,      // commits after both issuers' last operations (count 2)
  kPFree = 39,      // [2]  commit after the P.V that read P buffer t mod 2
  kStageFull = 41,  // [3]  MXFP4: bytes of a staged half tile (or the producer's arrival)
  kStageEmpty = 44, // [3]  MXFP4: the converter warps of that half read it (4 warps)
  kConvFull = 47,   // [2]  MXFP4: tile t converted into the ring (8 warps)
  kOFree2 = 49,     // epilogue group: kOFree of the second O^T buffer
  kOLast2 = 50,     // epilogue group: kOLast of the second O^T buffer
  kEpiReady = 51,   // [2]  epilogue group: a unit's l and m handed over, per O^T buffer (1)
  kConvQK = 53,     // [2]  block-scaled MXFP4: tile t's scale chunks, row exponents and rope block written (8 warps)
};
// block-scaled MXFP4 reuses the staging barriers for the rope block: kStageFull
// + (t mod 2) counts its TMA bytes, kStageEmpty + (t mod 2) the 8 converter
// warps that laid it out
__device__ __forceinline__ int ofree_bar(int obuf) { return obuf ? kOFree2 : kOFree; }
__device__ __forceinline__ int olast_bar(int obuf) { return obuf ? kOLast2 : kOLast; }


struct Ctx {
  uint8_t* smem;
  const UnitDesc* units;
  int nunits;
  uint64_t* bar;
  volatile int* abort_flag;
  uint32_t tmem;
  int early_row;  // one token, contiguous cache: the first tile's row, its copy (e4m3: the tile; converted
                  // MXFP4: its two staging halves) issued before the unit scan (-1: none)
};

__device__ __forceinline__ int tiles_of(const UnitDesc& d) { return (d.end - d.start + kTileRows - 1) / kTileRows; }

// ------------------------------------------------------------------ producer
// Column blocks of tile t: pair f (features [128 f, 128 f + 128)) goes to pair
// slot (4t + f) mod S (S = 11 for e4m3, 9 with two tokens, 10 for block-scaled
// MXFP4, 8 for MXFP4 converted from staging), the rope block to rope
// slot t mod 2; each slot is re-filled as soon as the MMA that read it has
// completed.
template <bool kMx, int kTok = 1, int kPath = kPathRows>
__device__ __forceinline__ int pair_slot(int t, int f) { return (4 * t + f) % Geo<kMx, kTok, kPath>::pair_slots; }
template <bool kMx, int kTok = 1, int kPath = kPathRows>
__device__ __forceinline__ int pair_use(int t, int f) { return (4 * t + f) / Geo<kMx, kTok, kPath>::pair_slots; }
template <bool kMx, int kTok = 1, int kPath = kPathRows>
__device__ __forceinline__ int wrap_slot(int s) {
  return s >= Geo<kMx, kTok, kPath>::pair_slots ? s - Geo<kMx, kTok, kPath>::pair_slots : s;
}

// The CTA's tiles in order (unit by unit): each tile's first row-space
// position and its unit's end.
struct TileWalk {
  int k = 0, t0 = -1;
  __device__ bool next(const Ctx& x, int& tile0, int& end) {
    while (k < x.nunits) {
      const UnitDesc d = x.units[k];
      if (t0 < 0) t0 = d.start;
      if (t0 >= d.end) {
        ++k;
        t0 = -1;
        continue;
      }
      tile0 = t0;
      end = d.end;
      t0 += kTileRows;
      return true;
    }
    return false;
  }
};

// Cache rows of a tile: one 128-row box at r0, or (64-row pages) two 64-row
// boxes at r0 and r1, the second only when the tile has rows there (r1 < 0).
struct TileRows {
  int r0, r1;
};
__device__ __forceinline__ TileRows tile_rows(const Stage1Params& p, int t0, int end) {
  TileRows r;
  r.r0 = cache_row(p, t0);
  r.r1 = (p.paged && p.page_shift == 6 && t0 + 64 < end) ? cache_row(p, t0 + 64) : -1;
  return r;
}

template <int kTok>
__device__ void producer_e4m3(const Stage1Params& p, const Ctx& x) {
  using L = Layout<false, kTok>;
  constexpr int kPairSlots = Geo<false, kTok>::pair_slots;
  const uint64_t pol = policy_evict_first();  // KV rows are read once
  const bool paged64 = p.paged && p.page_shift == 6;
  // one 64-byte column block of the tile (and the bytes it brings)
  auto load_block = [&](uint8_t* dst, int col, const TileRows& r, uint64_t* bar) {
    if (!paged64) {
      tma_load_2d(dst, &p.tmap_kv64, col, r.r0, bar, pol);
    } else {
      tma_load_2d(dst, &p.tmap_kv16, col, r.r0, bar, pol);
      if (r.r1 >= 0) tma_load_2d(dst + 64 * 64, &p.tmap_kv16, col, r.r1, bar, pol);
    }
  };
  int armed[kPairSlots + kRopeSlots];
  for (int i = 0; i < kPairSlots + kRopeSlots; ++i) armed[i] = 0;
  // the cache rows of the next tile are looked up one tile ahead (a paged
  // cache reads the page table; otherwise they are the tile's own rows)
  TileWalk walk;
  int nt0 = 0, nend = 0;
  bool have = walk.next(x, nt0, nend);
  TileRows nrows = have ? tile_rows(p, nt0, nend) : TileRows{0, -1};
  bool early_pending = x.early_row >= 0;  // the tile copied on entry is not yet accounted for
  for (int it = 0; have && !*x.abort_flag; ++it) {
    if (it == 0 && early_pending) {
      // the kernel prologue copied the tile the plan names into pair slots 0..3
      // and rope slot 0; the scan must agree (it does unless the device
      // kv_indptr differs from the plan's), else flag it and stop
      early_pending = false;
      for (int f = 0; f < 4; ++f) ++armed[f];
      ++armed[kPairSlots];
      if (!paged64 && nrows.r0 == x.early_row) {
        have = walk.next(x, nt0, nend);
        if (have) nrows = tile_rows(p, nt0, nend);
        continue;
      }
      flag_error(p.ws_err, kErrDeviceIndex, kTagFirstTile, x.early_row);
      *x.abort_flag = 1;
      break;
    }
    const TileRows rows = nrows;
    have = walk.next(x, nt0, nend);
    if (have) nrows = tile_rows(p, nt0, nend);
    const uint32_t block_bytes = (paged64 && rows.r1 < 0) ? kChunkBytes / 2 : kChunkBytes;
    for (int f = 0; f < 4; ++f) {
      const int sl = pair_slot<false, kTok>(it, f), use = pair_use<false, kTok>(it, f);
      if (use >= 1) wait_phase(&x.bar[kPairEmpty + sl], (use - 1) & 1, x.abort_flag, p.ws_err);
      if (*x.abort_flag) break;
      uint8_t* dst = x.smem + L::pairs + sl * kPairBytes;
      mbar_arrive_expect_tx(&x.bar[kPairFull + sl], 2 * block_bytes);
      load_block(dst, 128 * f, rows, &x.bar[kPairFull + sl]);
      load_block(dst + kChunkBytes, 128 * f + 64, rows, &x.bar[kPairFull + sl]);
      ++armed[sl];
      if (it == 0 && f == 0) trace_stamp(p, kTrFirstLoad);
    }
    const int rs = it % kRopeSlots, ruse = it / kRopeSlots;
    if (ruse >= 1) wait_phase(&x.bar[kRopeEmpty + rs], (ruse - 1) & 1, x.abort_flag, p.ws_err);
    if (*x.abort_flag) break;
    mbar_arrive_expect_tx(&x.bar[kRopeFull + rs], block_bytes);
    load_block(x.smem + L::rope + rs * kChunkBytes, 512, rows, &x.bar[kRopeFull + rs]);
    ++armed[kPairSlots + rs];
  }
  if (early_pending) {
    // the plan named a tile that this CTA's scan does not have: flag it, and
    // let the copy land before leaving
    flag_error(p.ws_err, kErrDeviceIndex, kTagFirstTile, x.early_row);
    *x.abort_flag = 1;
    for (int f = 0; f < 4; ++f) ++armed[f];
    ++armed[kPairSlots];
  }
  if (*x.abort_flag) {
    // a wait gave up somewhere: never leave with copies in flight (bounded wait per slot)
    for (int i = 0; i < kPairSlots + kRopeSlots; ++i) {
      if (armed[i] == 0) continue;
      uint64_t* bar = i < kPairSlots ? &x.bar[kPairFull + i] : &x.bar[kRopeFull + i - kPairSlots];
      const uint64_t t0 = global_timer_ns();
      while (!mbar_try_wait(bar, (armed[i] - 1) & 1) && global_timer_ns() - t0 < kWaitTimeoutNs) {
      }
    }
  }
}


// Pages of fewer than 64 rows: a tile's rows lie in many pages, so the 32
// lanes of warp 0 fetch them together, once lane 0 has waited for the tile's
// slots and armed their barriers.  The pair slots hold 128-byte rows (both
// column blocks of a pair side by side, 128-byte swizzle; the MMA descriptors
// of this instance say so), so that one copy brings both blocks of a pair.
// - Pages of 8 to 32 rows: lane l < 128 / P looks up page l of the tile and
//   issues one box of 128 B x P rows per pair and one of 64 B x P rows for the
//   rope block: 5 x 128 / P copies per tile.
// - Pages of 1 to 4 rows: lane l looks up the cache rows of tile rows
//   [4 l, 4 l + 4) and issues one four-row gather per pair (128 B wide) and
//   one for the rope block (64 B wide), the maps' boxes one row high: 160
//   copies per tile.
// Rows past the unit's end repeat its last row, or page (the softmax masks
// them and zeroes their V part).
template <int kTok>
__device__ void producer_e4m3_gather(const Stage1Params& p, const Ctx& x, int lane) {
  using L = Layout<false, kTok>;
  constexpr int kPairSlots = Geo<false, kTok>::pair_slots;
  const uint64_t pol = policy_evict_first();  // KV rows are read once
  int armed[kPairSlots + kRopeSlots];         // lane 0: fills issued per slot
  for (int i = 0; i < kPairSlots + kRopeSlots; ++i) armed[i] = 0;
  const bool per_page = p.page_shift >= 3;
  const int page_mask = (1 << p.page_shift) - 1;
  TileWalk walk;
  int t0 = 0, end = 0;
  for (int it = 0; walk.next(x, t0, end); ++it) {
    int cr[4];
    if (per_page) {
      // the first cache row of page `lane` of the tile (tiles start on page boundaries)
      const int v = min(t0 + (lane << p.page_shift), end - 1);
      cr[0] = cache_row(p, v) - (v & page_mask);
    } else {
#pragma unroll
      for (int j = 0; j < 4; ++j) cr[j] = cache_row(p, min(t0 + 4 * lane + j, end - 1));
    }
    int sl[4];
#pragma unroll
    for (int f = 0; f < 4; ++f) sl[f] = pair_slot<false, kTok>(it, f);
    const int rs = it % kRopeSlots;
    if (lane == 0) {
#pragma unroll
      for (int f = 0; f < 4; ++f) {
        const int use = pair_use<false, kTok>(it, f);
        if (use >= 1) wait_phase(&x.bar[kPairEmpty + sl[f]], (use - 1) & 1, x.abort_flag, p.ws_err);
      }
      const int ruse = it / kRopeSlots;
      if (ruse >= 1) wait_phase(&x.bar[kRopeEmpty + rs], (ruse - 1) & 1, x.abort_flag, p.ws_err);
      if (!*x.abort_flag) {
#pragma unroll
        for (int f = 0; f < 4; ++f) {
          mbar_arrive_expect_tx(&x.bar[kPairFull + sl[f]], 2 * kChunkBytes);
          ++armed[sl[f]];
        }
        mbar_arrive_expect_tx(&x.bar[kRopeFull + rs], kChunkBytes);
        ++armed[kPairSlots + rs];
      }
    }
    if (__shfl_sync(0xffffffffu, lane == 0 ? *x.abort_flag : 0, 0)) break;
    if (per_page) {
      if (lane < (kTileRows >> p.page_shift)) {
        // page `lane`: tile rows [lane P, lane P + P)
        const int r_tile = lane << p.page_shift;
#pragma unroll
        for (int f = 0; f < 4; ++f)
          tma_load_2d(x.smem + L::pairs + sl[f] * kPairBytes + r_tile * 128, &p.tmap_kv16, 128 * f, cr[0],
                      &x.bar[kPairFull + sl[f]], pol);
        tma_load_2d(x.smem + L::rope + rs * kChunkBytes + r_tile * 64, &p.tmap_kv64, 512, cr[0],
                    &x.bar[kRopeFull + rs], pol);
      }
    } else {
      // tile rows [4 lane, 4 lane + 4)
#pragma unroll
      for (int f = 0; f < 4; ++f)
        tma_gather4(x.smem + L::pairs + sl[f] * kPairBytes + 512 * lane, &p.tmap_kv16, 128 * f, cr[0], cr[1], cr[2],
                    cr[3], &x.bar[kPairFull + sl[f]], pol);
      tma_gather4(x.smem + L::rope + rs * kChunkBytes + 256 * lane, &p.tmap_kv64, 512, cr[0], cr[1], cr[2], cr[3],
                  &x.bar[kRopeFull + rs], pol);
    }
    if (it == 0 && lane == 0) trace_stamp(p, kTrFirstLoad);
  }
  if (lane == 0 && *x.abort_flag) {
    // a wait gave up somewhere: never leave with copies in flight (bounded wait per slot)
    for (int i = 0; i < kPairSlots + kRopeSlots; ++i) {
      if (armed[i] == 0) continue;
      uint64_t* bar = i < kPairSlots ? &x.bar[kPairFull + i] : &x.bar[kRopeFull + i - kPairSlots];
      const uint64_t tw = global_timer_ns();
      while (!mbar_try_wait(bar, (armed[i] - 1) & 1) && global_timer_ns() - tw < kWaitTimeoutNs) {
      }
    }
  }
}

// ------------------------------------------------------- MXFP4 converters
// Walks the CTA's half tiles in order: unit k, rows [t0 + 64 h, ...) of its
// tile starting at t0.
struct HalfCursor {
  int k = 0, t0 = -1, h = 0;
  __device__ bool next(const Ctx& x, int& r0, int& rows) {
    while (k < x.nunits) {
      const UnitDesc d = x.units[k];
      if (t0 < 0) t0 = d.start;
      if (t0 >= d.end) {
        ++k;
        t0 = -1;
        h = 0;
        continue;
      }
      r0 = t0 + h * kHalfRows;
      rows = max(0, min(kHalfRows, d.end - r0));
      if (++h == 2) {
        h = 0;
        t0 += kTileRows;
      }
      return true;
    }
    return false;
  }
};

// ------------------------------------------------------- MXFP4 producers
// Block-scaled MXFP4 (contiguous caches, pages of 64 rows or more), one lane:
// per tile, each 128-feature pair of e2m1 as one box of the 16U4_ALIGN16B map
// (tmap_kv64: 16 elements = 8 packed bytes land in 16 bytes of shared memory,
// the upper 8 zero, which is the tensor core's layout for a 4-bit operand;
// the barrier counts the 8 packed bytes), into the pair ring as 128-byte rows
// with the 128-byte swizzle; the rope block's 32 packed bytes a row as one box
// of the byte map (tmap_kv16) into a staging slot, which the converter warps
// lay out for the tensor core.  Pages of 64 rows: two 64-row boxes per tile.  The scale rows of the tile
// three ahead are prefetched into L2 for the converter warps.
static __device__ void producer_mx_bs(const Stage1Params& p, const Ctx& x) {
  using L = Layout<true, 1, kPathBlockScaled>;
  constexpr int kPairSlots = Geo<true, 1, kPathBlockScaled>::pair_slots;
  const uint64_t pol = policy_evict_first();  // KV rows are read once
  const bool paged64 = p.paged && p.page_shift == 6;
  const uint8_t* sc = static_cast<const uint8_t*>(p.kv_scale);
  const size_t ss = (size_t)p.scale_stride;
  const int cache_rows = p.paged ? (p.num_pages << p.page_shift) : p.total_kv;
  const size_t scale_end = ((size_t)cache_rows * ss) & ~(size_t)15;
  // one bulk L2 prefetch per box: the 16-byte-aligned part of its scale rows
  // that lies inside the tensor (the scale base is 16-byte aligned)
  auto prefetch_scales = [&](int c0, int rows) {
    if (c0 < 0 || rows <= 0) return;
    const size_t lo = ((size_t)c0 * ss) & ~(size_t)15;
    size_t hi = ((size_t)(c0 + rows) * ss + 15) & ~(size_t)15;
    if (hi > scale_end) hi = scale_end;
    if (hi > lo) bulk_prefetch_l2(sc + lo, (uint32_t)(hi - lo));
  };
  constexpr int kScaleAhead = 3;  // tiles
  TileWalk pre;
  auto prefetch_next = [&]() {
    int t0, end;
    if (!pre.next(x, t0, end)) return;
    const TileRows r = tile_rows(p, t0, end);
    if (!paged64) {
      prefetch_scales(r.r0, min(kTileRows, cache_rows - r.r0));
    } else {
      prefetch_scales(r.r0, 64);
      if (r.r1 >= 0) prefetch_scales(r.r1, 64);
    }
  };
  for (int i = 0; i < kScaleAhead; ++i) prefetch_next();
  int armed[kPairSlots + kRopeSlots];
  for (int i = 0; i < kPairSlots + kRopeSlots; ++i) armed[i] = 0;
  // the rope block of tile t + 2 is requested before the pairs of tile t: its
  // staging slot was laid out by the converters' step 1 for tile t, which
  // needs nothing requested later than tile t - 2, while the pairs of tile t
  // wait for the P.V of tiles t - 2 and t - 3
  TileWalk rope_walk;
  int rope_it = 0;
  auto request_rope = [&]() {
    int t0, end;
    if (!rope_walk.next(x, t0, end)) return;
    const TileRows rows = tile_rows(p, t0, end);
    const int rs = rope_it % kRopeSlots, ruse = rope_it / kRopeSlots;
    ++rope_it;
    if (ruse >= 1) wait_phase(&x.bar[kStageEmpty + rs], (ruse - 1) & 1, x.abort_flag, p.ws_err);
    if (*x.abort_flag) return;
    const uint32_t box_rows = (paged64 && rows.r1 < 0) ? 64u : 128u;
    uint8_t* dst = x.smem + L::stage + rs * kRopeStageBytes;
    mbar_arrive_expect_tx(&x.bar[kStageFull + rs], box_rows * 32);
    tma_load_2d(dst, &p.tmap_kv16, 256, rows.r0, &x.bar[kStageFull + rs], pol);
    if (paged64 && rows.r1 >= 0) tma_load_2d(dst + 64 * 32, &p.tmap_kv16, 256, rows.r1, &x.bar[kStageFull + rs], pol);
    ++armed[kPairSlots + rs];
  };
  request_rope();
  request_rope();
  TileWalk walk;
  int nt0 = 0, nend = 0;
  bool have = walk.next(x, nt0, nend);
  TileRows nrows = have ? tile_rows(p, nt0, nend) : TileRows{0, -1};
  for (int it = 0; have && !*x.abort_flag; ++it) {
    const TileRows rows = nrows;
    have = walk.next(x, nt0, nend);
    if (have) nrows = tile_rows(p, nt0, nend);
    prefetch_next();
    request_rope();
    if (*x.abort_flag) break;
    const uint32_t box_rows = (paged64 && rows.r1 < 0) ? 64u : 128u;  // rows the copies bring
    for (int f = 0; f < 4; ++f) {
      const int sl = pair_slot<true, 1, kPathBlockScaled>(it, f), use = pair_use<true, 1, kPathBlockScaled>(it, f);
      if (use >= 1) wait_phase(&x.bar[kPairEmpty + sl], (use - 1) & 1, x.abort_flag, p.ws_err);
      if (*x.abort_flag) break;
      uint8_t* dst = x.smem + L::pairs + sl * kPairBytes;
      mbar_arrive_expect_tx(&x.bar[kPairFull + sl], box_rows * 64);
      tma_load_3d(dst, &p.tmap_kv64, 0, f, rows.r0, &x.bar[kPairFull + sl], pol);
      if (paged64 && rows.r1 >= 0) tma_load_3d(dst + 64 * 128, &p.tmap_kv64, 0, f, rows.r1, &x.bar[kPairFull + sl], pol);
      ++armed[sl];
      if (it == 0 && f == 0) trace_stamp(p, kTrFirstLoad);
    }
  }
  if (*x.abort_flag) {
    // a wait gave up somewhere: never leave with copies in flight (bounded wait per slot)
    for (int i = 0; i < kPairSlots + kRopeSlots; ++i) {
      if (armed[i] == 0) continue;
      uint64_t* bar = i < kPairSlots ? &x.bar[kPairFull + i] : &x.bar[kStageFull + i - kPairSlots];
      const uint64_t t0 = global_timer_ns();
      while (!mbar_try_wait(bar, (armed[i] - 1) & 1) && global_timer_ns() - t0 < kWaitTimeoutNs) {
      }
    }
  }
}

// Converted MXFP4, contiguous caches and pages of 64 rows or more: half tiles
// (64 packed rows, 18 KB) into a ring of 3 staging slots by 1-D bulk copies (a
// half's rows are contiguous in the cache: a unit's rows, or one page of at
// least 64 rows); one lane issues them.  The rows' scale bytes are prefetched
// into L2 for the converter warps.  A half with no rows (the second half of a
// short tile) is signalled by a plain arrival.  With one token and a
// contiguous cache the kernel prologue has already copied the first tile's
// two halves (the plan's first row); the producer checks that row against its
// scan and goes on from the third half.
static __device__ void producer_mx(const Stage1Params& p, const Ctx& x) {
  using L = Layout<true>;
  const uint64_t pol = policy_evict_first();  // KV rows are read once
  const uint8_t* sc = static_cast<const uint8_t*>(p.kv_scale);
  const size_t ss = (size_t)p.scale_stride;
  int uses[kStageSlots] = {0, 0, 0};
  // the scale bytes of the half kScalePrefetch ahead go to L2 (the converters
  // read them a half ahead; this keeps those reads L2 hits)
  constexpr int kScalePrefetch = 6;
  // one bulk L2 prefetch per half: the 16-byte-aligned part of its scale rows
  // that lies inside the tensor (the base is 16-byte aligned)
  const int cache_rows = p.paged ? (p.num_pages << p.page_shift) : p.total_kv;
  const size_t scale_end = ((size_t)cache_rows * ss) & ~(size_t)15;
  auto prefetch_scales = [&](int c0, int rows) {
    if (rows <= 0) return;
    const size_t lo = ((size_t)c0 * ss) & ~(size_t)15;
    size_t hi = ((size_t)(c0 + rows) * ss + 15) & ~(size_t)15;
    if (hi > scale_end) hi = scale_end;
    if (hi > lo) bulk_prefetch_l2(sc + lo, (uint32_t)(hi - lo));
  };
  // cache rows are looked up one half before they are used (a paged cache
  // reads the page table; otherwise a half's cache rows are its own rows)
  HalfCursor pre;
  int pf_row = 0, pf_rows = 0;  // the half whose prefetch is issued next
  auto advance_prefetch = [&]() {
    prefetch_scales(pf_row, pf_rows);
    int r0, rows;
    pf_rows = pre.next(x, r0, rows) ? rows : 0;
    pf_row = pf_rows > 0 ? cache_row(p, r0) : 0;
  };
  for (int i = 0; i <= kScalePrefetch; ++i) advance_prefetch();
  HalfCursor cur;
  int nr0 = 0, nrows = 0;
  bool have = cur.next(x, nr0, nrows);
  int ncrow = (have && nrows > 0) ? cache_row(p, nr0) : 0;
  const bool early = x.early_row >= 0;  // the prologue copied the first tile's two halves
  for (int hh = 0; have && !*x.abort_flag; ++hh) {
    const int rows = nrows, crow = ncrow;
    have = cur.next(x, nr0, nrows);
    if (have) ncrow = nrows > 0 ? cache_row(p, nr0) : 0;
    const int sl = hh % kStageSlots, use = hh / kStageSlots;
    if (early && hh < 2) {
      // the scan must agree with the plan's first row (it does unless the
      // device kv_indptr differs from the plan's), else flag it and stop
      if (hh == 0 && (rows <= 0 || crow != x.early_row)) {
        flag_error(p.ws_err, kErrDeviceIndex, kTagFirstTile, x.early_row);
        *x.abort_flag = 1;
        uses[0] = uses[1] = 1;
        break;
      }
      ++uses[sl];
      advance_prefetch();
      continue;
    }
    if (use >= 1) wait_phase(&x.bar[kStageEmpty + sl], (use - 1) & 1, x.abort_flag, p.ws_err);
    if (*x.abort_flag) break;
    if (rows > 0) {
      mbar_arrive_expect_tx(&x.bar[kStageFull + sl], (uint32_t)(rows * kPackedRowBytes));
      bulk_g2s(x.smem + L::stage + sl * kStageBytes, p.kv + (size_t)crow * kPackedRowBytes,
               (uint32_t)(rows * kPackedRowBytes), &x.bar[kStageFull + sl], pol);
      if (hh == 0) trace_stamp(p, kTrFirstLoad);
    } else {
      mbar_arrive(&x.bar[kStageFull + sl]);
    }
    ++uses[sl];
    advance_prefetch();
  }
  if (early && uses[0] == 0) {
    // the plan named a tile that this CTA's scan does not have: flag it, and
    // let the two copies land before leaving
    flag_error(p.ws_err, kErrDeviceIndex, kTagFirstTile, x.early_row);
    *x.abort_flag = 1;
    uses[0] = uses[1] = 1;
  }
  if (*x.abort_flag) {
    // a wait gave up somewhere: never leave with copies in flight (bounded wait per slot)
    for (int i = 0; i < kStageSlots; ++i) {
      if (uses[i] == 0) continue;
      const uint64_t t0 = global_timer_ns();
      while (!mbar_try_wait(&x.bar[kStageFull + i], (uses[i] - 1) & 1) && global_timer_ns() - t0 < kWaitTimeoutNs) {
      }
    }
  }
}

// Converted MXFP4, pages of fewer than 64 rows: half tiles as above.  A half's rows
// lie in 64 / P pages, so the 32 lanes copy one page's rows each (two pages per
// lane for P = 1), through their own page-table lookups, once lane 0 has
// waited for the staging slot and armed its barrier; a half with no rows (the
// second half of a short tile) is signalled by a plain arrival.  No scale
// prefetch: the converters look up their rows' scales themselves.
static __device__ void producer_mx_rows(const Stage1Params& p, const Ctx& x, int lane) {
  using L = Layout<true, 1, kPathSmallPages>;
  const uint64_t pol = policy_evict_first();  // KV rows are read once
  int uses[kStageSlots] = {0, 0, 0};
  HalfCursor cur;
  int r0 = 0, rows = 0;
  for (int hh = 0; cur.next(x, r0, rows); ++hh) {
    const int sl = hh % kStageSlots, use = hh / kStageSlots;
    int armed_ok = 0;
    if (lane == 0) {
      if (use >= 1) wait_phase(&x.bar[kStageEmpty + sl], (use - 1) & 1, x.abort_flag, p.ws_err);
      if (!*x.abort_flag) {
        armed_ok = 1;
        if (rows > 0) {
          mbar_arrive_expect_tx(&x.bar[kStageFull + sl], (uint32_t)(rows * kPackedRowBytes));
          if (hh == 0) trace_stamp(p, kTrFirstLoad);
        } else {
          mbar_arrive(&x.bar[kStageFull + sl]);
        }
        ++uses[sl];
      }
    }
    if (!__shfl_sync(0xffffffffu, armed_ok, 0)) break;
    // page k of the half: rows [k P, k P + P) (halves start on page boundaries)
    for (int r = lane << p.page_shift; r < rows; r += 32 << p.page_shift) {
      const int n = min(1 << p.page_shift, rows - r);
      bulk_g2s(x.smem + L::stage + sl * kStageBytes + r * kPackedRowBytes,
               p.kv + (size_t)cache_row(p, r0 + r) * kPackedRowBytes, (uint32_t)(n * kPackedRowBytes),
               &x.bar[kStageFull + sl], pol);
    }
  }
  if (lane == 0 && *x.abort_flag) {
    // a wait gave up somewhere: never leave with copies in flight (bounded wait per slot)
    for (int i = 0; i < kStageSlots; ++i) {
      if (uses[i] == 0) continue;
      const uint64_t t0 = global_timer_ns();
      while (!mbar_try_wait(&x.bar[kStageFull + i], (uses[i] - 1) & 1) && global_timer_ns() - t0 < kWaitTimeoutNs) {
      }
    }
  }
}

// The 18 scale bytes of a row as nine pairs (byte 2i in bits 0-7 of e[i], byte
// 2i+1 in bits 8-15), by 16-bit loads when the row start is even; 127 for a row
// past the half's end.
__device__ __forceinline__ void load_row_scales(const uint8_t* sc, size_t ss, int grow_row, bool valid,
                                                uint32_t (&e)[9]) {
  const uint8_t* a = sc + (size_t)grow_row * ss;
  if (!valid) {
#pragma unroll
    for (int i = 0; i < 9; ++i) e[i] = 0x7f7fu;
  } else if ((reinterpret_cast<uintptr_t>(a) & 1) == 0) {
#pragma unroll
    for (int i = 0; i < 9; ++i) e[i] = __ldg(reinterpret_cast<const unsigned short*>(a) + i);
  } else {
#pragma unroll
    for (int i = 0; i < 9; ++i) e[i] = (uint32_t)__ldg(a + 2 * i) | ((uint32_t)__ldg(a + 2 * i + 1) << 8);
  }
}

// Eight e2m1 codes (one 32-bit word, element 2i in the low nibble of byte i)
// to eight e4m3 bytes for the shift whose magnitude table is (lo, hi).
__device__ __forceinline__ uint2 e2m1x8_to_e4m3(uint32_t w, uint32_t lut_lo, uint32_t lut_hi) {
  // prmt picks byte (nibble & 7) of {lut_lo, lut_hi} for each element; a
  // selector nibble with bit 3 (the e2m1 sign) set instead replicates the
  // picked byte's msb, which from 0x80808080 gives 0xff for a negative element
  // and 0x80 otherwise: bit 6 of that byte, moved up by one, is the e4m3 sign
  const uint32_t wm = w & 0x77777777u, w1 = w >> 16;
  const uint32_t m0 = prmt(lut_lo, lut_hi, wm), m1 = prmt(lut_lo, lut_hi, wm >> 16);
  const uint32_t s0 = prmt(0x80808080u, 0x80808080u, w), s1 = prmt(0x80808080u, 0x80808080u, w1);
  return make_uint2(m0 | ((s0 << 1) & 0x80808080u), m1 | ((s1 << 1) & 0x80808080u));
}

// Converted MXFP4: converter warp cw (0..7) converts half cw / 4 of every tile (tile rows
// [64 (cw / 4), +64)): rows [16 (cw % 4), +16) of that half.  Lane pair
// (2i, 2i+1) shares row 16 (cw % 4) + i, lane 2i + hp taking the row's blocks
// 2j + hp (j = 0..8).  Block 2j + hp holds features [64 j + 32 hp, +32),
// columns [32 hp, 32 hp + 32) of column block j, so the destination block of
// each is fixed at compile time.  Eight warps, two per SM sub-partition (one
// per half tile): the conversion is bound by each sub-partition's integer
// pipe, and a second warp keeps it busy while the first waits.
template <bool kSmallPages>
static __device__ void converter_mx(const Stage1Params& p, const Ctx& x, int cw, int lane) {
  using L = Layout<true>;
  const uint8_t* sc = static_cast<const uint8_t*>(p.kv_scale);
  const size_t ss = (size_t)p.scale_stride;
  const uint32_t lut0 = smem_u32(x.smem + L::lut), stage0 = smem_u32(x.smem + L::stage);
  const uint32_t pairs0 = smem_u32(x.smem + L::pairs), rope0 = smem_u32(x.smem + L::rope);
  int8_t* grow = reinterpret_cast<int8_t*>(x.smem + L::grow);
  const int hsel = cw >> 2;                                    // the half of every tile this warp converts
  const int lr = 16 * (cw & 3) + (lane >> 1), hp = lane & 1;  // row within the half, which half of the row
  HalfCursor cur, pre;
  int r0 = 0, rows = 0, pr0 = 0, prows = 0, pre_hh = 0;
  // the row's scale bytes are loaded one tile ahead of their use (the producer
  // has already brought them into L2, except for pages of fewer than 64 rows);
  // a half lies inside one page unless its pages are that small
  auto load_next_scales = [&](uint32_t (&dst)[9]) {
    while (pre.next(x, pr0, prows)) {
      if ((pre_hh++ & 1) != hsel) continue;  // the other half's rows
      const int crow = kSmallPages ? (lr < prows ? cache_row(p, pr0 + lr) : 0)
                                   : (prows > 0 ? cache_row(p, pr0) : 0) + lr;
      load_row_scales(sc, ss, crow, lr < prows, dst);
      return;
    }
  };
  uint32_t e_next[9];
#pragma unroll
  for (int i = 0; i < 9; ++i) e_next[i] = 0x7f7fu;
  load_next_scales(e_next);
  for (int hh = 0; cur.next(x, r0, rows) && !*x.abort_flag; ++hh) {
    const int it = hh >> 1, h = hh & 1;
    if (h != hsel) continue;
    uint32_t e[9];
#pragma unroll
    for (int i = 0; i < 9; ++i) e[i] = e_next[i];
    load_next_scales(e_next);
    {
      // the tile's ring slots must have been released by the MMAs that read them
#pragma unroll
      for (int f = 0; f < 4; ++f) {
        const int use = pair_use<true>(it, f);
        if (use >= 1)
          wait_phase(&x.bar[kPairEmpty + pair_slot<true>(it, f)], (use - 1) & 1, x.abort_flag, p.ws_err);
      }
      const int ruse = it / kRopeSlots;
      if (ruse >= 1) wait_phase(&x.bar[kRopeEmpty + it % kRopeSlots], (ruse - 1) & 1, x.abort_flag, p.ws_err);
    }
    const int sl = hh % kStageSlots;
    wait_phase(&x.bar[kStageFull + sl], (hh / kStageSlots) & 1, x.abort_flag, p.ws_err);
    const int row = h * kHalfRows + lr;  // row within the tile
    uint32_t g = 1;
#pragma unroll
    for (int i = 0; i < 9; ++i) g = max(g, max(e[i] & 0xffu, e[i] >> 8));
    const bool valid = lr < rows;
    if (hp == 0) grow[(it & 1) * 128 + row] = (int8_t)(valid ? (int)min(g, 254u) - 127 : 0);
    // a row past the end takes the all-zero table: its stale staging bytes
    // (in bounds) become zeros of either sign
    const uint32_t lutv = lut0 + (valid ? 0u : 128u);
    const uint32_t src = stage0 + sl * kStageBytes + lr * kPackedRowBytes + 16 * hp;
    uint4 w[9];
    uint2 lt[9];
#pragma unroll
    for (int j = 0; j < 9; ++j) {
      w[j] = lds128(src + 32 * j);
      const uint32_t eb = (e[j] >> (8 * hp)) & 0xffu;  // scale byte 2j + hp
      lt[j] = lds64(lutv + 8 * min(g - eb, 15u));
    }
    const uint32_t off0 = sw64_off(row, 32 * hp), off1 = sw64_off(row, 32 * hp + 16);
#pragma unroll
    for (int j = 0; j < 9; ++j) {
      const uint2 a = e2m1x8_to_e4m3(w[j].x, lt[j].x, lt[j].y), b = e2m1x8_to_e4m3(w[j].y, lt[j].x, lt[j].y);
      const uint2 c = e2m1x8_to_e4m3(w[j].z, lt[j].x, lt[j].y), d = e2m1x8_to_e4m3(w[j].w, lt[j].x, lt[j].y);
      const uint32_t base = j < 8 ? pairs0 + (uint32_t)(pair_slot<true>(it, j >> 1) * kPairBytes + (j & 1) * kChunkBytes)
                                  : rope0 + (uint32_t)((it % kRopeSlots) * kChunkBytes);
      sts128(base + off0, a.x, a.y, b.x, b.y);
      sts128(base + off1, c.x, c.y, d.x, d.y);
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&x.bar[kStageEmpty + sl]);
    tc::fence_proxy_async();  // the tensor core reads the ring through the async proxy
    __syncwarp();
    if (lane == 0) mbar_arrive(&x.bar[kConvFull + (it & 1)]);
  }
}

// Block-scaled MXFP4: converter warp cw (0..7) serves tile rows [16 cw, +16);
// lane 2i + hp takes row 16 cw + i and, of each of the row's 16 V blocks kb
// (32 features), the 16 features [32 kb + 16 hp, +16).  Per tile t:
//  1. for tile t + 1, first (so that its QK can overlap the conversion of
//     tile t): the row's scale bytes into that tile's five chunks, its row
//     exponent G - 127 (G: the largest scale byte of its 16 V blocks) and its
//     rope bytes laid out as the 4-bit operand (8 packed bytes, then 8 zero
//     bytes, per 16 elements) in the rope slot; then kConvQK;
//  2. once the QK of tile t is complete (its e2m1 bytes have been read), each
//     16-element group of the row's V blocks is rewritten in place as 16 e4m3
//     bytes n * 2^(e-G) (element n of a block with scale byte e; exact while
//     e is within 8 of G, smaller ones rounding to e4m3's subnormal grid) for
//     the P.V; then kConvFull.
// The scale chunks, rope slot and row exponents of tile t + 1 are those of
// tile t - 1: its QK completed before its conversion, and its softmax had
// read the row exponents (kSEmpty).  A row past the unit's end takes scale
// bytes 127 and the all-zero conversion table.
__device__ __forceinline__ uint32_t bs_scale_word(const uint32_t (&e)[9], int g) {
  return g < 4 ? (e[2 * g] | (e[2 * g + 1] << 16)) : (e[8] | 0x7f7f0000u);
}
static __device__ void converter_mx_bs(const Stage1Params& p, const Ctx& x, int cw, int lane) {
  using L = Layout<true, 1, kPathBlockScaled>;
  const uint8_t* sc = static_cast<const uint8_t*>(p.kv_scale);
  const size_t ss = (size_t)p.scale_stride;
  const uint32_t lut0 = smem_u32(x.smem + L::lut), pairs0 = smem_u32(x.smem + L::pairs);
  const uint32_t rope0 = smem_u32(x.smem + L::rope), stage0 = smem_u32(x.smem + L::stage);
  int8_t* grow = reinterpret_cast<int8_t*>(x.smem + L::grow);
  const int row = 16 * cw + (lane >> 1), hp = lane & 1;
  // the scale bytes of the row, two tiles ahead of the conversion
  TileWalk wl;
  auto next_scales = [&](uint32_t (&e)[9], bool& v) -> bool {
    int t0, end;
    if (!wl.next(x, t0, end)) return false;
    v = t0 + row < end;
    load_row_scales(sc, ss, v ? cache_row(p, t0 + row) : 0, v, e);
    return true;
  };
  // step 1 for tile t (scale bytes e, row valid v): returns G
  auto prepare = [&](int t, const uint32_t (&e)[9], bool v) -> uint32_t {
    const int sb = t & 1;
    uint32_t g = 1;
#pragma unroll
    for (int i = 0; i < 8; ++i) g = max(g, max(e[i] & 0xffu, e[i] >> 8));
    // the softmax of tile t - 2 has read its row exponents
    if (t >= 2) wait_phase(&x.bar[kSEmpty + sb], ((t >> 1) - 1) & 1, x.abort_flag, p.ws_err);
    if (hp == 0) grow[sb * 128 + row] = (int8_t)(v ? (int)min(g, 254u) - 127 : 0);
    uint8_t* chunk = x.smem + L::sf + sb * kSfTileBytes + (row & 31) * 16 + (row >> 5) * 4;
    if (hp == 0) {
#pragma unroll
      for (int c = 0; c < 3; ++c) *reinterpret_cast<uint32_t*>(chunk + 512 * c) = bs_scale_word(e, c);
    } else {
#pragma unroll
      for (int c = 3; c < kSfChunks; ++c) *reinterpret_cast<uint32_t*>(chunk + 512 * c) = bs_scale_word(e, c);
    }
    // the rope block: 16 packed bytes (32 elements) of the row per lane
    wait_phase(&x.bar[kStageFull + sb], (t >> 1) & 1, x.abort_flag, p.ws_err);
    const uint4 w = lds128(stage0 + sb * kRopeStageBytes + row * 32 + 16 * hp);
    const uint32_t rb = rope0 + sb * kChunkBytes;
    sts128(rb + sw64_off(row, 32 * hp), w.x, w.y, 0u, 0u);
    sts128(rb + sw64_off(row, 32 * hp + 16), w.z, w.w, 0u, 0u);
    __syncwarp();
    if (lane == 0) mbar_arrive(&x.bar[kStageEmpty + sb]);
    tc::fence_proxy_async();  // the tensor core reads the chunks and the rope slot through the async proxy
    __syncwarp();
    if (lane == 0) mbar_arrive(&x.bar[kConvQK + sb]);
    return g;
  };
  uint32_t ec[9], en[9];
  bool vc = false, vn = false;
  bool hc = next_scales(ec, vc);
  uint32_t gc = hc ? prepare(0, ec, vc) : 1u;
  bool hn = next_scales(en, vn);
  for (int it = 0; hc && !*x.abort_flag; ++it) {
    uint32_t e2[9];
    bool v2 = false;
    const bool h2 = hn && next_scales(e2, v2);
    const uint32_t gn = hn ? prepare(it + 1, en, vn) : 1u;
    // step 2 for tile it
    const int sb = it & 1;
    wait_phase(&x.bar[kSFull + sb], (it >> 1) & 1, x.abort_flag, p.ws_err);
    uint32_t base[4];
#pragma unroll
    for (int f = 0; f < 4; ++f) {
      const int sl = pair_slot<true, 1, kPathBlockScaled>(it, f);
      wait_phase(&x.bar[kPairFull + sl], pair_use<true, 1, kPathBlockScaled>(it, f) & 1, x.abort_flag, p.ws_err);
      base[f] = pairs0 + (uint32_t)sl * kPairBytes + row * 128;
    }
    if (*x.abort_flag) break;
    const uint32_t lutv = lut0 + (vc ? 0u : 128u);
#pragma unroll
    for (int kb = 0; kb < 16; ++kb) {
      const int u = 2 * (kb & 3) + hp;  // 16-element group of the 128-byte row
      const uint32_t a = base[kb >> 2] + ((u ^ (row & 7)) << 4);
      const uint2 w = lds64(a);
      const uint32_t eb = (ec[kb >> 1] >> (8 * (kb & 1))) & 0xffu;
      const uint2 lt = lds64(lutv + 8 * min(gc - eb, 15u));
      const uint2 lo = e2m1x8_to_e4m3(w.x, lt.x, lt.y), hi = e2m1x8_to_e4m3(w.y, lt.x, lt.y);
      sts128(a, lo.x, lo.y, hi.x, hi.y);
    }
    tc::fence_proxy_async();
    __syncwarp();
    if (lane == 0) mbar_arrive(&x.bar[kConvFull + sb]);
#pragma unroll
    for (int i = 0; i < 9; ++i) {
      ec[i] = en[i];
      en[i] = e2[i];
    }
    vc = vn;
    vn = v2;
    gc = gn;
    hc = hn;
    hn = h2;
  }
}

// ---------------------------------------------------------- query loader
// One thread: the query of unit k, prepared by mla_prep_q_kernel as the exact
// shared-memory image (two-term e4m3, 64-byte swizzle) plus its 16 score
// factors, comes in by two bulk copies per token once the last QK of unit k-1
// has completed and the softmax has taken unit k-1's factors (token i of a
// two-token unit of sequence b: the prepared output row 2 b + i).  The
// prepared queries are the one input written by the preceding grid, so this
// is the one thread that waits for it.
template <bool kMx, int kTok, int kPath>
__device__ void q_loader(const Stage1Params& p, const Ctx& x) {
  using L = Layout<kMx, kTok, kPath>;
  const uint64_t pol = policy_evict_last();  // a query serves every split of its sequence
  pdl_wait_primary();
  trace_stamp(p, kTrQueryReady);
  int uses = 0;
  for (int k = 0; k < x.nunits && !*x.abort_flag; ++k) {
    if (k >= 1) {
      wait_phase(&x.bar[kQEmpty], (k - 1) & 1, x.abort_flag, p.ws_err);
      wait_phase(&x.bar[kRFree], (k - 1) & 1, x.abort_flag, p.ws_err);
      if (*x.abort_flag) break;
    }
    mbar_arrive_expect_tx(&x.bar[kQFull], (uint32_t)(kTok * kQPrepBytes));
#pragma unroll
    for (int i = 0; i < kTok; ++i) {
      const uint8_t* src = p.ws_q + ((size_t)x.units[k].b * kTok + i) * kQPrepBytes;
      if constexpr (kTok == 1) {
        bulk_g2s(x.smem + L::qs, src, (uint32_t)kQImageBytes, &x.bar[kQFull], pol);
      } else {
        // K block c of both tokens side by side (rows 32 i + r): the N = 64 B operand
        for (int c = 0; c < 9; ++c)
          bulk_g2s(x.smem + L::qs + c * 2048 * kTok + i * 2048, src + c * 2048, 2048u, &x.bar[kQFull], pol);
      }
      bulk_g2s(x.smem + L::rq + i * 16 * sizeof(float), src + kQImageBytes, 16 * sizeof(float), &x.bar[kQFull],
               pol);
    }
    ++uses;
  }
  if (*x.abort_flag && uses > 0) {
    // never leave with a copy in flight (bounded)
    const uint64_t t0 = global_timer_ns();
    while (!mbar_try_wait(&x.bar[kQFull], (uses - 1) & 1) && global_timer_ns() - t0 < kWaitTimeoutNs) {
    }
  }
}

// ------------------------------------------------------------------ MMA issuers
// Two threads issue the tensor-core operations: warp 1 the QK of every tile,
// warp 2 the P.V of every tile, each in tile order.  Operands are described by
// descriptors built once per tile from templates and moved by constant
// offsets (a few instructions per MMA).
//
// Descriptors as (low word, high word): the high word is fixed per operand
// kind and the low word is the template's low bits plus (address >> 4), so
// every operand move below is a 32-bit add of a constant.
constexpr uint64_t kTplK64 = tc::desc_template(16, 512, 4);          // K-major, 64 B swizzle
constexpr uint64_t kTplV = tc::desc_template(kChunkBytes, 512, 4);   // V^T, MN-major, 64 B swizzle
constexpr uint64_t kTplP = tc::desc_template(1024, 256, 6);          // P^T, MN-major, 32 B swizzle
constexpr uint64_t kTplP2 = tc::desc_template(kPBytes, 256, 6);      // two tokens' P^T: 32-byte atoms kPBytes apart
// pair slots as 128-byte rows (pages of fewer than 64 rows, e4m3): both column
// blocks of a row side by side, [16 groups][8 rows x 128 B] with the 128-byte
// swizzle; column block 2 f + 1 starts 64 B into the row, and an 8-row group
// is 1024 B on.  The V^T block of the pair is one MN-major atom wide.
constexpr uint64_t kTplK128 = tc::desc_template(16, 1024, 2);        // K-major, 128 B swizzle
constexpr uint64_t kTplV128 = tc::desc_template(16, 1024, 2);        // V^T, MN-major, 128 B swizzle
__host__ __device__ constexpr uint32_t lo_word(uint64_t d) { return (uint32_t)d; }
__host__ __device__ constexpr uint32_t hi_word(uint64_t d) { return (uint32_t)(d >> 32); }


// QK of every tile: S^T(t) into TMEM columns [blk (t mod 2), +blk), token i's
// scores at +32 i (two tokens: one N = 64 MMA per k step over both query images).
template <bool kMx, int kTok, int kPath>
__device__ void qk_issuer(const Stage1Params& p, const Ctx& x) {
  constexpr bool kSmallPages = kPath == kPathSmallPages;
  using L = Layout<kMx, kTok, kPath>;
  constexpr bool kBs = Geo<kMx, kTok, kPath>::bs;  // block-scaled e2m1 scores
  constexpr bool kR128 = (kSmallPages && !kMx) || kBs;    // pair slots of 128-byte rows
  constexpr uint64_t kTplA = kR128 ? kTplK128 : kTplK64;
  using TM = Tmem<kTok>;
  constexpr int kPairSlots = Geo<kMx, kTok, kPath>::pair_slots;
  const uint32_t pairs0 = smem_u32(x.smem + L::pairs), rope0 = smem_u32(x.smem + L::rope);
  const uint32_t bq = lo_word(kTplK64) + (smem_u32(x.smem + L::qs) >> 4);
  int it = 0;
  for (int k = 0; k < x.nunits && !*x.abort_flag; ++k) {
    const int nt = tiles_of(x.units[k]);
    wait_phase(&x.bar[kQFull], k & 1, x.abort_flag, p.ws_err);
    for (int t = 0; t < nt; ++t, ++it) {
      const int s0 = (4 * it) % kPairSlots, use0 = (4 * it) / kPairSlots;
      if constexpr (kMx && !kBs) {
        // the converter warps filled all of the tile's slots
        wait_phase(&x.bar[kConvFull + (it & 1)], (it >> 1) & 1, x.abort_flag, p.ws_err);
      } else {
#pragma unroll
        for (int f = 0; f < 4; ++f) {
          const int sl = s0 + f;
          wait_phase(&x.bar[kPairFull + wrap_slot<kMx, kTok, kPath>(sl)], (use0 + (sl >= kPairSlots)) & 1,
                     x.abort_flag, p.ws_err);
        }
        if constexpr (kBs)  // the tile's scale chunks and rope block are laid out
          wait_phase(&x.bar[kConvQK + (it & 1)], (it >> 1) & 1, x.abort_flag, p.ws_err);
        else
          wait_phase(&x.bar[kRopeFull + it % kRopeSlots], (it / kRopeSlots) & 1, x.abort_flag, p.ws_err);
      }
      if (it >= 2) wait_phase(&x.bar[kSEmpty + (it & 1)], ((it >> 1) - 1) & 1, x.abort_flag, p.ws_err);
      if (*x.abort_flag) break;
      if (it < 32) trace_stamp(p, kTrTileData + it);
      tc::fence_after();
      uint32_t ap[4];
#pragma unroll
      for (int f = 0; f < 4; ++f)
        ap[f] = lo_word(kTplA) + ((pairs0 + (uint32_t)wrap_slot<kMx, kTok, kPath>(s0 + f) * kPairBytes) >> 4);
      const uint32_t ar = lo_word(kTplK64) + ((rope0 + (uint32_t)(it % kRopeSlots) * kChunkBytes) >> 4);
      const uint32_t d = x.tmem + TM::s + TM::blk * (it & 1);
      if constexpr (kBs) {
        // scale factors into TMEM (executed before the MMAs that follow):
        // the B factors (all 2^0) once, the tile's A chunks per tile
        const uint32_t sfa = x.tmem + TM::sfa + 32 * (it & 1), sfb = x.tmem + TM::sfb;
        if (it == 0) tc::cp_32x128b_warpx4(sfb, tc::smem_desc(smem_u32(x.smem + L::sfb), 128, 128, 0));
        const uint32_t chunks = smem_u32(x.smem + L::sf + (it & 1) * kSfTileBytes);
#pragma unroll
        for (int g = 0; g < kSfChunks; ++g)
          tc::cp_32x128b_warpx4(sfa + 4 * g, tc::smem_desc(chunks + 512 * g, 128, 128, 0));
        // 18 k32 steps, K-block kb's scales in byte kb mod 4 of chunk kb / 4:
        // the pairs' e2m1 (128-byte rows), then the rope block (64-byte rows)
#pragma unroll
        for (int kb = 0; kb < 18; ++kb) {
          const uint32_t a = kb < 16 ? ap[kb >> 2] + ((32 * (kb & 3)) >> 4) : ar + ((32 * (kb - 16)) >> 4);
          tc::mma_mx_words(d, a, kb < 16 ? hi_word(kTplK128) : hi_word(kTplK64),
                           bq + (((kb >> 1) * 2048 + 32 * (kb & 1)) >> 4), hi_word(kTplK64),
                           tc::idesc_mx_e2m1_e4m3(128, 32, kb & 3, 0), sfa + 4 * (kb >> 2), sfb, kb > 0 ? 1u : 0u);
        }
        tc::commit(&x.bar[kSFull + (it & 1)]);
      } else {
#pragma unroll
        for (int ks = 0; ks < 18; ++ks) {
          const int c = ks >> 1, half = ks & 1;
          constexpr int kBlockStride = kR128 ? 64 : kChunkBytes;  // column block 2 f + 1 within pair f
          const uint32_t a =
              c < 8 ? ap[c >> 1] + (((c & 1) * kBlockStride + 32 * half) >> 4) : ar + ((32 * half) >> 4);
          // both tokens' query rows form one B operand (block c: 32 kTok rows of 64 B)
          tc::mma_f8_words(d, a, c < 8 ? hi_word(kTplA) : hi_word(kTplK64),
                           bq + ((c * 2048 * kTok + 32 * half) >> 4), hi_word(kTplK64),
                           kTok == 1 ? kIdescQK : kIdescQK2, ks > 0 ? 1u : 0u);
        }
        tc::commit(&x.bar[kSFull + (it & 1)]);
        tc::commit(&x.bar[kRopeEmpty + it % kRopeSlots]);
      }
    }
    tc::commit(&x.bar[kQEmpty]);  // the query buffer may be refilled
  }
}

// P.V of every tile: O^T += V^T(t) . P^T(t) (token i: its own P buffer and O^T
// columns, both in one N = 64 MMA); releases the tile's ring slots, its P
// buffers and, on a unit's last tile, the unit's O^T.
template <bool kMx, int kTok, int kPath>
__device__ void pv_issuer(const Stage1Params& p, const Ctx& x) {
  constexpr bool kSmallPages = kPath == kPathSmallPages;
  using L = Layout<kMx, kTok, kPath>;
  constexpr bool kBs = Geo<kMx, kTok, kPath>::bs;  // block-scaled e2m1 scores, V converted in place
  constexpr bool kR128 = (kSmallPages && !kMx) || kBs;    // pair slots of 128-byte rows
  constexpr uint64_t kTplA = kR128 ? kTplV128 : kTplV;
  constexpr uint32_t kRows32 = kR128 ? 4 * 1024 : 2048;  // bytes of 32 rows of V^T in a slot
  using TM = Tmem<kTok>;
  constexpr int kPairSlots = Geo<kMx, kTok, kPath>::pair_slots;
  const uint32_t pairs0 = smem_u32(x.smem + L::pairs), pb0 = smem_u32(x.smem + L::pb);
  constexpr bool kEpi = Geo<kMx, kTok, kPath>::epi;
  int it = 0, ordinal = 0;
  for (int k = 0; k < x.nunits && !*x.abort_flag; ++k) {
    const int nt = tiles_of(x.units[k]);
    if (nt == 0) continue;
    // the unit's O^T buffer, and how many units used it before
    const int obuf = kEpi ? (ordinal & 1) : 0, use = kEpi ? (ordinal >> 1) : ordinal;
    const uint32_t od = x.tmem + TM::o + obuf * TM::obuf;
    for (int t = 0; t < nt; ++t, ++it) {
      wait_phase(&x.bar[kPFull + (it & 1)], (it >> 1) & 1, x.abort_flag, p.ws_err);
      // block-scaled MXFP4: the converter warps have rewritten the tile's V as e4m3
      if (kBs) wait_phase(&x.bar[kConvFull + (it & 1)], (it >> 1) & 1, x.abort_flag, p.ws_err);
      // a unit's first P.V overwrites O^T: the epilogue of the buffer's previous unit must have read it
      if (t == 0 && use > 0) wait_phase(&x.bar[ofree_bar(obuf)], (use - 1) & 1, x.abort_flag, p.ws_err);
      if (*x.abort_flag) break;
      tc::fence_after();
      constexpr uint64_t kTplPT = kTok == 1 ? kTplP : kTplP2;
      const uint32_t bp = lo_word(kTplPT) + ((pb0 + (uint32_t)(it & 1) * kTok * kPBytes) >> 4);
      const int s0 = (4 * it) % kPairSlots;
#pragma unroll
      for (int fb = 0; fb < 4; ++fb) {
        const int sl = wrap_slot<kMx, kTok, kPath>(s0 + fb);

        // V^T block: features [128 fb, 128 fb + 128) = the slot's two column blocks (LBO)
        const uint32_t av = lo_word(kTplA) + ((pairs0 + (uint32_t)sl * kPairBytes) >> 4);
#pragma unroll
        for (int q = 0; q < 4; ++q)  // rows [32 q, 32 q + 32): +kRows32 B of V^T, +1024 B of P^T (every token)
          tc::mma_f8_words(od + TM::blk * fb, av + q * (kRows32 >> 4), hi_word(kTplA), bp + q * (1024 >> 4),
                           hi_word(kTplPT), kTok == 1 ? kIdescPV : kIdescPV2, (t == 0 && q == 0) ? 0u : 1u);
        tc::commit(&x.bar[kPairEmpty + sl]);
      }
      tc::commit(&x.bar[kODone]);
      tc::commit(&x.bar[kPFree + (it & 1)]);
      if (t == nt - 1) tc::commit(&x.bar[olast_bar(obuf)]);
    }
    ++ordinal;
  }
}

// ------------------------------------------------------------------ unit output
// A unit's output from O^T in TMEM: this thread's lane is feature row `row` of
// each 128-feature block, the block's 32 columns at tl_o + blk fb (16 heads x
// the query's two terms).  An unsplit sequence gets bf16 out and lse; a split
// one an fp32 partial and lse in partial slot u.  l, m: the unit's softmax sum
// and reference per head (log2 units); out_scale: the factor O^T carries.
template <bool kTwo>
__device__ __forceinline__ void write_unit(const Stage1Params& p, uint32_t tl_o, uint32_t blk, int row, bool final_out,
                                           int ob, int u, const float (&l)[16], const float (&m)[16],
                                           float out_scale) {
  float inv[16];
#pragma unroll
  for (int h = 0; h < 16; ++h) inv[h] = l[h] > 0.f ? out_scale * __frcp_rn(l[h]) : 0.f;
  // kTwo: two blocks of 128 features per TMEM round trip (MXFP4: 0.1-0.5 us
  // off a bs32/kv8192 split stage in two A/B runs; the e4m3 kernel, which
  // needs four more registers for it, ran bs4/kv8192 1.4 us slower and keeps
  // one block per round trip)
  constexpr int kPer = kTwo ? 2 : 1;
#pragma unroll 1
  for (int fp = 0; fp < 4; fp += kPer) {
    uint32_t o[kPer][32];
#pragma unroll
    for (int j = 0; j < kPer; ++j) tc::ld32(tl_o + blk * (fp + j), o[j]);
    tc::wait_ld();
#pragma unroll
    for (int j = 0; j < kPer; ++j) {
      const int f = 128 * (fp + j) + row;
      if (final_out) {
        uint16_t* op = p.out + (size_t)ob * kHeads * kVDim + f;
#pragma unroll
        for (int h = 0; h < 16; ++h) {
          const float v = (__uint_as_float(o[j][h]) + __uint_as_float(o[j][16 + h])) * inv[h];
          op[h * kVDim] = (uint16_t)(pack_bf16x2(v, 0.f) & 0xffffu);
        }
      } else {
        float* op = p.ws_o + (size_t)u * kHeads * kVDim + f;
#pragma unroll
        for (int h = 0; h < 16; ++h)
          op[h * kVDim] = (__uint_as_float(o[j][h]) + __uint_as_float(o[j][16 + h])) * inv[h];
      }
    }
  }
  // lse of head h is written by row h (every row holds all 16 values): pick
  // this row's head with selects, no divergent branches
  if (row < kHeads) {
    float lh = l[0], mh = m[0];
#pragma unroll
    for (int h = 1; h < 16; ++h) {
      lh = row == h ? l[h] : lh;
      mh = row == h ? m[h] : mh;
    }
    const float lse = lh > 0.f ? (mh + fast_log2(lh)) * kLn2 : -INFINITY;
    if (final_out) {
      if (p.lse) p.lse[ob * kHeads + row] = lse;
    } else {
      p.ws_lse[(size_t)u * kHeads + row] = lse;
    }
  }
}

// Epilogue group (e4m3, one token per unit; warps 8-11, warp w reading TMEM
// lanes [32 (w mod 4), +32)): for each unit with tiles, in order, takes the
// softmax's l and m (kEpiReady), waits for the unit's last P.V, writes the
// unit's output from its O^T buffer and frees the buffer.  A CTA with two
// units whose second has four tiles or more writes the first unit's output
// after the second's: 32 KB of stores issued mid-stream delayed the copies of
// the next tiles (a per-CTA trace at bs64/kv8192 showed the unit boundary
// about 1.8 us longer with them), while at the end they follow the last P.V.
template <bool kMx, int kTok>
__device__ void epilogue_group(const Stage1Params& p, const Ctx& x, int ww, int lane) {
  using L = Layout<kMx, kTok>;
  using TM = Tmem<kTok>;
  const int row = 32 * ww + lane;
  const uint32_t tl = x.tmem + ((uint32_t)(32 * ww) << 16);
  const float kv_scale = *static_cast<const float*>(p.kv_scale);
  const float* hand = reinterpret_cast<const float*>(x.smem + L::hand);
  const bool defer = x.nunits == 2 && tiles_of(x.units[0]) > 0 && tiles_of(x.units[1]) >= 4;
  int ordinal = 0;
  for (int k = 0; k < x.nunits + (defer ? 1 : 0); ++k) {
    if (defer && k == 0) {
      // the first unit's hand-over and last P.V; its buffer is not taken again
      wait_phase(&x.bar[kEpiReady], 0, x.abort_flag, p.ws_err);
      wait_phase(&x.bar[olast_bar(0)], 0, x.abort_flag, p.ws_err);
      if (row == 0) trace_stamp(p, kTrUnitLastPV);
      ++ordinal;
      continue;
    }
    const bool late0 = defer && k == 2;  // the first unit's output, from buffer 0 (no waits left)
    if (late0) ordinal = 0;
    const int ku = late0 ? 0 : k;
    const UnitDesc d = x.units[ku];
    if (tiles_of(d) == 0) continue;
    const int obuf = ordinal & 1, use = ordinal >> 1;
    if (!late0) wait_phase(&x.bar[kEpiReady + obuf], use & 1, x.abort_flag, p.ws_err);
    float l[16], m[16];
#pragma unroll
    for (int h = 0; h < 16; ++h) {
      l[h] = hand[32 * obuf + h];
      m[h] = hand[32 * obuf + 16 + h];
    }
    if (!late0) wait_phase(&x.bar[olast_bar(obuf)], use & 1, x.abort_flag, p.ws_err);
    if (row == 0 && k < 8 && !late0) trace_stamp(p, kTrUnitLastPV + k);
    tc::fence_after();
    write_unit<false>(p, tl + TM::o + obuf * TM::obuf, TM::blk, row, (d.u & kFinalFlag) != 0, d.b, d.u & ~kFinalFlag, l, m,
               kv_scale);
    if (row == 0 && ku < 8) trace_stamp(p, kTrUnitDone + ku);
    tc::fence_before();
    __syncwarp();
    if (lane == 0 && !late0) mbar_arrive(&x.bar[ofree_bar(obuf)]);
    ++ordinal;
  }
}

// ------------------------------------------------------------------ softmax
// Max (or sum) over the 128 rows of the tile for 16 heads: butterfly within the
// warp, then across the 4 warps through smem.
template <bool kMax>
__device__ __forceinline__ void group_reduce16(float (&v)[16], float* red, int ww, int lane, uint32_t bar) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1)
#pragma unroll
    for (int h = 0; h < 16; ++h) {
      const float w = __shfl_xor_sync(0xffffffffu, v[h], o);
      v[h] = kMax ? fmaxf(v[h], w) : v[h] + w;
    }
  if (lane == 0) {
#pragma unroll
    for (int h = 0; h < 16; h += 4)
      *reinterpret_cast<float4*>(red + ww * 16 + h) = make_float4(v[h], v[h + 1], v[h + 2], v[h + 3]);
  }
  named_bar_sync(bar, 128);
#pragma unroll
  for (int h = 0; h < 16; h += 4) {
    float4 r = *reinterpret_cast<const float4*>(red + h);
#pragma unroll
    for (int w = 1; w < 4; ++w) {
      const float4 y = *reinterpret_cast<const float4*>(red + w * 16 + h);
      r.x = kMax ? fmaxf(r.x, y.x) : r.x + y.x;
      r.y = kMax ? fmaxf(r.y, y.y) : r.y + y.y;
      r.z = kMax ? fmaxf(r.z, y.z) : r.z + y.z;
      r.w = kMax ? fmaxf(r.w, y.w) : r.w + y.w;
    }
    v[h] = r.x;
    v[h + 1] = r.y;
    v[h + 2] = r.z;
    v[h + 3] = r.w;
  }
}

// 2^e for an integer e in [-126, 127] (exact).
__device__ __forceinline__ float exp2_int(int e) { return __int_as_float((e + 127) << 23); }

// Softmax group ti (four warps; one group per query token of the unit):
// thread `row` owns tile row `row` (its TMEM lane) for the token's 16 heads,
// in TMEM columns [32 ti, +32) of the S^T buffers and O^T blocks.  With two
// tokens, token 0 does not see the last row of its sequence (token 1's own
// entry), and token ti's partial slot is u + ti S_b.
template <bool kMx, int kTok, int kPath>
__device__ void softmax_epilogue(const Stage1Params& p, const Ctx& x, int ww, int lane, int ti) {
  constexpr bool kSmallPages = kPath == kPathSmallPages;
  constexpr bool kR128 = kSmallPages && !kMx;  // e4m3 pair slots of 128-byte rows
  constexpr bool kBs = Geo<kMx, kTok, kPath>::bs;  // block-scaled e2m1 scores
  using L = Layout<kMx, kTok, kPath>;
  using TM = Tmem<kTok>;
  constexpr int kGvNone = -1000;   // no MXFP4 reference yet
  const int row = 32 * ww + lane;  // tile row == TMEM lane of this thread
  const uint32_t tl = x.tmem + ((uint32_t)(32 * ww) << 16) + 32 * ti;
  const uint32_t bar = kBarSoftmax + ti;  // the group's named barrier
  const float kv_scale = kMx ? 1.f : *static_cast<const float*>(p.kv_scale);
  const int8_t* grow = reinterpret_cast<const int8_t*>(x.smem + L::grow);
  int* gred = reinterpret_cast<int*>(x.smem + L::gred);
  const float* rq = reinterpret_cast<const float*>(x.smem + L::rq) + 16 * ti;
  float* redbuf = reinterpret_cast<float*>(x.smem + L::red) + 128 * ti;
  constexpr bool kEpi = Geo<kMx, kTok, kPath>::epi;
  int it = 0, red_par = 0, ordinal = 0;
  for (int k = 0; k < x.nunits; ++k) {
    const UnitDesc d = x.units[k];
    wait_phase(&x.bar[kQFull], k & 1, x.abort_flag, p.ws_err);
    float r[16];
#pragma unroll
    for (int h = 0; h < 16; ++h) r[h] = rq[h];
    __syncwarp();
    if (lane == 0) mbar_arrive(&x.bar[kRFree]);
    const bool final_out = (d.u & kFinalFlag) != 0;
    // output row and partial slot of this group's token; the rows it does not
    // see at the end of the sequence's last unit
    const int ob = d.b * kTok + ti;
    const int u = (d.u & ~kFinalFlag) + (kTok > 1 ? ti * (d.qrow & ~kLastUnitBit) : 0);
    const int hidden = (kTok > 1 && (d.qrow & kLastUnitBit) != 0) ? kTok - 1 - ti : 0;
    const int nt = tiles_of(d);
    if (nt == 0) {
      // empty sequence: out = 0, lse = -inf
      for (int i = row; i < kHeads * kVDim; i += 128) {
        if (final_out)
          p.out[(size_t)ob * kHeads * kVDim + i] = 0;
        else
          p.ws_o[(size_t)u * kHeads * kVDim + i] = 0.f;
      }
      if (row < kHeads) {
        if (final_out) {
          if (p.lse) p.lse[ob * kHeads + row] = -INFINITY;
        } else {
          p.ws_lse[(size_t)u * kHeads + row] = -INFINITY;
        }
      }
      continue;
    }
    float m_ref[16], l_part[16];
#pragma unroll
    for (int h = 0; h < 16; ++h) {
      m_ref[h] = -INFINITY;
      l_part[h] = 0.f;
    }
    int gv = kGvNone;  // MXFP4: P.V reference exponent of the unit
    const int obuf = kEpi ? (ordinal & 1) : 0;  // the unit's O^T buffer
    const uint32_t tl_o = tl + TM::o + obuf * TM::obuf;
    for (int t = 0; t < nt; ++t, ++it) {
      const int sb = it & 1;
      const int t0 = d.start + t * kTileRows;
      const int valid = min(kTileRows, d.end - t0);
      const int vis = min(valid, d.end - hidden - t0);  // rows of the tile this token sees
      wait_phase(&x.bar[kSFull + sb], (it >> 1) & 1, x.abort_flag, p.ws_err);
      if (row == 0 && ti == 0 && it < 64) trace_stamp(p, kTrTileS + it);
      tc::fence_after();
      uint32_t acc[32];
      tc::ld32(tl + TM::s + TM::blk * sb, acc);
      tc::wait_ld();
      // MXFP4: the row's exponent G - 127, written by the converter warps before
      // they released the tile (waited for here too, so that the bytes are
      // visible); block-scaled: read before kSEmpty, which lets them reuse it
      if (kBs) wait_phase(&x.bar[kConvQK + sb], (it >> 1) & 1, x.abort_flag, p.ws_err);
      const int gsh_bs = kBs ? max(-126, (int)grow[sb * 128 + row]) : 0;
      tc::fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&x.bar[kSEmpty + sb]);
      if (kMx && !kBs) wait_phase(&x.bar[kConvFull + sb], (it >> 1) & 1, x.abort_flag, p.ws_err);
      const int gsh = kBs ? gsh_bs : (kMx ? max(-126, (int)grow[sb * 128 + row]) : 0);
      // the scores of block-scaled MMAs carry no row factor
      const float row_fac = (kMx && !kBs) ? exp2_int(gsh) : 1.f;
      float sv[16];
      uint32_t need = 0;  // heads with a score above m_ref + 8 in this row (bit 16: G above gv)
#pragma unroll
      for (int h = 0; h < 16; ++h) {
        sv[h] = row < vis ? (__uint_as_float(acc[h]) + __uint_as_float(acc[16 + h])) * (r[h] * row_fac)
                          : -INFINITY;
        need |= (sv[h] > m_ref[h] + kRescaleLog2 ? 1u : 0u) << h;
      }
      if (kMx && row < valid && gsh > gv) need |= 1u << 16;
      // heads whose reference rises: OR over the warp, then over the 4 warps
      need = __reduce_or_sync(0xffffffffu, need);
      {
        uint32_t* fl = reinterpret_cast<uint32_t*>(redbuf + red_par * 64);
        if (lane == 0) fl[ww] = need;
        named_bar_sync(bar, 128);
        need = fl[0] | fl[1] | fl[2] | fl[3];
        red_par ^= 1;
      }
      // P buffer it mod 2 was read by P.V(it-2); waiting for it here also makes
      // the o_done wait below exact (the barrier is then one phase behind at most)
      if (it >= 2) wait_phase(&x.bar[kPFree + sb], ((it >> 1) - 1) & 1, x.abort_flag, p.ws_err);
      if (need) {
        // tile max of the rising heads: redux over the warp (order-preserving
        // integer image of the float), then over the 4 warps through smem
        // (all 16 heads, without per-head branches: on a unit's first tile all rise)
        int* mx = reinterpret_cast<int*>(redbuf + red_par * 64);
        int wmax[16];
#pragma unroll
        for (int h = 0; h < 16; ++h) wmax[h] = __reduce_max_sync(0xffffffffu, float_order_key(sv[h]));
        if (lane == 0) {
#pragma unroll
          for (int h = 0; h < 16; h += 4)
            *reinterpret_cast<int4*>(mx + ww * 16 + h) = make_int4(wmax[h], wmax[h + 1], wmax[h + 2], wmax[h + 3]);
        }
        if (kMx && ((need >> 16) & 1u)) {
          const int w = __reduce_max_sync(0xffffffffu, row < valid ? gsh : kGvNone);
          if (lane == 0) gred[red_par * 4 + ww] = w;
        }
        named_bar_sync(bar, 128);
        float fac[16];
#pragma unroll
        for (int h = 0; h < 16; ++h) {
          fac[h] = 1.f;
          if ((need >> h) & 1u) {
            const float mn = float_from_order_key(max(max(mx[h], mx[16 + h]), max(mx[32 + h], mx[48 + h])));
            fac[h] = (m_ref[h] == -INFINITY) ? 0.f : fast_exp2(m_ref[h] - mn);
            m_ref[h] = mn;
            l_part[h] *= fac[h];
          }
        }
        if (kMx && ((need >> 16) & 1u)) {
          // raise the P.V reference: O^T so far is scaled down by 2^(gv_old - gv_new)
          const int* g4 = gred + red_par * 4;
          const int gnew = max(max(g4[0], g4[1]), max(g4[2], g4[3]));
          const float facg = gv == kGvNone ? 0.f : exp2_int(max(-126, gv - gnew));
          gv = gnew;
#pragma unroll
          for (int h = 0; h < 16; ++h) fac[h] *= facg;
        }
        red_par ^= 1;
        if (t > 0) {
          // rescale O^T in TMEM once the previous tile's P.V is complete
          wait_phase(&x.bar[kODone], (it - 1) & 1, x.abort_flag, p.ws_err);
          tc::fence_after();
#pragma unroll 1
          for (int fb = 0; fb < 4; ++fb) {
            uint32_t o[32];
            tc::ld32(tl_o + TM::blk * fb, o);
            tc::wait_ld();
#pragma unroll
            for (int h = 0; h < 16; ++h) {
              o[h] = __float_as_uint(__uint_as_float(o[h]) * fac[h]);
              o[16 + h] = __float_as_uint(__uint_as_float(o[16 + h]) * fac[h]);
            }
            tc::st32(tl_o + TM::blk * fb, o);
          }
          tc::wait_st();
        }
      }
      // probabilities (<= 256), two e4m3 terms, MN-major B operand row = this row;
      // MXFP4 weights for P.V carry the row's 2^(G-127) relative to 2^gv (<= 1)
      const float pv_fac = kMx ? exp2_int(max(-126, gsh - gv)) : 1.f;
      uint32_t hi[4], lo[4];
#pragma unroll
      for (int g = 0; g < 4; ++g) {
        float pv[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int h = 4 * g + e;
          const float pr = (m_ref[h] == -INFINITY) ? 0.f : fast_exp2(sv[h] - m_ref[h]);
          l_part[h] += pr;
          pv[e] = pr * pv_fac;
        }
        two_term_e4m3(pv[0], pv[1], pv[2], pv[3], hi[g], lo[g]);
      }
      uint8_t* pbuf = x.smem + L::pb + (sb * kTok + ti) * kPBytes + row * 32;
      const int xr = (row >> 2) & 1;  // 32 B swizzle: the 16-byte units of the row swap
      *reinterpret_cast<uint4*>(pbuf + 16 * xr) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
      *reinterpret_cast<uint4*>(pbuf + 16 * (xr ^ 1)) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
      if (!kMx && ti == 0 && row >= valid) {
        // rows past the unit's end hold other rows' data: zero their V part so
        // that P = 0 cannot meet a non-finite value (the MXFP4 converters write zeros)
        if constexpr (kR128) {
          // the row's 128 bytes in each pair slot (all eight 16-byte units, whatever the swizzle)
#pragma unroll
          for (int f = 0; f < 4; ++f) {
            uint8_t* rb = x.smem + L::pairs + pair_slot<kMx, kTok, kPath>(it, f) * kPairBytes + row * 128;
#pragma unroll
            for (int uu = 0; uu < 8; ++uu) *reinterpret_cast<uint4*>(rb + 16 * uu) = make_uint4(0, 0, 0, 0);
          }
        } else {
#pragma unroll
          for (int c = 0; c < 8; ++c) {
            uint8_t* blk =
                x.smem + L::pairs + pair_slot<kMx, kTok, kPath>(it, c >> 1) * kPairBytes + (c & 1) * kChunkBytes;
#pragma unroll
            for (int uu = 0; uu < 4; ++uu)
              *reinterpret_cast<uint4*>(blk + sw64_off(row, 16 * uu)) = make_uint4(0, 0, 0, 0);
          }
        }
      }
      tc::fence_proxy_async();
      tc::fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&x.bar[kPFull + sb]);
    }
    // unit epilogue: l per head over the 128 rows, O^T -> output
    group_reduce16<false>(l_part, redbuf + red_par * 64, ww, lane, bar);
    red_par ^= 1;
    if constexpr (kEpi) {
      // hand l and m to the epilogue group (its buffer slot is free once the
      // epilogue of the slot's previous unit has run) and go on to the next unit
      if (row == 0) {
        if (ordinal >= 2) wait_phase(&x.bar[ofree_bar(obuf)], ((ordinal >> 1) - 1) & 1, x.abort_flag, p.ws_err);
        float* hand = reinterpret_cast<float*>(x.smem + L::hand) + 32 * obuf;
#pragma unroll
        for (int h = 0; h < 16; ++h) {
          hand[h] = l_part[h];
          hand[16 + h] = m_ref[h];
        }
        mbar_arrive(&x.bar[kEpiReady + obuf]);
      }
      ++ordinal;
    } else {
      // the unit's last P.V: its own barrier completes once per unit, so the parity
      // of the unit's ordinal names it exactly (o_done may be a phase further on)
      wait_phase(&x.bar[kOLast], ordinal & 1, x.abort_flag, p.ws_err);
      if (row == 0 && ti == 0 && k < 8) trace_stamp(p, kTrUnitLastPV + k);
      ++ordinal;
      tc::fence_after();
      const float out_scale = kMx ? exp2_int(max(-126, min(127, gv))) : kv_scale;
      write_unit<kMx>(p, tl_o, TM::blk, row, final_out, ob, u, l_part, m_ref, out_scale);
      if (row == 0 && ti == 0 && k < 8) trace_stamp(p, kTrUnitDone + k);
      tc::fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&x.bar[kOFree]);
    }
  }
  if (row == 0 && ti == 0) trace_value(p, kTrTiles, (uint64_t)it);
}

// kPath: the instance -- kPathSmallPages for paged caches with pages of fewer
// than 64 rows (one token per unit), whose producer warp fetches rows page by
// page; kPathBlockScaled for MXFP4 scores from block-scaled MMAs.  Separate
// instances, so that the others carry none of their code.
template <bool kMx, int kTok, int kPath>
__global__ void __launch_bounds__(Geo<kMx, kTok, kPath>::threads, 1)
    mla_split_tc_kernel(const __grid_constant__ Stage1Params p) {
  constexpr bool kSmallPages = kPath == kPathSmallPages;
  using L = Layout<kMx, kTok, kPath>;
  constexpr bool kBs = Geo<kMx, kTok, kPath>::bs;
  extern __shared__ __align__(1024) uint8_t smem[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  Ctx x;
  x.smem = smem;
  x.units = reinterpret_cast<const UnitDesc*>(smem + L::units);
  x.bar = reinterpret_cast<uint64_t*>(smem + L::bars);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::misc);
  int* misc = reinterpret_cast<int*>(smem + L::misc);
  x.abort_flag = misc + 1;
  int* s_nunits = misc + 2;
  if (threadIdx.x == 0) {
    trace_stamp(p, kTrEntry);
    trace_smid(p);
  }

  if (threadIdx.x == 0) {
    uint32_t counts[L::nbars];
    for (int i = 0; i < L::nbars; ++i) counts[i] = 1;
    counts[kQFull] = 1;
    counts[kFinal] = 2;
    counts[kSEmpty] = counts[kSEmpty + 1] = 4 * kTok;  // every softmax warp
    counts[kPFull] = counts[kPFull + 1] = 4 * kTok;
    counts[kOFree] = 4 * kTok;
    if constexpr (Geo<kMx, kTok, kPath>::epi) counts[kOFree2] = 4 * kTok;
    counts[kRFree] = 4 * kTok;
    // staging halves: the 4 converter warps of a half; rope blocks (block-scaled): all 8
    for (int i = 0; i < kStageSlots; ++i) counts[kStageEmpty + i] = kBs ? 8 : 4;
    counts[kConvFull] = counts[kConvFull + 1] = 8;
    if constexpr (kBs) counts[kConvQK] = counts[kConvQK + 1] = 8;
    for (int i = 0; i < L::nbars; ++i) mbar_init(&x.bar[i], counts[i]);
    *x.abort_flag = 0;
    fence_mbar_init();
    misc[3] = -1;
    if constexpr (!kMx && kTok == 1 && !kSmallPages) {
      // the first tile's copy starts now, before the unit scan: the plan names
      // its row (the producer checks it against the scan), into pair slots
      // 0..3 and rope slot 0, where the producer would put tile 0
      const int r0 = blockIdx.x < MLA_PLAN_FIRST_ROWS ? p.first_row[blockIdx.x] : -1;
      if (r0 >= 0 && !p.paged) {
        const uint64_t pol = policy_evict_first();
        for (int f = 0; f < 4; ++f) {
          uint8_t* dst = smem + L::pairs + f * kPairBytes;
          mbar_arrive_expect_tx(&x.bar[kPairFull + f], 2 * kChunkBytes);
          tma_load_2d(dst, &p.tmap_kv64, 128 * f, r0, &x.bar[kPairFull + f], pol);
          tma_load_2d(dst + kChunkBytes, &p.tmap_kv64, 128 * f + 64, r0, &x.bar[kPairFull + f], pol);
        }
        mbar_arrive_expect_tx(&x.bar[kRopeFull], kChunkBytes);
        tma_load_2d(smem + L::rope, &p.tmap_kv64, 512, r0, &x.bar[kRopeFull], pol);
        trace_stamp(p, kTrFirstLoad);
        misc[3] = r0;
      }
    }
    if constexpr (kMx && !kBs && kTok == 1 && !kSmallPages) {
      // converted MXFP4: both staging halves of the first tile (64 packed rows
      // each, fewer at the cache's end), before the unit scan, into staging
      // slots 0 and 1 where the producer would put them
      const int r0 = blockIdx.x < MLA_PLAN_FIRST_ROWS ? p.first_row[blockIdx.x] : -1;
      if (r0 >= 0 && !p.paged) {
        const uint64_t pol = policy_evict_first();
        for (int hh = 0; hh < 2; ++hh) {
          const int rr = r0 + hh * kHalfRows, n = max(0, min(kHalfRows, p.total_kv - rr));
          if (n > 0) {
            mbar_arrive_expect_tx(&x.bar[kStageFull + hh], (uint32_t)(n * kPackedRowBytes));
            bulk_g2s(smem + L::stage + hh * kStageBytes, p.kv + (size_t)rr * kPackedRowBytes,
                     (uint32_t)(n * kPackedRowBytes), &x.bar[kStageFull + hh], pol);
          } else {
            mbar_arrive(&x.bar[kStageFull + hh]);
          }
        }
        trace_stamp(p, kTrFirstLoad);
        misc[3] = r0;
      }
    }
  }
  if (warp == 0) {
    // no grid-dependency wait here: this kernel is launched only once the
    // query-preparation grid has itself waited for all earlier work, so every
    // input but the prepared queries is complete (the query loader waits for those)
    scan_units<kTileRows, Geo<kMx, kTok, kPath>::max_units, kTok>(p, reinterpret_cast<UnitDesc*>(smem + L::units), s_nunits,
                                                     lane);
    if (lane == 0) trace_stamp(p, kTrScanDone);
    if (lane == 0 && !kMx) prefetch_tensormap(&p.tmap_kv64);
  }
  if (kMx && threadIdx.x >= 128 && threadIdx.x < 384) {
    // e4m3 bytes of the e2m1 magnitudes {0, .5, 1, 1.5, 2, 3, 4, 6} times
    // 2^-shift for shifts 0..15, then 16 all-zero entries (rows past the end)
    const int i = threadIdx.x - 128, shift = i >> 3, m = i & 7;
    const float mag = m < 4 ? 0.5f * (float)m : (float)(2 << ((m - 4) >> 1)) * ((m & 1) ? 1.5f : 1.f);
    smem[L::lut + i] = shift < 16 ? (uint8_t)(f32x2_to_e4m3x2(ldexpf(mag, -shift), 0.f) & 0xffu) : (uint8_t)0;
  }
  if (kBs && threadIdx.x >= 384) {
    // the query's scale factors, all 2^0 (e8m0 127): one 512-byte chunk
    reinterpret_cast<uint32_t*>(smem + L::sfb)[threadIdx.x - 384] = 0x7f7f7f7fu;
    tc::fence_proxy_async();  // read by tcgen05.cp (async proxy)
  }
  if (warp == 1) {
    tc::alloc(tmem_slot, Tmem<kTok>::cols);
    tc::relinquish();
  }
  // __syncthreads is an aligned barrier: every warp must reach it converged
  // (single-lane work above and below rejoins its warp first)
  __syncwarp();
  tc::fence_before();
  __syncthreads();
  tc::fence_after();
  pdl_launch_dependents();
  x.tmem = *tmem_slot;
  x.nunits = *s_nunits;
  x.early_row = misc[3];
  if (threadIdx.x == 0) {
    trace_stamp(p, kTrSetup);
    trace_value(p, kTrUnits, (uint64_t)x.nunits);
  }

  if (warp == 0) {
    if constexpr (kSmallPages) {
      if constexpr (kMx)
        producer_mx_rows(p, x, lane);
      else
        producer_e4m3_gather<kTok>(p, x, lane);
    } else if (lane == 0) {
      if constexpr (kBs)
        producer_mx_bs(p, x);
      else if constexpr (kMx)
        producer_mx(p, x);
      else
        producer_e4m3<kTok>(p, x);
    }
  } else if (warp == 1) {
    if (lane == 0) qk_issuer<kMx, kTok, kPath>(p, x);
  } else if (warp == 2) {
    if (lane == 0) pv_issuer<kMx, kTok, kPath>(p, x);
  } else if (warp == 3) {
    if (lane == 0) q_loader<kMx, kTok, kPath>(p, x);
  } else if (warp < 4 + 4 * (kMx ? 1 : kTok)) {
    // softmax group (warp - 4) / 4: one per query token of the unit (one call
    // site, so that both groups run the same code)
    softmax_epilogue<kMx, kTok, kPath>(p, x, warp & 3, lane, kTok == 1 ? 0 : (warp - 4) >> 2);
  } else {
    if constexpr (kBs)
      converter_mx_bs(p, x, warp - 8, lane);
    else if constexpr (kMx)
      converter_mx<kSmallPages>(p, x, warp - 8, lane);
    else if constexpr (Geo<kMx, kTok, kPath>::epi)
      epilogue_group<kMx, kTok>(p, x, warp & 3, lane);
  }

  if ((warp == 1 || warp == 2) && lane == 0) {
    // every tensor-core operation of this CTA is complete before TMEM is freed
    tc::commit(&x.bar[kFinal]);
    const uint64_t t0 = global_timer_ns();
    while (!mbar_try_wait(&x.bar[kFinal], 0) && global_timer_ns() - t0 < kWaitTimeoutNs) {
    }
  }
  __syncwarp();  // the single-lane roles rejoin their warps before the CTA barrier
  tc::fence_before();
  __syncthreads();
  tc::fence_after();
  if (threadIdx.x == 0) trace_stamp(p, kTrExit);
  if (warp == 1) tc::dealloc(x.tmem, Tmem<kTok>::cols);
}

}  // namespace tcfp8

template <bool kMx, int kTok = 1, int kPath = tcfp8::kPathRows>
inline cudaError_t launch_split_tc(const Stage1Params& p, cudaStream_t stream) {
  using L = tcfp8::Layout<kMx, kTok, kPath>;
  static_assert(L::total <= 232448, "shared memory carve-up exceeds the 227 KB per-CTA limit");
  static_assert(L::qs % 1024 == 0 && L::pb % 1024 == 0 && L::rope % 1024 == 0, "swizzled operand alignment");
  static_assert(L::stage % 128 == 0 && L::sf % 16 == 0 && L::sfb % 16 == 0, "copy source / destination alignment");
  static_assert(kPath != tcfp8::kPathSmallPages || kTok == 1, "paged caches take one token per sequence");
  auto* kernel = tcfp8::mla_split_tc_kernel<kMx, kTok, kPath>;
  cudaError_t e = smem_opt_in<tcfp8::mla_split_tc_kernel<kMx, kTok, kPath>>(L::total);
  if (e != cudaSuccess) return e;
  e = launch_overlapped(kernel, dim3(p.grid), dim3(tcfp8::Geo<kMx, kTok, kPath>::threads), L::total, stream, p);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace mla
