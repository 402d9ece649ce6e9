// mla_stage1.cuh -- split-K MLA decode kernel for sm_103a (one template per KV
// storage format).
//
// Computes, for every work unit (a contiguous range of KV rows of one sequence),
// the softmax attention of the sequence's 16 query heads over those rows
// (kernelindex "amd-mixed-mla" submission 593653, "Slow fallback" for the
// definition and "_flash_fp8_split_s1" for the split form: a normalised partial
// output plus lse = max + ln(sum) per head).  A sequence that is not split writes
// its bf16 output and lse directly; split sequences leave fp32 partials in the
// workspace for the log-sum-exp combine kernel.
//
// CTA organisation (persistent, one CTA of 12 warps per SM; CTA c owns units
// c, c+grid, c+2 grid, ...; tiles are 64 KV rows):
//   * KV tiles stream through a ring of smem stages, each filled by one 3-D
//     tensor-map TMA copy (64-row box; ragged tails use 16-row boxes) that
//     lands rows densely with the hardware swizzle, which keeps the 8-row
//     ldmatrix patterns below free of bank conflicts.  The last P.V warp to
//     finish a stage (an smem ticket) re-arms it with the tile kStages ahead.
//   * warps 0..3 (the score group) are 2 pairs; pair p scores rows
//     [32p, 32p+32) of a tile.  Warp (p, h) holds half h of the query
//     (features [288h, 288h+288)) in registers and contracts it with the K
//     rows on the tensor cores; the pair swaps partial scores through smem so
//     that warp (p, h) finishes head rows 8h..8h+7; a group-wide max gives the
//     running softmax max; probabilities go to smem as MMA A-fragments with the
//     per-head rescale factor.  The score group runs up to two tiles ahead.
//   * warps 4..11 (the P.V group): warp w accumulates output features
//     [64(w-4), 64(w-4)+64) for all 16 heads from the same smem tile
//     (V = the first 512 columns), so each KV byte is read from HBM once per
//     unit and from smem once for QK^T and once for P.V.
//   Hand-offs between the groups are mbarriers (P buffer full / empty, double
//   buffered); the score group's internal steps use named barriers.
//
// Tensor-core operands: mma.sync m16n8k16 bf16, Q and P in bf16.  This is the
// bf16 KV kernel; e4m3 and MXFP4 KV run the tcgen05 kernel of mla_tc.cuh.  The
// template parameter is the KV storage format, 0 (bf16) being the only one.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>

#include "mla_common.cuh"

namespace mla {

constexpr int kQRowStride = 1168;                   // bf16 query row (1152 B) padded by 16 B
constexpr int kQBufBytes = kHeads * kQRowStride;
constexpr int kScoreWarps = 4;
constexpr int kPvWarps = 8;
constexpr int kWarps = kScoreWarps + kPvWarps;
constexpr int kCtaThreads = kWarps * 32;
constexpr uint32_t kBarScore = 1;   // named barrier of the score group (128 threads)
constexpr uint32_t kBarPair0 = 2;   // named barriers of the two pairs (64 threads)

template <int KV>
struct KvTraits;  // defined for KV = 0 (bf16) only
template <>
struct KvTraits<0> {  // bf16 rows of 576 x 2 B, 9 chunks of 128 B, 128 B swizzle
  static constexpr int kRowBytes = 1152, kSpan = 128, kStages = 2;
};

// Byte offset of (row, byte column) inside a stage written by the swizzled TMA
// copy: the row is 9 consecutive 128-byte lines (line index rho = 9 row +
// chunk); the 16-byte unit inside a line is XOR-ed with the low 3 bits of the
// line index, as the hardware's 128-byte swizzle does.
template <int KV>
__device__ __forceinline__ uint32_t swz(int row, int col) {
  constexpr int span = KvTraits<KV>::kSpan;
  static_assert(span == 128, "bf16 rows: 128-byte lines");
  const int chunk = col / span;
  const int u = (col % span) >> 4;
  const int rho = 9 * row + chunk;
  return (uint32_t)(rho * span + ((u ^ (rho & 7)) << 4) + (col & 15));
}

// Shared-memory carve-up (byte offsets).
template <int KV>
struct Smem {
  using T = KvTraits<KV>;
  static constexpr int kStageBytes = kTile * T::kRowBytes;
  static constexpr int stages = 0;
  static constexpr int qbuf = stages + T::kStages * kStageBytes;
  static constexpr int xbuf = qbuf + 2 * kQBufBytes;        // float [2 pairs][2 halves][32 lanes][8]
  static constexpr int tmax = xbuf + 2 * 2 * 32 * 32;       // float [2 tile parities][16][2]
  static constexpr int lsum = tmax + 2 * 16 * 2 * 4;        // float [16][2]
  static constexpr int qsc = lsum + 16 * 2 * 4;             // float [2 unit parities][2][16]
  static constexpr int pbuf = qsc + 2 * 2 * 16 * 4;         // 2 x 2048 B of P A-fragments
  static constexpr int pside = pbuf + 2 * 2048;             // 2 x {alpha[16], l[16], pad}
  static constexpr int tickets = pside + 2 * 256;           // int [16]
  static constexpr int armed = tickets + 16 * 4;            // int [16] arm counts (stages, then queries)
  static constexpr int units = armed + 16 * 4;
  static constexpr int bars = units + kMaxUnitsPerCta * (int)sizeof(UnitDesc);
  static constexpr int nbars = T::kStages + 6;              // full[], pfull[2], pempty[2], qfull[2]
  static constexpr int misc = bars + nbars * 8;
  static constexpr int total = misc + 16;
};

// One thread: arms a stage's mbarrier and issues the tensor-map copies of the
// tile whose first row is cache row `crow` (a 64-row box, or 16-row boxes for
// a short tail; pages of 64 rows or more keep a tile inside one page).  Pages
// of fewer than 64 rows: one box per page (16 rows per box for 16- and 32-row
// pages), each page looked up from the tile's first row-space position `pos`.
// Rows past the unit's end come from the next rows of the tensor or page (or
// are zero past the tensor's end); the kernel masks them.
template <int KV>
__device__ __forceinline__ void issue_tile(const Stage1Params& p, uint8_t* st, uint64_t* bar, int crow, int rows,
                                           int* armed_count, int pos) {
  using T = KvTraits<KV>;
  const uint64_t pol = policy_evict_first();  // KV rows are read once
  if (p.paged && p.page_shift < 6) {
    const int bp = min(1 << p.page_shift, 16);  // rows per box; a tile starts on a page boundary
    const int nbox = (rows + bp - 1) / bp;
    ++*armed_count;
    mbar_arrive_expect_tx(bar, (uint32_t)(nbox * bp * T::kRowBytes));
    // the page lookups of 16 boxes are independent loads, issued before their copies
    for (int i0 = 0; i0 < nbox; i0 += 16) {
      int cr[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) cr[i] = i0 + i < nbox ? cache_row(p, pos + (i0 + i) * bp) : 0;
#pragma unroll
      for (int i = 0; i < 16; ++i)
        if (i0 + i < nbox) tma_load_3d(st + (i0 + i) * bp * T::kRowBytes, &p.tmap_kv16, 0, 0, cr[i], bar, pol);
    }
    return;
  }
  const int boxes16 = (rows + 15) / 16;
  const bool big = boxes16 == 4;
  const uint32_t bytes = (big ? kTile : 16 * boxes16) * T::kRowBytes;
  ++*armed_count;
  mbar_arrive_expect_tx(bar, bytes);
  if (big) {
    tma_load_3d(st, &p.tmap_kv64, 0, 0, crow, bar, pol);
  } else {
    for (int i = 0; i < boxes16; ++i)
      tma_load_3d(st + i * 16 * T::kRowBytes, &p.tmap_kv16, 0, 0, crow + 16 * i, bar, pol);
  }
}

// One thread: the copy of a unit's query row (16 heads x 1152 B, padded rows).
__device__ __forceinline__ void issue_q(const Stage1Params& p, uint8_t* qbuf, uint64_t* bar, int qrow,
                                        int* armed_count, uint64_t pol) {
  ++*armed_count;
  mbar_arrive_expect_tx(bar, kHeads * 1152);
  for (int h = 0; h < kHeads; ++h)
    bulk_g2s(qbuf + h * kQRowStride, p.q + ((size_t)qrow * kHeads + h) * 1152, 1152, bar, pol);
}

// ---------------------------------------------------------------- score group
template <int KV>
struct QFrag;
template <>
struct QFrag<0> {
  uint32_t a[18][4];  // 18 k16 steps, bf16 A fragments
};

// Loads this warp's query half into registers.  rf: per-row score factors
// (rows g and g+8): sm_scale * log2(e).
template <int KV>
__device__ __forceinline__ void load_q(const uint8_t* qs, int hf, int lane, float base_factor, QFrag<KV>& qf,
                                       float (&rf)[2]) {
  const int g = lane >> 2, c = lane & 3;
  if constexpr (KV == 0) {
    const int head = (lane & 7) + 8 * ((lane >> 3) & 1);
    const uint32_t a0 = smem_u32(qs + head * kQRowStride + 2 * (288 * hf + 8 * (lane >> 4)));
#pragma unroll
    for (int kk = 0; kk < 18; ++kk) ldsm_x4(a0 + 32 * kk, qf.a[kk][0], qf.a[kk][1], qf.a[kk][2], qf.a[kk][3]);
    rf[0] = rf[1] = base_factor;
  }
}

// Partial scores of this warp's query half for n-tiles j = 0..3 (rows
// 32p + 8j + n of the tile): acc[j] = C fragment (rows g / g+8 = heads).
// MMAs are issued so that consecutive ones write different accumulators
// (8 independent chains): issue is in order, so a dependent pair would stall
// for the whole MMA latency.
template <int KV>
__device__ __forceinline__ void qk_tile(const uint8_t* st, int pr, int hf, int lane, const QFrag<KV>& qf,
                                        float (&acc)[4][4]) {
  float a2[2][4][4];
#pragma unroll
  for (int t = 0; t < 2; ++t)
#pragma unroll
    for (int j = 0; j < 4; ++j)
#pragma unroll
      for (int e = 0; e < 4; ++e) a2[t][j][e] = 0.f;
  const uint32_t sbase = smem_u32(st);
  const int mi = lane >> 3;  // which 8x8 matrix of an x4 load this lane addresses
  const int rbase = 32 * pr + (lane & 7);
  if constexpr (KV == 0) {
    // x4 = 8 rows x 32 features: matrices = feature blocks of 8 (k16 steps 2kp, 2kp+1)
#pragma unroll
    for (int kp = 0; kp < 9; ++kp) {
      uint32_t b[4][4];
#pragma unroll
      for (int j = 0; j < 4; ++j)
        ldsm_x4(sbase + swz<KV>(rbase + 8 * j, 2 * (288 * hf + 32 * kp + 8 * mi)), b[j][0], b[j][1], b[j][2],
                b[j][3]);
#pragma unroll
      for (int j = 0; j < 4; ++j) mma_bf16_16816(a2[0][j], qf.a[2 * kp], b[j][0], b[j][1]);
#pragma unroll
      for (int j = 0; j < 4; ++j) mma_bf16_16816(a2[1][j], qf.a[2 * kp + 1], b[j][2], b[j][3]);
    }
  }
#pragma unroll
  for (int j = 0; j < 4; ++j)
#pragma unroll
    for (int e = 0; e < 4; ++e) acc[j][e] = a2[0][j][e] + a2[1][j][e];
}

// Writes this thread's probabilities (head g + 8h; rows 32p + 8j + 2c, +1 of
// n-tiles j = 0..3) as pieces of the P.V A fragments.
template <int KV>
__device__ __forceinline__ void store_p(uint8_t* pb, int pr, int hf, int lane, const float (&pv)[4][2]) {
  if constexpr (KV == 0) {
    // uint4 [4 k16 steps][32 lanes] = {a0, a2, a1, a3}; step 2p + (j >> 1), piece j & 1
#pragma unroll
    for (int jj = 0; jj < 2; ++jj) {
      const uint2 w = make_uint2(pack_bf16x2(pv[2 * jj][0], pv[2 * jj][1]),
                                 pack_bf16x2(pv[2 * jj + 1][0], pv[2 * jj + 1][1]));
      *reinterpret_cast<uint2*>(pb + ((2 * pr + jj) * 32 + lane) * 16 + 8 * hf) = w;
    }
  }
}

// ---------------------------------------------------------------- P.V group
__device__ __forceinline__ uint32_t half_mask2(int t0, int t1, int valid) {
  return (t0 < valid ? 0x0000ffffu : 0u) | (t1 < valid ? 0xffff0000u : 0u);
}

// o[nt] += P . V for output features [64v, 64v+64).  Rows >= valid hold data of
// other rows (or zeros) and are masked out of the V operand.  Consecutive MMAs
// write different accumulators (see qk_tile).
template <int KV>
__device__ __forceinline__ void pv_tile(const uint8_t* st, const uint8_t* pb, int v, int lane, int valid,
                                        float (&o)[8][4]) {
  const int c = lane & 3;
  const uint32_t sbase = smem_u32(st);
  if constexpr (KV == 0) {
#pragma unroll
    for (int kp = 0; kp < 4; ++kp) {
      const uint4 w = *reinterpret_cast<const uint4*>(pb + (kp * 32 + lane) * 16);
      const uint32_t a[4] = {w.x, w.z, w.y, w.w};
      const int row = 16 * kp + 8 * ((lane >> 3) & 1) + (lane & 7);
      uint32_t m0 = 0xffffffffu, m1 = 0xffffffffu;
      if (valid < kTile) {
        m0 = half_mask2(16 * kp + 2 * c, 16 * kp + 2 * c + 1, valid);
        m1 = half_mask2(16 * kp + 8 + 2 * c, 16 * kp + 9 + 2 * c, valid);
      }
      uint32_t r[4][4];
#pragma unroll
      for (int fg = 0; fg < 4; ++fg)
        ldsm_x4_t(sbase + swz<KV>(row, 2 * (64 * v + 16 * fg + 8 * (lane >> 4))), r[fg][0], r[fg][1], r[fg][2],
                  r[fg][3]);
#pragma unroll
      for (int fg = 0; fg < 4; ++fg) mma_bf16_16816(o[2 * fg], a, r[fg][0] & m0, r[fg][1] & m1);
#pragma unroll
      for (int fg = 0; fg < 4; ++fg) mma_bf16_16816(o[2 * fg + 1], a, r[fg][2] & m0, r[fg][3] & m1);
    }
  }
}

// Final (or partial) output of one unit: o * scale for heads g, g+8.
template <int KV>
__device__ __forceinline__ void store_out(const Stage1Params& p, const UnitDesc& d, int v, int lane,
                                          const float (&o)[8][4], float s0, float s1) {
  const int g = lane >> 2, c = lane & 3;
  const bool final_out = (d.u & kFinalFlag) != 0;
  const int u = d.u & ~kFinalFlag;
  if constexpr (KV == 0) {
#pragma unroll
    for (int nt = 0; nt < 8; ++nt) {
      const int f = 64 * v + 8 * nt + 2 * c;
      if (final_out) {
        uint16_t* ob = p.out + (size_t)d.b * kHeads * kVDim;
        *reinterpret_cast<uint32_t*>(ob + g * kVDim + f) = pack_bf16x2(o[nt][0] * s0, o[nt][1] * s0);
        *reinterpret_cast<uint32_t*>(ob + (g + 8) * kVDim + f) = pack_bf16x2(o[nt][2] * s1, o[nt][3] * s1);
      } else {
        float* ob = p.ws_o + (size_t)u * kHeads * kVDim;
        *reinterpret_cast<float2*>(ob + g * kVDim + f) = make_float2(o[nt][0] * s0, o[nt][1] * s0);
        *reinterpret_cast<float2*>(ob + (g + 8) * kVDim + f) = make_float2(o[nt][2] * s1, o[nt][3] * s1);
      }
    }
  }
}

struct Ctx {
  uint8_t* smem;
  const UnitDesc* units;
  int nunits;
  uint64_t* full;
  uint64_t* pfull;
  uint64_t* pempty;
  uint64_t* qfull;
  volatile int* abort_flag;
  int* armed;  // [kStages] stage arm counts, then [2] query-buffer arm counts
};

template <int KV>
__device__ __forceinline__ void score_loop(const Stage1Params& p, const Ctx& x, int warp, int lane) {
  using T = KvTraits<KV>;
  using L = Smem<KV>;
  uint8_t* smem = x.smem;
  const int pr = warp >> 1, hf = warp & 1;
  const int g = lane >> 2, c = lane & 3;
  const int hd = g + 8 * hf;  // the head row this thread finalises
  const uint32_t pair_bar = kBarPair0 + pr;
  float* xbuf = reinterpret_cast<float*>(smem + L::xbuf);
  float* tmax = reinterpret_cast<float*>(smem + L::tmax);
  float* lsum = reinterpret_cast<float*>(smem + L::lsum);
  float* qsc = reinterpret_cast<float*>(smem + L::qsc);
  const float base_factor = p.sm_scale * kLog2e;
  const uint64_t pol_keep = policy_evict_last();

  int it = 0;
  for (int k = 0; k < x.nunits; ++k) {
    const UnitDesc d = x.units[k];
    const int qb = k & 1;
    wait_phase(&x.qfull[qb], (k >> 1) & 1, x.abort_flag, p.ws_err);
    if (k == 0 && warp == 0 && lane == 0) trace_stamp(p, kTrQueryReady);
    QFrag<KV> qf;
    float rf[2];
    load_q<KV>(smem + L::qbuf + qb * kQBufBytes, hf, lane, base_factor, qf, rf);
    float* qs_k = qsc + (k & 1) * 32;  // by unit parity: a slow warp may still read unit k-1's
    if (c == 0) {
      qs_k[hf * 16 + g] = rf[0];
      qs_k[hf * 16 + g + 8] = rf[1];
    }
    named_bar_sync(kBarScore, kScoreWarps * 32);
    // every score warp has read query buffer qb: it takes unit k+2's query
    if (warp == 0 && lane == 0 && k + 2 < x.nunits && !*x.abort_flag)
      issue_q(p, smem + L::qbuf + qb * kQBufBytes, &x.qfull[qb], x.units[k + 2].qrow, &x.armed[T::kStages + qb],
              pol_keep);
    const float r_mine = qs_k[hf * 16 + hd], r_part = qs_k[(1 - hf) * 16 + hd];

    float m_run = -INFINITY, l_run = 0.f;
    for (int t0 = d.start; t0 < d.end; t0 += kTile, ++it) {
      const int s = it % T::kStages;
      const int pbi = it & 1;
      wait_phase(&x.full[s], (it / T::kStages) & 1, x.abort_flag, p.ws_err);
      if (warp == 0 && lane == 0 && it < 32) trace_stamp(p, kTrTileData + it);
      const uint8_t* st = smem + L::stages + s * L::kStageBytes;
      const int valid = min(kTile, d.end - t0);

      float acc[4][4];
      qk_tile<KV>(st, pr, hf, lane, qf, acc);
      // swap head rows with the partner: half 0 finishes rows g, half 1 rows g+8
      float* xs = xbuf + ((pr * 2 + (1 - hf)) * 32 + lane) * 8;
      const float* xr = xbuf + ((pr * 2 + hf) * 32 + lane) * 8;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        xs[2 * j] = hf == 0 ? acc[j][2] : acc[j][0];
        xs[2 * j + 1] = hf == 0 ? acc[j][3] : acc[j][1];
      }
      named_bar_sync(pair_bar, 64);
      float sv[4][2];
      float mx = -INFINITY;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const float m0 = hf == 0 ? acc[j][0] : acc[j][2];
        const float m1 = hf == 0 ? acc[j][1] : acc[j][3];
        const int tk = 32 * pr + 8 * j + 2 * c;
        sv[j][0] = tk < valid ? m0 * r_mine + xr[2 * j] * r_part : -INFINITY;
        sv[j][1] = tk + 1 < valid ? m1 * r_mine + xr[2 * j + 1] * r_part : -INFINITY;
        mx = fmaxf(mx, fmaxf(sv[j][0], sv[j][1]));
      }
      mx = quad_max(mx);
      float* tm = tmax + (it & 1) * 32;  // by tile parity: the other pair may still read tile it-1's
      if (c == 0) tm[hd * 2 + pr] = mx;
      named_bar_sync(kBarScore, kScoreWarps * 32);
      const float mt = fmaxf(tm[hd * 2], tm[hd * 2 + 1]);
      const float mn = fmaxf(m_run, mt);
      const float alpha = (mn == -INFINITY) ? 1.f : fast_exp2(m_run - mn);
      m_run = mn;
      float pv[4][2];
      float ls = 0.f;
#pragma unroll
      for (int j = 0; j < 4; ++j)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          pv[j][e] = (mn == -INFINITY) ? 0.f : fast_exp2(sv[j][e] - mn);
          ls += pv[j][e];
        }
      l_run = l_run * alpha + ls;
      // the P buffer of this tile is free once the P.V group finished tile it-2
      if (it >= 2) wait_phase(&x.pempty[pbi], ((it >> 1) - 1) & 1, x.abort_flag, p.ws_err);
      uint8_t* pb = smem + L::pbuf + pbi * 2048;
      float* side = reinterpret_cast<float*>(smem + L::pside + pbi * 256);
      store_p<KV>(pb, pr, hf, lane, pv);
      if (pr == 0 && c == 0) side[hd] = alpha;
      if (t0 + kTile >= d.end) {
        // unit epilogue: l per head = sum over the pairs; l to the P.V group, lse out
        const float lq = quad_sum(l_run);
        if (c == 0) lsum[hd * 2 + pr] = lq;
        named_bar_sync(kBarScore, kScoreWarps * 32);
        const float lt = lsum[hd * 2] + lsum[hd * 2 + 1];
        if (pr == 0 && c == 0) {
          side[16 + hd] = lt;
          const float lse = lt > 0.f ? (m_run + fast_log2(lt)) * kLn2 : -INFINITY;
          if (d.u & kFinalFlag) {
            if (p.lse) p.lse[d.b * kHeads + hd] = lse;
          } else {
            p.ws_lse[(size_t)(d.u & ~kFinalFlag) * kHeads + hd] = lse;
          }
        }
      }
      __syncwarp();
      if (warp == 0 && lane == 0 && it < 64) trace_stamp(p, kTrTileS + it);
      if (lane == 0) mbar_arrive(&x.pfull[pbi]);
    }
    if (d.start >= d.end && warp == 0 && c == 0) {
      // empty sequence: no tile, lse = -inf
      if (d.u & kFinalFlag) {
        if (p.lse) {
          p.lse[d.b * kHeads + g] = -INFINITY;
          p.lse[d.b * kHeads + g + 8] = -INFINITY;
        }
      } else {
        p.ws_lse[(size_t)(d.u & ~kFinalFlag) * kHeads + g] = -INFINITY;
        p.ws_lse[(size_t)(d.u & ~kFinalFlag) * kHeads + g + 8] = -INFINITY;
      }
    }
  }
  if (warp == 0 && lane == 0) trace_value(p, kTrTiles, (uint64_t)it);
}

template <int KV>
__device__ __forceinline__ void pv_loop(const Stage1Params& p, const Ctx& x, int v, int lane) {
  using T = KvTraits<KV>;
  using L = Smem<KV>;
  uint8_t* smem = x.smem;
  const int g = lane >> 2;
  int* tickets = reinterpret_cast<int*>(smem + L::tickets);
  const float out_mult = 1.f;  // bf16 P and V carry no extra factor
  // refill cursor: the tile kStages ahead of the one being consumed
  TileCursor cur;
  cur.k = 0;
  cursor_skip_empty(cur, x.units, x.nunits);
  for (int n = 0; n < T::kStages && cur.k < x.nunits; ++n) cursor_next<kTile>(cur, x.units, x.nunits);

  int it = 0;
  for (int k = 0; k < x.nunits; ++k) {
    const UnitDesc d = x.units[k];
    float o[8][4];
#pragma unroll
    for (int nt = 0; nt < 8; ++nt)
#pragma unroll
      for (int e = 0; e < 4; ++e) o[nt][e] = 0.f;
    float l0 = 0.f, l1 = 0.f;
    for (int t0 = d.start; t0 < d.end; t0 += kTile, ++it) {
      const int s = it % T::kStages;
      const int pbi = it & 1;
      // cache row of the refill tile, looked up before this tile's work
      const int refill_row = (lane == 0 && cur.k < x.nunits) ? cache_row(p, cur.t0) : 0;
      wait_phase(&x.pfull[pbi], (it >> 1) & 1, x.abort_flag, p.ws_err);
      wait_phase(&x.full[s], (it / T::kStages) & 1, x.abort_flag, p.ws_err);
      const uint8_t* st = smem + L::stages + s * L::kStageBytes;
      const uint8_t* pb = smem + L::pbuf + pbi * 2048;
      const float* side = reinterpret_cast<const float*>(smem + L::pside + pbi * 256);
      const float a0 = side[g], a1 = side[g + 8];
#pragma unroll
      for (int nt = 0; nt < 8; ++nt) {
        o[nt][0] *= a0;
        o[nt][1] *= a0;
        o[nt][2] *= a1;
        o[nt][3] *= a1;
      }
      pv_tile<KV>(st, pb, v, lane, min(kTile, d.end - t0), o);
      if (t0 + kTile >= d.end) {
        l0 = side[16 + g];
        l1 = side[16 + g + 8];
      }
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&x.pempty[pbi]);
        // the last P.V warp done with this stage re-arms it with the tile kStages ahead
        if (atomicAdd(&tickets[s], 1) == kPvWarps - 1) {
          tickets[s] = 0;
          if (cur.k < x.nunits && !*x.abort_flag)
            issue_tile<KV>(p, smem + L::stages + s * L::kStageBytes, &x.full[s], refill_row,
                           min(kTile, x.units[cur.k].end - cur.t0), &x.armed[s], cur.t0);
        }
      }
      if (cur.k < x.nunits) cursor_next<kTile>(cur, x.units, x.nunits);
    }
    const float s0 = l0 > 0.f ? out_mult / l0 : 0.f;
    const float s1 = l1 > 0.f ? out_mult / l1 : 0.f;
    store_out<KV>(p, d, v, lane, o, s0, s1);
    if (v == 0 && lane == 0 && k < 8) trace_stamp(p, kTrUnitDone + k);
  }
}

template <int KV>
__global__ void __launch_bounds__(kCtaThreads, 1) mla_split_kernel(const __grid_constant__ Stage1Params p) {
  using T = KvTraits<KV>;
  using L = Smem<KV>;
  extern __shared__ __align__(1024) uint8_t smem[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::bars);
  Ctx x;
  x.smem = smem;
  x.units = reinterpret_cast<const UnitDesc*>(smem + L::units);
  x.full = bars;
  x.pfull = bars + T::kStages;
  x.pempty = x.pfull + 2;
  x.qfull = x.pempty + 2;
  int* misc = reinterpret_cast<int*>(smem + L::misc);
  x.abort_flag = misc;
  int* s_nunits = misc + 1;
  x.armed = reinterpret_cast<int*>(smem + L::armed);

  if (threadIdx.x == 0) {
    trace_stamp(p, kTrEntry);
    trace_smid(p);
    for (int s = 0; s < T::kStages; ++s) mbar_init(&x.full[s], 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&x.pfull[i], kScoreWarps);
      mbar_init(&x.pempty[i], kPvWarps);
      mbar_init(&x.qfull[i], 1);
    }
    int* tickets = reinterpret_cast<int*>(smem + L::tickets);
    for (int s = 0; s < 16; ++s) {
      tickets[s] = 0;
      x.armed[s] = 0;
    }
    *x.abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0) {
    pdl_wait_primary();  // the previous kernel's writes are visible from here on
    scan_units<kTile>(p, reinterpret_cast<UnitDesc*>(smem + L::units), s_nunits, lane);
    __syncwarp();
    if (lane == 0) {
      trace_stamp(p, kTrScanDone);
      // prologue copies: queries of units 0 and 1, the first kStages tiles
      prefetch_tensormap(&p.tmap_kv64);
      prefetch_tensormap(&p.tmap_kv16);
      const int nu = *s_nunits;
      const uint64_t pol_keep = policy_evict_last();
      const UnitDesc* units = reinterpret_cast<const UnitDesc*>(smem + L::units);
      for (int k = 0; k < 2 && k < nu; ++k)
        issue_q(p, smem + L::qbuf + k * kQBufBytes, &x.qfull[k], units[k].qrow, &x.armed[T::kStages + k], pol_keep);
      TileCursor cur;
      cur.k = 0;
      cursor_skip_empty(cur, units, nu);
      // all the first tiles' cache rows are looked up before any is issued
      int crow[T::kStages], rows[T::kStages], pos[T::kStages];
      int nfirst = 0;
#pragma unroll
      for (int s = 0; s < T::kStages; ++s) {
        if (cur.k < nu) {
          crow[s] = cache_row(p, cur.t0);
          pos[s] = cur.t0;
          rows[s] = min(kTile, units[cur.k].end - cur.t0);
          nfirst = s + 1;
          cursor_next<kTile>(cur, units, nu);
        }
      }
#pragma unroll
      for (int s = 0; s < T::kStages; ++s)
        if (s < nfirst)
          issue_tile<KV>(p, smem + L::stages + s * L::kStageBytes, &x.full[s], crow[s], rows[s], &x.armed[s],
                         pos[s]);
      trace_stamp(p, kTrFirstLoad);
    }
  }
  __syncwarp();  // lane 0's prologue copies rejoin the warp before the aligned CTA barrier
  __syncthreads();
  pdl_wait_primary();
  pdl_launch_dependents();
  x.nunits = *s_nunits;
  if (threadIdx.x == 0) {
    trace_stamp(p, kTrSetup);
    trace_value(p, kTrUnits, (uint64_t)x.nunits);
  }
  if (warp < kScoreWarps)
    score_loop<KV>(p, x, warp, lane);
  else
    pv_loop<KV>(p, x, warp - kScoreWarps, lane);

  __syncwarp();
  __syncthreads();
  if (threadIdx.x == 0) trace_stamp(p, kTrExit);
  if (*x.abort_flag && threadIdx.x == 0) {
    // a wait gave up: never leave with copies in flight (bounded wait per barrier)
    for (int s = 0; s < T::kStages + 2; ++s) {
      const int n = x.armed[s];
      if (n == 0) continue;
      uint64_t* bar = s < T::kStages ? &x.full[s] : &x.qfull[s - T::kStages];
      const uint64_t t0 = global_timer_ns();
      while (!mbar_try_wait(bar, (n - 1) & 1) && global_timer_ns() - t0 < kWaitTimeoutNs) {
      }
    }
  }
}

template <int KV>
cudaError_t launch_split(const Stage1Params& p, cudaStream_t stream) {
  using L = Smem<KV>;
  static_assert(L::total <= 232448, "shared memory carve-up exceeds the 227 KB per-CTA limit");
  static_assert(L::qbuf % 1024 == 0 && L::kStageBytes % 1024 == 0, "TMA swizzle alignment");
  cudaError_t e = smem_opt_in<mla_split_kernel<KV>>(L::total);
  if (e != cudaSuccess) return e;
  e = launch_overlapped(mla_split_kernel<KV>, dim3(p.grid), dim3(kCtaThreads), L::total, stream, p);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace mla
