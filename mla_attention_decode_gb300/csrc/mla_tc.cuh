// mla_tc.cuh -- split-K MLA decode for e4m3 KV on the 5th-generation tensor
// cores (tcgen05, accumulators in tensor memory), sm_103a.
//
// Same contract as the split kernel in mla_stage1.cuh (kernelindex
// "amd-mixed-mla" submission 593653, "Slow fallback" for the definition and
// "_flash_fp8_split_s1" for the split form): per work unit, softmax attention of
// the 16 query heads over a contiguous range of KV rows; final bf16 output and
// lse for unsplit sequences, fp32 partials and lse for split ones.
//
// Per 128-row tile t of a unit (one CTA of 8 warps per SM, persistent):
//   scores  S^T[128 rows x 32] = K_t[128 x 576] . [Q_hi | Q_lo]^T   (tcgen05 kind::f8f6f4,
//           18 k32 steps; K straight from the TMA stage, K-major, 64 B swizzle;
//           the query as two e4m3 terms x = hi + lo with a power-of-two scale
//           per head, 32 "columns" = 16 heads x 2 terms, in TMEM)
//   softmax one thread per row reads its 32 accumulators, builds the scores,
//           the per-head tile max (warp shuffles + smem), exponentials and row
//           sums, and writes P^T[128 rows x 32] = [P_hi | P_lo] (two e4m3 terms)
//           as the MN-major B operand
//   P.V     O^T[512 features x 32] += V_t^T[512 x 128] . P^T   (4 blocks of 128
//           features x 4 k32 steps; V^T read MN-major from the same stage --
//           V is the first 512 columns of K -- so each KV byte is read from HBM
//           once per unit), O^T resident in TMEM across the unit's tiles
// The running max is applied lazily: P = 2^(s - m_ref) with m_ref raised (and
// O^T, l rescaled in place) only when a head's tile max exceeds m_ref by more
// than 8 (log2 units), which keeps P <= 256 inside e4m3 range.  Scores are in
// log2 units: s = (q . k) * sm_scale * log2(e) * kv_scale.
//
// Warp roles: 0 TMA producer (9 column boxes of 64 B x 128 rows per tile into
// a 2-stage ring); 1 MMA issuer (QK of tile t, then PV of tile t-1) and TMEM
// owner; 2-3 query preparation (two-term query per unit, double buffered);
// 4-7 softmax, O^T rescale and the unit epilogue.  Hand-offs are mbarriers
// (TMA transaction bytes, tcgen05.commit, thread arrivals).
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>

#include "mla_common.cuh"

namespace mla {
namespace tcfp8 {

constexpr int kTileRows = 128;
constexpr int kStages = 2;
constexpr int kChunkBytes = kTileRows * 64;  // one 64-byte feature column block of a tile
constexpr int kStageBytes = 9 * kChunkBytes;
constexpr int kQsBytes = 9 * 32 * 64;        // two-term query: 32 rows x 576 B, K-major, 64 B swizzle
constexpr int kPBytes = kTileRows * 32;      // two-term P^T: 128 rows x 32 B, MN-major, 32 B swizzle
constexpr int kThreads = 256;
constexpr uint32_t kTmemCols = 256;
constexpr uint32_t kColS = 0;   // S^T double buffer: columns [0, 32) and [32, 64)
constexpr uint32_t kColO = 64;  // O^T: 4 feature blocks x 32 columns
constexpr float kRescaleLog2 = 8.f;
constexpr uint32_t kBarSoftmax = 1;  // named barrier of the softmax warps (128 threads)
constexpr uint32_t kIdescQK = tc::idesc_e4m3(128, 32, 0, 0);
constexpr uint32_t kIdescPV = tc::idesc_e4m3(128, 32, 1, 1);

struct Layout {
  static constexpr int stages = 0;                           // 1024-aligned
  static constexpr int qs = stages + kStages * kStageBytes;  // [2]
  static constexpr int pb = qs + 2 * kQsBytes;               // [2]
  static constexpr int rq = pb + 2 * kPBytes;                // float [2][16] score factor per head
  static constexpr int red = rq + 2 * 16 * 4;                // float [2][4 warps][16]
  static constexpr int units = red + 2 * 4 * 16 * 4;
  static constexpr int bars = units + kMaxUnitsPerCta * (int)sizeof(UnitDesc);
  static constexpr int nbars = 19;
  static constexpr int misc = bars + nbars * 8;  // tmem slot, abort flag, unit count
  static constexpr int total = misc + 16;
};

// mbarrier slots
enum {
  kKvFull = 0,    // [2] TMA bytes of a stage
  kKvEmpty = 2,   // [2] commit after the P.V of the stage's tile
  kQFull = 4,     // [2] query prepared (2 warps)
  kQEmpty = 6,    // [2] commit after the unit's last QK
  kSFull = 8,     // [2] commit after QK
  kSEmpty = 10,   // [2] softmax read S (4 warps)
  kPFull = 12,    // [2] P written, O^T rescaled (4 warps)
  kODone = 14,    // commit after each P.V
  kOFree = 15,    // unit epilogue read O^T (4 warps)
  kRFree = 16,    // [2] softmax copied the unit's score factors (4 warps)
  kFinal = 18,    // commit after the MMA issuer's last operation
};

__device__ __forceinline__ uint32_t sw64_off(int row, int col) {  // byte (row, col) of a 64 B-row, 64 B-swizzled block
  return (uint32_t)(row * 64 + ((((col >> 4) ^ (row >> 1)) & 3) << 4) + (col & 15));
}

struct Ctx {
  uint8_t* smem;
  const UnitDesc* units;
  int nunits;
  uint64_t* bar;
  volatile int* abort_flag;
  uint32_t tmem;
};

__device__ __forceinline__ int tiles_of(const UnitDesc& d) { return (d.end - d.start + kTileRows - 1) / kTileRows; }

// ------------------------------------------------------------------ producer
__device__ void producer(const Stage1Params& p, const Ctx& x) {
  const uint64_t pol = policy_evict_first();  // KV rows are read once
  int it = 0;
  int armed[2] = {0, 0};
  for (int k = 0; k < x.nunits && !*x.abort_flag; ++k) {
    const UnitDesc d = x.units[k];
    for (int t0 = d.start; t0 < d.end; t0 += kTileRows, ++it) {
      const int s = it & 1;
      if (it >= 2) wait_phase(&x.bar[kKvEmpty + s], ((it >> 1) - 1) & 1, x.abort_flag, p.ws_err);
      if (*x.abort_flag) break;
      uint8_t* st = x.smem + Layout::stages + s * kStageBytes;
      mbar_arrive_expect_tx(&x.bar[kKvFull + s], kStageBytes);
      for (int c = 0; c < 9; ++c) tma_load_2d(st + c * kChunkBytes, &p.tmap_kv64, 64 * c, t0, &x.bar[kKvFull + s], pol);
      ++armed[s];
    }
  }
  if (*x.abort_flag) {
    // a wait gave up somewhere: never leave with copies in flight (bounded wait per stage)
    for (int s = 0; s < 2; ++s) {
      if (armed[s] == 0) continue;
      const uint64_t t0 = global_timer_ns();
      while (!mbar_try_wait(&x.bar[kKvFull + s], (armed[s] - 1) & 1) && global_timer_ns() - t0 < kWaitTimeoutNs) {
      }
    }
  }
}

// ---------------------------------------------------------- query preparation
// 64 threads: thread j handles head j/4, features [144 (j%4), 144 (j%4) + 144).
__device__ void prep_query(const Stage1Params& p, const Ctx& x, int j) {
  const int h = j >> 2, part = j & 3;
  const float kv_scale = *static_cast<const float*>(p.kv_scale);
  const float base_factor = p.sm_scale * kLog2e * kv_scale;
  float* rq = reinterpret_cast<float*>(x.smem + Layout::rq);
  for (int k = 0; k < x.nunits; ++k) {
    const int qb = k & 1;
    if (k >= 2) {
      wait_phase(&x.bar[kQEmpty + qb], ((k >> 1) - 1) & 1, x.abort_flag, p.ws_err);
      wait_phase(&x.bar[kRFree + qb], ((k >> 1) - 1) & 1, x.abort_flag, p.ws_err);
    }
    const int qrow = p.qo_indptr[x.units[k].b];
    const uint4* src = reinterpret_cast<const uint4*>(p.q + (((size_t)qrow * kHeads + h) * kQkDim + 144 * part) * 2);
    uint4 raw[18];
#pragma unroll
    for (int i = 0; i < 18; ++i) raw[i] = __ldg(src + i);
    float amax = 0.f;
#pragma unroll
    for (int i = 0; i < 18; ++i) {
      const float4 a = bf16x4_to_f4(make_uint2(raw[i].x, raw[i].y));
      const float4 b = bf16x4_to_f4(make_uint2(raw[i].z, raw[i].w));
      amax = fmaxf(amax, fmaxf(fmaxf(fmaxf(fabsf(a.x), fabsf(a.y)), fmaxf(fabsf(a.z), fabsf(a.w))),
                               fmaxf(fmaxf(fabsf(b.x), fabsf(b.y)), fmaxf(fabsf(b.z), fabsf(b.w)))));
    }
    amax = quad_max(amax);
    // power-of-two scale with amax * scale <= 448 (e4m3 max); 1 for an all-zero head
    float sc = 1.f;
    if (amax > 0.f) {
      sc = exp2f(floorf(log2f(448.f / amax)));
      if (amax * sc > 448.f) sc *= 0.5f;
    }
    uint8_t* qs = x.smem + Layout::qs + qb * kQsBytes;
#pragma unroll
    for (int i = 0; i < 18; ++i) {
      const int f0 = 144 * part + 8 * i;  // 8 features, inside one 16-byte unit of a 64-byte chunk
      const float4 a = bf16x4_to_f4(make_uint2(raw[i].x, raw[i].y));
      const float4 b = bf16x4_to_f4(make_uint2(raw[i].z, raw[i].w));
      uint32_t hi0, lo0, hi1, lo1;
      two_term_e4m3(a.x * sc, a.y * sc, a.z * sc, a.w * sc, hi0, lo0);
      two_term_e4m3(b.x * sc, b.y * sc, b.z * sc, b.w * sc, hi1, lo1);
      const int chunk = f0 >> 6, col = f0 & 63;
      *reinterpret_cast<uint2*>(qs + chunk * 2048 + sw64_off(h, col)) = make_uint2(hi0, hi1);
      *reinterpret_cast<uint2*>(qs + chunk * 2048 + sw64_off(16 + h, col)) = make_uint2(lo0, lo1);
    }
    if (part == 0) rq[qb * 16 + h] = base_factor / sc;
    tc::fence_proxy_async();  // the tensor core reads the query through the async proxy
    __syncwarp();
    if ((j & 31) == 0) mbar_arrive(&x.bar[kQFull + qb]);
  }
}

// ------------------------------------------------------------------ MMA issuer
struct PvJob {
  int it;       // tile index (P buffer / o_done phase)
  int stage;
  int first;    // first tile of its unit
  int ordinal;  // index of its unit among the CTA's units with tiles
};

__device__ __forceinline__ void issue_pv(const Stage1Params& p, const Ctx& x, const PvJob& j) {
  wait_phase(&x.bar[kPFull + (j.it & 1)], (j.it >> 1) & 1, x.abort_flag, p.ws_err);
  if (j.first && j.ordinal > 0) wait_phase(&x.bar[kOFree], (j.ordinal - 1) & 1, x.abort_flag, p.ws_err);
  tc::fence_after();
  const uint32_t st = smem_u32(x.smem + Layout::stages + j.stage * kStageBytes);
  const uint32_t pb = smem_u32(x.smem + Layout::pb + (j.it & 1) * kPBytes);
#pragma unroll
  for (int fb = 0; fb < 4; ++fb)
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      // V^T block: features [128 fb, 128 fb + 128) = chunks 2fb, 2fb+1 (LBO), rows [32q, 32q+32)
      const uint64_t a = tc::smem_desc(st + 2 * fb * kChunkBytes + q * 32 * 64, kChunkBytes, 512, 4);
      const uint64_t b = tc::smem_desc(pb + q * 32 * 32, 1024, 256, 6);
      tc::mma_f8(x.tmem + kColO + 32 * fb, a, b, kIdescPV, (j.first && q == 0) ? 0u : 1u);
    }
  tc::commit(&x.bar[kODone]);
  tc::commit(&x.bar[kKvEmpty + j.stage]);
}

__device__ void mma_issuer(const Stage1Params& p, const Ctx& x) {
  int it = 0, ordinal = 0;
  PvJob prev{0, 0, 0, 0};
  bool have_prev = false;
  for (int k = 0; k < x.nunits; ++k) {
    const UnitDesc d = x.units[k];
    const int qb = k & 1;
    wait_phase(&x.bar[kQFull + qb], (k >> 1) & 1, x.abort_flag, p.ws_err);
    tc::fence_after();
    const uint32_t qs = smem_u32(x.smem + Layout::qs + qb * kQsBytes);
    const int nt = tiles_of(d);
    for (int t = 0; t < nt; ++t, ++it) {
      const int s = it & 1;
      wait_phase(&x.bar[kKvFull + s], (it >> 1) & 1, x.abort_flag, p.ws_err);
      if (it >= 2) wait_phase(&x.bar[kSEmpty + s], ((it >> 1) - 1) & 1, x.abort_flag, p.ws_err);
      tc::fence_after();
      const uint32_t st = smem_u32(x.smem + Layout::stages + s * kStageBytes);
#pragma unroll
      for (int ks = 0; ks < 18; ++ks) {
        const int c = ks >> 1, half = ks & 1;
        const uint64_t a = tc::smem_desc(st + c * kChunkBytes + 32 * half, 16, 512, 4);
        const uint64_t b = tc::smem_desc(qs + c * 2048 + 32 * half, 16, 512, 4);
        tc::mma_f8(x.tmem + kColS + 32 * s, a, b, kIdescQK, ks > 0 ? 1u : 0u);
      }
      tc::commit(&x.bar[kSFull + s]);
      if (t == nt - 1) tc::commit(&x.bar[kQEmpty + qb]);
      if (have_prev) issue_pv(p, x, prev);
      prev = PvJob{it, s, t == 0, ordinal};
      have_prev = true;
    }
    if (nt == 0) tc::commit(&x.bar[kQEmpty + qb]);
    else ++ordinal;
  }
  if (have_prev) issue_pv(p, x, prev);
}

// ------------------------------------------------------------------ softmax
// Max (or sum) over the 128 rows of the tile for 16 heads: butterfly within the
// warp, then across the 4 warps through smem.
template <bool kMax>
__device__ __forceinline__ void group_reduce16(float (&v)[16], float* red, int ww, int lane) {
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
  named_bar_sync(kBarSoftmax, 128);
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

__device__ void softmax_epilogue(const Stage1Params& p, const Ctx& x, int ww, int lane) {
  const int row = 32 * ww + lane;  // tile row == TMEM lane of this thread
  const uint32_t tl = x.tmem + ((uint32_t)(32 * ww) << 16);
  const float kv_scale = *static_cast<const float*>(p.kv_scale);
  const float* rq = reinterpret_cast<const float*>(x.smem + Layout::rq);
  float* redbuf = reinterpret_cast<float*>(x.smem + Layout::red);
  int it = 0, red_par = 0;
  for (int k = 0; k < x.nunits; ++k) {
    const UnitDesc d = x.units[k];
    const int qb = k & 1;
    wait_phase(&x.bar[kQFull + qb], (k >> 1) & 1, x.abort_flag, p.ws_err);
    float r[16];
#pragma unroll
    for (int h = 0; h < 16; ++h) r[h] = rq[qb * 16 + h];
    __syncwarp();
    if (lane == 0) mbar_arrive(&x.bar[kRFree + qb]);
    const bool final_out = (d.u & kFinalFlag) != 0;
    const int u = d.u & ~kFinalFlag;
    const int nt = tiles_of(d);
    if (nt == 0) {
      // empty sequence: out = 0, lse = -inf
      for (int i = row; i < kHeads * kVDim; i += 128) {
        if (final_out)
          p.out[(size_t)d.b * kHeads * kVDim + i] = 0;
        else
          p.ws_o[(size_t)u * kHeads * kVDim + i] = 0.f;
      }
      if (row < kHeads) {
        if (final_out) {
          if (p.lse) p.lse[d.b * kHeads + row] = -INFINITY;
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
    for (int t = 0; t < nt; ++t, ++it) {
      const int sb = it & 1;
      const int t0 = d.start + t * kTileRows;
      const int valid = min(kTileRows, d.end - t0);
      wait_phase(&x.bar[kSFull + sb], (it >> 1) & 1, x.abort_flag, p.ws_err);
      tc::fence_after();
      uint32_t acc[32];
      tc::ld32(tl + kColS + 32 * sb, acc);
      tc::wait_ld();
      tc::fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&x.bar[kSEmpty + sb]);
      float sv[16], mx[16];
#pragma unroll
      for (int h = 0; h < 16; ++h) {
        sv[h] = row < valid ? (__uint_as_float(acc[h]) + __uint_as_float(acc[16 + h])) * r[h] : -INFINITY;
        mx[h] = sv[h];
      }
      group_reduce16<true>(mx, redbuf + red_par * 64, ww, lane);
      red_par ^= 1;
      // lazy running max: raise m_ref only when a head's tile max exceeds it by > 8
      bool any = false;
      float fac[16];
#pragma unroll
      for (int h = 0; h < 16; ++h) {
        const bool up = mx[h] > m_ref[h] + kRescaleLog2;
        const float mn = up ? mx[h] : m_ref[h];
        fac[h] = (m_ref[h] == -INFINITY) ? 0.f : fast_exp2(m_ref[h] - mn);
        any |= up;
        m_ref[h] = mn;
      }
      if (any && t > 0) {
        // rescale O^T in TMEM once the previous tile's P.V is complete
        wait_phase(&x.bar[kODone], (it - 1) & 1, x.abort_flag, p.ws_err);
        tc::fence_after();
#pragma unroll 1
        for (int fb = 0; fb < 4; ++fb) {
          uint32_t o[32];
          tc::ld32(tl + kColO + 32 * fb, o);
          tc::wait_ld();
#pragma unroll
          for (int h = 0; h < 16; ++h) {
            o[h] = __float_as_uint(__uint_as_float(o[h]) * fac[h]);
            o[16 + h] = __float_as_uint(__uint_as_float(o[16 + h]) * fac[h]);
          }
          tc::st32(tl + kColO + 32 * fb, o);
        }
        tc::wait_st();
      }
      if (any) {
#pragma unroll
        for (int h = 0; h < 16; ++h) l_part[h] *= fac[h];
      }
      // probabilities (<= 256), two e4m3 terms, MN-major B operand row = this row
      uint32_t hi[4], lo[4];
#pragma unroll
      for (int g = 0; g < 4; ++g) {
        float pv[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int h = 4 * g + e;
          pv[e] = (m_ref[h] == -INFINITY) ? 0.f : fast_exp2(sv[h] - m_ref[h]);
          l_part[h] += pv[e];
        }
        two_term_e4m3(pv[0], pv[1], pv[2], pv[3], hi[g], lo[g]);
      }
      uint8_t* pbuf = x.smem + Layout::pb + sb * kPBytes + row * 32;
      const int xr = (row >> 2) & 1;  // 32 B swizzle: the 16-byte units of the row swap
      *reinterpret_cast<uint4*>(pbuf + 16 * xr) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
      *reinterpret_cast<uint4*>(pbuf + 16 * (xr ^ 1)) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
      if (row >= valid) {
        // rows past the unit's end hold other rows' data: zero their V part so
        // that P = 0 cannot meet a non-finite value
        uint8_t* st = x.smem + Layout::stages + (it & 1) * kStageBytes;
#pragma unroll
        for (int c = 0; c < 8; ++c)
#pragma unroll
          for (int uu = 0; uu < 4; ++uu)
            *reinterpret_cast<uint4*>(st + c * kChunkBytes + sw64_off(row, 16 * uu)) = make_uint4(0, 0, 0, 0);
      }
      tc::fence_proxy_async();
      tc::fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&x.bar[kPFull + sb]);
    }
    // unit epilogue: l per head over the 128 rows, O^T -> output
    group_reduce16<false>(l_part, redbuf + red_par * 64, ww, lane);
    red_par ^= 1;
    wait_phase(&x.bar[kODone], (it - 1) & 1, x.abort_flag, p.ws_err);
    tc::fence_after();
    float inv[16];
#pragma unroll
    for (int h = 0; h < 16; ++h) inv[h] = l_part[h] > 0.f ? kv_scale / l_part[h] : 0.f;
#pragma unroll 1
    for (int fb = 0; fb < 4; ++fb) {
      uint32_t o[32];
      tc::ld32(tl + kColO + 32 * fb, o);
      tc::wait_ld();
      const int f = 128 * fb + row;
      if (final_out) {
        uint16_t* ob = p.out + (size_t)d.b * kHeads * kVDim + f;
#pragma unroll
        for (int h = 0; h < 16; ++h) {
          const float v = (__uint_as_float(o[h]) + __uint_as_float(o[16 + h])) * inv[h];
          ob[h * kVDim] = (uint16_t)(pack_bf16x2(v, 0.f) & 0xffffu);
        }
      } else {
        float* ob = p.ws_o + (size_t)u * kHeads * kVDim + f;
#pragma unroll
        for (int h = 0; h < 16; ++h) ob[h * kVDim] = (__uint_as_float(o[h]) + __uint_as_float(o[16 + h])) * inv[h];
      }
    }
    if (row == 0) {
#pragma unroll
      for (int h = 0; h < 16; ++h) {
        const float lse = l_part[h] > 0.f ? (m_ref[h] + log2f(l_part[h])) * kLn2 : -INFINITY;
        if (final_out) {
          if (p.lse) p.lse[d.b * kHeads + h] = lse;
        } else {
          p.ws_lse[(size_t)u * kHeads + h] = lse;
        }
      }
    }
    tc::fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(&x.bar[kOFree]);
  }
}

__global__ void __launch_bounds__(kThreads, 1) mla_split_tc_kernel(const __grid_constant__ Stage1Params p) {
  extern __shared__ __align__(1024) uint8_t smem[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  Ctx x;
  x.smem = smem;
  x.units = reinterpret_cast<const UnitDesc*>(smem + Layout::units);
  x.bar = reinterpret_cast<uint64_t*>(smem + Layout::bars);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + Layout::misc);
  int* misc = reinterpret_cast<int*>(smem + Layout::misc);
  x.abort_flag = misc + 1;
  int* s_nunits = misc + 2;

  if (threadIdx.x == 0) {
    const uint32_t counts[Layout::nbars] = {1, 1, 1, 1, 2, 2, 1, 1, 1, 1, 4, 4, 4, 4, 1, 4, 4, 4, 1};
    for (int i = 0; i < Layout::nbars; ++i) mbar_init(&x.bar[i], counts[i]);
    *x.abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0) {
    scan_units<kTileRows>(p, reinterpret_cast<UnitDesc*>(smem + Layout::units), s_nunits, lane);
    if (lane == 0) prefetch_tensormap(&p.tmap_kv64);
  }
  if (warp == 1) {
    tc::alloc(tmem_slot, kTmemCols);
    tc::relinquish();
  }
  tc::fence_before();
  __syncthreads();
  tc::fence_after();
  pdl_launch_dependents();
  x.tmem = *tmem_slot;
  x.nunits = *s_nunits;

  if (warp == 0) {
    if (lane == 0) producer(p, x);
  } else if (warp == 1) {
    if (lane == 0) mma_issuer(p, x);
  } else if (warp < 4) {
    prep_query(p, x, threadIdx.x - 64);
  } else {
    softmax_epilogue(p, x, warp - 4, lane);
  }

  if (warp == 1 && lane == 0) {
    // every tensor-core operation of this CTA is complete before TMEM is freed
    tc::commit(&x.bar[kFinal]);
    const uint64_t t0 = global_timer_ns();
    while (!mbar_try_wait(&x.bar[kFinal], 0) && global_timer_ns() - t0 < kWaitTimeoutNs) {
    }
  }
  tc::fence_before();
  __syncthreads();
  tc::fence_after();
  if (warp == 1) tc::dealloc(x.tmem, kTmemCols);
}

}  // namespace tcfp8

inline cudaError_t launch_split_tc_fp8(const Stage1Params& p, cudaStream_t stream) {
  using L = tcfp8::Layout;
  static_assert(L::total <= 232448, "shared memory carve-up exceeds the 227 KB per-CTA limit");
  static_assert(L::qs % 1024 == 0 && L::pb % 1024 == 0, "swizzled operand alignment");
  cudaError_t e =
      cudaFuncSetAttribute(tcfp8::mla_split_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, L::total);
  if (e != cudaSuccess) return e;
  tcfp8::mla_split_tc_kernel<<<p.grid, tcfp8::kThreads, L::total, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace mla
