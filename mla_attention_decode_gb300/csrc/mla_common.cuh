// mla_common.cuh -- pieces shared by the decode kernels: the work-unit list,
// bounded mbarrier waits, small warp reductions and the two-term e4m3 encoding.
#pragma once
#include <cuda_runtime.h>

#include "mla_internal.h"
#include "mla_ptx.cuh"

namespace mla {

#ifndef MLA_TRACE
#define MLA_TRACE 0
#endif

// Trace builds: the global time (ns) at `slot` of this CTA's stamp row, or a
// count when `value` is given.  Compiled out of normal builds.
__device__ __forceinline__ void trace_stamp(const Stage1Params& p, int slot) {
#if MLA_TRACE
  if (p.trace != nullptr && slot >= 0 && slot < kTraceSlots)
    p.trace[(size_t)blockIdx.x * kTraceSlots + slot] = global_timer_ns();
#else
  (void)p;
  (void)slot;
#endif
}
__device__ __forceinline__ void trace_value(const Stage1Params& p, int slot, uint64_t value) {
#if MLA_TRACE
  if (p.trace != nullptr && slot >= 0 && slot < kTraceSlots) p.trace[(size_t)blockIdx.x * kTraceSlots + slot] = value;
#else
  (void)p;
  (void)slot;
  (void)value;
#endif
}

// Trace builds: the SM this CTA runs on.
__device__ __forceinline__ void trace_smid(const Stage1Params& p) {
#if MLA_TRACE
  uint32_t smid;
  asm volatile("mov.u32 %0, %%smid;" : "=r"(smid));
  trace_value(p, kTrSmid, smid);
#else
  (void)p;
#endif
}

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr uint64_t kWaitTimeoutNs = 4000000000ull;  // 4 s: a wait this long means a lost copy

struct UnitDesc {
  int32_t b, start, end, u;  // u: work unit index (two tokens per unit: token 0's partial slot);
                             // bit 31 set when the sequence has one split
  int32_t qrow;              // qo_indptr[b]: the sequence's query row; two tokens per unit:
                             // S_b, plus kLastUnitBit on the sequence's last unit
};
constexpr int32_t kFinalFlag = (int32_t)0x80000000;
constexpr int32_t kLastUnitBit = 1 << 30;

// Error tags (word 4 of the workspace) naming where an index error was seen
// (the bounded waits and the page lookups only set the error word: the
// recording below, inlined at their many call sites, cost the e4m3 split
// kernel registers and about 2 us at bs64/kv8192).
enum : int32_t {
  kTagScan = 3,         // the device kv_indptr / qo_indptr disagree with the plan (round-robin scan)
  kTagScanContig = 4,   // the same, contiguous-range scan
  kTagFirstTile = 5,    // the plan's first tile row is not the scan's (word 5: the row)
};
// Sets the workspace's error word to `code` unless an error is already there;
// the first error also leaves where it was seen: words 2-5 = CTA, thread, tag,
// detail.
__device__ __forceinline__ void flag_error(int32_t* ws_err, int32_t code, int32_t tag, int32_t detail) {
  if (atomicCAS(ws_err, 0, code) == 0) {
    ws_err[2] = (int32_t)blockIdx.x;
    ws_err[3] = (int32_t)threadIdx.x;
    ws_err[4] = tag;
    ws_err[5] = detail;
  }
}

// Bounded mbarrier wait.  Returns false (after flagging the error) if the phase
// did not complete within kWaitTimeoutNs, or immediately if another thread of
// the CTA already gave up; the caller then carries on without the data so that
// every warp still reaches the same named barriers and the kernel ends.
// The slow path of wait_phase, out of line: the many inlined waits then carry
// only the first try and a call (measured: 4 us off a bs32/kv8192 MXFP4 call,
// 1.2 us off bs64/kv8192 e4m3; the kernels' code size matters).
static __device__ __noinline__ bool wait_phase_slow(uint64_t* bar, uint32_t parity, volatile int* abort_flag,
                                                    int32_t* ws_err) {
  const uint64_t t0 = global_timer_ns();
  while (true) {
    if (*abort_flag) return false;
    // sleep in the barrier (up to 0.1 ms per try) instead of spinning, so that
    // waiting warps leave the issue slots to the warps doing work
    if (mbar_try_wait_sleep(bar, parity, 100000u)) return true;
    if (global_timer_ns() - t0 > kWaitTimeoutNs) {
      *abort_flag = 1;
      atomicCAS(ws_err, 0, kErrDeviceTimeout);
      return false;
    }
  }
}
__device__ __forceinline__ bool wait_phase(uint64_t* bar, uint32_t parity, volatile int* abort_flag,
                                           int32_t* ws_err) {
  if (mbar_try_wait(bar, parity)) return true;
  return wait_phase_slow(bar, parity, abort_flag, ws_err);
}

// Rows [start, end) of sequence b in the row space the tiles walk: the cache
// rows themselves, or for a paged cache the page-ordered positions
// kv_indptr[b] * P + i (i below the sequence's token count: P rows per page,
// kv_last[b] in the last one).  False for a layout the rules forbid.
__device__ __forceinline__ bool seq_rows(const Stage1Params& p, int b, int& start, int& end) {
  if (p.q_len > 1) {
    // token b % q_len of sequence b / q_len: the rows up to its own entry
    const int s = b / p.q_len, i = b - s * p.q_len;
    const int a = p.kv_indptr[s], z = p.kv_indptr[s + 1];
    start = a;
    end = max(a, z - (p.q_len - 1 - i));
    return a >= 0 && z >= a;
  }
  const int a = p.kv_indptr[b], z = p.kv_indptr[b + 1];
  if (!p.paged) {
    start = a;
    end = z;
    return a >= 0 && z >= a;
  }
  if (a < 0 || z < a || z > (p.total_kv >> p.page_shift)) return false;
  start = a << p.page_shift;
  end = start;
  if (z > a) {
    const int last = p.kv_last[b];
    if (last < 1 || last > (1 << p.page_shift)) return false;
    end = start + ((z - a - 1) << p.page_shift) + last;
  }
  return true;
}

// Query row of output row b (a sequence, or with several tokens per sequence
// token b % q_len of sequence b / q_len).
__device__ __forceinline__ int query_row(const Stage1Params& p, int b) {
  if (p.q_len > 1) {
    const int s = b / p.q_len;
    return p.qo_indptr[s] + (b - s * p.q_len);
  }
  return p.qo_indptr[b];
}

// Rows and query check of unit-list entry b: output row b (its own rows,
// query row qo_indptr-derived), or with TOK = 2 tokens per unit sequence b,
// whose full rows both tokens' units cover; qrow < 0 flags a bad query row.
template <int TOK>
__device__ __forceinline__ bool entry_rows(const Stage1Params& p, int b, int& start, int& end, int& qrow) {
  if constexpr (TOK > 1) {
    const int a = p.kv_indptr[b], z = p.kv_indptr[b + 1];
    start = a;
    end = z;
    qrow = query_row(p, TOK * b);  // the sequence's tokens are query rows qrow, qrow + 1, ...
    return a >= 0 && z >= a;
  } else {
    qrow = query_row(p, b);
    return seq_rows(p, b, start, end);
  }
}

// Cache row of row-space position v (a row of some sequence): v itself, or for
// a paged cache row v % P of page kv_indices[v / P].  A page index outside
// [0, num_pages) is flagged and page 0 is read instead.
__device__ __forceinline__ int cache_row(const Stage1Params& p, int v) {
  if (!p.paged) return v;
  int pg = __ldg(p.kv_indices + (v >> p.page_shift));
  if ((unsigned)pg >= (unsigned)p.num_pages) {
    atomicCAS(p.ws_err, 0, kErrDeviceIndex);
    pg = 0;
  }
  return (pg << p.page_shift) | (v & ((1 << p.page_shift) - 1));
}

// Order-preserving map of floats (no NaN) to signed integers, for integer
// max reductions (redux.sync): non-negative floats keep their bits, negative
// ones have the magnitude bits flipped.
__device__ __forceinline__ int float_order_key(float f) {
  const int i = __float_as_int(f);
  return i >= 0 ? i : i ^ 0x7FFFFFFF;
}
__device__ __forceinline__ float float_from_order_key(int k) { return __int_as_float(k >= 0 ? k : k ^ 0x7FFFFFFF); }

__device__ __forceinline__ float quad_max(float v) {
  v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 1));
  v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 2));
  return v;
}
__device__ __forceinline__ float quad_sum(float v) {
  v += __shfl_xor_sync(0xffffffffu, v, 1);
  v += __shfl_xor_sync(0xffffffffu, v, 2);
  return v;
}

// Byte (row, col) of a block of 64-byte rows in the tcgen05 64-byte swizzle
// (16-byte units of a row permuted by bits 1-2 of the row; block 512-byte aligned).
__device__ __forceinline__ uint32_t sw64_off(int row, int col) {
  return (uint32_t)(row * 64 + ((((col >> 4) ^ (row >> 1)) & 3) << 4) + (col & 15));
}

// Two-term e4m3 encoding of four floats: hi = e4m3(x), lo = e4m3(x - hi).
// Byte i of each word holds element i.
__device__ __forceinline__ void two_term_e4m3(float x0, float x1, float x2, float x3, uint32_t& hi,
                                              uint32_t& lo) {
  const uint32_t h01 = f32x2_to_e4m3x2(x0, x1), h23 = f32x2_to_e4m3x2(x2, x3);
  const float2 b01 = __half22float2(e4m3x2_to_h2(h01));
  const float2 b23 = __half22float2(e4m3x2_to_h2(h23));
  hi = h01 | (h23 << 16);
  lo = f32x2_to_e4m3x2(x0 - b01.x, x1 - b01.y) | (f32x2_to_e4m3x2(x2 - b23.x, x3 - b23.y) << 16);
}

__device__ __forceinline__ float4 bf16x4_to_f4(uint2 v) {
  return make_float4(__uint_as_float(v.x << 16), __uint_as_float(v.x & 0xffff0000u),
                     __uint_as_float(v.y << 16), __uint_as_float(v.y & 0xffff0000u));
}

// ------------------------------------------------------------- unit list
// Walks kv_indptr (one warp, 32 sequences per step) and writes the units owned
// by this CTA to smem; CTA 0 also writes the per-sequence split table used by
// the combine kernel.  Sequence b is cut into S_b splits on TILE-row tile
// boundaries.  Inconsistent index data raises MLA_ERR_DEVICE_INDEX and the
// affected sequences are treated as empty.
template <int TILE>
__device__ __forceinline__ int splits_of(int len, int chunk, int cap) {
  if (len <= 0) return 1;
  const int tiles = (len + TILE - 1) / TILE;
  int s = (int)(((long long)len + chunk - 1) / chunk);
  s = min(s, cap);
  s = min(s, tiles);
  return max(s, 1);
}

// Schedule 1 (contiguous tile ranges): sequence b weighs w_b = max(1, T_b)
// tiles, laid end to end with unit_cost empty positions between consecutive
// sequences (C positions in all); CTA c owns positions [B(c), B(c+1)) with
// B(c) = floor(c C' / G) - D max(0, c - (G - L)), C' = C + L D (the last L =
// late_ctas CTAs, which start behind the others, own D = late_tiles positions
// fewer), and takes one unit from every sequence whose tiles overlap its range.
template <int TILE, int MAX_UNITS, int TOK>
__device__ __forceinline__ void scan_units_contiguous(const Stage1Params& p, UnitDesc* units, int* s_nunits,
                                                      int lane) {
  const long long T = p.total_tiles, G = p.grid, c = blockIdx.x, U = p.unit_cost;
  const int nseq = p.batch / TOK;       // unit-list entries: sequences of a two-token plan
  const int nunits = p.num_work / TOK;  // work units (num_work counts partial slots)
  const long long C = T + U * (nseq > 0 ? nseq - 1 : 0);
  const long long L = p.late_ctas, D = p.late_tiles, Cp = C + L * D;
  auto bound = [&](long long k) { return k * Cp / G - D * (k > G - L ? k - (G - L) : 0); };
  const long long lo = bound(c), hi = bound(c + 1), late0 = bound(G - L);
  auto cta_of = [&](long long x) {
    return (D == 0 || x < late0) ? ((x + 1) * G - 1) / Cp : ((x - D * (G - L) + 1) * G - 1) / (Cp - D * G);
  };
  long long tprefix = 0;  // tiles of the sequences before this chunk of 32
  int uprefix = 0, count = 0;
  bool bad = false;
  for (int b0 = 0; b0 < nseq; b0 += 32) {
    const int b = b0 + lane;
    int start = 0, end = 0, qrow = 0, w = 0;
    if (b < nseq) {
      if (!entry_rows<TOK>(p, b, start, end, qrow) || end > p.total_kv || qrow < 0) {
        bad = true;
        start = end = qrow = 0;
      }
      w = end > start ? (end - start + TILE - 1) / TILE : 1;
    }
    int wincl = w;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int t = __shfl_up_sync(0xffffffffu, wincl, o);
      if (lane >= o) wincl += t;
    }
    const long long P = tprefix + wincl - w;  // tiles before sequence b
    const long long X = P + U * b;            // position of its first tile
    int sb = 0, cf = 0;
    if (b < nseq) {
      if (P + w > T) {
        bad = true;  // the device kv_indptr holds more tiles than the plan
      } else {
        cf = (int)cta_of(X);
        sb = (int)(cta_of(X + w - 1) - cf + 1);
      }
    }
    int sincl = sb;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int t = __shfl_up_sync(0xffffffffu, sincl, o);
      if (lane >= o) sincl += t;
    }
    const int ub = uprefix + sincl - sb;  // first unit of sequence b
    if (blockIdx.x == 0 && b < nseq) {
      // split table for the combine kernel, per output row (token i of a
      // two-token entry: slots TOK ub + i S_b ..); never point past the plan's slots
      const bool fits = ub + sb <= nunits;
#pragma unroll
      for (int i = 0; i < TOK; ++i) {
        p.ws_seq[2 * (TOK * b + i)] = fits ? TOK * ub + i * sb : 0;
        p.ws_seq[2 * (TOK * b + i) + 1] = fits ? sb : 0;
      }
    }
    // a unit past the plan's slots is not taken, and not counted (the list stays gap-free)
    const bool over = sb > 0 && c >= cf && c < cf + sb && ub + (int)(c - cf) >= nunits;
    if (over) bad = true;
    const bool mine = sb > 0 && c >= cf && c < cf + sb && !over;
    const unsigned m = __ballot_sync(0xffffffffu, mine);
    if (mine) {
      const int pos = count + __popc(m & ((1u << lane) - 1));
      const int u = ub + (int)(c - cf);
      if (pos >= MAX_UNITS) {
        bad = true;
      } else {
        const long long a = (lo > X ? lo : X) - X, e = (hi < X + w ? hi : X + w) - X;  // the sequence's tiles here
        UnitDesc d;
        d.b = b;
        d.start = end > start ? start + TILE * (int)a : start;
        d.end = end > start ? min(end, start + TILE * (int)e) : start;
        d.u = (TOK * ub + (u - ub)) | (sb == 1 ? kFinalFlag : 0);
        d.qrow = TOK > 1 ? (sb | (c == cf + sb - 1 ? kLastUnitBit : 0)) : qrow;
        units[pos] = d;
      }
    }
    count += __popc(m);
    tprefix += __shfl_sync(0xffffffffu, wincl, 31);
    uprefix += __shfl_sync(0xffffffffu, sincl, 31);
  }
  if (tprefix != T || uprefix != nunits) bad = true;
  bad = __any_sync(0xffffffffu, bad);
  if (lane == 0) {
    if (bad) flag_error(p.ws_err, kErrDeviceIndex, kTagScanContig, 0);
    *s_nunits = min(count, MAX_UNITS);
  }
}

// TOK: output rows per unit-list entry (2: a two-token plan, whose entries are
// sequences and whose units serve both tokens; compile-time, so that the
// one-token scan carries none of it).
template <int TILE, int MAX_UNITS = kMaxUnitsPerCta, int TOK = 1>
__device__ __forceinline__ void scan_units(const Stage1Params& p, UnitDesc* units, int* s_nunits, int lane) {
  if (p.schedule == 1) {
    scan_units_contiguous<TILE, MAX_UNITS, TOK>(p, units, s_nunits, lane);
    return;
  }
  const int nseq = p.batch / TOK;       // unit-list entries: sequences of a two-token plan
  const int nunits = p.num_work / TOK;  // work units (num_work counts partial slots)
  int prefix = 0, count = 0;
  bool bad = false;
  for (int b0 = 0; b0 < nseq; b0 += 32) {
    const int b = b0 + lane;
    int start = 0, end = 0, sb = 0, qrow = 0;
    if (b < nseq) {
      if (!entry_rows<TOK>(p, b, start, end, qrow) || end > p.total_kv || qrow < 0) {
        bad = true;
        start = end = 0;
        qrow = 0;
      }
      sb = splits_of<TILE>(end - start, p.chunk_tokens, p.max_splits);
    }
    int incl = sb;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int t = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += t;
    }
    const int pb = prefix + incl - sb;
    if (blockIdx.x == 0 && b < nseq) {
      // split table for the combine kernel (as in the contiguous schedule);
      // never point past the plan's slots
      const bool fits = pb + sb <= nunits;
#pragma unroll
      for (int i = 0; i < TOK; ++i) {
        p.ws_seq[2 * (TOK * b + i)] = fits ? TOK * pb + i * sb : 0;
        p.ws_seq[2 * (TOK * b + i) + 1] = fits ? sb : 0;
      }
    }
    int n = 0, first = 0;
    if (b < nseq) {
      int off = (int)(((long long)blockIdx.x - pb) % p.grid);
      if (off < 0) off += p.grid;
      first = pb + off;
      if (first < pb + sb) n = (pb + sb - 1 - first) / p.grid + 1;
      // units past the plan's slots (a device kv_indptr with more splits than
      // the plan's) are not taken, and not counted: the list stays gap-free
      if (n > 0 && first + (n - 1) * p.grid >= nunits) {
        bad = true;
        n = first < nunits ? (nunits - 1 - first) / p.grid + 1 : 0;
      }
    }
    int nincl = n;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int t = __shfl_up_sync(0xffffffffu, nincl, o);
      if (lane >= o) nincl += t;
    }
    const int pos = count + nincl - n;
    const int tiles = (end - start + TILE - 1) / TILE;
    for (int k = 0; k < n; ++k) {
      const int u = first + k * p.grid;
      const int s = u - pb;
      if (pos + k >= MAX_UNITS) {
        bad = true;
        continue;
      }
      UnitDesc d;
      d.b = b;
      d.start = start + TILE * (int)((long long)s * tiles / sb);
      d.end = min(end, start + TILE * (int)((long long)(s + 1) * tiles / sb));
      d.u = (TOK * pb + s) | (sb == 1 ? kFinalFlag : 0);
      d.qrow = TOK > 1 ? (sb | (s == sb - 1 ? kLastUnitBit : 0)) : qrow;
      units[pos + k] = d;
    }
    count += __shfl_sync(0xffffffffu, nincl, 31);
    prefix += __shfl_sync(0xffffffffu, incl, 31);
  }
  if (prefix != nunits) bad = true;
  bad = __any_sync(0xffffffffu, bad);
  if (lane == 0) {
    if (bad) flag_error(p.ws_err, kErrDeviceIndex, kTagScan, 0);
    *s_nunits = min(count, MAX_UNITS);
  }
}

// Cursor over the CTA's KV tiles in consumption order (unit by unit, TILE rows
// at a time).  Warps that need it keep identical copies.
struct TileCursor {
  int k;   // unit index in the CTA's list
  int t0;  // first row of the tile
};
__device__ __forceinline__ void cursor_skip_empty(TileCursor& c, const UnitDesc* units, int nunits) {
  while (c.k < nunits && units[c.k].start >= units[c.k].end) ++c.k;
  c.t0 = c.k < nunits ? units[c.k].start : 0;
}
template <int TILE>
__device__ __forceinline__ void cursor_next(TileCursor& c, const UnitDesc* units, int nunits) {
  c.t0 += TILE;
  if (c.t0 >= units[c.k].end) {
    ++c.k;
    cursor_skip_empty(c, units, nunits);
  }
}

}  // namespace mla
