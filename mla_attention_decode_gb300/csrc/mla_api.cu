// mla_api.cu -- C ABI of libmla_decode.so: split planner, workspace sizing,
// argument validation and kernel launches (see include/mla_decode.h).
#include <cmath>
#include <cstdint>
#include <cstring>
#include <vector>

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include "mla_decode.h"
#include "mla_internal.h"

namespace {

using mla::kHeads;
using mla::kTile;
using mla::kVDim;

constexpr int32_t kNoCap = 1 << 30;

// KV rows per pipeline tile of each kernel: 64 (bf16, warp-level MMA) or 128
// (e4m3 and e2m1, one tcgen05 M=128 block).  Splits end on tile boundaries.
int tile_rows(int kv_dtype) { return kv_dtype == MLA_KV_BF16 ? 64 : 128; }

int rows_bytes(int kv_dtype) {
  switch (kv_dtype) {
    case MLA_KV_BF16: return 1152;
    case MLA_KV_FP8_E4M3: return 576;
    default: return 288 + 18;
  }
}

// Split count of a sequence of `len` rows (the rule stated in mla_decode.h):
// ceil(len / chunk), capped by `cap` and by the number of 64-row tiles.
int32_t splits_for(int64_t len, int32_t chunk, int32_t cap, int tile) {
  if (len <= 0) return 1;
  int64_t s = (len + chunk - 1) / chunk;
  const int64_t tiles = (len + tile - 1) / tile;
  if (s > cap) s = cap;
  if (s > tiles) s = tiles;
  return static_cast<int32_t>(s < 1 ? 1 : s);
}

// Rows of split i of S of a sequence of len rows (splits end on tile boundaries).
int64_t split_rows(int64_t len, int32_t i, int32_t s, int tile) {
  if (len <= 0) return 0;
  const int64_t tiles = (len + tile - 1) / tile;
  const int64_t a = tile * (i * tiles / s);
  int64_t b = tile * ((i + 1) * tiles / s);
  if (b > len) b = len;
  return b - a;
}

// Modelled duration (in units of one pipeline tile of this dtype) of a plan:
// the busiest CTA's tiles plus a fixed cost per unit, plus the combine kernel
// when any sequence is split (a fixed part and its partial traffic spread over
// the SMs).  Units are dealt round-robin, as the kernel does.
double plan_cost(const std::vector<int64_t>& lens, int32_t chunk, int32_t cap, int num_sms, int kv_dtype,
                 int64_t* work_out) {
  const double kUnitCost = 0.5, kCombineFixed = 2.0;
  const int tile = tile_rows(kv_dtype);
  int64_t work = 0, split_units = 0;
  for (int64_t L : lens) {
    const int32_t s = splits_for(L, chunk, cap, tile);
    work += s;
    if (s > 1) split_units += s;
  }
  *work_out = work;
  if (work == 0) return 0.0;
  const int64_t grid = work < num_sms ? work : num_sms;
  std::vector<double> load(static_cast<size_t>(grid), 0.0);
  int64_t u = 0;
  for (int64_t L : lens) {
    const int32_t s = splits_for(L, chunk, cap, tile);
    for (int32_t i = 0; i < s; ++i, ++u) {
      const int64_t rows = split_rows(L, i, s, tile);
      load[static_cast<size_t>(u % grid)] += (double)((rows + tile - 1) / tile) + kUnitCost;
    }
  }
  double mk = 0.0;
  for (double v : load) mk = v > mk ? v : mk;
  if (split_units > 0) {
    const double tile_bytes = (double)tile * rows_bytes(kv_dtype);
    const double partial_bytes = (double)kHeads * (kVDim + 1) * 4.0;
    mk += kCombineFixed + (double)split_units * partial_bytes / ((double)num_sms * tile_bytes);
  }
  return mk;
}

// Schedule 1 (contiguous tile ranges, see mla_decode.h): the sequences' tiles
// laid end to end with unit_cost empty positions between consecutive
// sequences, C positions in all; CTA c of G owns positions [lo(c), lo(c+1)),
// the last L CTAs (late_ctas) D positions (late_tiles) fewer than the others,
// and cta(x) is the CTA owning position x.
struct Partition {
  int64_t C, G, L, D;
  int64_t lo(int64_t c) const {
    const int64_t Cp = C + L * D;
    return c * Cp / G - D * (c > G - L ? c - (G - L) : 0);
  }
  int64_t cta(int64_t x) const {
    const int64_t Cp = C + L * D;
    if (D == 0 || x < lo(G - L)) return ((x + 1) * G - 1) / Cp;
    return ((x - D * (G - L) + 1) * G - 1) / (Cp - D * G);
  }
};
// The late CTAs: e4m3 and MXFP4 plans start the split kernel while the
// query-preparation grid (one CTA per output row) still holds SMs, and the
// hardware places the split CTAs of the highest indices on those SMs once
// they are free; a per-CTA trace puts them about 3.3 us behind (two e4m3
// tiles, one MXFP4 or two-token tile).  Those CTAs get D positions fewer.
int64_t late_ctas(int64_t G, int64_t prep_rows, int64_t num_sms) {
  const int64_t l = G + prep_rows - num_sms;
  return l <= 0 ? 0 : (l < G ? l : G);
}

struct BalancedPlan {
  int64_t T = 0, C = 0, G = 0, work = 0, L = 0, D = 0;
  int32_t smax = 0, max_units = 0, unit_cost = 0;
  double cost = -1.0;
};

// A unit boundary inside a CTA (the epilogue of one unit, the next unit's
// query and the refill of the ring) costs about two e4m3 tiles of pipeline
// time, and about one of MXFP4's longer tiles; schedule 1 gives each boundary
// that weight when the CTAs have at least U + 2 tiles each (below that the
// weight would leave CTAs without tiles).  Measured against weights one
// higher and one lower: e4m3 bs64/kv8192 split stage 65.5 us against 66.6 (1)
// and 66.1 (3); MXFP4 bs32/kv8192 51.6 us (1) against 53.6 (2) and 54.5 (3).
#ifndef MLA_UNIT_COST
#define MLA_UNIT_COST 2
#endif
#ifndef MLA_UNIT_COST_MXFP4
#define MLA_UNIT_COST_MXFP4 1
#endif
int32_t schedule_unit_cost(int kv_dtype) {
  return kv_dtype == MLA_KV_MXFP4 ? MLA_UNIT_COST_MXFP4 : MLA_UNIT_COST;
}

// The busiest CTA's tiles plus kUnitCost per unit it owns, plus the combine
// (same model as plan_cost).
BalancedPlan plan_balanced(const std::vector<int64_t>& lens, int num_sms, int kv_dtype, int64_t prep_rows,
                           int64_t late_tiles) {
  const double kUnitCost = 0.5, kCombineFixed = 2.0;
  const int tile = tile_rows(kv_dtype);
  BalancedPlan bp;
  for (int64_t L : lens) bp.T += L > 0 ? (L + tile - 1) / tile : 1;
  if (bp.T == 0) return bp;
  bp.G = bp.T < num_sms ? bp.T : num_sms;
  const int64_t B = static_cast<int64_t>(lens.size());
  const int32_t U = schedule_unit_cost(kv_dtype);
  bp.unit_cost = bp.T >= (U + 2) * bp.G ? U : 0;
  bp.C = bp.T + bp.unit_cost * (B - 1);
  // the late CTAs' share, when every CTA keeps at least two positions
  bp.L = late_ctas(bp.G, prep_rows, num_sms);
  bp.D = (bp.L > 0 && bp.C + bp.L * late_tiles >= (late_tiles + 2) * bp.G) ? late_tiles : 0;
  if (bp.D == 0) bp.L = 0;
  const Partition part{bp.C, bp.G, bp.L, bp.D};
  std::vector<int64_t> tiles(static_cast<size_t>(bp.G), 0);
  std::vector<int32_t> units(static_cast<size_t>(bp.G), 0);
  int64_t P = 0, split_units = 0;
  for (int64_t b = 0; b < B; ++b) {
    const int64_t L = lens[static_cast<size_t>(b)];
    const int64_t w = L > 0 ? (L + tile - 1) / tile : 1;
    const int64_t x = P + bp.unit_cost * b;  // position of the sequence's first tile
    const int64_t cf = part.cta(x), cl = part.cta(x + w - 1);
    const int64_t s = cl - cf + 1;
    bp.work += s;
    if (s > 1) split_units += s;
    bp.smax = s > bp.smax ? static_cast<int32_t>(s) : bp.smax;
    for (int64_t c = cf; c <= cl; ++c) {
      const int64_t lo = part.lo(c), hi = part.lo(c + 1);
      tiles[static_cast<size_t>(c)] += (hi < x + w ? hi : x + w) - (lo > x ? lo : x);
      units[static_cast<size_t>(c)] += 1;
    }
    P += w;
  }
  double mk = 0.0;
  for (int64_t c = 0; c < bp.G; ++c) {
    const double load = (double)tiles[static_cast<size_t>(c)] + kUnitCost * units[static_cast<size_t>(c)];
    mk = load > mk ? load : mk;
    bp.max_units = units[static_cast<size_t>(c)] > bp.max_units ? units[static_cast<size_t>(c)] : bp.max_units;
  }
  if (split_units > 0) {
    const double tile_bytes = (double)tile * rows_bytes(kv_dtype);
    const double partial_bytes = (double)kHeads * (kVDim + 1) * 4.0;
    mk += kCombineFixed + (double)split_units * partial_bytes / ((double)num_sms * tile_bytes);
  }
  bp.cost = mk;
  return bp;
}

// cuTensorMapEncodeTiled from the driver, fetched through the runtime once.
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = []() -> PFN_cuTensorMapEncodeTiled_v12000 {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess) {
      cudaGetLastError();
      return nullptr;
    }
    return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  }();
  return fn;
}

// KV rows viewed as (span bytes, 9 chunks, rows) with the matching swizzle, so a
// box of `box_rows` rows lands densely in smem with 16-byte units permuted.
// e4m3 KV rows as a 2-D byte tensor (576, rows); a box is one 64-byte column
// block of box_rows rows, landed with the 64-byte swizzle (the tcgen05 operand layout).
bool encode_kv_map_tc(CUtensorMap* m, const void* kv, int32_t total_kv, uint32_t box_rows) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
  if (!enc) return false;
  const cuuint64_t dims[2] = {576, (cuuint64_t)(total_kv > 0 ? total_kv : 1)};
  const cuuint64_t strides[1] = {576};
  const cuuint32_t box[2] = {64, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(kv), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// e4m3 rows, a box of 128 B (both column blocks of a pair) x box_rows rows
// with the 128-byte swizzle.
bool encode_kv_map_pairs(CUtensorMap* m, const void* kv, int32_t total_kv, uint32_t box_rows) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
  if (!enc) return false;
  const cuuint64_t dims[2] = {576, (cuuint64_t)(total_kv > 0 ? total_kv : 1)};
  const cuuint64_t strides[1] = {576};
  const cuuint32_t box[2] = {128, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(kv), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// MXFP4 rows (288 packed bytes, element 2i in the low nibble of byte i) for the
// block-scaled kernel: the 512 V features as 4 groups of 128 e2m1 elements in
// the 16U4_ALIGN16B form (each 16 elements land in 16 bytes of shared memory,
// 8 packed bytes then 8 zero bytes; 128-byte swizzle), one group x box_rows
// rows per box (kv 32-byte aligned); and the rows as bytes, for the rope
// block's 32 bytes (at byte 256) x box_rows rows.
constexpr cuuint64_t kMxRowBytes = MLA_QK_DIM / 2;
bool encode_kv_maps_mx(CUtensorMap* m4, CUtensorMap* m8, const void* kv, int32_t total_kv, uint32_t box_rows) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
  if (!enc) return false;
  const cuuint64_t rows = (cuuint64_t)(total_kv > 0 ? total_kv : 1);
  const cuuint64_t dims4[3] = {128, 4, rows};
  const cuuint64_t strides4[2] = {64, kMxRowBytes};
  const cuuint32_t box4[3] = {128, 1, box_rows};
  const cuuint32_t estr[3] = {1, 1, 1};
  if (enc(m4, CU_TENSOR_MAP_DATA_TYPE_16U4_ALIGN16B, 3, const_cast<void*>(kv), dims4, strides4, box4, estr,
          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return false;
  const cuuint64_t dims8[2] = {kMxRowBytes, rows};
  const cuuint64_t strides8[1] = {kMxRowBytes};
  const cuuint32_t box8[2] = {32, box_rows};
  return enc(m8, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(kv), dims8, strides8, box8, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool encode_kv_map(CUtensorMap* m, const void* kv, int kv_dtype, int32_t total_kv, uint32_t box_rows) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
  if (!enc) return false;
  const uint32_t span = kv_dtype == MLA_KV_BF16 ? 128 : (kv_dtype == MLA_KV_FP8_E4M3 ? 64 : 32);
  const CUtensorMapSwizzle sw = kv_dtype == MLA_KV_BF16 ? CU_TENSOR_MAP_SWIZZLE_128B
                                : (kv_dtype == MLA_KV_FP8_E4M3 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_32B);
  const cuuint64_t dims[3] = {span, 9, (cuuint64_t)(total_kv > 0 ? total_kv : 1)};
  const cuuint64_t strides[2] = {span, 9ull * span};
  const cuuint32_t box[3] = {span, 9, box_rows};
  const cuuint32_t estr[3] = {1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(kv), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int device_sm_count(int32_t* out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return MLA_ERR_NO_DEVICE;
  }
  int n = 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) {
    cudaGetLastError();
    return MLA_ERR_CUDA;
  }
  *out = n;
  return MLA_OK;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// plan->first_row (mla_decode.h): the first row of the first non-empty unit of
// each CTA, by the unit rules of the plan's schedule (contiguous single-token
// plans; the others say -1).
void fill_first_rows(mla_plan* plan, const int32_t* kv_indptr_host) {
  for (int c = 0; c < MLA_PLAN_FIRST_ROWS; ++c) plan->first_row[c] = -1;
  if (!kv_indptr_host || plan->batch <= 0 || plan->grid <= 0) return;
  const int64_t B = plan->batch, G = plan->grid, R = plan->tile_tokens;
  auto set = [&](int64_t c, int64_t row) {
    if (c >= 0 && c < MLA_PLAN_FIRST_ROWS && plan->first_row[c] < 0) plan->first_row[c] = static_cast<int32_t>(row);
  };
  if (plan->schedule == 1) {
    const int64_t U = plan->unit_cost, T = plan->total_tiles, C = T + U * (B - 1);
    const int64_t D = plan->late_tiles, L = D > 0 ? late_ctas(G, plan->batch, plan->num_sms) : 0;
    const Partition part{C, G, L, D};
    int64_t P = 0;
    for (int64_t b = 0; b < B; ++b) {
      const int64_t L = (int64_t)kv_indptr_host[b + 1] - kv_indptr_host[b];
      const int64_t w = L > 0 ? (L + R - 1) / R : 1;
      const int64_t X = P + U * b;
      if (L > 0)
        for (int64_t c = part.cta(X); c <= part.cta(X + w - 1); ++c) {
          const int64_t lo = part.lo(c);
          set(c, kv_indptr_host[b] + R * ((lo > X ? lo : X) - X));
        }
      P += w;
    }
  } else {
    int64_t u = 0;
    for (int64_t b = 0; b < B; ++b) {
      const int64_t L = (int64_t)kv_indptr_host[b + 1] - kv_indptr_host[b];
      const int32_t S = splits_for(L, plan->chunk_tokens, plan->max_splits, static_cast<int>(R));
      const int64_t t = (L + R - 1) / R;
      for (int32_t sp = 0; sp < S; ++sp, ++u)
        if (L > 0) set(u % G, kv_indptr_host[b] + R * ((int64_t)sp * t / S));
    }
  }
}

// Trace builds: the stamp buffer of the split kernel's launches (null: off).
uint64_t* g_trace = nullptr;

// The plan of a batch of sequences with lengths `lens` whose rows span
// [0, total_kv) of the row space the kernels walk (see mla_decode.h).
// Positions a late CTA gives up (see late_ctas): e4m3 one token per unit,
// MXFP4 and the two-token e4m3 form; none for bf16 (no query preparation).
#ifndef MLA_LATE_TILES_E4M3
#define MLA_LATE_TILES_E4M3 2
#endif
#ifndef MLA_LATE_TILES_OTHER
#define MLA_LATE_TILES_OTHER 1
#endif
int64_t late_tiles_for(int32_t kv_dtype, bool fused) {
  if (kv_dtype == MLA_KV_BF16) return 0;
  return (kv_dtype == MLA_KV_FP8_E4M3 && !fused) ? MLA_LATE_TILES_E4M3 : MLA_LATE_TILES_OTHER;
}

// prep_rows: output rows (the query-preparation grid); fused: the two-token e4m3 form
int plan_lengths(const std::vector<int64_t>& lens, int32_t total_kv, int32_t kv_dtype, int32_t num_sms,
                 int32_t num_splits, mla_plan* plan, int64_t prep_rows, bool fused = false) {
  const int32_t batch = static_cast<int32_t>(lens.size());
  int64_t lmax = 0;
  for (int64_t L : lens) lmax = L > lmax ? L : lmax;
  int32_t sms = num_sms;
  if (sms <= 0) {
    const int rc = device_sm_count(&sms);
    if (rc != MLA_OK) return rc;
  }
  const int64_t unit_cap = (int64_t)sms * mla::max_units_per_cta(kv_dtype);

  int32_t chunk = 1, cap = kNoCap;
  int64_t work = 0;
  double rr_cost = -1.0;
  if (num_splits > 0) {
    chunk = 1;
    cap = num_splits;
    plan_cost(lens, chunk, cap, sms, kv_dtype, &work);
    if (work > unit_cap) return MLA_ERR_UNSUPPORTED;
  } else {
    const int tile = tile_rows(kv_dtype);
    // candidates: split counts 1..256 of the longest sequence, as 64-row multiples
    double best = -1.0;
    int32_t best_chunk = 0;
    int32_t prev = -1;
    const int64_t lref = lmax > 0 ? lmax : 1;
    for (int s = 1; s <= 256; ++s) {
      int64_t c = (lref + s - 1) / s;
      c = (c + tile - 1) / tile * tile;
      if (c > lref) c = lref;
      if (c < 1) c = 1;
      if (c == prev) continue;
      prev = static_cast<int32_t>(c);
      int64_t w = 0;
      const double cost = plan_cost(lens, static_cast<int32_t>(c), kNoCap, sms, kv_dtype, &w);
      if (w > unit_cap) continue;
      if (best < 0.0 || cost < best - 1e-9) {
        best = cost;
        best_chunk = static_cast<int32_t>(c);
      }
      if (c <= tile) break;
    }
    chunk = best_chunk;
    cap = kNoCap;
    rr_cost = best;
    if (best >= 0.0) plan_cost(lens, chunk, cap, sms, kv_dtype, &work);
    // the contiguous schedule, when it is cheaper (or the only one that fits)
    const BalancedPlan bp = plan_balanced(lens, sms, kv_dtype, prep_rows, late_tiles_for(kv_dtype, fused));
    if (bp.cost >= 0.0 && bp.max_units <= mla::max_units_per_cta(kv_dtype) && bp.work <= INT32_MAX &&
        bp.C <= INT32_MAX && (rr_cost < 0.0 || bp.cost < rr_cost - 1e-9)) {
      mla_plan p;
      std::memset(&p, 0, sizeof p);
      p.batch = batch;
      p.kv_dtype = kv_dtype;
      p.total_kv = total_kv;
      p.chunk_tokens = tile_rows(kv_dtype);
      p.max_splits = kNoCap;
      p.num_work = static_cast<int32_t>(bp.work);
      p.grid = static_cast<int32_t>(bp.G);
      p.num_sms = sms;
      p.splits_max = bp.smax;
      p.tile_tokens = tile_rows(kv_dtype);
      p.units_per_cta = bp.max_units;
      p.schedule = 1;
      p.total_tiles = static_cast<int32_t>(bp.T);
      p.unit_cost = bp.unit_cost;
      p.late_tiles = static_cast<int32_t>(bp.D);
      for (int c = 0; c < MLA_PLAN_FIRST_ROWS; ++c) p.first_row[c] = -1;
      *plan = p;
      return MLA_OK;
    }
    if (best < 0.0) return MLA_ERR_UNSUPPORTED;  // too many sequences for the unit table
  }
  if (work > INT32_MAX) return MLA_ERR_UNSUPPORTED;
  int32_t smax = 0;
  for (int64_t L : lens) {
    const int32_t s = splits_for(L, chunk, cap, tile_rows(kv_dtype));
    smax = s > smax ? s : smax;
  }
  mla_plan p;
  std::memset(&p, 0, sizeof p);
  p.batch = batch;
  p.kv_dtype = kv_dtype;
  p.total_kv = total_kv;
  p.chunk_tokens = chunk;
  p.max_splits = cap;
  p.num_work = static_cast<int32_t>(work);
  p.grid = static_cast<int32_t>(work < sms ? work : sms);
  p.num_sms = sms;
  p.splits_max = smax;
  p.tile_tokens = tile_rows(kv_dtype);
  p.units_per_cta = p.grid > 0 ? (p.num_work + p.grid - 1) / p.grid : 0;
  for (int c = 0; c < MLA_PLAN_FIRST_ROWS; ++c) p.first_row[c] = -1;
  *plan = p;
  return MLA_OK;
}

}  // namespace

extern "C" {

int mla_decode_plan(const int32_t* kv_indptr_host, int32_t batch, int32_t kv_dtype, int32_t num_sms,
                    int32_t num_splits, mla_plan* plan) {
  if (!kv_indptr_host || !plan) return MLA_ERR_INVALID_ARG;
  if (batch < 0 || batch > MLA_MAX_BATCH) return MLA_ERR_INVALID_ARG;
  if (kv_dtype < MLA_KV_BF16 || kv_dtype > MLA_KV_MXFP4) return MLA_ERR_UNSUPPORTED;
  if (num_splits < 0) return MLA_ERR_INVALID_ARG;
  if (kv_indptr_host[0] < 0) return MLA_ERR_INVALID_ARG;
  std::vector<int64_t> lens(static_cast<size_t>(batch));
  for (int32_t b = 0; b < batch; ++b) {
    const int64_t L = (int64_t)kv_indptr_host[b + 1] - kv_indptr_host[b];
    if (L < 0) return MLA_ERR_INVALID_ARG;
    lens[static_cast<size_t>(b)] = L;
  }
  const int rc = plan_lengths(lens, kv_indptr_host[batch], kv_dtype, num_sms, num_splits, plan, batch);
  if (rc == MLA_OK) fill_first_rows(plan, kv_indptr_host);
  return rc;
}

int mla_decode_plan_multi(const int32_t* kv_indptr_host, int32_t num_seqs, int32_t q_len, int32_t kv_dtype,
                          int32_t num_sms, int32_t num_splits, mla_plan* plan) {
  if (!kv_indptr_host || !plan) return MLA_ERR_INVALID_ARG;
  if (q_len < 1 || q_len > 16) return MLA_ERR_UNSUPPORTED;
  if (num_seqs < 0 || (int64_t)num_seqs * q_len > MLA_MAX_BATCH) return MLA_ERR_INVALID_ARG;
  if (kv_dtype < MLA_KV_BF16 || kv_dtype > MLA_KV_MXFP4) return MLA_ERR_UNSUPPORTED;
  if (num_splits < 0) return MLA_ERR_INVALID_ARG;
  if (kv_indptr_host[0] < 0) return MLA_ERR_INVALID_ARG;
  // e4m3, two tokens: one unit list over the sequences' rows serves both
  // tokens (the split kernel reads each row once); otherwise one entry per
  // token over the rows up to its own entry
  const bool fused = q_len == 2 && kv_dtype == MLA_KV_FP8_E4M3;
  std::vector<int64_t> lens(static_cast<size_t>(num_seqs) * (fused ? 1 : q_len));
  for (int32_t b = 0; b < num_seqs; ++b) {
    const int64_t L = (int64_t)kv_indptr_host[b + 1] - kv_indptr_host[b];
    if (L < 0) return MLA_ERR_INVALID_ARG;
    if (fused) {
      lens[static_cast<size_t>(b)] = L;
      continue;
    }
    for (int32_t i = 0; i < q_len; ++i) {
      const int64_t Li = L - (q_len - 1 - i);  // the rows up to token i's own entry
      lens[static_cast<size_t>(b) * q_len + i] = Li > 0 ? Li : 0;
    }
  }
  mla_plan p;
  const int rc = plan_lengths(lens, kv_indptr_host[num_seqs], kv_dtype, num_sms, num_splits, &p,
                              (int64_t)num_seqs * q_len, fused);
  if (rc != MLA_OK) return rc;
  if (fused) {
    if (2 * (int64_t)p.num_work > INT32_MAX) return MLA_ERR_UNSUPPORTED;
    p.batch = 2 * num_seqs;
    p.num_work *= 2;  // partial slots: two per work unit
    p.tokens_fused = 2;
  }
  p.q_len = q_len;
  *plan = p;
  return MLA_OK;
}

int mla_decode_plan_paged(const int32_t* kv_page_indptr_host, const int32_t* kv_last_page_len_host, int32_t batch,
                          int32_t page_size, int32_t num_pages, int32_t kv_dtype, int32_t num_sms,
                          int32_t num_splits, mla_plan* plan) {
  if (!kv_page_indptr_host || !plan || (batch > 0 && !kv_last_page_len_host)) return MLA_ERR_INVALID_ARG;
  if (batch < 0 || batch > MLA_MAX_BATCH || num_pages < 0 || num_splits < 0) return MLA_ERR_INVALID_ARG;
  if (kv_dtype < MLA_KV_BF16 || kv_dtype > MLA_KV_MXFP4) return MLA_ERR_UNSUPPORTED;
  if (page_size < 1 || page_size > (1 << 20) || (page_size & (page_size - 1)) != 0) return MLA_ERR_UNSUPPORTED;
  if (kv_page_indptr_host[0] < 0) return MLA_ERR_INVALID_ARG;
  if ((int64_t)kv_page_indptr_host[batch] * page_size > INT32_MAX || (int64_t)num_pages * page_size > INT32_MAX)
    return MLA_ERR_UNSUPPORTED;
  std::vector<int64_t> lens(static_cast<size_t>(batch));
  for (int32_t b = 0; b < batch; ++b) {
    const int64_t np = (int64_t)kv_page_indptr_host[b + 1] - kv_page_indptr_host[b];
    if (np < 0) return MLA_ERR_INVALID_ARG;
    int64_t L = 0;
    if (np > 0) {
      const int32_t last = kv_last_page_len_host[b];
      if (last < 1 || last > page_size) return MLA_ERR_INVALID_ARG;
      L = (np - 1) * page_size + last;
    }
    lens[static_cast<size_t>(b)] = L;
  }
  const int32_t total = static_cast<int32_t>((int64_t)kv_page_indptr_host[batch] * page_size);
  mla_plan p;
  const int rc = plan_lengths(lens, total, kv_dtype, num_sms, num_splits, &p, batch);
  if (rc != MLA_OK) return rc;
  p.page_size = page_size;
  p.num_pages = num_pages;
  *plan = p;
  return MLA_OK;
}

size_t mla_decode_workspace_bytes(const mla_plan* plan) {
  if (!plan) return 0;
  return mla::ws_layout(plan->batch, plan->num_work).total;
}

}  // extern "C"

namespace {

// The page table of a paged cache (null for a contiguous one).
struct PagedArgs {
  const int32_t* kv_indices;
  const int32_t* kv_last_page_len;
};

// Validates the arguments of one decode and fills the split-kernel parameters.
int prepare(const void* q, const void* kv, const void* kv_scale, int32_t scale_stride, const int32_t* kv_indptr,
            const int32_t* qo_indptr, void* out, float* lse, float sm_scale, const mla_plan* plan, void* workspace,
            size_t workspace_bytes, mla::Stage1Params* p, bool* nothing_to_do, const PagedArgs* paged = nullptr) {
  *nothing_to_do = false;
  if (!plan) return MLA_ERR_INVALID_ARG;
  // a paged plan goes with the paged entry point only, and the reverse
  if ((plan->page_size != 0) != (paged != nullptr)) return MLA_ERR_INVALID_ARG;
  int32_t cache_rows = plan->total_kv;
  int32_t page_shift = 0;
  if (paged) {
    const int32_t P = plan->page_size;
    if (P < 1 || (P & (P - 1)) != 0 || plan->num_pages < 0 || (int64_t)plan->num_pages * P > INT32_MAX)
      return MLA_ERR_INVALID_ARG;
    if (plan->total_kv > 0 && plan->num_pages == 0) return MLA_ERR_INVALID_ARG;  // pages with no cache
    if (plan->total_kv > 0 && (!paged->kv_indices || !paged->kv_last_page_len ||
                               !aligned(paged->kv_indices, 4) || !aligned(paged->kv_last_page_len, 4)))
      return MLA_ERR_INVALID_ARG;
    while ((1 << page_shift) < P) ++page_shift;
    cache_rows = plan->num_pages * P;
  }
  if (plan->kv_dtype < MLA_KV_BF16 || plan->kv_dtype > MLA_KV_MXFP4) return MLA_ERR_UNSUPPORTED;
  if (plan->batch < 0 || plan->num_work < 0 || plan->grid < 0 || plan->chunk_tokens <= 0 || plan->max_splits <= 0)
    return MLA_ERR_INVALID_ARG;
  if (plan->batch == 0 || plan->num_work == 0) {
    *nothing_to_do = true;
    return MLA_OK;
  }
  if (plan->units_per_cta > mla::max_units_per_cta(plan->kv_dtype) || plan->grid <= 0) return MLA_ERR_INVALID_ARG;
  if (!q || !kv || !kv_indptr || !qo_indptr || !out || !workspace) return MLA_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(kv, 16) || !aligned(out, 8) || !aligned(workspace, 256)) return MLA_ERR_INVALID_ARG;
  if (!aligned(kv_indptr, 4) || !aligned(qo_indptr, 4) || (lse && !aligned(lse, 4))) return MLA_ERR_INVALID_ARG;
  if (!std::isfinite(sm_scale)) return MLA_ERR_INVALID_ARG;
  if (plan->kv_dtype == MLA_KV_FP8_E4M3 && (!kv_scale || !aligned(kv_scale, 4))) return MLA_ERR_INVALID_ARG;
  if (plan->kv_dtype == MLA_KV_MXFP4 && (!kv_scale || !aligned(kv_scale, 16) || scale_stride < MLA_MX_SCALES_PER_ROW))
    return MLA_ERR_INVALID_ARG;
  const mla::WsLayout w = mla::ws_layout(plan->batch, plan->num_work);
  if (workspace_bytes < w.total) return MLA_ERR_WORKSPACE_TOO_SMALL;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  p->q = static_cast<const uint8_t*>(q);
  p->kv = static_cast<const uint8_t*>(kv);
  p->kv_scale = kv_scale;
  p->scale_stride = plan->kv_dtype == MLA_KV_MXFP4 ? scale_stride : 0;
  p->kv_indptr = kv_indptr;
  p->qo_indptr = qo_indptr;
  p->kv_indices = paged ? paged->kv_indices : nullptr;
  p->kv_last = paged ? paged->kv_last_page_len : nullptr;
  p->paged = paged ? 1 : 0;
  p->page_shift = page_shift;
  p->num_pages = paged ? plan->num_pages : 0;
  p->out = static_cast<uint16_t*>(out);
  p->lse = lse;
  p->sm_scale = sm_scale;
  p->ws_err = reinterpret_cast<int32_t*>(ws + w.err);
  p->ws_seq = reinterpret_cast<int32_t*>(ws + w.seq);
  p->ws_lse = reinterpret_cast<float*>(ws + w.lse);
  p->ws_o = reinterpret_cast<float*>(ws + w.o);
  p->ws_q = ws + w.q;
  p->batch = plan->batch;
  p->total_kv = plan->total_kv;
  p->chunk_tokens = plan->chunk_tokens;
  p->max_splits = plan->max_splits;
  p->num_work = plan->num_work;
  p->grid = plan->grid;
  p->schedule = plan->schedule;
  p->total_tiles = plan->total_tiles;
  p->unit_cost = plan->unit_cost;
  p->trace = g_trace;
  p->q_len = plan->q_len > 1 ? plan->q_len : 1;
  if (plan->q_len > 16 || (p->q_len > 1 && (paged || plan->batch % p->q_len != 0))) return MLA_ERR_INVALID_ARG;
  // a two-token plan: e4m3 KV, q_len 2, two partial slots per work unit
  p->tok = plan->tokens_fused == 2 ? 2 : 1;
  // MXFP4 scores by block-scaled MMAs (pages of fewer than 64 rows take the copy)
  if (plan->mx_scores != 0 && (plan->mx_scores != 1 || plan->kv_dtype != MLA_KV_MXFP4)) return MLA_ERR_INVALID_ARG;
  p->mx_bs = (plan->mx_scores == 1 && !(paged && page_shift < 6)) ? 1 : 0;
  // the first tile rows of a contiguous single-token plan (the e4m3 split
  // kernel starts those copies before its unit scan)
  const bool first_rows = !paged && p->q_len == 1 && p->tok == 1;
  for (int c = 0; c < MLA_PLAN_FIRST_ROWS; ++c) {
    const int32_t r = first_rows ? plan->first_row[c] : -1;
    if (r < -1 || r >= plan->total_kv) return MLA_ERR_INVALID_ARG;  // a row of the cache, or none
    p->first_row[c] = r;
  }
  if (plan->tokens_fused != 0 && (plan->tokens_fused != 2 || plan->kv_dtype != MLA_KV_FP8_E4M3 ||
                                  plan->q_len != 2 || plan->num_work % 2 != 0))
    return MLA_ERR_INVALID_ARG;
  const int32_t entries = plan->batch / p->tok;  // sequences in the unit list
  if (plan->schedule != 0 && (plan->schedule != 1 || plan->total_tiles < plan->grid)) return MLA_ERR_INVALID_ARG;
  // schedule 1's late CTAs (see late_ctas): every CTA keeps at least two positions
  p->late_tiles = plan->late_tiles;
  p->late_ctas = plan->late_tiles > 0 ? static_cast<int32_t>(late_ctas(plan->grid, plan->batch, plan->num_sms)) : 0;
  if (plan->late_tiles < 0 || (plan->late_tiles > 0 && (plan->schedule != 1 || plan->late_tiles > 64 ||
                                                        p->late_ctas == 0 || plan->num_sms <= 0)))
    return MLA_ERR_INVALID_ARG;
  if (plan->unit_cost < 0 || (plan->schedule == 1 && (int64_t)plan->total_tiles +
                              (int64_t)plan->unit_cost * (entries > 0 ? entries - 1 : 0) > INT32_MAX))
    return MLA_ERR_INVALID_ARG;
  if (plan->late_tiles > 0) {
    const int64_t C = (int64_t)plan->total_tiles + (int64_t)plan->unit_cost * (entries > 0 ? entries - 1 : 0);
    if (C + (int64_t)p->late_ctas * plan->late_tiles < (int64_t)(plan->late_tiles + 2) * plan->grid ||
        C + (int64_t)p->late_ctas * plan->late_tiles > INT32_MAX)
      return MLA_ERR_INVALID_ARG;
  }
  if (plan->kv_dtype == MLA_KV_FP8_E4M3) {
    if (!encode_kv_map_tc(&p->tmap_kv64, kv, cache_rows, 128)) return MLA_ERR_CUDA;
    if (paged && page_shift == 6) {
      // 64-row pages: a tile is two 64-row boxes
      if (!encode_kv_map_tc(&p->tmap_kv16, kv, cache_rows, 64)) return MLA_ERR_CUDA;
    } else if (paged && page_shift < 6) {
      // smaller pages: a pair of column blocks (128 B) and the rope block (64 B)
      // per box, one page high for pages of 8 to 32 rows, one row high (for
      // four-row gathers) for pages of 1 to 4 rows
      const uint32_t rows = page_shift >= 3 ? (1u << page_shift) : 1u;
      if (!encode_kv_map_pairs(&p->tmap_kv16, kv, cache_rows, rows) ||
          !encode_kv_map_tc(&p->tmap_kv64, kv, cache_rows, rows))
        return MLA_ERR_CUDA;
    } else {
      std::memcpy(&p->tmap_kv16, &p->tmap_kv64, sizeof(CUtensorMap));
    }
  } else if (plan->kv_dtype == MLA_KV_MXFP4) {
    if (!p->mx_bs) {
      // the e4m3 copy: packed rows by 1-D bulk copies, no tensor map
      std::memset(&p->tmap_kv64, 0, sizeof(CUtensorMap));
      std::memset(&p->tmap_kv16, 0, sizeof(CUtensorMap));
    } else {
      // the block-scaled kernel: 128-row boxes (two 64-row boxes per tile for 64-row pages)
      if (!aligned(kv, 32)) return MLA_ERR_INVALID_ARG;
      if (!encode_kv_maps_mx(&p->tmap_kv64, &p->tmap_kv16, kv, cache_rows, (paged && page_shift == 6) ? 64u : 128u))
        return MLA_ERR_CUDA;
    }
  } else {
    // bf16: 64-row boxes, and 16-row boxes for short tails; pages of fewer
    // than 16 rows come in one page per box
    const uint32_t small = (paged && page_shift < 4) ? (1u << page_shift) : 16u;
    if (!encode_kv_map(&p->tmap_kv64, kv, plan->kv_dtype, cache_rows, 64) ||
        !encode_kv_map(&p->tmap_kv16, kv, plan->kv_dtype, cache_rows, small))
      return MLA_ERR_CUDA;
  }
  return MLA_OK;
}

// The split stage: for e4m3 and MXFP4 KV the query preparation, then the split
// kernel (which overlaps its set-up with the preparation).
int launch_split_stage(const mla::Stage1Params& p, int kv_dtype, cudaStream_t s) {
  cudaError_t e;
  switch (kv_dtype) {
    case MLA_KV_BF16: e = mla::launch_stage1_bf16(p, s); break;
    case MLA_KV_FP8_E4M3:
      e = mla::launch_prep_q(p, false, s);
      if (e == cudaSuccess) e = mla::launch_stage1_fp8(p, s);
      break;
    default:
      e = mla::launch_prep_q(p, true, s);
      if (e == cudaSuccess) e = mla::launch_stage1_mxfp4(p, s);
      break;
  }
  if (e != cudaSuccess) {
    cudaGetLastError();
    return MLA_ERR_CUDA;
  }
  return MLA_OK;
}

int launch_combine_stage(const mla::Stage1Params& p, const mla_plan* plan, cudaStream_t s) {
  if (plan->splits_max <= 1) return MLA_OK;
  mla::CombineParams c;
  c.ws_seq = p.ws_seq;
  c.ws_lse = p.ws_lse;
  c.ws_o = p.ws_o;
  c.out = p.out;
  c.lse = p.lse;
  c.batch = plan->batch;
  c.few_splits = plan->splits_max <= 4 ? 1 : 0;
  if (mla::launch_combine(c, s, true) != cudaSuccess) {
    cudaGetLastError();
    return MLA_ERR_CUDA;
  }
  return MLA_OK;
}

}  // namespace

extern "C" {

int mla_decode_fwd(const void* q, const void* kv, const void* kv_scale, int32_t scale_stride,
                   const int32_t* kv_indptr, const int32_t* qo_indptr, void* out, float* lse, float sm_scale,
                   const mla_plan* plan, void* workspace, size_t workspace_bytes, void* stream) {
  mla::Stage1Params p;
  bool noop = false;
  int rc = prepare(q, kv, kv_scale, scale_stride, kv_indptr, qo_indptr, out, lse, sm_scale, plan, workspace,
                   workspace_bytes, &p, &noop);
  if (rc != MLA_OK || noop) return rc;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  rc = launch_split_stage(p, plan->kv_dtype, s);
  if (rc != MLA_OK) return rc;
  return launch_combine_stage(p, plan, s);
}

int mla_decode_fwd_paged(const void* q, const void* kv_pages, const void* kv_scale, int32_t scale_stride,
                         const int32_t* kv_page_indptr, const int32_t* kv_indices, const int32_t* kv_last_page_len,
                         const int32_t* qo_indptr, void* out, float* lse, float sm_scale, const mla_plan* plan,
                         void* workspace, size_t workspace_bytes, void* stream) {
  mla::Stage1Params p;
  bool noop = false;
  const PagedArgs paged{kv_indices, kv_last_page_len};
  int rc = prepare(q, kv_pages, kv_scale, scale_stride, kv_page_indptr, qo_indptr, out, lse, sm_scale, plan,
                   workspace, workspace_bytes, &p, &noop, &paged);
  if (rc != MLA_OK || noop) return rc;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  rc = launch_split_stage(p, plan->kv_dtype, s);
  if (rc != MLA_OK) return rc;
  return launch_combine_stage(p, plan, s);
}

int mla_decode_split(const void* q, const void* kv, const void* kv_scale, int32_t scale_stride,
                     const int32_t* kv_indptr, const int32_t* qo_indptr, void* out, float* lse, float sm_scale,
                     const mla_plan* plan, void* workspace, size_t workspace_bytes, void* stream) {
  mla::Stage1Params p;
  bool noop = false;
  int rc = prepare(q, kv, kv_scale, scale_stride, kv_indptr, qo_indptr, out, lse, sm_scale, plan, workspace,
                   workspace_bytes, &p, &noop);
  if (rc != MLA_OK || noop) return rc;
  return launch_split_stage(p, plan->kv_dtype, static_cast<cudaStream_t>(stream));
}

int mla_decode_combine(void* out, float* lse, const mla_plan* plan, void* workspace, size_t workspace_bytes,
                       void* stream) {
  if (!plan) return MLA_ERR_INVALID_ARG;
  if (plan->batch <= 0 || plan->num_work <= 0 || plan->splits_max <= 1) return MLA_OK;
  if (!out || !workspace || !aligned(out, 8) || !aligned(workspace, 256) || (lse && !aligned(lse, 4)))
    return MLA_ERR_INVALID_ARG;
  const mla::WsLayout w = mla::ws_layout(plan->batch, plan->num_work);
  if (workspace_bytes < w.total) return MLA_ERR_WORKSPACE_TOO_SMALL;
  mla::Stage1Params p;
  std::memset(&p, 0, sizeof p);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  p.ws_seq = reinterpret_cast<int32_t*>(ws + w.seq);
  p.ws_lse = reinterpret_cast<float*>(ws + w.lse);
  p.ws_o = reinterpret_cast<float*>(ws + w.o);
  p.out = static_cast<uint16_t*>(out);
  p.lse = lse;
  return launch_combine_stage(p, plan, static_cast<cudaStream_t>(stream));
}

int mla_decode_poll_error(void* workspace, void* stream) {
  if (!workspace) return MLA_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(s) != cudaSuccess) {
    cudaGetLastError();
    return MLA_ERR_CUDA;
  }
  int32_t word = 0;
  if (cudaMemcpy(&word, workspace, sizeof word, cudaMemcpyDeviceToHost) != cudaSuccess) {
    cudaGetLastError();
    return MLA_ERR_CUDA;
  }
  if (word != 0) {
    if (cudaMemset(workspace, 0, sizeof word) != cudaSuccess) {
      cudaGetLastError();
      return MLA_ERR_CUDA;
    }
  }
  return word;
}

const char* mla_status_string(int status) {
  switch (status) {
    case MLA_OK: return "ok";
    case MLA_ERR_INVALID_ARG: return "invalid argument (null or misaligned pointer, bad size or layout)";
    case MLA_ERR_UNSUPPORTED: return "unsupported shape or dtype";
    case MLA_ERR_WORKSPACE_TOO_SMALL: return "workspace smaller than mla_decode_workspace_bytes(plan)";
    case MLA_ERR_CUDA: return "CUDA runtime call or kernel launch failed";
    case MLA_ERR_DEVICE_INDEX: return "kernel found kv_indptr inconsistent with the plan";
    case MLA_ERR_DEVICE_TIMEOUT: return "kernel timed out waiting for its own copies";
    case MLA_ERR_NO_DEVICE: return "no CUDA device visible";
    default: return "unknown status";
  }
}

const char* mla_decode_version(void) { return "0.2.0"; }

int mla_decode_set_trace(uint64_t* buffer) {
#if defined(MLA_TRACE) && MLA_TRACE
  g_trace = buffer;
  return MLA_OK;
#else
  if (buffer) return MLA_ERR_UNSUPPORTED;
  g_trace = nullptr;
  return MLA_OK;
#endif
}

}  // extern "C"
