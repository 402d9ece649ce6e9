// mla_internal.h -- parameters shared by the host API and the kernel launchers.
#pragma once
#include <atomic>
#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "mla_decode.h"

namespace mla {

constexpr int kHeads = 16;
constexpr int kQkDim = 576;
constexpr int kVDim = 512;
constexpr int kTile = 64;              // KV rows per pipeline stage
constexpr int kConsumerWarps = 8;      // 4 pairs; pair p scores rows [16p, 16p+16) of a tile
constexpr int kThreads = kConsumerWarps * 32;
constexpr int kMaxUnitsPerCta = 256;   // work units one CTA may own (unit table in smem)
constexpr int kMaxUnitsPerCtaMx = 64;  // the same for MXFP4 KV (its staging ring leaves less smem)
inline int max_units_per_cta(int kv_dtype) { return kv_dtype == 2 ? kMaxUnitsPerCtaMx : kMaxUnitsPerCta; }

// Workspace layout (byte offsets from the 256-aligned base).
struct WsLayout {
  size_t err;      // int32 error word
  size_t seq;      // int32 [batch][2] = {first unit, split count}
  size_t lse;      // fp32 [num_work][16] partial lse (natural log)
  size_t o;        // fp32 [num_work][16][512] normalised partial outputs
  size_t q;        // [batch] prepared queries (e4m3 and MXFP4 KV): two-term e4m3 image + 16 fp32 factors
  size_t total;
};

// A prepared query: the two-term e4m3 query exactly as the tensor cores read
// it from shared memory (32 rows x 576 B, K-major, 64 B swizzle: 9 blocks of
// 2048 B), followed by the 16 per-head score factors.
constexpr size_t kQImageBytes = 9 * 32 * 64;
constexpr size_t kQPrepBytes = kQImageBytes + 16 * sizeof(float);

inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

inline WsLayout ws_layout(int batch, int num_work) {
  WsLayout w;
  w.err = 0;
  w.seq = 256;
  w.lse = align_up(w.seq + sizeof(int32_t) * 2 * static_cast<size_t>(batch), 256);
  w.o = align_up(w.lse + sizeof(float) * kHeads * static_cast<size_t>(num_work), 256);
  w.q = align_up(w.o + sizeof(float) * kHeads * kVDim * static_cast<size_t>(num_work), 1024);
  w.total = align_up(w.q + kQPrepBytes * static_cast<size_t>(batch), 256);
  return w;
}

struct Stage1Params {
  CUtensorMap tmap_kv64;     // KV rows as (span bytes, 9 chunks, rows), swizzled; 64-row box
                             // (e4m3: 64-byte column blocks of 128 rows)
  CUtensorMap tmap_kv16;     // the same with a 16-row box (ragged tails); e4m3 over a
                             // 64-row paged cache: 64-byte column blocks of 64 rows
  const uint8_t* q;          // bf16 [*, 16, 576]
  const uint8_t* kv;         // row bytes depend on the dtype
  const void* kv_scale;      // fp32[1] (fp8) or e8m0 [rows, scale_stride] (mxfp4)
  int32_t scale_stride;
  const int32_t* kv_indptr;  // rows per sequence; for a paged cache, pages per sequence
  const int32_t* qo_indptr;
  const int32_t* kv_indices; // paged cache: the page table (else null)
  const int32_t* kv_last;    // paged cache: rows in each sequence's last page
  int32_t paged;             // 1: a paged cache (kv_indices, kv_last); 0: contiguous rows
  int32_t page_shift;        // paged cache: log2(page size); 0 for a contiguous cache
  int32_t num_pages;         // paged cache: pages in the cache tensor
  uint16_t* out;             // bf16 [batch, 16, 512]
  float* lse;                // fp32 [batch, 16] or null
  float sm_scale;
  int32_t* ws_err;
  int32_t* ws_seq;
  float* ws_lse;
  float* ws_o;
  uint8_t* ws_q;             // prepared queries [batch][kQPrepBytes] (e4m3 / MXFP4 KV)
  int32_t batch;
  int32_t total_kv;
  int32_t chunk_tokens;
  int32_t max_splits;
  int32_t num_work;
  int32_t grid;
  int32_t schedule;     // 0: round-robin splits, 1: contiguous tile ranges
  int32_t total_tiles;  // schedule 1: sum of the sequences' weights in tiles
  int32_t unit_cost;    // schedule 1: empty positions between consecutive sequences
  int32_t q_len;        // query tokens per sequence; batch counts tokens
  int32_t tok;          // tokens one work unit serves (2: fused two-token e4m3 plan, else 1);
                        // num_work then counts partial slots, tok per unit
  int32_t mx_bs;        // MXFP4 (contiguous, pages >= 64 rows): 1 = scores by block-scaled MMAs
  int32_t late_ctas;    // schedule 1: the last late_ctas CTAs own late_tiles positions fewer
  int32_t late_tiles;
  uint64_t* trace;      // trace builds only: [grid][kTraceSlots] global-timer stamps (else null)
  int32_t first_row[MLA_PLAN_FIRST_ROWS];  // the plan's first tile row per CTA (-1: none; see mla_plan)
};

// Per-CTA stamp slots of a trace build (compiled with MLA_TRACE=1).
constexpr int kTraceSlots = 128;
enum TraceSlot {
  kTrEntry = 0,        // kernel entry
  kTrSetup = 1,        // set-up done (barriers, unit list, TMEM)
  kTrFirstLoad = 2,    // producer issued the first KV copy
  kTrQueryReady = 3,   // query loader: the query-preparation grid is complete
  kTrUnits = 4,        // (a count) work units of the CTA
  kTrTiles = 5,        // (a count) tiles of the CTA
  kTrExit = 6,         // every role done, before TMEM is freed
  kTrScanDone = 7,     // the unit list is in shared memory
  kTrUnitDone = 8,     // [8] unit k's epilogue written
  kTrTileS = 16,       // [64] softmax: tile t's scores ready
  kTrTileData = 80,    // [32] QK issuer: tile t's data landed and its S buffer free
  kTrUnitLastPV = 112, // [8] unit k's last P.V complete (its epilogue starts)
  kTrPrepEntry = 120,  // query-preparation CTA of the same index: entry,
  kTrPrepWaited = 121, //   past its wait for earlier work,
  kTrPrepDone = 122,   //   and its image written
  kTrSmid = 127,       // (a value) the SM the CTA ran on
};

struct CombineParams {
  const int32_t* ws_seq;
  const float* ws_lse;
  const float* ws_o;
  uint16_t* out;
  float* lse;
  int32_t batch;
  int32_t few_splits;  // the plan splits no sequence more than 4 times
};

// Device error codes written to the workspace error word (match mla_status).
constexpr int32_t kErrDeviceIndex = 5;
constexpr int32_t kErrDeviceTimeout = 6;

cudaError_t launch_stage1_bf16(const Stage1Params& p, cudaStream_t s);
cudaError_t launch_stage1_fp8(const Stage1Params& p, cudaStream_t s);
cudaError_t launch_stage1_fp8_t2(const Stage1Params& p, cudaStream_t s);  // p.tok == 2
cudaError_t launch_stage1_mxfp4(const Stage1Params& p, cudaStream_t s);
// paged caches with pages of fewer than 64 rows (e4m3 or MXFP4, one token)
cudaError_t launch_stage1_small_pages(const Stage1Params& p, bool mx, cudaStream_t s);
// MXFP4 scores by block-scaled MMAs on the e2m1 tile (p.mx_bs)
cudaError_t launch_stage1_mxfp4_bs(const Stage1Params& p, cudaStream_t s);
// Two-term e4m3 query of every sequence into the workspace (e4m3 / MXFP4 KV).
cudaError_t launch_prep_q(const Stage1Params& p, bool mx, cudaStream_t s);
cudaError_t launch_combine(const CombineParams& p, cudaStream_t s, bool pdl);

// Sets kernel K's dynamic shared-memory opt-in once per device and process
// (the attribute belongs to the function in each device's context; setting it
// on every call costs host time between two dependent launches).
template <auto K>
inline cudaError_t smem_opt_in(int bytes) {
  static std::atomic<uint64_t> done{0};  // bit d: set on device d
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const uint64_t bit = dev < 64 ? (1ull << dev) : 0;
  if (bit != 0 && (done.load(std::memory_order_acquire) & bit) != 0) return cudaSuccess;
  e = cudaFuncSetAttribute(K, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess && bit != 0) done.fetch_or(bit, std::memory_order_release);
  return e;
}

// Launch with programmatic dependent launch allowed: the kernel may start while
// the previous kernel on the stream finishes, and waits (griddepcontrol.wait)
// before it reads memory.
template <class Kernel>
inline cudaError_t launch_overlapped(Kernel kernel, dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                                     const Stage1Params& p) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, p);
}

}  // namespace mla
