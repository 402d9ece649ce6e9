/*
 * mla_decode.h -- C ABI of libmla_decode.so: multi-head latent attention
 * decode (one query token per sequence, or a few) on a GB300 (sm_103a).
 *
 * The operation (kernelindex "amd-mixed-mla" submission 593653, section
 * "Slow fallback", _bmm_reference; constants from its "Constants" section):
 * for every sequence b and query head h < 16,
 *
 *   s_t        = (q[qo_indptr[b], h, :576] . dequant(kv[t, :576])) * sm_scale
 *   out[b,h,:] = sum_t softmax(s)_t * dequant(kv[t, :512])
 *   lse[b,h]   = ln sum_t exp(s_t)                      (natural log)
 *
 * over the KV rows t in [kv_indptr[b], kv_indptr[b+1]) -- one latent KV head
 * shared by all 16 query heads, QK dim 576 (512 latent + 64 rope), V = the first
 * 512 columns of the same row, page size 1, sm_scale = 1/sqrt(576) = 1/24.
 * An empty sequence gives out = 0 and lse = -inf.  Extensions below: a paged
 * cache (mla_decode_plan_paged / mla_decode_fwd_paged) and several query
 * tokens per sequence (mla_decode_plan_multi).
 *
 * KV storage (submission 593653 "Dispatch" and submission 754939 "Stage 1"):
 *   MLA_KV_BF16      bf16 [rows, 576]
 *   MLA_KV_FP8_E4M3  OCP e4m3fn bytes [rows, 576] times one fp32 per-tensor scale
 *   MLA_KV_MXFP4     packed e2m1 [rows, 288] (element 2i = low nibble of byte i)
 *                    with one e8m0 byte per 32 elements, [rows, scale_stride],
 *                    scale_stride >= 18 (only the first 18 bytes are read).
 *
 * Calling sequence: mla_decode_plan() (or mla_decode_plan_multi /
 * mla_decode_plan_paged) on the host for a batch layout (it reads only the
 * host copy of the index arrays), mla_decode_workspace_bytes() for the size
 * of the caller-owned device workspace, then mla_decode_fwd() for each call on
 * that layout.  The library never allocates device memory, never synchronises
 * the stream and never exits the process: every entry point returns an
 * mla_status.  All device buffers are owned by the caller.
 *
 * Threading: entry points are reentrant.  Calls that share one workspace must
 * be ordered on the GPU (same stream, or events); overlapping calls on one
 * workspace race.
 */
#ifndef MLA_DECODE_H
#define MLA_DECODE_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define MLA_API __attribute__((visibility("default")))
#else
#define MLA_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

#define MLA_NUM_HEADS 16
#define MLA_QK_DIM 576
#define MLA_V_DIM 512
#define MLA_MX_BLOCK 32
#define MLA_MX_SCALES_PER_ROW 18
#define MLA_MAX_BATCH 65536
#define MLA_PLAN_FIRST_ROWS 256

typedef enum {
  MLA_KV_BF16 = 0,
  MLA_KV_FP8_E4M3 = 1,
  MLA_KV_MXFP4 = 2
} mla_kv_dtype;

typedef enum {
  MLA_OK = 0,
  MLA_ERR_INVALID_ARG = 1,          /* null/misaligned pointer, bad size or layout */
  MLA_ERR_UNSUPPORTED = 2,          /* a shape or dtype this library does not implement */
  MLA_ERR_WORKSPACE_TOO_SMALL = 3,  /* workspace_bytes < mla_decode_workspace_bytes(plan) */
  MLA_ERR_CUDA = 4,                 /* a CUDA runtime call or a kernel launch failed */
  MLA_ERR_DEVICE_INDEX = 5,         /* a kernel found kv_indptr inconsistent with the plan */
  MLA_ERR_DEVICE_TIMEOUT = 6,       /* a kernel gave up waiting for its own copies */
  MLA_ERR_NO_DEVICE = 7             /* no CUDA device is visible */
} mla_status;

/*
 * The work decomposition of one batch layout (split-K over the KV sequence).
 * With R = tile_tokens (64 rows for bf16 KV, 128 for e4m3 and e2m1 KV),
 * sequence b with L_b = kv_indptr[b+1] - kv_indptr[b] rows and
 * T_b = ceil(L_b / R) row tiles is cut into
 *   S_b = L_b == 0 ? 1 : min(max_splits, ceil(L_b / chunk_tokens), T_b)
 * contiguous splits on tile boundaries, split s covering rows
 *   [kv_indptr[b] + R floor(s T_b / S_b), kv_indptr[b] + min(L_b, R floor((s+1) T_b / S_b))),
 * so no split is empty when L_b > 0.  Work unit u (0 <= u < num_work) is split
 * s of sequence b with u = sum_{b' < b} S_b' + s; CTA c of the grid processes
 * units c, c + grid, c + 2 grid, ...  (schedule 0).
 *
 * Schedule 1 (contiguous tile ranges) instead lays the sequences' tiles end to
 * end, each sequence weighing w_b = max(1, T_b) tiles, T = sum_b w_b, with
 * U = unit_cost empty positions between consecutive sequences (the weight of
 * a unit boundary), C = T + U (batch - 1) positions in all, and gives CTA c of
 * G = grid the positions [B(c), B(c+1)) with
 *   B(c) = floor(c C' / G) - D max(0, c - (G - L)),  C' = C + L D,
 * D = late_tiles and L = min(G, max(0, G + batch - num_sms)) when D > 0 (else
 * L = 0): the last L CTAs, which the hardware places on the SMs the
 * query-preparation grid (one CTA per output row) holds and so start later,
 * own D positions fewer.  Sequence b's tiles sit at positions X_b + i,
 * X_b = P_b + U b with P_b = sum_{b' < b} w_b'; it is split where CTA ranges
 * cut it: with cta(x) the CTA whose range holds x,
 * S_b = cta(X_b + w_b - 1) - cta(X_b) + 1, split s covers the sequence's tiles
 * in CTA cta(X_b) + s's range, and unit u = sum_{b' < b} S_b' + s.  The planner takes whichever schedule its cost
 * model (the busiest CTA's tiles and units, plus the combine) prefers; a forced
 * split count always uses schedule 0.  Fields are filled by mla_decode_plan and
 * must not be edited.
 */
typedef struct {
  int32_t batch;          /* output rows: sequences (times q_len for mla_decode_plan_multi) */
  int32_t kv_dtype;       /* mla_kv_dtype */
  int32_t total_kv;       /* kv_indptr[batch]: rows of the KV tensor that are read */
  int32_t chunk_tokens;   /* split length target (tokens) */
  int32_t max_splits;     /* cap on S_b */
  int32_t num_work;       /* sum_b S_b = work units = partial slots in the workspace */
  int32_t grid;           /* CTAs of the split kernel (<= num_sms) */
  int32_t num_sms;        /* SM count the plan was made for */
  int32_t splits_max;     /* max_b S_b (1: no combine kernel is launched) */
  int32_t tile_tokens;    /* R: KV rows per pipeline tile (splits end on tile boundaries) */
  int32_t units_per_cta;  /* the most units any CTA owns */
  int32_t schedule;       /* 0: splits dealt round-robin (rule above); 1: contiguous tile ranges */
  int32_t total_tiles;    /* schedule 1: T = sum_b max(1, T_b) */
  int32_t page_size;      /* 0: contiguous cache (mla_decode_plan); P >= 1: paged (mla_decode_plan_paged) */
  int32_t num_pages;      /* paged: pages in the cache tensor; 0 otherwise */
  int32_t unit_cost;      /* schedule 1: U, empty tile positions between consecutive sequences */
  int32_t q_len;          /* query tokens per sequence (0 or 1: one; see mla_decode_plan_multi) */
  int32_t tokens_fused;   /* 2: a two-token e4m3 plan whose split kernel reads each cache row once
                             for both tokens (see mla_decode_plan_multi); 0 otherwise */
  int32_t mx_scores;      /* mxfp4 only, set by the caller after planning (the planners write 0):
                             0: both tensor-core products read an e4m3 copy of each tile made
                             in shared memory; 1: the scores q.k come from block-scaled MMAs
                             (tcgen05 kind::mxf8f6f4) on the e2m1 tile with the cache's e8m0
                             block scales, only the V part being converted for P.V (needs kv
                             32-byte aligned).  Paged caches with pages of fewer than 64 rows
                             always take the copy. */
  int32_t late_tiles;     /* schedule 1: D, the positions each late CTA gives up (rule above); 0: none */
  /* first_row[c] (c < MLA_PLAN_FIRST_ROWS): the row-space row of the first tile
   * CTA c of the split kernel reads, -1 when it reads none or the plan does not
   * say (paged and multi-token plans).  The e4m3 split kernel starts that
   * tile's copy on entry, before its unit scan; the device kv_indptr must then
   * hold the values the plan was made from (as it must anyway). */
  int32_t first_row[MLA_PLAN_FIRST_ROWS];
} mla_plan;

/*
 * mla_decode_plan -- host only; reads kv_indptr_host[0..batch] (int32, the host
 * copy of the device kv_indptr passed to mla_decode_fwd).  kv_indptr must be
 * non-decreasing with kv_indptr[0] >= 0.  num_sms <= 0 queries the current
 * device.  num_splits > 0 forces S_b = min(num_splits, T_b) (at least 1);
 * num_splits == 0 lets the planner choose a split length that balances the
 * units over num_sms CTAs.  Returns MLA_OK and fills *plan, or an error code and
 * leaves *plan untouched.  Never calls CUDA when num_sms > 0.
 */
MLA_API int mla_decode_plan(const int32_t* kv_indptr_host, int32_t batch, int32_t kv_dtype,
                    int32_t num_sms, int32_t num_splits, mla_plan* plan);

/* Bytes of device workspace mla_decode_fwd needs for this plan (0 on a null plan).
 * The workspace holds fp32 partial outputs and lse values of the split units, a
 * per-sequence split table and an error word; its content between calls is
 * irrelevant except for the error word (see mla_decode_poll_error). */
MLA_API size_t mla_decode_workspace_bytes(const mla_plan* plan);

/*
 * mla_decode_fwd -- enqueue one decode on `stream` (a cudaStream_t; NULL = the
 * legacy default stream).  Asynchronous: returns after launching.
 *
 * "device" below means memory the GPU can address: device memory, or pinned
 * (page-locked, CUDA-registered) host memory, which the kernels then read or
 * write across the host link.  The KV cache, its scales and the workspace
 * must be device memory, and so must q for bf16 KV (fetched by bulk copies).
 *
 *   q          device, bf16 [*, 16, 576] row-major; sequence b uses row qo_indptr[b].
 *              16-byte aligned.
 *   kv         device, see the storage table above; rows [0, plan->total_kv) are read.
 *              16-byte aligned; 32-byte aligned for mxfp4 (the 4-bit tensor-map
 *              form the block-scaled kernel reads).
 *   kv_scale   device: NULL for bf16; fp32[1] for fp8 (dequant = e4m3 * kv_scale[0]);
 *              uint8 e8m0 [plan->total_kv, scale_stride] for mxfp4 (16-byte aligned).
 *   scale_stride  mxfp4: bytes between scale rows, >= 18; otherwise 0.
 *   kv_indptr  device int32 [batch+1], equal to the host copy the plan was made from.
 *   qo_indptr  device int32 [batch+1]; only qo_indptr[b] (the query row of b) is read.
 *   out        device, bf16 [batch, 16, 512] row-major (written).  8-byte aligned.
 *   lse        device fp32 [batch, 16] (written) or NULL.
 *   sm_scale   softmax scale (1/24 for this problem).
 *   workspace  device, >= mla_decode_workspace_bytes(plan) bytes, 256-byte aligned.
 *
 * Returns MLA_OK, MLA_ERR_INVALID_ARG / MLA_ERR_WORKSPACE_TOO_SMALL (nothing was
 * launched) or MLA_ERR_CUDA (a launch failed).  Device-side faults in the index
 * data are reported by mla_decode_poll_error, not here.
 */
MLA_API int mla_decode_fwd(const void* q, const void* kv, const void* kv_scale, int32_t scale_stride,
                   const int32_t* kv_indptr, const int32_t* qo_indptr, void* out, float* lse,
                   float sm_scale, const mla_plan* plan, void* workspace, size_t workspace_bytes,
                   void* stream);

/*
 * The two stages of mla_decode_fwd, for callers that schedule them separately
 * (e.g. to time or overlap them).  mla_decode_split takes exactly the arguments
 * of mla_decode_fwd and launches only the split kernel: sequences with one
 * split get their final out/lse, split sequences leave fp32 partials in the
 * workspace.  mla_decode_combine then merges those partials into out/lse
 * (log-sum-exp combine; submission 593653's stage-2 kernel _flash_fp8_split_s2)
 * and launches nothing when plan->splits_max <= 1.  It must follow the split
 * stage on the same stream with the same plan, workspace, out and lse.
 */
MLA_API int mla_decode_split(const void* q, const void* kv, const void* kv_scale, int32_t scale_stride,
                             const int32_t* kv_indptr, const int32_t* qo_indptr, void* out, float* lse,
                             float sm_scale, const mla_plan* plan, void* workspace, size_t workspace_bytes,
                             void* stream);
MLA_API int mla_decode_combine(void* out, float* lse, const mla_plan* plan, void* workspace,
                               size_t workspace_bytes, void* stream);

/*
 * mla_decode_poll_error -- synchronises `stream`, reads and clears the error
 * word a kernel leaves in `workspace` (MLA_ERR_DEVICE_INDEX when kv_indptr on
 * the device disagreed with the plan -- the offending units are skipped;
 * MLA_ERR_DEVICE_TIMEOUT when a kernel stopped waiting for its own copies).
 * Returns MLA_OK when the word was clear.  For tests and debugging: the first
 * error found by a unit scan also leaves int32 words 2-5 of the workspace =
 * the CTA, the thread, a tag (3 / 4: kv_indptr or qo_indptr disagree with the
 * plan in the round-robin / contiguous unit scan; 5: the plan's first tile row
 * is not the scan's, word 5 = the row), which this call does not clear.
 */
MLA_API int mla_decode_poll_error(void* workspace, void* stream);

/*
 * Several query tokens per sequence (q_len > 1), e.g. draft tokens checked in
 * one step.  The pages decode one token per sequence; this is the causal
 * reading for more: sequence b's tokens are query rows qo_indptr[b] + i
 * (i < q_len), the last q_len of its L_b cached rows are those tokens' own
 * entries, and token i attends to the first L_b - (q_len - 1 - i) rows
 * [kv_indptr[b], kv_indptr[b+1] - (q_len - 1 - i)) (none when that is not
 * positive: out = 0, lse = -inf).
 *
 * Two forms.  With e4m3 KV and q_len = 2 the plan is fused (tokens_fused = 2):
 * the rule applies to the sequences' full row ranges, one work unit serves both
 * tokens, and the split kernel reads each cache row once, masking token 0's
 * last row; partial slot of token i of unit s of sequence b is
 * 2 sum_{b' < b} S_b' + i S_b + s (num_work counts slots, 2 per unit).
 * Otherwise each token is decoded as a sequence of its own over its visible
 * rows, so the cache rows of a sequence are read once per token.
 *
 * mla_decode_plan_multi -- as mla_decode_plan for num_seqs sequences of
 * q_len (1..16) tokens each; the plan's batch is num_seqs * q_len (one output
 * row per token) and its rule applies to the tokens' row ranges in (b, i)
 * order (fused form: to the sequences' rows).  mla_decode_fwd with such a
 * plan reads q rows qo_indptr[b] + i and writes out [num_seqs * q_len, 16, 512]
 * and lse [num_seqs * q_len, 16] in (b, i) order.  Returns the status codes of
 * mla_decode_plan.
 */
MLA_API int mla_decode_plan_multi(const int32_t* kv_indptr_host, int32_t num_seqs, int32_t q_len, int32_t kv_dtype,
                                  int32_t num_sms, int32_t num_splits, mla_plan* plan);

/*
 * Paged KV cache (kernelindex "amd-mixed-mla" submission 703488: AITER's
 * mla_decode_fwd over kv_buffer = kv.view(num_pages, page_size, 1, 576) with
 * kv_indptr counted in pages, kv_indices and kv_last_page_lens).  The cache is
 * num_pages * page_size rows in the storage format of the dtype (scales: one
 * row of scale_stride bytes per cache row for MXFP4).  Sequence b owns the
 * pages kv_indices[kv_page_indptr[b] .. kv_page_indptr[b+1]) in that order;
 * its tokens are those pages' rows in order: page_size rows of every page but
 * the last, kv_last_page_len[b] (1..page_size) rows of the last.  A sequence
 * with no pages is empty (out = 0, lse = -inf).
 *
 * page_size must be a power of two (1, 2, 4, ...; MLA_ERR_UNSUPPORTED
 * otherwise).  Pages of 64 rows or more hold whole tiles of the copies into
 * shared memory; smaller pages are gathered row by row (e4m3: four-row tensor
 * gathers, MXFP4: one bulk copy per row, bf16: one box per page), each row
 * through the page table.  The plan's splits and rule are those of
 * mla_decode_plan with start_b = kv_page_indptr[b] * page_size (a position in
 * the sequences' page-ordered row space) and L_b the token count above;
 * total_kv is kv_page_indptr[batch] * page_size.  Both that and
 * num_pages * page_size must fit in int32.
 *
 * mla_decode_plan_paged -- host only; kv_page_indptr_host[0..batch] and
 * kv_last_page_len_host[0..batch-1] are the host copies of the device arrays
 * passed to mla_decode_fwd_paged.  Returns MLA_OK, MLA_ERR_INVALID_ARG (a bad
 * layout) or MLA_ERR_UNSUPPORTED (page size, or a layout the unit table cannot
 * hold).  Never calls CUDA when num_sms > 0.
 */
MLA_API int mla_decode_plan_paged(const int32_t* kv_page_indptr_host, const int32_t* kv_last_page_len_host,
                                  int32_t batch, int32_t page_size, int32_t num_pages, int32_t kv_dtype,
                                  int32_t num_sms, int32_t num_splits, mla_plan* plan);

/*
 * mla_decode_fwd_paged -- mla_decode_fwd over a paged cache; the plan must come
 * from mla_decode_plan_paged.  Arguments as for mla_decode_fwd, except
 *   kv_pages          device, the cache: num_pages * page_size rows, 16-byte aligned
 *                     (mxfp4 with pages of 64 rows or more: 32-byte aligned).
 *   kv_scale          fp8: fp32[1]; mxfp4: uint8 e8m0 [num_pages * page_size, scale_stride].
 *   kv_page_indptr    device int32 [batch+1], equal to the host copy the plan was made from.
 *   kv_indices        device int32 [kv_page_indptr[batch]], each in [0, num_pages).
 *   kv_last_page_len  device int32 [batch].
 * A page index outside [0, num_pages) or layouts that disagree with the plan are
 * reported by mla_decode_poll_error (MLA_ERR_DEVICE_INDEX); the affected rows
 * read page 0 instead.  Only the rows of the sequences' pages are used: other
 * pages, and the rows of a last page past kv_last_page_len, may hold anything.
 */
MLA_API int mla_decode_fwd_paged(const void* q, const void* kv_pages, const void* kv_scale, int32_t scale_stride,
                                 const int32_t* kv_page_indptr, const int32_t* kv_indices,
                                 const int32_t* kv_last_page_len, const int32_t* qo_indptr, void* out, float* lse,
                                 float sm_scale, const mla_plan* plan, void* workspace, size_t workspace_bytes,
                                 void* stream);

/*
 * mla_decode_fwd_static -- mla_decode_fwd for callers that cannot allocate
 * device memory.  The paper has no counterpart; it exists for code that runs
 * where it gets no allocator: a plugin or custom-operator interface of a host
 * runtime that hands it only its inputs and outputs, or a latency-critical loop
 * where cudaMalloc (which may synchronise the whole device and has unbounded
 * latency) is not allowed.  Instead of a caller-owned workspace it uses one
 * device array of MLA_STATIC_WORKSPACE_BYTES inside this library (held by
 * every GPU that loads the library until the process exits).  It allocates
 * nothing and calls no allocating routine.
 *
 * Arguments are those of mla_decode_fwd without workspace/workspace_bytes, plus
 *   device_error  device int32[1] or NULL: receives this call's device error word
 *                 (0, MLA_ERR_DEVICE_INDEX or MLA_ERR_DEVICE_TIMEOUT) in stream order.
 *
 * The first call on a device looks up the array's device address (once per
 * device, with that device current); make that first call before any stream
 * capture.  The address is kept with the id of the device's context: after
 * the context changes (the application called cudaDeviceReset, or released
 * and re-created the primary context) the next call looks it up again, so
 * that call, too, belongs before any capture.  Each call clears the array's
 * error word and overwrites the rest,
 * so nothing carries over between calls -- but every call on a device shares
 * the one array: calls that may overlap on the GPU (different streams without
 * ordering, or several host threads) race and give wrong results.
 *
 * Returns MLA_ERR_WORKSPACE_TOO_SMALL, launching nothing, when
 * mla_decode_workspace_bytes(plan) > MLA_STATIC_WORKSPACE_BYTES (a plan with
 * more split units than fit: plan with fewer SMs or fewer splits, or use
 * mla_decode_fwd); otherwise the status codes of mla_decode_fwd.
 */
#define MLA_STATIC_WORKSPACE_BYTES (16u << 20)
MLA_API int mla_decode_fwd_static(const void* q, const void* kv, const void* kv_scale, int32_t scale_stride,
                                  const int32_t* kv_indptr, const int32_t* qo_indptr, void* out, float* lse,
                                  float sm_scale, const mla_plan* plan, int32_t* device_error, void* stream);

/*
 * mla_decode_set_trace -- diagnostics, for the library's trace build only
 * (compiled with MLA_TRACE=1; the normal build returns MLA_ERR_UNSUPPORTED for
 * a non-null buffer and records nothing).  The pages have no counterpart.
 * While `buffer` is set, every launch of the tensor-core split kernel (e4m3
 * and MXFP4 KV) writes global-timer stamps (ns) into
 *   buffer[cta * MLA_TRACE_SLOTS + slot]   (device uint64, grid * MLA_TRACE_SLOTS entries)
 * for slot: 0 kernel entry, 1 set-up done, 2 first KV copy issued, 3 query
 * preparation complete, 4 the CTA's unit count (a count, not a time),
 * 5 its tile count (a count), 6 exit, 7 unit list built, 8 + k unit k's
 * epilogue written (k < 8), 16 + t tile t's scores ready for the softmax
 * (t < 64), 80 + t tile t's KV landed with its score buffer free (t < 32),
 * 112 + k unit k's last P.V complete (k < 8), 127 the SM id (a value).  Slots a launch does not reach
 * keep their old contents.  Process-wide; not thread-safe; NULL turns it off.
 */
#define MLA_TRACE_SLOTS 128
MLA_API int mla_decode_set_trace(uint64_t* buffer);

/* Static, NUL-terminated description of a status code. */
MLA_API const char* mla_status_string(int status);

/* Library version, "major.minor.patch". */
MLA_API const char* mla_decode_version(void);

#ifdef __cplusplus
}
#endif

#endif /* MLA_DECODE_H */
