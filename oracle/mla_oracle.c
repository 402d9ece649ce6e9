/*
 * mla_oracle.c -- plain, slow, fp64 CPU oracle for single-token MLA decode.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the checker the CUDA path is compared
 * against.  Only the test suite, the smoke check and the benchmark's CPU-baseline
 * leg may load it.  It shares no code, header, table or helper with the CUDA
 * library: nothing here is included by, or includes, anything under the package.
 *
 * What it computes (kernelindex "amd-mixed-mla" submission 593653, section
 * "Slow fallback", function _bmm_reference; constants from the same page's
 * "Constants" section):
 *
 *   for each sequence b and query head h < 16:
 *     k_t      = dequant(kv[t])                  t in [kv_indptr[b], kv_indptr[b+1])
 *     s_t      = (sum_{d<576} q[qo_indptr[b], h, d] * k_t[d]) * sm_scale
 *     m        = max_t s_t
 *     w_t      = exp(s_t - m),   l = sum_t w_t
 *     out[b,h,j] = sum_t w_t * k_t[j] / l         j < 512  (V = first 512 columns)
 *     lse[b,h]   = m + ln(l)                      (natural log, sm_scale included)
 *
 * The page's reference rounds the softmax to bf16 before the second bmm; this
 * oracle does not round anywhere (pure real-valued definition, evaluated in fp64).
 * An empty sequence gives out = 0 and lse = -inf (the split kernels on submission
 * 593653 guard the normaliser with max(esum, 1e-12) and skip splits whose lse is
 * below -1e30, which yields exactly that).
 *
 * Dequantisation, element by element, in fp64:
 *   bf16 : widen the 16 stored bits (exact).
 *   fp8  : OCP e4m3fn (bias 7, subnormals, max 448, S.1111.111 = NaN, no inf),
 *          times the per-tensor fp32 scale (submission 754939, quantize_fp8:
 *          x ~= fp8 * scale with scale = amax / 448).
 *   mxfp4: element 2i is the low nibble of byte i, element 2i+1 the high nibble
 *          (submission 754939, stage-1 kernel mla_s1, V unpack/join); a nibble is
 *          e2m1 decoded by the page's _dq4 rule (e = (n>>1)&3, m = n&1,
 *          e==0 ? m/2 : (1+m/2)*2^(e-1), bit 3 = sign); block j = elements
 *          32j..32j+31 uses scale byte j of the row, worth 2^(byte-127) (the same
 *          kernel's "vsc_exp = scale - 127; exp2").  Byte 255 decodes to NaN.
 *
 * Parallelism: an OpenMP loop over (b, h) pairs only; each pair is evaluated by
 * the straight loops above, with no blocking, fusion or reordering.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORACLE_NUM_HEADS 16
#define ORACLE_QK_DIM 576
#define ORACLE_V_DIM 512
#define ORACLE_MX_BLOCK 32

enum { ORACLE_KV_BF16 = 0, ORACLE_KV_FP8_E4M3 = 1, ORACLE_KV_MXFP4 = 2 };

/* Planted mistakes for the pin self-test: compiled only with -DORACLE_MUTANT=n.
 * The default build has ORACLE_MUTANT == 0 and none of them is active. */
#ifndef ORACLE_MUTANT
#define ORACLE_MUTANT 0
#endif

/* ---------------------------------------------------------------- decoders */

double oracle_bf16_to_double(uint16_t bits) {
  uint32_t u = (uint32_t)bits << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

double oracle_e4m3_to_double(uint8_t code) {
  int sign = (code >> 7) & 1;
  int e = (code >> 3) & 0xF;
  int m = code & 0x7;
  double v;
  if (e == 0xF && m == 0x7) return NAN;
#if ORACLE_MUTANT == 10
  v = ldexp(1.0 + m / 8.0, e - 7); /* mistake: subnormals decoded as normals */
#else
  if (e == 0)
    v = ldexp(m / 8.0, 1 - 7); /* subnormal: 0.m * 2^(1-bias) */
  else
    v = ldexp(1.0 + m / 8.0, e - 7);
#endif
  return sign ? -v : v;
}

double oracle_e2m1_to_double(uint8_t nibble) {
  int sign = (nibble >> 3) & 1;
  int e = (nibble >> 1) & 3;
  int m = nibble & 1;
  double v = (e == 0) ? 0.5 * m : ldexp(1.0 + 0.5 * m, e - 1);
  return sign ? -v : v;
}

double oracle_e8m0_to_double(uint8_t e) {
  if (e == 255) return NAN;
#if ORACLE_MUTANT == 6
  return ldexp(1.0, (int)e - 128); /* mistake: wrong bias */
#else
  return ldexp(1.0, (int)e - 127);
#endif
}

/* Element-wise array forms, for the decoder pins. */
void oracle_decode_bf16_array(const uint16_t* in, double* out, int64_t n) {
  for (int64_t i = 0; i < n; ++i) out[i] = oracle_bf16_to_double(in[i]);
}
void oracle_decode_e4m3_array(const uint8_t* in, double* out, int64_t n) {
  for (int64_t i = 0; i < n; ++i) out[i] = oracle_e4m3_to_double(in[i]);
}
void oracle_decode_e2m1_array(const uint8_t* in, double* out, int64_t n) {
  for (int64_t i = 0; i < n; ++i) out[i] = oracle_e2m1_to_double(in[i]);
}
void oracle_decode_e8m0_array(const uint8_t* in, double* out, int64_t n) {
  for (int64_t i = 0; i < n; ++i) out[i] = oracle_e8m0_to_double(in[i]);
}

/* One cached KV row, dequantised to 576 doubles. */
static void dequant_row(int kv_dtype, const void* kv, const uint8_t* block_scales,
                        int64_t scale_stride, double kv_scale, int64_t row, double* k) {
  if (kv_dtype == ORACLE_KV_BF16) {
    const uint16_t* p = (const uint16_t*)kv + row * ORACLE_QK_DIM;
    for (int d = 0; d < ORACLE_QK_DIM; ++d) k[d] = oracle_bf16_to_double(p[d]);
  } else if (kv_dtype == ORACLE_KV_FP8_E4M3) {
    const uint8_t* p = (const uint8_t*)kv + row * ORACLE_QK_DIM;
    for (int d = 0; d < ORACLE_QK_DIM; ++d) {
#if ORACLE_MUTANT == 4
      k[d] = oracle_e4m3_to_double(p[d]); /* mistake: per-tensor scale dropped */
#else
      k[d] = oracle_e4m3_to_double(p[d]) * kv_scale;
#endif
    }
  } else {
    const uint8_t* p = (const uint8_t*)kv + row * (ORACLE_QK_DIM / 2);
    const uint8_t* s = block_scales + row * scale_stride;
    for (int d = 0; d < ORACLE_QK_DIM; ++d) {
      uint8_t byte = p[d / 2];
#if ORACLE_MUTANT == 5
      uint8_t nib = (d % 2 == 0) ? (uint8_t)(byte >> 4) : (uint8_t)(byte & 0xF); /* mistake: nibble order */
#else
      uint8_t nib = (d % 2 == 0) ? (uint8_t)(byte & 0xF) : (uint8_t)(byte >> 4);
#endif
      k[d] = oracle_e2m1_to_double(nib) * oracle_e8m0_to_double(s[d / ORACLE_MX_BLOCK]);
    }
  }
}

/* Attention of one query row over KV rows [start, end), one head -- or, when
 * `rows` is not NULL, over the rows rows[0..end-start) in that order (a paged
 * cache).  Writes the normalised output (512 values) and the natural-log lse. */
static void attend_one(int kv_dtype, const double* qv, const void* kv, const uint8_t* block_scales,
                       int64_t scale_stride, double kv_scale, int64_t start, int64_t end,
                       const int64_t* rows, double sm_scale, double* o, double* lse, double* scores,
                       double* k) {
  int64_t L = end - start;
  if (L <= 0) {
    for (int j = 0; j < ORACLE_V_DIM; ++j) o[j] = 0.0;
    *lse = -INFINITY;
    return;
  }
  /* pass 1: scores */
  for (int64_t t = 0; t < L; ++t) {
    dequant_row(kv_dtype, kv, block_scales, scale_stride, kv_scale, rows ? rows[t] : start + t, k);
    double acc = 0.0;
#if ORACLE_MUTANT == 1
    for (int d = 0; d < 512; ++d) acc += qv[d] * k[d]; /* mistake: rope part dropped */
#else
    for (int d = 0; d < ORACLE_QK_DIM; ++d) acc += qv[d] * k[d];
#endif
#if ORACLE_MUTANT == 3
    scores[t] = acc; /* mistake: sm_scale ignored */
#else
    scores[t] = acc * sm_scale;
#endif
  }
  /* softmax statistics */
  double m = -INFINITY;
  for (int64_t t = 0; t < L; ++t)
    if (scores[t] > m) m = scores[t];
  double l = 0.0;
  for (int64_t t = 0; t < L; ++t) {
#if ORACLE_MUTANT == 7
    scores[t] = exp(scores[t]); /* mistake: no max subtraction (overflows) */
#else
    scores[t] = exp(scores[t] - m);
#endif
    l += scores[t];
  }
  /* pass 2: weighted sum of V = first 512 columns of the same rows */
  for (int j = 0; j < ORACLE_V_DIM; ++j) o[j] = 0.0;
  for (int64_t t = 0; t < L; ++t) {
    dequant_row(kv_dtype, kv, block_scales, scale_stride, kv_scale, rows ? rows[t] : start + t, k);
    for (int j = 0; j < ORACLE_V_DIM; ++j) {
#if ORACLE_MUTANT == 2
      o[j] += scores[t] * k[j + 64]; /* mistake: V taken from the wrong columns */
#else
      o[j] += scores[t] * k[j];
#endif
    }
  }
  for (int j = 0; j < ORACLE_V_DIM; ++j) o[j] /= l;
#if ORACLE_MUTANT == 7
  *lse = log(l);
#elif ORACLE_MUTANT == 8
  *lse = m + log2(l); /* mistake: wrong logarithm base */
#else
  *lse = m + log(l);
#endif
}

static void widen_q(const uint16_t* q, int64_t qrow, int h, double* qv) {
#if ORACLE_MUTANT == 9
  h = 0; /* mistake: every head reads head 0 */
#endif
  const uint16_t* p = q + (qrow * ORACLE_NUM_HEADS + h) * ORACLE_QK_DIM;
  for (int d = 0; d < ORACLE_QK_DIM; ++d) qv[d] = oracle_bf16_to_double(p[d]);
}

static int64_t max_len(const int32_t* kv_indptr, int batch) {
  int64_t mx = 0;
  for (int b = 0; b < batch; ++b) {
    int64_t L = (int64_t)kv_indptr[b + 1] - kv_indptr[b];
    if (L > mx) mx = L;
  }
  return mx;
}

/*
 * Full decode.  q: bf16 bits [*, 16, 576]; kv: bf16 bits / e4m3 bytes [*, 576] or
 * packed e2m1 bytes [*, 288]; block_scales: e8m0 bytes [*, scale_stride] (mxfp4 only);
 * kv_scale: per-tensor scale (fp8 only).  out: [batch, 16, 512]; lse: [batch, 16].
 * Returns 0, or -1 on an invalid argument.
 */
int oracle_mla_decode(int kv_dtype, const uint16_t* q, const void* kv, const uint8_t* block_scales,
                      int64_t scale_stride, double kv_scale, const int32_t* kv_indptr,
                      const int32_t* qo_indptr, int batch, double sm_scale, double* out,
                      double* lse, int num_threads) {
  if (batch < 0 || !kv_indptr || !qo_indptr || !out || !lse) return -1;
  if (kv_dtype < 0 || kv_dtype > 2) return -1;
  if (kv_dtype == ORACLE_KV_MXFP4 && (!block_scales || scale_stride < ORACLE_QK_DIM / ORACLE_MX_BLOCK)) return -1;
  int64_t Lmax = max_len(kv_indptr, batch);
  int64_t pairs = (int64_t)batch * ORACLE_NUM_HEADS;
#ifdef _OPENMP
  if (num_threads > 0) omp_set_num_threads(num_threads);
#pragma omp parallel
#endif
  {
    double* scores = (double*)malloc(sizeof(double) * (size_t)(Lmax > 0 ? Lmax : 1));
    double qv[ORACLE_QK_DIM], k[ORACLE_QK_DIM];
#ifdef _OPENMP
#pragma omp for schedule(dynamic, 1)
#endif
    for (int64_t pr = 0; pr < pairs; ++pr) {
      int b = (int)(pr / ORACLE_NUM_HEADS), h = (int)(pr % ORACLE_NUM_HEADS);
      widen_q(q, qo_indptr[b], h, qv);
      attend_one(kv_dtype, qv, kv, block_scales, scale_stride, kv_scale, kv_indptr[b],
                 kv_indptr[b + 1], NULL, sm_scale, out + pr * ORACLE_V_DIM, lse + pr, scores, k);
    }
    free(scores);
  }
  return 0;
}

/*
 * Paged cache (kernelindex "amd-mixed-mla" submission 703488's AITER call and
 * its page_size variants: kv_buffer = kv.view(num_pages, page_size, 1, 576)
 * with kv_indptr counted in pages, kv_indices and kv_last_page_lens).  Sequence
 * b owns the pages kv_indices[page_indptr[b] .. page_indptr[b+1]) in that order;
 * its tokens are those pages' rows in order, all page_size rows of every page
 * but the last, and last_page_len[b] rows of the last.  Row i of sequence b is
 * therefore cache row kv_indices[page_indptr[b] + i / P] * P + i % P, and the
 * attention is the definition above over those rows.  A sequence with no pages
 * is empty.  Returns 0, or -1 on an invalid argument (including a page index
 * outside [0, num_pages) or a last-page length outside [1, P]).
 */
int oracle_mla_decode_paged(int kv_dtype, const uint16_t* q, const void* kv, const uint8_t* block_scales,
                            int64_t scale_stride, double kv_scale, const int32_t* page_indptr,
                            const int32_t* kv_indices, const int32_t* last_page_len, int page_size,
                            int64_t num_pages, const int32_t* qo_indptr, int batch, double sm_scale,
                            double* out, double* lse, int num_threads) {
  if (batch < 0 || !page_indptr || !qo_indptr || !out || !lse || page_size < 1) return -1;
  if (kv_dtype < 0 || kv_dtype > 2) return -1;
  if (kv_dtype == ORACLE_KV_MXFP4 && (!block_scales || scale_stride < ORACLE_QK_DIM / ORACLE_MX_BLOCK)) return -1;
  /* the rows of every sequence, in order */
  int64_t* first = (int64_t*)malloc(sizeof(int64_t) * (size_t)(batch + 1));
  first[0] = 0;
  for (int b = 0; b < batch; ++b) {
    int64_t np = (int64_t)page_indptr[b + 1] - page_indptr[b];
    if (np < 0 || (np > 0 && (!kv_indices || !last_page_len))) {
      free(first);
      return -1;
    }
    int64_t L = 0;
    if (np > 0) {
      if (last_page_len[b] < 1 || last_page_len[b] > page_size) {
        free(first);
        return -1;
      }
#if ORACLE_MUTANT == 11
      L = np * page_size; /* mistake: the last page read in full */
#else
      L = (np - 1) * page_size + last_page_len[b];
#endif
    }
    first[b + 1] = first[b] + L;
  }
  int64_t* rows = (int64_t*)malloc(sizeof(int64_t) * (size_t)(first[batch] > 0 ? first[batch] : 1));
  for (int b = 0; b < batch; ++b) {
    for (int64_t i = 0; i < first[b + 1] - first[b]; ++i) {
#if ORACLE_MUTANT == 12
      int64_t page = (int64_t)page_indptr[b] + i / page_size; /* mistake: page table ignored */
#else
      int64_t page = kv_indices[page_indptr[b] + i / page_size];
#endif
      if (page < 0 || page >= num_pages) {
        free(rows);
        free(first);
        return -1;
      }
      rows[first[b] + i] = page * page_size + i % page_size;
    }
  }
  int64_t Lmax = 0;
  for (int b = 0; b < batch; ++b)
    if (first[b + 1] - first[b] > Lmax) Lmax = first[b + 1] - first[b];
  int64_t pairs = (int64_t)batch * ORACLE_NUM_HEADS;
#ifdef _OPENMP
  if (num_threads > 0) omp_set_num_threads(num_threads);
#pragma omp parallel
#endif
  {
    double* scores = (double*)malloc(sizeof(double) * (size_t)(Lmax > 0 ? Lmax : 1));
    double qv[ORACLE_QK_DIM], k[ORACLE_QK_DIM];
#ifdef _OPENMP
#pragma omp for schedule(dynamic, 1)
#endif
    for (int64_t pr = 0; pr < pairs; ++pr) {
      int b = (int)(pr / ORACLE_NUM_HEADS), h = (int)(pr % ORACLE_NUM_HEADS);
      widen_q(q, qo_indptr[b], h, qv);
      attend_one(kv_dtype, qv, kv, block_scales, scale_stride, kv_scale, 0, first[b + 1] - first[b],
                 rows + first[b], sm_scale, out + pr * ORACLE_V_DIM, lse + pr, scores, k);
    }
    free(scores);
  }
  free(rows);
  free(first);
  return 0;
}

/*
 * Several query tokens per sequence (q_len > 1: the decode of q_len draft or
 * verification tokens at once).  The pages decode one token per sequence;
 * this is the plain causal reading for more: sequence b's tokens are query
 * rows qo_indptr[b] + i (i < q_len) and the last q_len of its L_b cached rows
 * are those tokens' own entries, so token i attends to the first
 * L_b - (q_len - 1 - i) rows [kv_indptr[b], kv_indptr[b+1] - (q_len - 1 - i))
 * (none when that is not positive: out = 0, lse = -inf).  Outputs are in
 * (b, i) order: out [batch * q_len, 16, 512], lse [batch * q_len, 16].
 */
int oracle_mla_decode_multi(int kv_dtype, const uint16_t* q, const void* kv, const uint8_t* block_scales,
                            int64_t scale_stride, double kv_scale, const int32_t* kv_indptr,
                            const int32_t* qo_indptr, int batch, int q_len, double sm_scale, double* out,
                            double* lse, int num_threads) {
  if (batch < 0 || q_len < 1 || !kv_indptr || !qo_indptr || !out || !lse) return -1;
  if (kv_dtype < 0 || kv_dtype > 2) return -1;
  if (kv_dtype == ORACLE_KV_MXFP4 && (!block_scales || scale_stride < ORACLE_QK_DIM / ORACLE_MX_BLOCK)) return -1;
  int64_t Lmax = max_len(kv_indptr, batch);
  int64_t pairs = (int64_t)batch * q_len * ORACLE_NUM_HEADS;
#ifdef _OPENMP
  if (num_threads > 0) omp_set_num_threads(num_threads);
#pragma omp parallel
#endif
  {
    double* scores = (double*)malloc(sizeof(double) * (size_t)(Lmax > 0 ? Lmax : 1));
    double qv[ORACLE_QK_DIM], k[ORACLE_QK_DIM];
#ifdef _OPENMP
#pragma omp for schedule(dynamic, 1)
#endif
    for (int64_t pr = 0; pr < pairs; ++pr) {
      const int64_t t = pr / ORACLE_NUM_HEADS;  /* (b, i) in order */
      const int b = (int)(t / q_len), i = (int)(t % q_len), h = (int)(pr % ORACLE_NUM_HEADS);
#if ORACLE_MUTANT == 13
      int64_t end = (int64_t)kv_indptr[b + 1] - (q_len - i); /* mistake: the token's own row left out */
#else
      int64_t end = (int64_t)kv_indptr[b + 1] - (q_len - 1 - i);
#endif
      if (end < kv_indptr[b]) end = kv_indptr[b];
      widen_q(q, (int64_t)qo_indptr[b] + i, h, qv);
      attend_one(kv_dtype, qv, kv, block_scales, scale_stride, kv_scale, kv_indptr[b], end, NULL, sm_scale,
                 out + pr * ORACLE_V_DIM, lse + pr, scores, k);
    }
    free(scores);
  }
  return 0;
}

/*
 * One split: the normalised partial attention of query row qrow over KV rows
 * [start, end), all 16 heads.  o: [16, 512]; lse: [16].  An empty range gives
 * o = 0 and lse = -inf.
 */
int oracle_mla_partial(int kv_dtype, const uint16_t* q, const void* kv, const uint8_t* block_scales,
                       int64_t scale_stride, double kv_scale, int64_t qrow, int64_t start,
                       int64_t end, double sm_scale, double* o, double* lse) {
  if (!o || !lse) return -1;
  int64_t L = end > start ? end - start : 1;
  double* scores = (double*)malloc(sizeof(double) * (size_t)L);
  double qv[ORACLE_QK_DIM], k[ORACLE_QK_DIM];
  for (int h = 0; h < ORACLE_NUM_HEADS; ++h) {
    widen_q(q, qrow, h, qv);
    attend_one(kv_dtype, qv, kv, block_scales, scale_stride, kv_scale, start, end, NULL, sm_scale,
               o + (int64_t)h * ORACLE_V_DIM, lse + h, scores, k);
  }
  free(scores);
  return 0;
}

/*
 * Log-sum-exp combine of n normalised partials (submission 593653, stage-2 kernel
 * _flash_fp8_split_s2, restated in its closed form): per head,
 *   M = max_s lse_s over splits with lse_s > -inf,  w_s = exp(lse_s - M),
 *   out = sum_s w_s o_s / sum_s w_s,  lse = M + ln(sum_s w_s).
 * All splits empty -> out = 0, lse = -inf.  o: [n, 16, 512]; lse: [n, 16].
 */
int oracle_mla_combine(int n, const double* o, const double* lse, double* out, double* lse_out) {
  if (n < 0 || !out || !lse_out) return -1;
  for (int h = 0; h < ORACLE_NUM_HEADS; ++h) {
    double M = -INFINITY;
    for (int s = 0; s < n; ++s) {
      double v = lse[(int64_t)s * ORACLE_NUM_HEADS + h];
      if (v > M) M = v;
    }
    double* dst = out + (int64_t)h * ORACLE_V_DIM;
    for (int j = 0; j < ORACLE_V_DIM; ++j) dst[j] = 0.0;
    if (M == -INFINITY) {
      lse_out[h] = -INFINITY;
      continue;
    }
    double wsum = 0.0;
    for (int s = 0; s < n; ++s) {
      double v = lse[(int64_t)s * ORACLE_NUM_HEADS + h];
      if (v == -INFINITY) continue;
      double w = exp(v - M);
      wsum += w;
      const double* src = o + ((int64_t)s * ORACLE_NUM_HEADS + h) * ORACLE_V_DIM;
      for (int j = 0; j < ORACLE_V_DIM; ++j) dst[j] += w * src[j];
    }
    for (int j = 0; j < ORACLE_V_DIM; ++j) dst[j] /= wsum;
    lse_out[h] = M + log(wsum);
  }
  return 0;
}

int oracle_mutant_id(void) { return ORACLE_MUTANT; }
