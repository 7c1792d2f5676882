/*
 * MLA decode oracle: plain, slow, float64 CPU reference for single-token
 * Multi-head Latent Attention decode over a paged latent KV cache.
 *
 * TEST INFRASTRUCTURE ONLY. Nothing on the product path may load or call
 * this library; only the tests, the smoke check and the benchmark's CPU
 * baseline leg use it. It shares no code, header or constant table with
 * the CUDA library.
 *
 * What it computes (kernelbot amd-mixed-mla submission 689529 "MLA decode
 * V3", module constants and custom_kernel; the same call appears in
 * submissions 690201 "V6c" and 641982 "v86"):
 *   16 query heads share one KV head; every KV row holds 576 values (a
 *   512-wide latent followed by a 64-wide rope part). For sequence b and head
 *   h the scores are s_t = sm_scale * sum_{d<576} q[b,h,d] * kv[row_t,d] with
 *   row_t = kv_indices[kv_indptr[b] + t], 0 <= t < kv_indptr[b+1]-kv_indptr[b]
 *   (page_size = 1: one token per page). The output is
 *   O[b,h,j] = sum_t softmax(s)_t * kv[row_t, j] for j < 512, i.e. the value
 *   vectors are the first 512 entries of the very rows used as keys
 *   (V3 passes the single kv buffer once; V6c views it as [pages,1,1,576]).
 *   Paged addressing (submission 641982 "v86", _run_a8w8, and 598454 "v12",
 *   custom_kernel): the KV buffer is viewed as [num_pages, page_size, 1, 576],
 *   kv_indptr counts pages, kv_indices holds page ids and kv_last_page_lens[b]
 *   is the number of tokens used in sequence b's last page. Token t is entry
 *   t % page_size of page kv_indices[kv_indptr[b] + t / page_size]; page_size
 *   1 with every last page full is the row addressing above.
 *   There is no mask: with one query token per sequence it sees all of its KV
 *   (the pages set is_causal both ways; with q_seq_len = 1 the two agree).
 *   logit_cap = 0 on the pages means no cap.
 *
 * Value modes (the dtype_mode argument):
 *   0  bf16 Q x bf16 KV. Inputs are used exactly (bf16 -> double is exact).
 *   1  fp8: Q is cast directly to OCP fp8 e4m3fn with scale 1 (no amax pass;
 *      V3 / V6c docstrings and custom_kernel, submission 598454 "v12" step 1)
 *      and KV holds e4m3fn bytes with one per-tensor fp32 kv_scale
 *      (kv_data["fp8"] = (buffer, scale) in every submission). Values are
 *      decode(byte) * kv_scale; attention on the dequantised values is the
 *      same as folding q_scale * kv_scale into the scores and kv_scale into
 *      the output.
 *   2  bf16 Q x fp8 KV (the "a16w8" naming in submission 598454 "v12").
 *
 * Readings where the pages are silent (also listed with the design notes):
 *   - the Q cast rounds to nearest, ties to even; magnitudes above 448 (which
 *     the pages argue cannot occur for randn Q) saturate to +-448;
 *   - an empty sequence yields O = 0 and LSE = -inf;
 *   - the log-sum-exp returned is natural-log based.
 *
 * Build: gcc -O2 -fopenmp -fPIC -shared mla_oracle.c -o liboracle.so -lm
 * (OpenMP only spreads independent (sequence, head) pairs over cores.)
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORACLE_HEADS 16
#define ORACLE_QK_DIM 576
#define ORACLE_V_DIM 512

/* bf16 is the upper 16 bits of an IEEE-754 binary32 value. */
double oracle_bf16_decode(uint16_t bits) {
  uint32_t u = (uint32_t)bits << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

/*
 * OCP 8-bit floating point, E4M3 ("e4m3fn"): 1 sign bit, 4 exponent bits with
 * bias 7, 3 mantissa bits. Exponent field 0 is subnormal (m/8 * 2^-6);
 * S.1111.111 is NaN; there is no infinity; the largest finite value is
 * S.1111.110 = 448.
 */
double oracle_e4m3_decode(uint8_t code) {
  int s = code >> 7, e = (code >> 3) & 15, m = code & 7;
  double v;
  if (e == 15 && m == 7) return NAN;
  if (e == 0)
    v = ldexp((double)m, -9);          /* (m/8) * 2^(1-7) */
  else
    v = ldexp(8.0 + (double)m, e - 10); /* (1 + m/8) * 2^(e-7) */
  return s ? -v : v;
}

/*
 * Round a real number to e4m3fn: nearest representable value, ties to the
 * even code (the one whose mantissa LSB is 0), and magnitudes above the
 * largest finite value saturate to +-448. NaN stays NaN.
 * Non-negative finite codes 0x00..0x7E are increasing in value, so the
 * result is found by bracketing |x| between two neighbouring codes.
 */
uint8_t oracle_e4m3_encode(double x) {
  uint8_t sign = signbit(x) ? 0x80 : 0x00;
  double a = fabs(x);
  int lo;
  double vlo, vhi;
  if (isnan(x)) return (uint8_t)(sign | 0x7F);
  if (a >= 448.0) return (uint8_t)(sign | 0x7E);
  lo = 0;
  while (lo < 0x7E && oracle_e4m3_decode((uint8_t)(lo + 1)) <= a) lo++;
  vlo = oracle_e4m3_decode((uint8_t)lo);
  vhi = oracle_e4m3_decode((uint8_t)(lo + 1));
  if (a - vlo < vhi - a) return (uint8_t)(sign | lo);
  if (vhi - a < a - vlo) return (uint8_t)(sign | (lo + 1));
  return (uint8_t)(sign | ((lo & 1) ? lo + 1 : lo));
}

/* Query element as the method sees it (mode 1: the direct e4m3 cast, scale 1). */
static double q_value(const uint16_t* q, int64_t i, int mode) {
  double v = oracle_bf16_decode(q[i]);
  if (mode == 1) v = oracle_e4m3_decode(oracle_e4m3_encode(v));
  return v;
}

/* KV element as the method sees it. */
static double kv_value(const void* kv, int64_t row, int d, int mode, double kv_scale) {
  if (mode == 0) return oracle_bf16_decode(((const uint16_t*)kv)[row * ORACLE_QK_DIM + d]);
  return oracle_e4m3_decode(((const uint8_t*)kv)[row * ORACLE_QK_DIM + d]) * kv_scale;
}

/* KV row of token t of a sequence whose page list starts at kv_indices[page_base]. */
static int64_t token_row(const int32_t* kv_indices, int64_t page_base, int64_t t, int page_size) {
  return (int64_t)kv_indices[page_base + t / page_size] * page_size + t % page_size;
}

/*
 * Tokens of sequence b: (pages - 1) * page_size + its last page length, or 0
 * when it has no pages. With no last_page_len array every last page is full.
 * Returns -1 for a negative page count or a last page length outside
 * [1, page_size].
 */
static int64_t seq_tokens(const int32_t* kv_indptr, const int32_t* last_page_len, int page_size, int b) {
  int64_t pages = (int64_t)kv_indptr[b + 1] - kv_indptr[b], last;
  if (pages == 0) return 0;
  if (pages < 0) return -1;
  last = last_page_len ? (int64_t)last_page_len[b] : (int64_t)page_size;
  if (last < 1 || last > page_size) return -1;
  return (pages - 1) * page_size + last;
}

/*
 * Attention of head h of query row q_row over the tokens t in [t_begin, t_end)
 * of sequence b. Writes out[0..511] and *lse (natural log of sum_t e^{s_t}).
 * Returns 0, or -1 if a token's row is outside [0, num_slots).
 */
static int attend_head(const uint16_t* q, const void* kv, int64_t num_slots, int mode, double kv_scale,
                       const int32_t* kv_indptr, const int32_t* kv_indices, int page_size, double sm_scale, int b,
                       int64_t q_row, int h, int64_t t_begin, int64_t t_end, double* out, double* lse) {
  int64_t n = t_end - t_begin, t;
  int d, j;
  double m, z, *s;
  const int64_t base = (int64_t)kv_indptr[b];
  double qh[ORACLE_QK_DIM];
  for (d = 0; d < ORACLE_QK_DIM; ++d) qh[d] = q_value(q, (q_row * ORACLE_HEADS + h) * ORACLE_QK_DIM + d, mode);
  for (j = 0; j < ORACLE_V_DIM; ++j) out[j] = 0.0;
  if (n <= 0) {
    *lse = -INFINITY;
    return 0;
  }
  s = (double*)malloc(sizeof(double) * (size_t)n);
  if (!s) return -2;
  /* scores */
  for (t = 0; t < n; ++t) {
    int64_t row = token_row(kv_indices, base, t_begin + t, page_size);
    double acc = 0.0;
    if (row < 0 || row >= num_slots) {
      free(s);
      return -1;
    }
    for (d = 0; d < ORACLE_QK_DIM; ++d) acc += qh[d] * kv_value(kv, row, d, mode, kv_scale);
    s[t] = sm_scale * acc;
  }
  /* softmax weights (shifted by the max so no exp overflows) */
  m = s[0];
  for (t = 1; t < n; ++t)
    if (s[t] > m) m = s[t];
  z = 0.0;
  for (t = 0; t < n; ++t) {
    s[t] = exp(s[t] - m);
    z += s[t];
  }
  /* weighted sum of the value vectors = first 512 entries of the same rows */
  for (t = 0; t < n; ++t) {
    int64_t row = token_row(kv_indices, base, t_begin + t, page_size);
    double w = s[t] / z;
    for (j = 0; j < ORACLE_V_DIM; ++j) out[j] += w * kv_value(kv, row, j, mode, kv_scale);
  }
  *lse = m + log(z);
  free(s);
  return 0;
}

/*
 * Full decode over a paged KV buffer for the sequences listed in seq_ids (all
 * B sequences, in order, when seq_ids is NULL). kv_indptr [B+1] counts pages,
 * kv_indices holds page ids, kv_last_page_len [B] the tokens used in each
 * last page (NULL: every last page is full); num_rows = num_pages * page_size.
 * out: [n_seq, 16, 512] float64; lse: [n_seq, 16] or NULL. Returns 0 on
 * success, -1 for a token row outside the buffer, -3 for bad arguments.
 */
int oracle_decode_paged(int batch, const uint16_t* q, const void* kv, int64_t num_rows, int mode, float kv_scale,
                        const int32_t* kv_indptr, const int32_t* kv_indices, const int32_t* kv_last_page_len,
                        int page_size, double sm_scale, const int32_t* seq_ids, int n_seq, double* out,
                        double* lse) {
  int i, bad = 0;
  if (batch < 0 || mode < 0 || mode > 2 || page_size < 1 || !out) return -3;
  if (!seq_ids) n_seq = batch;
  for (i = 0; i < n_seq; ++i) {
    int b = seq_ids ? seq_ids[i] : i;
    if (b < 0 || b >= batch || seq_tokens(kv_indptr, kv_last_page_len, page_size, b) < 0) return -3;
  }
#pragma omp parallel for schedule(dynamic, 1) reduction(| : bad)
  for (i = 0; i < n_seq * ORACLE_HEADS; ++i) {
    int k = i / ORACLE_HEADS, h = i % ORACLE_HEADS;
    int b = seq_ids ? seq_ids[k] : k;
    double l;
    int rc = attend_head(q, kv, num_rows, mode, (double)kv_scale, kv_indptr, kv_indices, page_size, sm_scale, b, b, h,
                         0, seq_tokens(kv_indptr, kv_last_page_len, page_size, b), out + (size_t)i * ORACLE_V_DIM,
                         &l);
    if (rc) bad |= 1;
    if (lse) lse[i] = l;
  }
  return bad ? -1 : 0;
}

/* The unpaged decode: page_size 1, so kv_indptr / kv_indices address single rows. */
int oracle_decode(int batch, const uint16_t* q, const void* kv, int64_t num_slots, int mode, float kv_scale,
                  const int32_t* kv_indptr, const int32_t* kv_indices, double sm_scale, const int32_t* seq_ids,
                  int n_seq, double* out, double* lse) {
  return oracle_decode_paged(batch, q, kv, num_slots, mode, kv_scale, kv_indptr, kv_indices, NULL, 1, sm_scale,
                             seq_ids, n_seq, out, lse);
}

/*
 * Multi-token decode (submission 690201 "V6c", _build_cache: qo_indptr =
 * arange(B + 1) * q_seq_len, handed to the stage-1 call with max_seqlen_q).
 * Sequence b has q_b = qo_indptr[b+1] - qo_indptr[b] query tokens, rows
 * qo_indptr[b] .. qo_indptr[b+1] - 1 of q and out. The query tokens are the
 * last q_b tokens of the sequence: with causal != 0, query token j sees the
 * first max(0, L_b - q_b + j + 1) of the sequence's L_b KV tokens; otherwise
 * every query token sees all L_b. KV addressing as oracle_decode_paged.
 * out: [qo_indptr[B], 16, 512] float64; lse: [qo_indptr[B], 16] or NULL.
 * Returns 0, -1 for a token row outside the buffer, -2 when out of memory,
 * -3 for bad arguments.
 */
int oracle_decode_multi(int batch, const uint16_t* q, const void* kv, int64_t num_rows, int mode, float kv_scale,
                        const int32_t* qo_indptr, const int32_t* kv_indptr, const int32_t* kv_indices,
                        const int32_t* kv_last_page_len, int page_size, int causal, double sm_scale, double* out,
                        double* lse) {
  int b, bad = 0;
  int64_t i, n_rows, *row_seq, *row_len;
  if (batch < 0 || mode < 0 || mode > 2 || page_size < 1 || !out || !qo_indptr) return -3;
  if (batch > 0 && qo_indptr[0] != 0) return -3;
  for (b = 0; b < batch; ++b)
    if (qo_indptr[b + 1] < qo_indptr[b] || seq_tokens(kv_indptr, kv_last_page_len, page_size, b) < 0) return -3;
  n_rows = batch > 0 ? qo_indptr[batch] : 0;
  row_seq = (int64_t*)malloc(sizeof(int64_t) * (size_t)(n_rows + 1));
  row_len = (int64_t*)malloc(sizeof(int64_t) * (size_t)(n_rows + 1));
  if (!row_seq || !row_len) {
    free(row_seq);
    free(row_len);
    return -2;
  }
  /* sequence and number of visible KV tokens of every query row */
  for (b = 0; b < batch; ++b) {
    const int64_t L = seq_tokens(kv_indptr, kv_last_page_len, page_size, b);
    const int64_t qb = (int64_t)qo_indptr[b + 1] - qo_indptr[b];
    int64_t j;
    for (j = 0; j < qb; ++j) {
      int64_t n = causal ? L - qb + j + 1 : L;
      row_seq[qo_indptr[b] + j] = b;
      row_len[qo_indptr[b] + j] = n < 0 ? 0 : (n > L ? L : n);
    }
  }
#pragma omp parallel for schedule(dynamic, 1) reduction(| : bad)
  for (i = 0; i < n_rows * ORACLE_HEADS; ++i) {
    const int64_t r = i / ORACLE_HEADS;
    const int h = (int)(i % ORACLE_HEADS);
    double l;
    int rc = attend_head(q, kv, num_rows, mode, (double)kv_scale, kv_indptr, kv_indices, page_size, sm_scale,
                         (int)row_seq[r], r, h, 0, row_len[r], out + (size_t)i * ORACLE_V_DIM, &l);
    if (rc) bad |= 1;
    if (lse) lse[i] = l;
  }
  free(row_seq);
  free(row_len);
  return bad ? -1 : 0;
}

/*
 * Attention of sequence b over its rows [t_begin, t_end) only: the partial
 * result one split of a split-KV decode must produce. out [16,512], lse [16].
 */
int oracle_decode_range(int batch, const uint16_t* q, const void* kv, int64_t num_slots, int mode, float kv_scale,
                        const int32_t* kv_indptr, const int32_t* kv_indices, double sm_scale, int b,
                        int64_t t_begin, int64_t t_end, double* out, double* lse) {
  int h, bad = 0;
  int64_t len;
  if (b < 0 || b >= batch || mode < 0 || mode > 2) return -3;
  len = (int64_t)kv_indptr[b + 1] - kv_indptr[b];
  if (t_begin < 0 || t_end > len || t_begin > t_end) return -3;
  for (h = 0; h < ORACLE_HEADS; ++h)
    if (attend_head(q, kv, num_slots, mode, (double)kv_scale, kv_indptr, kv_indices, 1, sm_scale, b, b, h, t_begin,
                    t_end,
                    out + (size_t)h * ORACLE_V_DIM, lse + h))
      bad = 1;
  return bad ? -1 : 0;
}

/*
 * Merge the softmax results of disjoint row sets of one sequence: with
 * L = log sum_s e^{lse_s}, O = sum_s e^{lse_s - L} O_s (each O_s is already
 * normalised over its own rows). Parts with lse = -inf (no rows) weigh 0.
 * part_out [n_parts,16,512], part_lse [n_parts,16] -> out [16,512], lse [16].
 */
int oracle_combine(int n_parts, const double* part_out, const double* part_lse, double* out, double* lse) {
  int h, j, s;
  for (h = 0; h < ORACLE_HEADS; ++h) {
    double m = -INFINITY, z = 0.0;
    for (s = 0; s < n_parts; ++s)
      if (part_lse[s * ORACLE_HEADS + h] > m) m = part_lse[s * ORACLE_HEADS + h];
    for (j = 0; j < ORACLE_V_DIM; ++j) out[h * ORACLE_V_DIM + j] = 0.0;
    if (m == -INFINITY) {
      lse[h] = -INFINITY;
      continue;
    }
    for (s = 0; s < n_parts; ++s) z += exp(part_lse[s * ORACLE_HEADS + h] - m);
    for (s = 0; s < n_parts; ++s) {
      double w = exp(part_lse[s * ORACLE_HEADS + h] - m) / z;
      for (j = 0; j < ORACLE_V_DIM; ++j)
        out[h * ORACLE_V_DIM + j] += w * part_out[((size_t)s * ORACLE_HEADS + h) * ORACLE_V_DIM + j];
    }
    lse[h] = m + log(z);
  }
  return 0;
}

/* The direct Q cast of mode 1, element-wise: bf16 bits -> e4m3 codes. */
void oracle_q_to_e4m3(const uint16_t* q, int64_t n, uint8_t* out) {
  int64_t i;
  for (i = 0; i < n; ++i) out[i] = oracle_e4m3_encode(oracle_bf16_decode(q[i]));
}

int oracle_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}
