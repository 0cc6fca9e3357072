/*
 * Paged MLA decode oracle: plain, slow, fp64 CPU implementation.
 *
 * TEST INFRASTRUCTURE ONLY. This file is the correctness oracle for the CUDA
 * path of paged_latent_attention_mla_gb300. It shares no code, header, table or
 * helper with that path. Only tests/, __graft_entry__.smoke() and bench.py's
 * CPU-baseline leg may load it.
 *
 * What it computes (the method, as the kv_balanced_mla kernel page of the vLLM
 * Kimi-K3 MLA docs defines it, BlackwellMultiHeadLatentAttentionForwardFP8):
 *
 *   for every batch row b, query token t < Sq and head h < H:
 *     visible keys j in [lo, hi) of sequence b (see oracle_visible_range),
 *     key j lives at page page_table[b][j / P], slot j % P
 *       (__call__ docstring: c_latent / c_rope are [num_pages, page_size, D],
 *        page_table is [batch, page_count]),
 *     s_j = scale * (q_latent . c_j + q_rope . kpe_j)
 *     O   = sum_j softmax(s)_j * c_j      (V is the latent c itself: the
 *                                          kernel's PV operand is the
 *                                          transposed view of c_latent)
 *     LSE = log(sum_j exp(s_j))           (natural log; empty rows: O = 0,
 *                                          LSE = -inf, write_empty_output)
 *
 * Two routes compute it:
 *   oracle_mla_decode        the definition above, one row at a time
 *                            (oracle_mla_decode_ex: the same with decode
 *                            context parallelism and per-token local bounds);
 *   oracle_mla_decode_split  the pages' split-KV route: get_k_tile_count's
 *                            tile ranges, a normalized partial (O_i, lse_i)
 *                            per split, then reduction_kernel's base-2
 *                            LSE-weighted combine.
 * Their agreement is one of the oracle's invariant pins.
 *
 * Inputs are raw element bits (bf16 or float8 e4m3fn) with per-tensor fp32
 * descales, exactly what the CUDA path receives.  Decoding bits to fp64 is the
 * first step (bf16 is exact in fp64; e4m3 follows the OCP 8-bit floating point
 * definition: 1 sign, 4 exponent bits with bias 7, 3 mantissa bits, subnormals,
 * S.1111.111 is NaN, no infinities).
 *
 * Parity pins (tests/test_oracle_pins.py): brute-force dense attention through
 * a library routine, single-key and equal-score closed forms, split
 * recombination, page permutation, window and causal special cases, and the
 * constant score shift.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORACLE_DC 512 /* latent width d_c: __init__ sets latent_dim = 512 */
#define ORACLE_DR 64  /* rope width d_r: __init__ sets rope_dim = 64      */

enum { ORACLE_BF16 = 0, ORACLE_E4M3 = 1 };

/* bf16 is the top half of an IEEE binary32: widen and convert. */
double oracle_bf16_to_f64(uint16_t bits) {
  uint32_t w = ((uint32_t)bits) << 16;
  float f;
  memcpy(&f, &w, sizeof f);
  return (double)f;
}

/* OCP float8 e4m3 ("fn": finite, one NaN pattern per sign). */
double oracle_e4m3_to_f64(uint8_t bits) {
  int sign = (bits >> 7) & 1;
  int exp = (bits >> 3) & 0xF;
  int man = bits & 0x7;
  double v;
  if (exp == 0xF && man == 0x7) return NAN;
  if (exp == 0)
    v = ldexp((double)man / 8.0, -6); /* subnormal: 0.m * 2^(1-7) */
  else
    v = ldexp(1.0 + (double)man / 8.0, exp - 7);
  return sign ? -v : v;
}

static double load_elem(const void *base, int64_t idx, int dtype) {
  if (dtype == ORACLE_BF16) return oracle_bf16_to_f64(((const uint16_t *)base)[idx]);
  return oracle_e4m3_to_f64(((const uint8_t *)base)[idx]);
}

static int elem_bytes(int dtype) { return dtype == ORACLE_BF16 ? 2 : 1; }

/*
 * Visible key range [lo, hi) of query token t of a request with K cached keys
 * (K counts the Sq new tokens too).
 *   causal: token t sits at position K - Sq + t and sees keys up to it, so
 *           hi = K - (Sq - 1 - t)       (softmax masking: a row's K bound is
 *                                        K - (S_q - 1 - q_tok))
 *   window: lo = max(0, K - Sq - window_left + t)   (__init__ docstring of
 *           window_left); window_left < 0 means full history, lo = 0.
 * Both ends are clamped to [0, K]; an empty range means an empty row.
 */
void oracle_visible_range(int K, int Sq, int t, int causal, int window_left, int *lo, int *hi) {
  int h = causal ? K - (Sq - 1 - t) : K;
  int l = 0;
  if (window_left >= 0) {
    l = K - Sq - window_left + t;
    if (l < 0) l = 0;
  }
  if (h > K) h = K;
  if (h < 0) h = 0;
  if (l > K) l = K;
  if (l > h) l = h;
  *lo = l;
  *hi = h;
}

typedef struct {
  const void *q_latent; /* [B, Sq, H, 512] */
  const void *q_rope;   /* [B, Sq, H, 64]  */
  const void *ckv;      /* [num_pages, P, 512] */
  const void *kpe;      /* [num_pages, P, 64]  */
  int dtype;
  double q_descale, ckv_descale, kpe_descale;
  const int32_t *page_table; /* [B, pt_stride] */
  int pt_stride;
  const int32_t *seq_lens; /* [B] */
  int B, Sq, H, page_size, num_pages;
  double scale;
  int causal, window_left;
  /* Decode context parallelism (kv_balanced_mla kernel page, __init__: cp_world,
   * cp_rank, cp_interleave_size; __call__: causal_seqs).  The sequence's keys are
   * dealt to cp_world ranks in runs of cp_interleave consecutive positions, run k
   * to rank k % cp_world; this rank's cache holds its keys in position order and
   * seq_lens counts them; global_seq_lens holds the whole sequence's length, which
   * the causal and window bounds are taken on.  cp_world <= 1: no context parallelism. */
  int cp_world, cp_rank, cp_interleave;
  const int32_t *global_seq_lens; /* [B], or NULL without context parallelism */
  /* __call__'s local_visible_lens: [B, Sq] exclusive bounds on the local key index,
   * one per query token, replacing the causal bound when given (NULL: not given). */
  const int32_t *local_visible_lens;
} oracle_problem;

/* Address of key j of request b: page_table[b][j / P], slot j % P. */
static int64_t key_row(const oracle_problem *p, int b, int j) {
  int32_t page = p->page_table[(int64_t)b * p->pt_stride + j / p->page_size];
  return (int64_t)page * p->page_size + (j % p->page_size);
}

/* Score s_j = scale * (q_latent . c_j + q_rope . kpe_j) in fp64. */
static double score(const oracle_problem *p, const double *ql, const double *qr, int64_t row) {
  double acc = 0.0;
  for (int d = 0; d < ORACLE_DC; d++)
    acc += ql[d] * (load_elem(p->ckv, row * ORACLE_DC + d, p->dtype) * p->ckv_descale);
  for (int d = 0; d < ORACLE_DR; d++)
    acc += qr[d] * (load_elem(p->kpe, row * ORACLE_DR + d, p->dtype) * p->kpe_descale);
  return p->scale * acc;
}

static void load_query(const oracle_problem *p, int b, int t, int h, double *ql, double *qr) {
  int64_t r = ((int64_t)b * p->Sq + t) * p->H + h;
  for (int d = 0; d < ORACLE_DC; d++) ql[d] = load_elem(p->q_latent, r * ORACLE_DC + d, p->dtype) * p->q_descale;
  for (int d = 0; d < ORACLE_DR; d++) qr[d] = load_elem(p->q_rope, r * ORACLE_DR + d, p->dtype) * p->q_descale;
}

/*
 * Softmax attention of one row over keys [lo, hi): writes O[512] and returns
 * the natural-log LSE.  Plain two-pass definition: max, then exp-sum.
 */
static double attend_range(const oracle_problem *p, int b, const double *ql, const double *qr, int lo, int hi,
                           double *o, double *s_buf) {
  for (int d = 0; d < ORACLE_DC; d++) o[d] = 0.0;
  if (hi <= lo) return -INFINITY;
  double m = -INFINITY;
  for (int j = lo; j < hi; j++) {
    s_buf[j - lo] = score(p, ql, qr, key_row(p, b, j));
    if (s_buf[j - lo] > m) m = s_buf[j - lo];
  }
  double z = 0.0;
  for (int j = lo; j < hi; j++) {
    double w = exp(s_buf[j - lo] - m);
    int64_t row = key_row(p, b, j);
    z += w;
    for (int d = 0; d < ORACLE_DC; d++) o[d] += w * (load_elem(p->ckv, row * ORACLE_DC + d, p->dtype) * p->ckv_descale);
  }
  for (int d = 0; d < ORACLE_DC; d++) o[d] /= z;
  return m + log(z);
}

static int max_len(const oracle_problem *p) {
  int m = 1;
  for (int b = 0; b < p->B; b++)
    if (p->seq_lens[b] > m) m = p->seq_lens[b];
  return m;
}

/*
 * The definition.  rows: optional list of flat row ids r = (b*Sq + t)*H + h
 * (NULL = all B*Sq*H rows, in order).  O is [n_rows, 512], LSE is [n_rows].
 */
int oracle_mla_decode(const void *q_latent, const void *q_rope, const void *ckv, const void *kpe, int dtype,
                      double q_descale, double ckv_descale, double kpe_descale, const int32_t *page_table,
                      int pt_stride, const int32_t *seq_lens, int B, int Sq, int H, int page_size, int num_pages,
                      double scale, int causal, int window_left, const int64_t *rows, int64_t n_rows,
                      int n_threads, double *O, double *LSE) {
  oracle_problem p = {q_latent, q_rope, ckv, kpe, dtype, q_descale, ckv_descale, kpe_descale, page_table,
                      pt_stride, seq_lens, B, Sq, H, page_size, num_pages, scale, causal, window_left,
                      1, 0, 1, NULL, NULL};
  int64_t total = (int64_t)B * Sq * H;
  if (!rows) n_rows = total;
  int kmax = max_len(&p);
#ifdef _OPENMP
  if (n_threads > 0) omp_set_num_threads(n_threads);
#pragma omp parallel
#endif
  {
    double *s_buf = (double *)malloc(sizeof(double) * (size_t)kmax);
    double ql[ORACLE_DC], qr[ORACLE_DR];
#ifdef _OPENMP
#pragma omp for schedule(dynamic, 1)
#endif
    for (int64_t i = 0; i < n_rows; i++) {
      int64_t r = rows ? rows[i] : i;
      int h = (int)(r % H);
      int t = (int)((r / H) % Sq);
      int b = (int)(r / ((int64_t)H * Sq));
      int lo, hi;
      oracle_visible_range(seq_lens[b], Sq, t, causal, window_left, &lo, &hi);
      load_query(&p, b, t, h, ql, qr);
      LSE[i] = attend_range(&p, b, ql, qr, lo, hi, O + i * ORACLE_DC, s_buf);
    }
    free(s_buf);
  }
  return 0;
}

/*
 * Global position of local key l of this rank: the rank owns runs of cp_interleave
 * consecutive positions, one run in every cycle of cp_world runs, so its local run
 * l / I sits in cycle l / I at offset cp_rank * I within the cycle.
 */
static int64_t global_position(const oracle_problem *p, int64_t l) {
  if (p->cp_world <= 1) return l;
  int64_t I = p->cp_interleave, W = p->cp_world;
  return (l / I) * W * I + (int64_t)p->cp_rank * I + l % I;
}

/*
 * Is local key l of request b visible to query token t?  The causal and window
 * bounds are the position rule of oracle_visible_range, taken on the global
 * sequence (its length and the key's global position) under context parallelism;
 * local_visible_lens, when given, replaces the causal bound with l < its entry.
 */
static int key_visible(const oracle_problem *p, int b, int t, int l) {
  if (l < 0 || l >= p->seq_lens[b]) return 0;
  int Kg = p->cp_world > 1 ? p->global_seq_lens[b] : p->seq_lens[b];
  int lo, hi;
  oracle_visible_range(Kg, p->Sq, t, p->causal, p->window_left, &lo, &hi);
  int64_t g = global_position(p, l);
  if (p->window_left >= 0 && g < lo) return 0;
  if (p->local_visible_lens) return l < p->local_visible_lens[(int64_t)b * p->Sq + t];
  if (p->causal) return g < hi;
  return 1;
}

/*
 * Softmax attention of row (b, t) over its visible keys, tested key by key:
 * writes O[512] and returns the natural-log LSE (-inf and O = 0 when none).
 */
static double attend_visible(const oracle_problem *p, int b, int t, const double *ql, const double *qr, double *o,
                             double *s_buf) {
  int K = p->seq_lens[b];
  for (int d = 0; d < ORACLE_DC; d++) o[d] = 0.0;
  double m = -INFINITY;
  int n = 0;
  for (int j = 0; j < K; j++) {
    if (!key_visible(p, b, t, j)) continue;
    s_buf[j] = score(p, ql, qr, key_row(p, b, j));
    if (s_buf[j] > m) m = s_buf[j];
    n++;
  }
  if (n == 0) return -INFINITY;
  double z = 0.0;
  for (int j = 0; j < K; j++) {
    if (!key_visible(p, b, t, j)) continue;
    double w = exp(s_buf[j] - m);
    int64_t row = key_row(p, b, j);
    z += w;
    for (int d = 0; d < ORACLE_DC; d++) o[d] += w * (load_elem(p->ckv, row * ORACLE_DC + d, p->dtype) * p->ckv_descale);
  }
  for (int d = 0; d < ORACLE_DC; d++) o[d] /= z;
  return m + log(z);
}

/*
 * The definition with context parallelism and local bounds: this rank's share
 * of every row (its visible keys only), or the whole row when cp_world <= 1.
 * Arguments as oracle_mla_decode, plus cp_world, cp_rank, cp_interleave,
 * global_seq_lens [B] (may be NULL when cp_world <= 1) and local_visible_lens
 * [B, Sq] (may be NULL).
 */
int oracle_mla_decode_ex(const void *q_latent, const void *q_rope, const void *ckv, const void *kpe, int dtype,
                         double q_descale, double ckv_descale, double kpe_descale, const int32_t *page_table,
                         int pt_stride, const int32_t *seq_lens, int B, int Sq, int H, int page_size, int num_pages,
                         double scale, int causal, int window_left, int cp_world, int cp_rank, int cp_interleave,
                         const int32_t *global_seq_lens, const int32_t *local_visible_lens, int n_threads, double *O,
                         double *LSE) {
  if (cp_world > 1 && (!global_seq_lens || cp_rank < 0 || cp_rank >= cp_world || cp_interleave < 1)) return 1;
  oracle_problem p = {q_latent, q_rope, ckv, kpe, dtype, q_descale, ckv_descale, kpe_descale, page_table,
                      pt_stride, seq_lens, B, Sq, H, page_size, num_pages, scale, causal, window_left,
                      cp_world, cp_rank, cp_interleave, global_seq_lens, local_visible_lens};
  int64_t total = (int64_t)B * Sq * H;
  int kmax = max_len(&p);
#ifdef _OPENMP
  if (n_threads > 0) omp_set_num_threads(n_threads);
#pragma omp parallel
#endif
  {
    double *s_buf = (double *)malloc(sizeof(double) * (size_t)kmax);
    double ql[ORACLE_DC], qr[ORACLE_DR];
#ifdef _OPENMP
#pragma omp for schedule(dynamic, 1)
#endif
    for (int64_t r = 0; r < total; r++) {
      int h = (int)(r % H);
      int t = (int)((r / H) % Sq);
      int b = (int)(r / ((int64_t)H * Sq));
      load_query(&p, b, t, h, ql, qr);
      LSE[r] = attend_visible(&p, b, t, ql, qr, O + r * ORACLE_DC, s_buf);
    }
    free(s_buf);
  }
  return 0;
}

/*
 * Combine pieces of the same rows computed over disjoint key sets (the ranks of
 * context parallelism): O_parts [world, rows, 512] normalized outputs and
 * L_parts [world, rows] natural-log LSEs.  lse = m + ln(sum_r e^(L_r - m)) with m
 * the largest L_r, O = sum_r e^(L_r - lse) O_r; pieces with L_r = -inf add
 * nothing, and rows where every piece is empty get O = 0, lse = -inf.
 */
int oracle_merge(const double *O_parts, const double *L_parts, int world, int64_t rows, double *O, double *L) {
  for (int64_t i = 0; i < rows; i++) {
    double m = -INFINITY;
    for (int r = 0; r < world; r++)
      if (L_parts[(int64_t)r * rows + i] > m) m = L_parts[(int64_t)r * rows + i];
    double *o = O + i * ORACLE_DC;
    for (int d = 0; d < ORACLE_DC; d++) o[d] = 0.0;
    if (m == -INFINITY) {
      L[i] = -INFINITY;
      continue;
    }
    double z = 0.0;
    for (int r = 0; r < world; r++) z += exp(L_parts[(int64_t)r * rows + i] - m);
    double lse = m + log(z);
    for (int r = 0; r < world; r++) {
      double lr = L_parts[(int64_t)r * rows + i];
      if (lr == -INFINITY) continue;
      double w = exp(lr - lse);
      const double *src = O_parts + ((int64_t)r * rows + i) * ORACLE_DC;
      for (int d = 0; d < ORACLE_DC; d++) o[d] += w * src[d];
    }
    L[i] = lse;
  }
  return 0;
}

/*
 * The split-KV route, following the page's planning and reduction steps:
 *
 * get_k_tile_count: with tile_n keys per tile,
 *   k_tile_total = ceil(K / tile_n)
 *   k_tile_lo    = window ? max(0, K - Sq - window_left) / tile_n : 0
 *   per_cta      = ceil((k_tile_total - k_tile_lo) / split_kv)
 *   k_index      = k_tile_lo + split * per_cta
 *   count        = max(0, min(k_tile_total, k_index + per_cta) - k_index)
 * Each split attends to the visible keys inside its tiles and yields a
 * normalized partial O_i with a base-2 log-sum-exp lse_i (O_i = 0 and
 * lse_i = -inf when it saw no visible key, write_empty_output).
 *
 * reduction_kernel: only the first ceil((k_tile_total - k_tile_lo) /
 * max(1, per_cta)) splits are read; lse_max = max_i lse_i (0 when every
 * lse_i is -inf); sum = sum_i 2^(lse_i - lse_max);
 * lse = lse_max + log2(sum) (or -inf when sum == 0);
 * O = sum_i 2^(lse_i - lse) * O_i.  The natural-log LSE is lse * ln 2.
 */
int oracle_mla_decode_split(const void *q_latent, const void *q_rope, const void *ckv, const void *kpe, int dtype,
                            double q_descale, double ckv_descale, double kpe_descale, const int32_t *page_table,
                            int pt_stride, const int32_t *seq_lens, int B, int Sq, int H, int page_size,
                            int num_pages, double scale, int causal, int window_left, int split_kv, int tile_n,
                            int n_threads, double *O, double *LSE) {
  oracle_problem p = {q_latent, q_rope, ckv, kpe, dtype, q_descale, ckv_descale, kpe_descale, page_table,
                      pt_stride, seq_lens, B, Sq, H, page_size, num_pages, scale, causal, window_left,
                      1, 0, 1, NULL, NULL};
  if (split_kv < 1 || tile_n < 1) return 1;
  int64_t total = (int64_t)B * Sq * H;
  int kmax = max_len(&p);
#ifdef _OPENMP
  if (n_threads > 0) omp_set_num_threads(n_threads);
#pragma omp parallel
#endif
  {
    double *s_buf = (double *)malloc(sizeof(double) * (size_t)kmax);
    double *part_o = (double *)malloc(sizeof(double) * (size_t)split_kv * ORACLE_DC);
    double *part_lse2 = (double *)malloc(sizeof(double) * (size_t)split_kv);
    double ql[ORACLE_DC], qr[ORACLE_DR];
#ifdef _OPENMP
#pragma omp for schedule(dynamic, 1)
#endif
    for (int64_t r = 0; r < total; r++) {
      int h = (int)(r % H);
      int t = (int)((r / H) % Sq);
      int b = (int)(r / ((int64_t)H * Sq));
      int K = seq_lens[b];
      int lo, hi;
      oracle_visible_range(K, Sq, t, causal, window_left, &lo, &hi);
      load_query(&p, b, t, h, ql, qr);

      int k_tile_total = (K + tile_n - 1) / tile_n;
      int k_tile_lo = 0;
      if (window_left >= 0) {
        int first = K - Sq - window_left;
        k_tile_lo = (first > 0 ? first : 0) / tile_n;
      }
      int span = k_tile_total - k_tile_lo;
      int per_cta = (span + split_kv - 1) / split_kv;
      for (int s = 0; s < split_kv; s++) {
        int k_index = k_tile_lo + s * per_cta;
        int end = k_index + per_cta < k_tile_total ? k_index + per_cta : k_tile_total;
        int count = end - k_index > 0 ? end - k_index : 0;
        int key_lo = k_index * tile_n, key_hi = (k_index + count) * tile_n;
        if (key_lo < lo) key_lo = lo;
        if (key_hi > hi) key_hi = hi;
        double lse_e = attend_range(&p, b, ql, qr, key_lo, key_hi > key_lo ? key_hi : key_lo,
                                    part_o + (int64_t)s * ORACLE_DC, s_buf);
        part_lse2[s] = lse_e / log(2.0);
      }

      int used = (per_cta > 0) ? (span + per_cta - 1) / per_cta : 0;
      if (used > split_kv) used = split_kv;
      double lse_max = -INFINITY;
      for (int s = 0; s < used; s++)
        if (part_lse2[s] > lse_max) lse_max = part_lse2[s];
      if (lse_max == -INFINITY) lse_max = 0.0;
      double sum = 0.0;
      for (int s = 0; s < used; s++) sum += exp2(part_lse2[s] - lse_max);
      double lse2 = sum != 0.0 ? lse_max + log2(sum) : -INFINITY;
      double *o = O + r * ORACLE_DC;
      for (int d = 0; d < ORACLE_DC; d++) o[d] = 0.0;
      for (int s = 0; s < used; s++) {
        if (part_lse2[s] == -INFINITY) continue; /* an empty partial adds nothing */
        double w = exp2(part_lse2[s] - lse2);
        for (int d = 0; d < ORACLE_DC; d++) o[d] += w * part_o[(int64_t)s * ORACLE_DC + d];
      }
      LSE[r] = lse2 * log(2.0);
    }
    free(s_buf);
    free(part_o);
    free(part_lse2);
  }
  return 0;
}

/*
 * Dense gather through the page table: out[b][j] = (c_j | kpe_j) as raw
 * element bytes, 576 elements per key, for j < seq_lens[b]; key rows
 * j >= seq_lens[b] (up to max_k) are zero bytes.
 */
int oracle_gather(const void *ckv, const void *kpe, int dtype, const int32_t *page_table, int pt_stride,
                  const int32_t *seq_lens, int B, int page_size, int max_k, void *out) {
  int eb = elem_bytes(dtype);
  uint8_t *dst = (uint8_t *)out;
  const uint8_t *c = (const uint8_t *)ckv, *k = (const uint8_t *)kpe;
  int row_bytes = (ORACLE_DC + ORACLE_DR) * eb;
  for (int b = 0; b < B; b++) {
    for (int j = 0; j < max_k; j++) {
      uint8_t *o = dst + ((int64_t)b * max_k + j) * row_bytes;
      if (j >= seq_lens[b]) {
        memset(o, 0, (size_t)row_bytes);
        continue;
      }
      int64_t row = (int64_t)page_table[(int64_t)b * pt_stride + j / page_size] * page_size + j % page_size;
      memcpy(o, c + row * ORACLE_DC * eb, (size_t)ORACLE_DC * eb);
      memcpy(o + ORACLE_DC * eb, k + row * ORACLE_DR * eb, (size_t)ORACLE_DR * eb);
    }
  }
  return 0;
}

/*
 * Visibility bits: bits[b][t][w] has bit i set iff key 32*w + i is in the
 * visible range of query token t of request b.  n_words = ceil(max_k / 32).
 */
int oracle_visibility_bits(const int32_t *seq_lens, int B, int Sq, int causal, int window_left, int max_k,
                           uint32_t *bits) {
  int n_words = (max_k + 31) / 32;
  for (int b = 0; b < B; b++) {
    for (int t = 0; t < Sq; t++) {
      int lo, hi;
      oracle_visible_range(seq_lens[b], Sq, t, causal, window_left, &lo, &hi);
      uint32_t *w = bits + ((int64_t)b * Sq + t) * n_words;
      for (int i = 0; i < n_words; i++) w[i] = 0u;
      for (int j = lo; j < hi && j < max_k; j++) w[j / 32] |= 1u << (j % 32);
    }
  }
  return 0;
}

/*
 * Visibility bits with context parallelism and local bounds: bit i of word w of
 * row (b, t) is set iff local key 32*w + i passes key_visible (the rule of
 * oracle_mla_decode_ex).  Arguments as there; bits [B, Sq, ceil(max_k / 32)].
 */
int oracle_visibility_bits_ex(const int32_t *seq_lens, int B, int Sq, int causal, int window_left, int cp_world,
                              int cp_rank, int cp_interleave, const int32_t *global_seq_lens,
                              const int32_t *local_visible_lens, int max_k, uint32_t *bits) {
  if (cp_world > 1 && (!global_seq_lens || cp_rank < 0 || cp_rank >= cp_world || cp_interleave < 1)) return 1;
  oracle_problem p;
  memset(&p, 0, sizeof p);
  p.seq_lens = seq_lens;
  p.B = B;
  p.Sq = Sq;
  p.causal = causal;
  p.window_left = window_left;
  p.cp_world = cp_world;
  p.cp_rank = cp_rank;
  p.cp_interleave = cp_interleave;
  p.global_seq_lens = global_seq_lens;
  p.local_visible_lens = local_visible_lens;
  int n_words = (max_k + 31) / 32;
  for (int b = 0; b < B; b++)
    for (int t = 0; t < Sq; t++) {
      uint32_t *w = bits + ((int64_t)b * Sq + t) * n_words;
      for (int i = 0; i < n_words; i++) w[i] = 0u;
      for (int j = 0; j < max_k; j++)
        if (key_visible(&p, b, t, j)) w[j / 32] |= 1u << (j % 32);
    }
  return 0;
}

int oracle_max_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}
