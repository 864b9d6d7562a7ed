/*
 * gqa_oracle.c -- plain, slow fp64 CPU oracle for grouped-query attention forward.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check and the
 * benchmark's CPU-baseline leg load this library.  The CUDA library never calls
 * it, and the two share no code, header, table or helper.
 *
 * Sources (page title, section):
 *   [AKL]  "Attention Kernel 계보" (study book V07)
 *            p.2 §1  scaled dot-product attention: S = Q K^T * tau, P = softmax(S), O = P V
 *            p.3 §2  safe softmax in three passes: max, sum of exp(x - max), divide
 *            p.3 §9  LSE = m + log(l) kept per query row
 *            p.4 §2-§8  partial (m_a, l_a, O_a) over a key subset and the merge
 *                    m = max(m_a, m_b), l = a_a l_a + a_b l_b, O = a_a O_a + a_b O_b
 *            p.4 §9  the merge has the identity (-inf, 0)
 *            p.13 §1 causal: key j is visible from query row i iff j <= i
 *            p.15 §2 query head h reads KV head floor(h / (H/g))
 *            p.18 §4 split-K decode: stage-1 partials, stage-2 merge
 *   [TFS]  "TileFoundry showcase: putting it all to work on one decode kernel",
 *            Stage0_Naive: repeat each KV head G times (repeat_interleave on the
 *            head axis), then max-subtracted exp, sum, weighted sum, divide.
 *
 * Precision: every input element is widened exactly to double (bf16 inputs are
 * widened bit-exactly); all arithmetic is fp64 with libm exp/log.  No exp2, no
 * tiling, no online update.  The repeated KV head of a query head is
 * materialised into a private contiguous buffer, one query head at a time, so
 * the memory held is bounded by one head's keys per worker thread.
 *
 * Layouts (row-major, innermost last):
 *   decode : q [B, H_q, d]; k, v [B, S_max, H_kv, d]; seq_lens [B] (int32)
 *            out [B, H_q, d] (double); lse [B, H_q] (double)
 *   prefill: q [B, S, H_q, d]; k, v [B, S, H_kv, d]; rows [n_rows] (int64 query positions)
 *            out [B, n_rows, H_q, d] (double); lse [B, H_q, n_rows] (double)
 *   chunk  : q [B, T_q, H_q, d]; k, v [B, S_max, H_kv, d]; seq_lens [B] or NULL;
 *            rows [n_rows] (chunk row indices); out, lse as for prefill
 *   paged  : q [B, H_q, d]; k_pool, v_pool [P, B_p, H_kv, d]; block_table [B, max_blocks]
 *            (int32); seq_lens [B]; out, lse as for decode
 *   fp8    : q [B, H_q, d] (bf16 bits or double); k8, v8 [B, S_max, H_kv, d] (e4m3 bytes);
 *            k_scale, v_scale [B, S_max] (double); out, lse as for decode
 *
 * Every entry point returns 0 on success and a negative number for invalid
 * arguments (nothing is written then).
 */
#include <math.h>
#include <pthread.h>
#include <stdatomic.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORC_F64 0  /* inputs are double */
#define ORC_BF16 1 /* inputs are bfloat16 bit patterns (uint16) */

/* Exact widening of one input element to double. */
static double widen(const void* base, int64_t idx, int dtype) {
  if (dtype == ORC_F64) return ((const double*)base)[idx];
  uint16_t bits = ((const uint16_t*)base)[idx];
  uint32_t u = (uint32_t)bits << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

/* ---------------------------------------------------------------------------
 * The three-pass safe softmax attention of one query row over n keys
 * ([AKL] p.2 §1 and p.3 §2; LSE from p.3 §9).  kh, vh hold the n visible keys
 * and values of this row's (repeated) KV head, contiguous [n][d].
 * ------------------------------------------------------------------------- */
static void attend_row(const double* qrow, const double* kh, const double* vh, int64_t n, int d,
                       double scale, double* s, double* out, double* lse) {
  /* scores s_j = tau * <q, k_j> */
  for (int64_t j = 0; j < n; ++j) {
    double acc = 0.0;
    for (int t = 0; t < d; ++t) acc += qrow[t] * kh[j * d + t];
    s[j] = scale * acc;
  }
  /* pass 1: m = max_j s_j */
  double m = -INFINITY;
  for (int64_t j = 0; j < n; ++j)
    if (s[j] > m) m = s[j];
  /* pass 2: l = sum_j exp(s_j - m) */
  double l = 0.0;
  for (int64_t j = 0; j < n; ++j) l += exp(s[j] - m);
  /* pass 3: O = sum_j (exp(s_j - m) / l) v_j */
  for (int t = 0; t < d; ++t) out[t] = 0.0;
  for (int64_t j = 0; j < n; ++j) {
    double p = exp(s[j] - m) / l;
    for (int t = 0; t < d; ++t) out[t] += p * vh[j * d + t];
  }
  *lse = m + log(l);
}

/* Copy keys [0, n) of KV head kv of batch b into contiguous [n][d] doubles:
 * the per-query-head slice of the repeated KV cache ([TFS] Stage0_Naive). */
static void repeat_head(const void* src, int dtype, int64_t b, int64_t n, int64_t S_stride,
                        int H_kv, int d, int kv, double* dst) {
  for (int64_t j = 0; j < n; ++j)
    for (int t = 0; t < d; ++t)
      dst[j * d + t] = widen(src, ((b * S_stride + j) * H_kv + kv) * d + t, dtype);
}

/* ------------------------------------------------------------------------- */
/* A minimal thread pool over task indices 0..n_tasks-1.                     */
typedef struct {
  void (*fn)(void* ctx, int64_t task, double* scratch);
  void* ctx;
  int64_t n_tasks;
  size_t scratch_doubles;
  atomic_llong next;
  atomic_int failed;
} pool_t;

static void* pool_worker(void* arg) {
  pool_t* p = (pool_t*)arg;
  double* scratch = (double*)malloc(p->scratch_doubles * sizeof(double) + 64);
  if (!scratch) {
    atomic_store(&p->failed, 1);
    return NULL;
  }
  for (;;) {
    int64_t t = atomic_fetch_add(&p->next, 1);
    if (t >= p->n_tasks) break;
    p->fn(p->ctx, t, scratch);
  }
  free(scratch);
  return NULL;
}

static int run_pool(void (*fn)(void*, int64_t, double*), void* ctx, int64_t n_tasks,
                    size_t scratch_doubles, int nthreads) {
  pool_t p;
  p.fn = fn;
  p.ctx = ctx;
  p.n_tasks = n_tasks;
  p.scratch_doubles = scratch_doubles;
  atomic_init(&p.next, 0);
  atomic_init(&p.failed, 0);
  if (nthreads < 1) nthreads = 1;
  if (nthreads > n_tasks) nthreads = (int)(n_tasks > 0 ? n_tasks : 1);
  pthread_t* th = (pthread_t*)malloc(sizeof(pthread_t) * (size_t)nthreads);
  if (!th) return -100;
  int started = 0;
  for (int i = 0; i < nthreads; ++i) {
    if (pthread_create(&th[i], NULL, pool_worker, &p) != 0) break;
    ++started;
  }
  if (started == 0) pool_worker(&p); /* no threads available: run inline */
  for (int i = 0; i < started; ++i) pthread_join(th[i], NULL);
  free(th);
  return atomic_load(&p.failed) ? -101 : 0;
}

/* ------------------------------------------------------------------------- */
/* Decode (one query row per (b, h)); visible keys are [0, L_b).             */
typedef struct {
  const void *q, *k, *v;
  int dtype;
  const int32_t* seq_lens;
  int B, S_max, H_q, H_kv, d;
  double scale;
  double *out, *lse;
} dec_ctx;

static void dec_task(void* vctx, int64_t task, double* scratch) {
  dec_ctx* c = (dec_ctx*)vctx;
  int64_t b = task / c->H_q;
  int h = (int)(task % c->H_q);
  int G = c->H_q / c->H_kv;
  int kv = h / G; /* [AKL] p.15 §2 */
  int64_t n = c->seq_lens[b];
  int d = c->d;
  double* qrow = scratch;
  double* kh = qrow + d;
  double* vh = kh + (size_t)c->S_max * d;
  double* s = vh + (size_t)c->S_max * d;
  for (int t = 0; t < d; ++t) qrow[t] = widen(c->q, (b * c->H_q + h) * d + t, c->dtype);
  repeat_head(c->k, c->dtype, b, n, c->S_max, c->H_kv, d, kv, kh);
  repeat_head(c->v, c->dtype, b, n, c->S_max, c->H_kv, d, kv, vh);
  attend_row(qrow, kh, vh, n, d, c->scale, s, c->out + (b * c->H_q + h) * d,
             c->lse + b * c->H_q + h);
}

static int check_heads(int B, int S, int H_q, int H_kv, int d) {
  if (B < 1 || S < 1 || H_q < 1 || H_kv < 1 || d < 1) return -1;
  if (H_q % H_kv != 0) return -2;
  return 0;
}

int orc_decode(const void* q, const void* k, const void* v, int dtype, const int32_t* seq_lens,
               int B, int S_max, int H_q, int H_kv, int d, double scale, double* out, double* lse,
               int nthreads) {
  int rc = check_heads(B, S_max, H_q, H_kv, d);
  if (rc) return rc;
  if (dtype != ORC_F64 && dtype != ORC_BF16) return -3;
  for (int b = 0; b < B; ++b)
    if (seq_lens[b] < 1 || seq_lens[b] > S_max) return -4;
  dec_ctx c = {q, k, v, dtype, seq_lens, B, S_max, H_q, H_kv, d, scale, out, lse};
  size_t scratch = (size_t)d + 3 * (size_t)S_max * d + (size_t)S_max;
  return run_pool(dec_task, &c, (int64_t)B * H_q, scratch, nthreads);
}

/* ------------------------------------------------------------------------- */
/* Decode partials: split s covers keys [s*chunk, min((s+1)*chunk, L_b)).     */
/* Per split, by definition ([AKL] p.4 §2, §8; p.18 §4 stage 1):             */
/*   m_s = max s_j,  l_s = sum exp(s_j - m_s),  O_s = sum exp(s_j - m_s) v_j  */
/* An empty split is the merge identity (-inf, 0, 0) ([AKL] p.4 §9).         */
/* Outputs: m, l [B, H_q, n_split]; O [B, H_q, n_split, d].                   */
typedef struct {
  dec_ctx base;
  int n_split, chunk;
  double *m, *l, *O;
} part_ctx;

static void part_task(void* vctx, int64_t task, double* scratch) {
  part_ctx* pc = (part_ctx*)vctx;
  dec_ctx* c = &pc->base;
  int64_t b = task / c->H_q;
  int h = (int)(task % c->H_q);
  int kv = h / (c->H_q / c->H_kv);
  int64_t n = c->seq_lens[b];
  int d = c->d;
  double* qrow = scratch;
  double* kh = qrow + d;
  double* vh = kh + (size_t)c->S_max * d;
  for (int t = 0; t < d; ++t) qrow[t] = widen(c->q, (b * c->H_q + h) * d + t, c->dtype);
  repeat_head(c->k, c->dtype, b, n, c->S_max, c->H_kv, d, kv, kh);
  repeat_head(c->v, c->dtype, b, n, c->S_max, c->H_kv, d, kv, vh);
  for (int sp = 0; sp < pc->n_split; ++sp) {
    int64_t idx = (b * c->H_q + h) * pc->n_split + sp;
    int64_t lo = (int64_t)sp * pc->chunk;
    int64_t hi = lo + pc->chunk;
    if (hi > n) hi = n;
    double* O = pc->O + idx * d;
    for (int t = 0; t < d; ++t) O[t] = 0.0;
    if (lo >= hi) {
      pc->m[idx] = -INFINITY;
      pc->l[idx] = 0.0;
      continue;
    }
    double m = -INFINITY;
    for (int64_t j = lo; j < hi; ++j) {
      double acc = 0.0;
      for (int t = 0; t < d; ++t) acc += qrow[t] * kh[j * d + t];
      double sj = c->scale * acc;
      if (sj > m) m = sj;
    }
    double l = 0.0;
    for (int64_t j = lo; j < hi; ++j) {
      double acc = 0.0;
      for (int t = 0; t < d; ++t) acc += qrow[t] * kh[j * d + t];
      double e = exp(c->scale * acc - m);
      l += e;
      for (int t = 0; t < d; ++t) O[t] += e * vh[j * d + t];
    }
    pc->m[idx] = m;
    pc->l[idx] = l;
  }
}

int orc_decode_partials(const void* q, const void* k, const void* v, int dtype,
                        const int32_t* seq_lens, int B, int S_max, int H_q, int H_kv, int d,
                        double scale, int n_split, int chunk, double* m, double* l, double* O,
                        int nthreads) {
  int rc = check_heads(B, S_max, H_q, H_kv, d);
  if (rc) return rc;
  if (dtype != ORC_F64 && dtype != ORC_BF16) return -3;
  if (n_split < 1 || chunk < 1) return -5;
  for (int b = 0; b < B; ++b)
    if (seq_lens[b] < 1 || seq_lens[b] > S_max) return -4;
  part_ctx pc;
  pc.base = (dec_ctx){q, k, v, dtype, seq_lens, B, S_max, H_q, H_kv, d, scale, NULL, NULL};
  pc.n_split = n_split;
  pc.chunk = chunk;
  pc.m = m;
  pc.l = l;
  pc.O = O;
  size_t scratch = (size_t)d + 2 * (size_t)S_max * d;
  return run_pool(part_task, &pc, (int64_t)B * H_q, scratch, nthreads);
}

/* ------------------------------------------------------------------------- */
/* Merge of split partials ([AKL] p.4 §3, §8; p.18 §4 stage 2), folded left  */
/* to right from the identity (-inf, 0, 0).  A side whose m is -inf has      */
/* l = 0 and O = 0 and gets the factor 0 (the identity of p.4 §9), so that   */
/* (-inf) - (-inf) is never evaluated.  Final O = O / l, LSE = m + ln l.     */
/* Inputs m, l [R, n_split], O [R, n_split, d]; outputs out [R, d], lse [R]. */
int orc_merge_partials(const double* m, const double* l, const double* O, int64_t R, int n_split,
                       int d, double* out, double* lse) {
  if (R < 1 || n_split < 1 || d < 1) return -1;
  double* acc = (double*)malloc(sizeof(double) * (size_t)d);
  if (!acc) return -100;
  for (int64_t r = 0; r < R; ++r) {
    double m_acc = -INFINITY, l_acc = 0.0;
    for (int t = 0; t < d; ++t) acc[t] = 0.0;
    for (int s = 0; s < n_split; ++s) {
      double m_s = m[r * n_split + s], l_s = l[r * n_split + s];
      const double* O_s = O + (r * n_split + s) * d;
      double M = m_acc > m_s ? m_acc : m_s;
      double a_acc = (m_acc == -INFINITY) ? 0.0 : exp(m_acc - M);
      double a_s = (m_s == -INFINITY) ? 0.0 : exp(m_s - M);
      l_acc = a_acc * l_acc + a_s * l_s;
      for (int t = 0; t < d; ++t) acc[t] = a_acc * acc[t] + a_s * O_s[t];
      m_acc = M;
    }
    for (int t = 0; t < d; ++t) out[r * d + t] = acc[t] / l_acc;
    lse[r] = m_acc + log(l_acc);
  }
  free(acc);
  return 0;
}

/* ------------------------------------------------------------------------- */
/* Causal prefill on selected query rows; row i sees keys [0, i]             */
/* ([AKL] p.13 §1, with S_q = S_kv so that query and key positions align).   */
typedef struct {
  const void *q, *k, *v;
  int dtype;
  int B, S, H_q, H_kv, d;
  double scale;
  const int64_t* rows;
  int n_rows;
  int64_t max_row;
  double *out, *lse;
} pre_ctx;

static void pre_task(void* vctx, int64_t task, double* scratch) {
  pre_ctx* c = (pre_ctx*)vctx;
  int64_t b = task / c->H_q;
  int h = (int)(task % c->H_q);
  int kv = h / (c->H_q / c->H_kv);
  int d = c->d;
  int64_t n_all = c->max_row + 1;
  double* qrow = scratch;
  double* kh = qrow + d;
  double* vh = kh + (size_t)n_all * d;
  double* s = vh + (size_t)n_all * d;
  repeat_head(c->k, c->dtype, b, n_all, c->S, c->H_kv, d, kv, kh);
  repeat_head(c->v, c->dtype, b, n_all, c->S, c->H_kv, d, kv, vh);
  for (int r = 0; r < c->n_rows; ++r) {
    int64_t i = c->rows[r];
    for (int t = 0; t < d; ++t)
      qrow[t] = widen(c->q, ((b * c->S + i) * c->H_q + h) * d + t, c->dtype);
    attend_row(qrow, kh, vh, i + 1, d, c->scale, s,
               c->out + ((b * c->n_rows + r) * c->H_q + h) * d,
               c->lse + (b * c->H_q + h) * c->n_rows + r);
  }
}

int orc_prefill_causal_rows(const void* q, const void* k, const void* v, int dtype, int B, int S,
                            int H_q, int H_kv, int d, double scale, const int64_t* rows,
                            int n_rows, double* out, double* lse, int nthreads) {
  int rc = check_heads(B, S, H_q, H_kv, d);
  if (rc) return rc;
  if (dtype != ORC_F64 && dtype != ORC_BF16) return -3;
  if (n_rows < 1) return -5;
  int64_t max_row = 0;
  for (int r = 0; r < n_rows; ++r) {
    if (rows[r] < 0 || rows[r] >= S) return -4;
    if (rows[r] > max_row) max_row = rows[r];
  }
  pre_ctx c = {q, k, v, dtype, B, S, H_q, H_kv, d, scale, rows, n_rows, max_row, out, lse};
  size_t scratch = (size_t)d + 3 * (size_t)(max_row + 1) * d;
  return run_pool(pre_task, &c, (int64_t)B * H_q, scratch, nthreads);
}

/* ------------------------------------------------------------------------- */
/* Chunked prefill with an optional sliding window.                          */
/* A chunk of T_q query tokens is the last T_q tokens of sequence b, whose    */
/* length (cache included) is L_b = seq_lens[b] (L_b = S_max when seq_lens is */
/* NULL): chunk row i sits at absolute position a = L_b - T_q + i and sees    */
/* keys j with a - W <= j <= a, W = window (no lower bound when window < 0).  */
/* Sources: ADR-0060 §0.5.3 (q_block_meta {q_start, T_q}) and §5.4 (query     */
/* block vs key tile causality); "Attention Kernel 계보" p.13 §1 (causal) and */
/* §7 (sliding window i - W <= j <= i).                                      */
typedef struct {
  const void *q, *k, *v;
  int dtype;
  const int32_t* seq_lens;
  int B, T_q, S_max, H_q, H_kv, d, window;
  double scale;
  const int64_t* rows;
  int n_rows;
  double *out, *lse;
} chunk_ctx;

static void chunk_task(void* vctx, int64_t task, double* scratch) {
  chunk_ctx* c = (chunk_ctx*)vctx;
  int64_t b = task / c->H_q;
  int h = (int)(task % c->H_q);
  int kv = h / (c->H_q / c->H_kv);
  int d = c->d;
  int64_t L = c->seq_lens ? c->seq_lens[b] : c->S_max;
  int64_t q0 = L - c->T_q; /* absolute position of chunk row 0 */
  double* qrow = scratch;
  double* kh = qrow + d;
  double* vh = kh + (size_t)c->S_max * d;
  double* s = vh + (size_t)c->S_max * d;
  repeat_head(c->k, c->dtype, b, L, c->S_max, c->H_kv, d, kv, kh);
  repeat_head(c->v, c->dtype, b, L, c->S_max, c->H_kv, d, kv, vh);
  for (int r = 0; r < c->n_rows; ++r) {
    int64_t i = c->rows[r];
    int64_t a = q0 + i;
    int64_t lo = (c->window >= 0 && a - c->window > 0) ? a - c->window : 0;
    for (int t = 0; t < d; ++t)
      qrow[t] = widen(c->q, ((b * c->T_q + i) * c->H_q + h) * d + t, c->dtype);
    attend_row(qrow, kh + lo * d, vh + lo * d, a - lo + 1, d, c->scale, s,
               c->out + ((b * c->n_rows + r) * c->H_q + h) * d,
               c->lse + (b * c->H_q + h) * c->n_rows + r);
  }
}

int orc_prefill_chunk_rows(const void* q, const void* k, const void* v, int dtype,
                           const int32_t* seq_lens, int B, int T_q, int S_max, int H_q, int H_kv,
                           int d, double scale, int window, const int64_t* rows, int n_rows,
                           double* out, double* lse, int nthreads) {
  int rc = check_heads(B, S_max, H_q, H_kv, d);
  if (rc) return rc;
  if (dtype != ORC_F64 && dtype != ORC_BF16) return -3;
  if (T_q < 1 || T_q > S_max || n_rows < 1) return -5;
  for (int b = 0; seq_lens && b < B; ++b)
    if (seq_lens[b] < T_q || seq_lens[b] > S_max) return -4;
  for (int r = 0; r < n_rows; ++r)
    if (rows[r] < 0 || rows[r] >= T_q) return -4;
  chunk_ctx c = {q, k, v, dtype, seq_lens, B, T_q, S_max, H_q, H_kv, d, window, scale,
                 rows, n_rows, out, lse};
  size_t scratch = (size_t)d + 3 * (size_t)S_max * d;
  return run_pool(chunk_task, &c, (int64_t)B * H_q, scratch, nthreads);
}

/* ------------------------------------------------------------------------- */
/* Paged decode ("Attention Kernel 계보", p.17 §2-§4, p.18 §1-§5): the keys   */
/* of sequence b live in fixed pages of B_p tokens; logical token t sits in   */
/* page block_table[b][t / B_p] at offset t % B_p.  The oracle gathers the    */
/* sequence's keys and values through the table into a contiguous repeated   */
/* head, then runs the same three-pass softmax as orc_decode.                 */
typedef struct {
  const void *q, *kp, *vp;
  int dtype;
  const int32_t *table, *seq_lens;
  int B, P, B_p, max_blocks, H_q, H_kv, d;
  double scale;
  double *out, *lse;
} paged_ctx;

static void paged_gather(const void* pool, int dtype, const int32_t* row_table, int64_t n,
                         int B_p, int H_kv, int d, int kv, double* dst) {
  for (int64_t t = 0; t < n; ++t) {
    int64_t page = row_table[t / B_p];
    int64_t off = t % B_p;
    for (int x = 0; x < d; ++x)
      dst[t * d + x] = widen(pool, ((page * B_p + off) * H_kv + kv) * d + x, dtype);
  }
}

static void paged_task(void* vctx, int64_t task, double* scratch) {
  paged_ctx* c = (paged_ctx*)vctx;
  int64_t b = task / c->H_q;
  int h = (int)(task % c->H_q);
  int kv = h / (c->H_q / c->H_kv);
  int d = c->d;
  int64_t n = c->seq_lens[b];
  int64_t cap = (int64_t)c->max_blocks * c->B_p;
  double* qrow = scratch;
  double* kh = qrow + d;
  double* vh = kh + (size_t)cap * d;
  double* s = vh + (size_t)cap * d;
  const int32_t* row_table = c->table + b * c->max_blocks;
  for (int x = 0; x < d; ++x) qrow[x] = widen(c->q, (b * c->H_q + h) * d + x, c->dtype);
  paged_gather(c->kp, c->dtype, row_table, n, c->B_p, c->H_kv, d, kv, kh);
  paged_gather(c->vp, c->dtype, row_table, n, c->B_p, c->H_kv, d, kv, vh);
  attend_row(qrow, kh, vh, n, d, c->scale, s, c->out + (b * c->H_q + h) * d,
             c->lse + b * c->H_q + h);
}

int orc_decode_paged(const void* q, const void* k_pool, const void* v_pool, int dtype,
                     const int32_t* block_table, int max_blocks, const int32_t* seq_lens, int B,
                     int P, int B_p, int H_q, int H_kv, int d, double scale, double* out,
                     double* lse, int nthreads) {
  int rc = check_heads(B, B_p, H_q, H_kv, d);
  if (rc) return rc;
  if (dtype != ORC_F64 && dtype != ORC_BF16) return -3;
  if (P < 1 || max_blocks < 1) return -5;
  for (int b = 0; b < B; ++b) {
    if (seq_lens[b] < 1 || seq_lens[b] > (int64_t)max_blocks * B_p) return -4;
    for (int j = 0; j < (seq_lens[b] + B_p - 1) / B_p; ++j) {
      int32_t page = block_table[(int64_t)b * max_blocks + j];
      if (page < 0 || page >= P) return -6;
    }
  }
  paged_ctx c = {q, k_pool, v_pool, dtype, block_table, seq_lens, B, P, B_p, max_blocks, H_q,
                 H_kv, d, scale, out, lse};
  size_t cap = (size_t)max_blocks * B_p;
  size_t scratch = (size_t)d + 3 * cap * d;
  return run_pool(paged_task, &c, (int64_t)B * H_q, scratch, nthreads);
}

/* ------------------------------------------------------------------------- */
/* FP8 KV cache ("Attention Kernel 계보", p.17 §7): keys and values stored as */
/* 8-bit floats with one scale per token; the value a kernel must use is      */
/* e4m3(byte) * scale.  E4M3 (the "fn" variant): 1 sign, 4 exponent bits with  */
/* bias 7, 3 mantissa bits; exponent 0 is subnormal (m/8 * 2^-6); the pattern  */
/* S.1111.111 is NaN; there is no infinity.                                    */
double orc_e4m3_to_double(uint8_t x) {
  int sign = x >> 7, e = (x >> 3) & 15, m = x & 7;
  double v;
  if (e == 15 && m == 7) return NAN;
  if (e == 0)
    v = ldexp((double)m / 8.0, -6);
  else
    v = ldexp(1.0 + (double)m / 8.0, e - 7);
  return sign ? -v : v;
}

typedef struct {
  const void* q;
  int qdtype;
  const uint8_t *k8, *v8;
  const double *ks, *vs;
  const int32_t* seq_lens;
  int B, S_max, H_q, H_kv, d;
  double scale;
  double *out, *lse;
} fp8_ctx;

static void fp8_task(void* vctx, int64_t task, double* scratch) {
  fp8_ctx* c = (fp8_ctx*)vctx;
  int64_t b = task / c->H_q;
  int h = (int)(task % c->H_q);
  int kv = h / (c->H_q / c->H_kv);
  int d = c->d;
  int64_t n = c->seq_lens[b];
  double* qrow = scratch;
  double* kh = qrow + d;
  double* vh = kh + (size_t)c->S_max * d;
  double* s = vh + (size_t)c->S_max * d;
  for (int t = 0; t < d; ++t) qrow[t] = widen(c->q, (b * c->H_q + h) * d + t, c->qdtype);
  for (int64_t j = 0; j < n; ++j) {
    double ksj = c->ks[b * c->S_max + j], vsj = c->vs[b * c->S_max + j];
    for (int t = 0; t < d; ++t) {
      int64_t idx = ((b * c->S_max + j) * c->H_kv + kv) * d + t;
      kh[j * d + t] = orc_e4m3_to_double(c->k8[idx]) * ksj;
      vh[j * d + t] = orc_e4m3_to_double(c->v8[idx]) * vsj;
    }
  }
  attend_row(qrow, kh, vh, n, d, c->scale, s, c->out + (b * c->H_q + h) * d,
             c->lse + b * c->H_q + h);
}

int orc_decode_fp8(const void* q, int qdtype, const uint8_t* k8, const uint8_t* v8,
                   const double* k_scale, const double* v_scale, const int32_t* seq_lens, int B,
                   int S_max, int H_q, int H_kv, int d, double scale, double* out, double* lse,
                   int nthreads) {
  int rc = check_heads(B, S_max, H_q, H_kv, d);
  if (rc) return rc;
  if (qdtype != ORC_F64 && qdtype != ORC_BF16) return -3;
  for (int b = 0; b < B; ++b)
    if (seq_lens[b] < 1 || seq_lens[b] > S_max) return -4;
  fp8_ctx c = {q, qdtype, k8, v8, k_scale, v_scale, seq_lens, B, S_max, H_q, H_kv, d, scale,
               out, lse};
  size_t scratch = (size_t)d + 3 * (size_t)S_max * d;
  return run_pool(fp8_task, &c, (int64_t)B * H_q, scratch, nthreads);
}
