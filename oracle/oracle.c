/*
 * oracle.c -- plain fp64 CPU reference for paged-KV split-KV decode attention.
 *
 * TEST INFRASTRUCTURE. Only the tests, the package's smoke check and the
 * benchmark's CPU-baseline leg load this file's library. The product path
 * (the CUDA library) shares no code, header or table with it, and neither
 * side includes or links the other.
 *
 * What it computes. One new query token per request is scored against the
 * request's paged KV cache, one score per key for each query head of a KV
 * group (TensorFold pull 1932, "What this changes": the planned decode walk's
 * Q.K gives one score per key for each query head of a KV group), and the
 * softmax-weighted sum of the value rows is returned with the log-sum-exp of
 * the scaled scores. Written out for request b and query head h:
 *
 *     g     = heads / kv_heads,      kv = h / g           (consecutive groups)
 *     row_t = (page_table[b][t / ps] * kv_heads + kv) * ps + t % ps
 *     s_t   = scale * sum_d q[b,h,d] * K[row_t, d]        t = 0 .. L_b - 1
 *     M     = max_t s_t,   Z = sum_t exp(s_t - M)
 *     out   = sum_t exp(s_t - M) * V[row_t, 0:Dv] / Z,    lse = M + ln Z
 *
 * An empty request (L_b = 0) gives out = 0 and lse = -inf. Everything is
 * double precision; bf16 and fp16 inputs convert to double exactly.
 *
 * Several query tokens per request (q_len >= 1: draft tokens checked in one
 * step; the TensorFold pull 1932 page serves its model with multi-token-
 * prediction drafts, Receipt, and asks that drafted output equal undrafted
 * output, Checklist). The request's last q_len tokens are its
 * queries, already in the cache: query token j (0-based) sits at position
 * L_b - q_len + j and attends to the keys at or before its own position,
 * t = 0 .. L_b - q_len + j. q is [B, q_len, Hq, D] and out / lse follow the
 * same (request, token, head) order; "virtual head" v = j * Hq + h indexes
 * the (token, head) pairs of one request. q_len = 1 is the plain decode.
 *
 * The split partial and the merge follow the aiter pull 4758 page
 * ("[Gluon][MLA] Deeper async-copy pipeline in the bh16 stage-1 decode
 * loop"), Motivation and Technical Details 3: each split of a request's
 * tokens yields a normalised partial output with its log-sum-exp, and the
 * merge re-derives the scalar statistics (the largest partial lse and the
 * weights' sum) and combines the partials with those weights.
 *
 * The `mutation` field plants one known mistake on request, so that the
 * test suite can show that each of its pins catches something (the
 * TensorFold page's "Tests run": the check must fail when a fold runs in
 * the wrong order or a block is skipped). 0 means faithful.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORC_BF16 0
#define ORC_FP16 1

/* Mistakes the test-of-tests can plant (mutation field). */
#define MUT_NONE 0
#define MUT_NO_SCALE 1        /* scores not multiplied by scale            */
#define MUT_HEAD_MAP_MOD 2    /* kv = h % kv_heads instead of h / g        */
#define MUT_SLOT_OFF_BY_ONE 3 /* slot = (t + 1) % ps                        */
#define MUT_LSE_LOG2 4        /* lse in base 2                              */
#define MUT_V_FROM_K 5        /* value rows read from the key pool          */
#define MUT_NO_MAX_SHIFT 6    /* exp(s_t) without subtracting the maximum   */
#define MUT_DIVIDE_BY_L 7     /* normalise by L instead of Z                */
#define MUT_PAGES_REVERSED 8  /* page_table walked from the far end         */
#define MUT_MERGE_NO_NORM 9   /* merge divides by the split count           */
#define MUT_DROP_LAST_KEY 10  /* the last token of a request is skipped      */
#define MUT_NO_CAUSAL 11      /* every query token sees all L_b keys         */

typedef struct {
  int32_t batch;
  int32_t heads;       /* query heads per request                        */
  int32_t kv_heads;    /* KV heads; heads % kv_heads == 0                 */
  int32_t head_dim;    /* D: length of q and of the K part of a row       */
  int32_t head_dim_v;  /* Dv: length of the V part of a row                */
  int32_t page_size;   /* ps: tokens per page                             */
  int32_t dtype;       /* ORC_BF16 or ORC_FP16 for q, K and V             */
  int32_t mutation;    /* MUT_* (0 = faithful)                            */
  int64_t max_pages;   /* row stride of page_table, in entries            */
  int64_t k_row_pitch; /* elements between consecutive K rows             */
  int64_t v_row_pitch; /* elements between consecutive V rows             */
  double scale;        /* multiplies q.k                                   */
  int32_t q_len;       /* query tokens per request; 0 counts as 1          */
} orc_problem;

static int q_len_of(const orc_problem *P) { return P->q_len > 0 ? P->q_len : 1; }

/* bf16 is the top half of an IEEE binary32: widen and reinterpret. */
static double bf16_to_double(uint16_t bits) {
  uint32_t u = (uint32_t)bits << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

/* IEEE binary16: 1 sign, 5 exponent (bias 15), 10 fraction bits. */
static double fp16_to_double(uint16_t bits) {
  int sign = bits >> 15;
  int expo = (bits >> 10) & 0x1f;
  int frac = bits & 0x3ff;
  double v;
  if (expo == 0)
    v = ldexp((double)frac, -24); /* zero or subnormal: frac * 2^-24 */
  else if (expo == 31)
    v = frac ? NAN : INFINITY;
  else
    v = ldexp((double)(frac | 0x400), expo - 25); /* 1.frac * 2^(e-15) */
  return sign ? -v : v;
}

static double elem(const uint16_t *p, int dtype) {
  return dtype == ORC_FP16 ? fp16_to_double(*p) : bf16_to_double(*p);
}

/* Exact widening of n stored elements; exported so the tests can check the
 * decoders against independent library conversions. */
void orc_to_double(const uint16_t *src, int64_t n, int32_t dtype, double *dst) {
  for (int64_t i = 0; i < n; ++i) dst[i] = elem(src + i, dtype);
}

/* Pool row holding logical token t of request b for KV head kv. */
static int64_t kv_row(const orc_problem *P, const int32_t *page_table,
                      const int32_t *seq_lens, int b, int64_t t, int kv) {
  int ps = P->page_size;
  int64_t page_idx = t / ps;
  int64_t slot = t % ps;
  if (P->mutation == MUT_SLOT_OFF_BY_ONE) slot = (t + 1) % ps;
  if (P->mutation == MUT_PAGES_REVERSED) {
    int64_t npages = ((int64_t)seq_lens[b] + ps - 1) / ps;
    page_idx = npages - 1 - page_idx;
  }
  int64_t page = page_table[(int64_t)b * P->max_pages + page_idx];
  return (page * P->kv_heads + kv) * ps + slot;
}

static int kv_head_of(const orc_problem *P, int h) {
  int g = P->heads / P->kv_heads;
  if (P->mutation == MUT_HEAD_MAP_MOD) return h % P->kv_heads;
  return h / g;
}

/* Scaled scores s_t for t in [t0, t1) of (b, v) into s[0 .. t1-t0), where
 * v = j * heads + h is query token j's head h. */
static void scores(const orc_problem *P, const uint16_t *q, const uint16_t *k,
                   const int32_t *page_table, const int32_t *seq_lens, int b,
                   int v, int64_t t0, int64_t t1, double *s) {
  int D = P->head_dim;
  int kv = kv_head_of(P, v % P->heads);
  const uint16_t *qrow = q + ((int64_t)b * q_len_of(P) * P->heads + v) * D;
  double scale = P->mutation == MUT_NO_SCALE ? 1.0 : P->scale;
  for (int64_t t = t0; t < t1; ++t) {
    const uint16_t *krow =
        k + kv_row(P, page_table, seq_lens, b, t, kv) * P->k_row_pitch;
    double dot = 0.0;
    for (int d = 0; d < D; ++d)
      dot += elem(qrow + d, P->dtype) * elem(krow + d, P->dtype);
    s[t - t0] = scale * dot;
  }
}

/* Softmax-weighted V over the tokens of [t0, t1) that (b, vh) may see:
 * out[0:Dv] and lse. vh = j * heads + h; query token j sees the tokens
 * t <= L_b - q_len + j. An empty range gives out = 0, lse = -inf. Returns 0,
 * or -1 on OOM. */
static int attend_range(const orc_problem *P, const uint16_t *q,
                        const uint16_t *k, const uint16_t *v,
                        const int32_t *page_table, const int32_t *seq_lens,
                        int b, int vh, int64_t t0, int64_t t1, double *out,
                        double *lse) {
  int Dv = P->head_dim_v;
  for (int d = 0; d < Dv; ++d) out[d] = 0.0;
  int64_t visible = (int64_t)seq_lens[b] - q_len_of(P) + vh / P->heads + 1;
  if (P->mutation == MUT_NO_CAUSAL) visible = seq_lens[b];
  if (t1 > visible) t1 = visible;
  if (P->mutation == MUT_DROP_LAST_KEY && t1 == seq_lens[b] && t1 > t0) --t1;
  int64_t n = t1 - t0;
  if (n <= 0) {
    *lse = -INFINITY;
    return 0;
  }
  double *s = (double *)malloc((size_t)n * sizeof(double));
  if (!s) return -1;
  scores(P, q, k, page_table, seq_lens, b, vh, t0, t1, s);

  double m = -INFINITY;
  for (int64_t i = 0; i < n; ++i)
    if (s[i] > m) m = s[i];
  if (P->mutation == MUT_NO_MAX_SHIFT) m = 0.0;

  const uint16_t *vpool = P->mutation == MUT_V_FROM_K ? k : v;
  int64_t vpitch = P->mutation == MUT_V_FROM_K ? P->k_row_pitch : P->v_row_pitch;
  int kv = kv_head_of(P, vh % P->heads);
  double z = 0.0;
  for (int64_t i = 0; i < n; ++i) {
    double w = exp(s[i] - m);
    z += w;
    const uint16_t *vrow =
        vpool + kv_row(P, page_table, seq_lens, b, t0 + i, kv) * vpitch;
    for (int d = 0; d < Dv; ++d) out[d] += w * elem(vrow + d, P->dtype);
  }
  double denom = P->mutation == MUT_DIVIDE_BY_L ? (double)n : z;
  for (int d = 0; d < Dv; ++d) out[d] /= denom;
  *lse = P->mutation == MUT_LSE_LOG2 ? (m + log(z)) / log(2.0) : m + log(z);
  free(s);
  return 0;
}

static int check_problem(const orc_problem *P) {
  if (P->batch < 0 || P->heads <= 0 || P->kv_heads <= 0 || P->head_dim <= 0 ||
      P->head_dim_v <= 0 || P->page_size <= 0)
    return -2;
  if (P->heads % P->kv_heads) return -2;
  if (P->dtype != ORC_BF16 && P->dtype != ORC_FP16) return -2;
  if (P->q_len < 0) return -2;
  return 0;
}

/* Full decode for every (b, v): out [B, q_len * Hq, Dv] (= [B, q_len, Hq,
 * Dv]), lse [B, q_len * Hq]. */
int orc_decode(const orc_problem *P, const uint16_t *q, const uint16_t *k,
               const uint16_t *v, const int32_t *page_table,
               const int32_t *seq_lens, double *out, double *lse) {
  int rc = check_problem(P);
  if (rc) return rc;
  int VH = q_len_of(P) * P->heads;
  for (int b = 0; b < P->batch; ++b)
    for (int h = 0; h < VH; ++h) {
      int64_t i = (int64_t)b * VH + h;
      rc = attend_range(P, q, k, v, page_table, seq_lens, b, h, 0, seq_lens[b],
                        out + i * P->head_dim_v, lse + i);
      if (rc) return rc;
    }
  return 0;
}

/* Decode for a list of (b, v) pairs: pairs[2i] = b, pairs[2i+1] = v (query
 * token v / Hq, head v % Hq); results go to out[i * Dv ...] and lse[i]. */
int orc_decode_pairs(const orc_problem *P, const uint16_t *q, const uint16_t *k,
                     const uint16_t *v, const int32_t *page_table,
                     const int32_t *seq_lens, const int32_t *pairs,
                     int64_t npairs, double *out, double *lse) {
  int rc = check_problem(P);
  if (rc) return rc;
  for (int64_t i = 0; i < npairs; ++i) {
    int b = pairs[2 * i], h = pairs[2 * i + 1];
    rc = attend_range(P, q, k, v, page_table, seq_lens, b, h, 0, seq_lens[b],
                      out + i * P->head_dim_v, lse + i);
    if (rc) return rc;
  }
  return 0;
}

/* One split's normalised partial over tokens [t0, t1) of (b, v). */
int orc_partial(const orc_problem *P, const uint16_t *q, const uint16_t *k,
                const uint16_t *v, const int32_t *page_table,
                const int32_t *seq_lens, int32_t b, int32_t h, int64_t t0,
                int64_t t1, double *o, double *lse) {
  int rc = check_problem(P);
  if (rc) return rc;
  return attend_range(P, q, k, v, page_table, seq_lens, b, h, t0, t1, o, lse);
}

/* Merge of nsplits normalised partials o_parts [nsplits, dv] with their
 * log-sum-exps: M = max lse_s, w_s = exp(lse_s - M),
 * out = sum_s w_s o_s / sum_s w_s, lse = M + ln sum_s w_s. Splits whose
 * lse is -inf carry no weight; all of them -inf gives out = 0, lse = -inf. */
int orc_merge(int32_t nsplits, int32_t dv, const double *o_parts,
              const double *lse_parts, int32_t mutation, double *out,
              double *lse) {
  double m = -INFINITY;
  for (int s = 0; s < nsplits; ++s)
    if (lse_parts[s] > m) m = lse_parts[s];
  for (int d = 0; d < dv; ++d) out[d] = 0.0;
  if (m == -INFINITY) {
    *lse = -INFINITY;
    return 0;
  }
  double wsum = 0.0;
  for (int s = 0; s < nsplits; ++s) {
    double w = exp(lse_parts[s] - m);
    wsum += w;
    for (int d = 0; d < dv; ++d) out[d] += w * o_parts[(int64_t)s * dv + d];
  }
  double denom = mutation == MUT_MERGE_NO_NORM ? (double)nsplits : wsum;
  for (int d = 0; d < dv; ++d) out[d] /= denom;
  *lse = m + log(wsum);
  return 0;
}

/* The same decode spread over threads by (b, h) pair, for timing the oracle
 * on all host cores. Each pair is computed exactly as in orc_decode. */
typedef struct {
  const orc_problem *P;
  const uint16_t *q, *k, *v;
  const int32_t *page_table, *seq_lens;
  double *out, *lse;
  int64_t first, last; /* pair range [first, last) in (b, v) order */
  int rc;
} orc_job;

static void *orc_worker(void *arg) {
  orc_job *J = (orc_job *)arg;
  const orc_problem *P = J->P;
  J->rc = 0;
  int VH = q_len_of(P) * P->heads;
  for (int64_t i = J->first; i < J->last && !J->rc; ++i) {
    int b = (int)(i / VH), h = (int)(i % VH);
    J->rc = attend_range(P, J->q, J->k, J->v, J->page_table, J->seq_lens, b, h,
                         0, J->seq_lens[b], J->out + i * P->head_dim_v,
                         J->lse + i);
  }
  return NULL;
}

int orc_decode_threads(const orc_problem *P, const uint16_t *q,
                       const uint16_t *k, const uint16_t *v,
                       const int32_t *page_table, const int32_t *seq_lens,
                       int32_t nthreads, double *out, double *lse) {
  int rc = check_problem(P);
  if (rc) return rc;
  int64_t npairs = (int64_t)P->batch * q_len_of(P) * P->heads;
  if (nthreads < 1) nthreads = 1;
  if (nthreads > npairs) nthreads = (int32_t)(npairs > 0 ? npairs : 1);
  orc_job *jobs = (orc_job *)calloc((size_t)nthreads, sizeof(orc_job));
  pthread_t *tid = (pthread_t *)calloc((size_t)nthreads, sizeof(pthread_t));
  if (!jobs || !tid) {
    free(jobs);
    free(tid);
    return -1;
  }
  for (int i = 0; i < nthreads; ++i) {
    orc_job *J = &jobs[i];
    J->P = P; J->q = q; J->k = k; J->v = v;
    J->page_table = page_table; J->seq_lens = seq_lens;
    J->out = out; J->lse = lse;
    J->first = npairs * i / nthreads;
    J->last = npairs * (i + 1) / nthreads;
  }
  int started = 0;
  for (; started < nthreads; ++started)
    if (pthread_create(&tid[started], NULL, orc_worker, &jobs[started])) break;
  if (started < nthreads) /* run what could not be started on this thread */
    for (int i = started; i < nthreads; ++i) orc_worker(&jobs[i]);
  for (int i = 0; i < started; ++i) pthread_join(tid[i], NULL);
  for (int i = 0; i < nthreads; ++i)
    if (jobs[i].rc) rc = jobs[i].rc;
  free(jobs);
  free(tid);
  return rc;
}
