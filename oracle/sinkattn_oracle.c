/*
 * Float64 CPU oracle for grouped-query attention with learned sinks.
 *
 * TEST INFRASTRUCTURE. This file is the slow, obviously correct statement of
 * what the sink-attention library computes. Only the test suite, the smoke
 * check and the benchmark's CPU-baseline leg load it. The library's product
 * path never calls, links or includes it, and it shares no code, header or
 * constant with the CUDA sources.
 *
 * What it computes. Page "GPT-OSS on day 0", section "Attention: GQA with
 * Attention Sinks": every attention head owns one trained sink parameter that
 * takes part in the softmax. Section "Kernels for GPT-OSS / Sink Attention":
 * the sink is one extra logit placed before the softmax next to the scaled
 * Q.K products; it has no value row, so it enlarges the denominator only.
 * Written out for one query row i of head h of sequence b:
 *
 *   g   = h / (Hq / Hkv)                      (grouped-query head sharing)
 *   p   = (Lk - Lq) + i                       (query position, bottom-right)
 *   J   = { j in [0, Lk) : (!causal || j <= p) && (W == 0 || j > p - W) }
 *   s_j = scale * sum_d q[i,h,d] * k[j,g,d]   (exact products of bf16 inputs)
 *   z   = max(sink_h, max_{j in J} s_j)
 *   den = exp(sink_h - z) + sum_{j in J} exp(s_j - z)
 *   out = sum_{j in J} exp(s_j - z) * v[j,g,:] / den
 *   lse = z + ln(den)                         (natural log, sink included)
 *
 * With no sink vector the sink term is absent (sink = -inf): an empty J then
 * gives out = 0 and lse = -inf. With a sink and an empty J, out = 0 and
 * lse = sink_h.
 *
 * The same section notes that when attention is split into blocks along the
 * KV sequence, the sink must be counted in one block only. The "partial" entry
 * below computes one such block: the softmax restricted to keys in
 * [kv_begin, kv_end) of J, with or without the sink, normalised within the
 * block, together with the block's log-sum-exp. The "merge" entry combines
 * such blocks by their log-sum-exp weights.
 *
 * Everything is computed in double precision from the exact values of the
 * bf16 inputs; exp and log come from the C library. Work items are spread
 * over POSIX threads; each item is computed independently, in the order the
 * definition above states.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* bf16 is the top half of an IEEE binary32; the conversion is exact. */
static double bf16_to_double(uint16_t bits) {
  uint32_t u = ((uint32_t)bits) << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

/* Where the K and V rows of one sequence live. Two layouts:
 *   contiguous: k[total_k, Hkv, D], sequence b occupies rows
 *               [cu_k[b], cu_k[b+1]);
 *   paged:      k[num_pages, Hkv, page_size, D], key j of sequence b lives in
 *               page block_table[b * max_pages + j / page_size] at slot
 *               j % page_size. */
typedef struct {
  const uint16_t *k, *v;
  const int32_t *cu_k;        /* contiguous layout, or NULL */
  const int32_t *block_table; /* paged layout, or NULL */
  const int32_t *seqlens_k;   /* paged layout: [batch] */
  int max_pages, page_size;
  int hkv, d;
} kv_source;

static int kv_len(const kv_source *s, int b) {
  if (s->cu_k) return s->cu_k[b + 1] - s->cu_k[b];
  return s->seqlens_k[b];
}

static size_t kv_row(const kv_source *s, int b, int j, int g) {
  if (s->cu_k) return ((size_t)(s->cu_k[b] + j) * s->hkv + g) * s->d;
  int page = s->block_table[(size_t)b * s->max_pages + j / s->page_size];
  return (((size_t)page * s->hkv + g) * s->page_size + j % s->page_size) * s->d;
}

typedef struct {
  const uint16_t *q;
  const int32_t *cu_q;
  kv_source kv;
  int batch, hq, d;
  const float *sinks; /* NULL: no sink */
  int use_sink;       /* 0: leave the sink out even if sinks != NULL */
  int causal, window;
  double scale;
  const int32_t *kv_begin, *kv_end; /* NULL, or per-sequence key range */
  /* rows to compute: (b, h, i) triples */
  const int32_t *rows;
  long nrows;
  double *out; /* [nrows, d] */
  double *lse; /* [nrows] */
} job;

/* One query row: the definition in the header comment, term by term. */
static void attend_row(const job *jb, int b, int h, int i, double *out, double *lse) {
  const int d = jb->d;
  const int group = jb->hq / jb->kv.hkv;
  const int g = h / group;
  const int lq = jb->cu_q[b + 1] - jb->cu_q[b];
  const int lk = kv_len(&jb->kv, b);
  const long p = (long)(lk - lq) + i;
  const uint16_t *qrow = jb->q + ((size_t)(jb->cu_q[b] + i) * jb->hq + h) * d;

  int j0 = 0, j1 = lk;
  if (jb->kv_begin) {
    if (jb->kv_begin[b] > j0) j0 = jb->kv_begin[b];
    if (jb->kv_end[b] < j1) j1 = jb->kv_end[b];
  }
  const int has_sink = jb->sinks != NULL && jb->use_sink;
  const double sink = has_sink ? (double)jb->sinks[h] : -INFINITY;

  /* scores of the visible keys */
  int n = 0;
  double *s = (double *)malloc(sizeof(double) * (size_t)(j1 > j0 ? j1 - j0 : 1));
  int *idx = (int *)malloc(sizeof(int) * (size_t)(j1 > j0 ? j1 - j0 : 1));
  for (int j = j0; j < j1; ++j) {
    if (jb->causal && (long)j > p) continue;
    if (jb->window > 0 && (long)j <= p - jb->window) continue;
    const uint16_t *krow = jb->kv.k + kv_row(&jb->kv, b, j, g);
    double dot = 0.0;
    for (int c = 0; c < d; ++c) dot += bf16_to_double(qrow[c]) * bf16_to_double(krow[c]);
    s[n] = jb->scale * dot;
    idx[n] = j;
    ++n;
  }

  double z = sink;
  for (int t = 0; t < n; ++t)
    if (s[t] > z) z = s[t];

  for (int c = 0; c < d; ++c) out[c] = 0.0;
  if (z == -INFINITY) { /* nothing visible and no sink */
    *lse = -INFINITY;
    free(s);
    free(idx);
    return;
  }
  double den = has_sink ? exp(sink - z) : 0.0;
  for (int t = 0; t < n; ++t) {
    const double w = exp(s[t] - z);
    den += w;
    const uint16_t *vrow = jb->kv.v + kv_row(&jb->kv, b, idx[t], g);
    for (int c = 0; c < d; ++c) out[c] += w * bf16_to_double(vrow[c]);
  }
  for (int c = 0; c < d; ++c) out[c] /= den;
  *lse = z + log(den);
  free(s);
  free(idx);
}

typedef struct {
  const job *jb;
  long begin, end;
} slice;

static void *run_slice(void *arg) {
  const slice *sl = (const slice *)arg;
  const job *jb = sl->jb;
  for (long r = sl->begin; r < sl->end; ++r) {
    const int32_t *t = jb->rows + 3 * r;
    attend_row(jb, t[0], t[1], t[2], jb->out + r * jb->d, jb->lse + r);
  }
  return NULL;
}

static void run_job(const job *jb, int nthreads) {
  if (nthreads < 1) nthreads = 1;
  if (nthreads > 256) nthreads = 256;
  if ((long)nthreads > jb->nrows) nthreads = jb->nrows > 0 ? (int)jb->nrows : 1;
  pthread_t th[256];
  slice sl[256];
  for (int t = 0; t < nthreads; ++t) {
    sl[t].jb = jb;
    sl[t].begin = jb->nrows * t / nthreads;
    sl[t].end = jb->nrows * (t + 1) / nthreads;
  }
  for (int t = 1; t < nthreads; ++t) pthread_create(&th[t], NULL, run_slice, &sl[t]);
  run_slice(&sl[0]);
  for (int t = 1; t < nthreads; ++t) pthread_join(th[t], NULL);
}

/* Enumerate every (b, h, i) row; returns the count, fills *rows_out. */
static long all_rows(const int32_t *cu_q, int batch, int hq, int32_t **rows_out) {
  long n = (long)(cu_q[batch] - cu_q[0]) * hq;
  int32_t *rows = (int32_t *)malloc(sizeof(int32_t) * 3 * (size_t)(n > 0 ? n : 1));
  long r = 0;
  for (int b = 0; b < batch; ++b) {
    const int lq = cu_q[b + 1] - cu_q[b];
    for (int i = 0; i < lq; ++i)
      for (int h = 0; h < hq; ++h) {
        rows[3 * r] = b;
        rows[3 * r + 1] = h;
        rows[3 * r + 2] = i;
        ++r;
      }
  }
  *rows_out = rows;
  return r;
}

static int check_common(const uint16_t *q, const int32_t *cu_q, const kv_source *kv, int batch,
                        int hq, int d) {
  if (!q || !cu_q || !kv->k || !kv->v || batch < 0 || d <= 0 || hq <= 0 || kv->hkv <= 0) return 1;
  if (cu_q[0] != 0) return 1;
  if (kv->cu_k && kv->cu_k[0] != 0) return 1;
  if (hq % kv->hkv) return 1;
  if (!kv->cu_k && (!kv->block_table || !kv->seqlens_k || kv->page_size <= 0)) return 1;
  return 0;
}

/*
 * Attention over packed variable-length sequences. Output rows follow the
 * packed query layout: out[(cu_q[b] + i) * hq + h][d], lse[(cu_q[b] + i) * hq + h].
 * K/V are contiguous (cu_k != NULL) or paged (block_table, seqlens_k).
 * sinks may be NULL. kv_begin/kv_end may be NULL (all keys) or restrict each
 * sequence's keys to [kv_begin[b], kv_end[b]); use_sink = 0 leaves the sink
 * out. With a restriction the result is the normalised partial of that block.
 */
int oracle_attention(const uint16_t *q, const int32_t *cu_q, const uint16_t *k, const uint16_t *v,
                     const int32_t *cu_k, const int32_t *block_table, const int32_t *seqlens_k,
                     int max_pages, int page_size, int batch, int hq, int hkv, int d,
                     const float *sinks, int use_sink, int causal, int window, double scale,
                     const int32_t *kv_begin, const int32_t *kv_end, double *out, double *lse,
                     int nthreads) {
  job jb;
  memset(&jb, 0, sizeof jb);
  jb.q = q;
  jb.cu_q = cu_q;
  jb.kv.k = k;
  jb.kv.v = v;
  jb.kv.cu_k = cu_k;
  jb.kv.block_table = block_table;
  jb.kv.seqlens_k = seqlens_k;
  jb.kv.max_pages = max_pages;
  jb.kv.page_size = page_size;
  jb.kv.hkv = hkv;
  jb.kv.d = d;
  if (check_common(q, cu_q, &jb.kv, batch, hq, d) || !out || !lse) return 1;
  jb.batch = batch;
  jb.hq = hq;
  jb.d = d;
  jb.sinks = sinks;
  jb.use_sink = use_sink;
  jb.causal = causal;
  jb.window = window;
  jb.scale = scale;
  jb.kv_begin = kv_begin;
  jb.kv_end = kv_end;
  int32_t *rows = NULL;
  jb.nrows = all_rows(cu_q, batch, hq, &rows);
  jb.rows = rows;
  /* all_rows enumerates rows in packed order, so row r of the job is
   * packed row r: (cu_q[b] + i) * hq + h. */
  jb.out = out;
  jb.lse = lse;
  run_job(&jb, nthreads);
  free(rows);
  return 0;
}

/*
 * The same definition for a chosen set of rows only: rows[r] = (b, h, i).
 * out[r * d ...], lse[r]. Used to check outputs of large problems one by one.
 */
int oracle_attention_rows(const uint16_t *q, const int32_t *cu_q, const uint16_t *k,
                          const uint16_t *v, const int32_t *cu_k, const int32_t *block_table,
                          const int32_t *seqlens_k, int max_pages, int page_size, int batch,
                          int hq, int hkv, int d, const float *sinks, int causal, int window,
                          double scale, const int32_t *rows, long nrows, double *out,
                          double *lse, int nthreads) {
  job jb;
  memset(&jb, 0, sizeof jb);
  jb.q = q;
  jb.cu_q = cu_q;
  jb.kv.k = k;
  jb.kv.v = v;
  jb.kv.cu_k = cu_k;
  jb.kv.block_table = block_table;
  jb.kv.seqlens_k = seqlens_k;
  jb.kv.max_pages = max_pages;
  jb.kv.page_size = page_size;
  jb.kv.hkv = hkv;
  jb.kv.d = d;
  if (check_common(q, cu_q, &jb.kv, batch, hq, d) || !out || !lse || (!rows && nrows)) return 1;
  for (long r = 0; r < nrows; ++r) {
    const int b = rows[3 * r], h = rows[3 * r + 1], i = rows[3 * r + 2];
    if (b < 0 || b >= batch || h < 0 || h >= hq || i < 0 || i >= cu_q[b + 1] - cu_q[b]) return 1;
  }
  jb.batch = batch;
  jb.hq = hq;
  jb.d = d;
  jb.sinks = sinks;
  jb.use_sink = 1;
  jb.causal = causal;
  jb.window = window;
  jb.scale = scale;
  jb.rows = rows;
  jb.nrows = nrows;
  jb.out = out;
  jb.lse = lse;
  run_job(&jb, nthreads);
  return 0;
}

/*
 * Merge of blocks computed along the KV sequence (same section: the sink must
 * enter exactly once). Each block k carries a normalised output o_k and its
 * log-sum-exp l_k. With M = max over l_k (and the sink, if given),
 *   w_k = exp(l_k - M),  W = sum_k w_k (+ exp(sink_h - M)),
 *   out = sum_k w_k o_k / W,  lse = M + ln W.
 * The sink, when given, is one more block with lse = sink_h and a zero output.
 * partial_o: [nsplit, rows, hq, d]; partial_lse: [nsplit, rows, hq].
 */
int oracle_merge(const double *partial_o, const double *partial_lse, int nsplit, long rows, int hq,
                 int d, const float *sinks, double *out, double *lse) {
  if (!partial_o || !partial_lse || !out || !lse || nsplit < 0 || rows < 0 || hq <= 0 || d <= 0)
    return 1;
  for (long r = 0; r < rows; ++r)
    for (int h = 0; h < hq; ++h) {
      const long rh = r * hq + h;
      double m = sinks ? (double)sinks[h] : -INFINITY;
      for (int k = 0; k < nsplit; ++k) {
        const double l = partial_lse[(long)k * rows * hq + rh];
        if (l > m) m = l;
      }
      double *o = out + rh * d;
      for (int c = 0; c < d; ++c) o[c] = 0.0;
      if (m == -INFINITY) {
        lse[rh] = -INFINITY;
        continue;
      }
      double wsum = sinks ? exp((double)sinks[h] - m) : 0.0;
      for (int k = 0; k < nsplit; ++k) {
        const double l = partial_lse[(long)k * rows * hq + rh];
        if (l == -INFINITY) continue;
        const double w = exp(l - m);
        wsum += w;
        const double *ok = partial_o + ((long)k * rows * hq + rh) * d;
        for (int c = 0; c < d; ++c) o[c] += w * ok[c];
      }
      for (int c = 0; c < d; ++c) o[c] /= wsum;
      lse[rh] = m + log(wsum);
    }
  return 0;
}
