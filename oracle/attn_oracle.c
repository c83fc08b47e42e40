/*
 * attn_oracle.c -- plain, slow fp64 CPU reference for paged attention.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the package smoke check and the
 * benchmark's CPU-baseline leg may load this code; the product path never does.
 * It shares no code, header or constant with the CUDA library.
 *
 * What it computes (AstrAI commit log, page "astrai/extension/backend/attention.py
 * @c9ceca1", batched-SDPA commit: one softmax attention per query row over the
 * request's cached keys, with the causal offset seq_len - q_len and exact-zero
 * weight for masked keys; page "astrai/extension @6f67ba8", CUDA-backend commit:
 * req_to_token is the page table at page_size = 1; same page, fallback-GQA bullet:
 * query heads share KV heads in consecutive groups, kvh = h / (Hq / Hkv)):
 *
 *   decode, request b, query head h:
 *     out[b,h,:] = sum_{j < seq_len_b} softmax_j( sm_scale * <q[b,h], K_j> ) * V_j
 *   prefill/extend, request b, local query row i (flat row qo_indptr[b] + i):
 *     same sum over j <= c_b + i,  c_b = seq_len_b - q_len_b   (bottom-right causal)
 *   with K_j = k_pool[req_to_token[b][j], kvh, :], V_j likewise, bf16 widened exactly.
 *
 * The softmax is the textbook stable one in fp64: subtract the max logit, exponentiate,
 * sum, divide.  An empty key set (seq_len = 0) yields a zero row (empty-sum reading).
 *
 * The split-KV functions follow the flash-decoding decomposition of the same page
 * (kernel-rename commit: per-split unnormalised partials plus a log-sum-exp combine):
 *   a split over keys [lo, hi) stores m = max logit (natural-log units),
 *   l = sum exp(logit - m) and o = sum exp(logit - m) V  (unnormalised);
 *   an empty split stores m = -inf, l = 0, o = 0;
 *   combine:  M = max_s m_s,  w_s = exp(m_s - M),  out = (sum_s w_s o_s) / (sum_s w_s l_s).
 *
 * Explicit masks (page "astrai/extension @6f67ba8", prefill-mask commit: 2-D [batch, kv_len]
 * and 3-D [batch, q_len, kv_len] masks, causal and mask able to coexist; unified causal
 * offset, -1 = off): key j of request b is visible to local query row i iff j < seq_len_b,
 * (causal off or j <= c_b + i), and the mask byte is nonzero -- mask[b][j] (2-D) or
 * mask[b][i][j] (3-D), rows kv_pitch bytes apart (3-D: q_pitch rows per request).  The row
 * attends over exactly its visible keys, in key order; no visible key gives a zero row.
 * Decode is the case q_len = 1, i = 0.
 *
 * The KV-append step (page "astrai/extension/attention_backend.py @47b3ed4",
 * write-then-gather helper commit: the new tokens' K and V are written into the pool
 * before attention gathers from it).  Reading: new token i of request b is the key at
 * position c_b + i of that request, so it is stored at slot req_to_token[b][c_b + i]:
 *   k_pool[slot, :, :] = k_new[qo_indptr[b] + i, :, :],  v_pool likewise;
 * every other pool row keeps its contents.
 *
 * Parallelism: independent output rows are spread over POSIX threads; each row is
 * computed start to finish by one thread in the order written above.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* bf16 bits -> double, exact (bf16 is the top half of an IEEE binary32). */
static double bf16_to_f64(uint16_t h) {
  uint32_t u = ((uint32_t)h) << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

typedef struct {
  int Hq, Hkv, D;
  const uint16_t *k_pool, *v_pool;  /* [num_slots, Hkv, D] */
  double sm_scale;
} pool_t;

/* Logit of query row q (already widened to double) against pool slot `slot`, head kvh. */
static double logit(const pool_t *P, const double *q, int32_t slot, int kvh) {
  const uint16_t *k = P->k_pool + ((int64_t)slot * P->Hkv + kvh) * P->D;
  double s = 0.0;
  for (int d = 0; d < P->D; ++d) s += q[d] * bf16_to_f64(k[d]);
  return P->sm_scale * s;
}

/* Full softmax attention of one query row over keys slots[0..n). */
static void attend(const pool_t *P, const double *q, int kvh, const int32_t *slots, int64_t n,
                   double *out /* [D] */) {
  const int D = P->D;
  for (int d = 0; d < D; ++d) out[d] = 0.0;
  if (n <= 0) return;
  double *s = (double *)malloc(sizeof(double) * (size_t)n);
  double m = -INFINITY;
  for (int64_t j = 0; j < n; ++j) {
    s[j] = logit(P, q, slots[j], kvh);
    if (s[j] > m) m = s[j];
  }
  double l = 0.0;
  for (int64_t j = 0; j < n; ++j) {
    s[j] = exp(s[j] - m);
    l += s[j];
  }
  for (int64_t j = 0; j < n; ++j) {
    const uint16_t *v = P->v_pool + ((int64_t)slots[j] * P->Hkv + kvh) * P->D;
    for (int d = 0; d < D; ++d) out[d] += s[j] * bf16_to_f64(v[d]);
  }
  for (int d = 0; d < D; ++d) out[d] /= l;
  free(s);
}

/* Unnormalised partial over keys slots[lo..hi): (o, m, l) as described in the header. */
static void partial(const pool_t *P, const double *q, int kvh, const int32_t *slots, int64_t lo,
                    int64_t hi, double *o, double *m_out, double *l_out) {
  const int D = P->D;
  for (int d = 0; d < D; ++d) o[d] = 0.0;
  if (hi <= lo) {
    *m_out = -INFINITY;
    *l_out = 0.0;
    return;
  }
  double m = -INFINITY;
  for (int64_t j = lo; j < hi; ++j) {
    double s = logit(P, q, slots[j], kvh);
    if (s > m) m = s;
  }
  double l = 0.0;
  for (int64_t j = lo; j < hi; ++j) {
    double w = exp(logit(P, q, slots[j], kvh) - m);
    l += w;
    const uint16_t *v = P->v_pool + ((int64_t)slots[j] * P->Hkv + kvh) * P->D;
    for (int d = 0; d < D; ++d) o[d] += w * bf16_to_f64(v[d]);
  }
  *m_out = m;
  *l_out = l;
}

static void widen_row(const uint16_t *src, int D, double *dst) {
  for (int d = 0; d < D; ++d) dst[d] = bf16_to_f64(src[d]);
}

/* ---------------------------------------------------------------- work items */

enum { JOB_DECODE = 0, JOB_PREFILL = 1, JOB_PARTIALS = 2, JOB_MASKED = 3, JOB_RANGES = 4 };

typedef struct {
  int kind;
  pool_t P;
  int B;
  const uint16_t *q;
  const int32_t *req_to_token;
  int64_t r2t_stride;
  const int32_t *seq_lens;
  const int32_t *qo_indptr;
  /* the rows to compute: decode (b,h); prefill (flat row, h) */
  int64_t n_items;
  const int32_t *item_row, *item_head;
  double *out;  /* [n_items, D] */
  /* partials */
  int S;
  double *o_part, *ml_part;
  /* key ranges (JOB_RANGES): item n covers keys [item_lo[n], item_hi[n]) of its request */
  const int64_t *item_lo, *item_hi;
  /* explicit mask (JOB_MASKED): kind 2 = [B, kv_pitch], 3 = [B, q_pitch, kv_pitch]; rows are
   * decode (b, h) pairs when is_decode, else (flat row, h) */
  const uint8_t *mask;
  int mask_dims, is_decode, causal;
  int64_t kv_pitch, q_pitch;
  int next_thread;
  int nthreads;
} job_t;

typedef struct {
  job_t *J;
  int tid;
} targ_t;

/* Request owning flat query row r (qo_indptr is non-decreasing, qo_indptr[0] = 0). */
static int request_of_row(const int32_t *qo_indptr, int B, int64_t r) {
  int lo = 0, hi = B - 1;
  while (lo < hi) {
    int mid = (lo + hi + 1) / 2;
    if ((int64_t)qo_indptr[mid] <= r) lo = mid; else hi = mid - 1;
  }
  while (lo < B - 1 && (int64_t)qo_indptr[lo + 1] <= r) ++lo;  /* skip empty requests */
  return lo;
}

static void run_item(job_t *J, int64_t it, double *qbuf) {
  const pool_t *P = &J->P;
  const int G = P->Hq / P->Hkv;
  const int D = P->D;
  int h = J->item_head[it];
  int kvh = h / G;
  if (J->kind == JOB_DECODE) {
    int b = J->item_row[it];
    widen_row(J->q + ((int64_t)b * P->Hq + h) * D, D, qbuf);
    attend(P, qbuf, kvh, J->req_to_token + (int64_t)b * J->r2t_stride, J->seq_lens[b], J->out + it * D);
  } else if (J->kind == JOB_PREFILL) {
    int64_t r = J->item_row[it];
    int b = request_of_row(J->qo_indptr, J->B, r);
    int64_t i = r - J->qo_indptr[b];
    int64_t q_len = (int64_t)J->qo_indptr[b + 1] - J->qo_indptr[b];
    int64_t c = (int64_t)J->seq_lens[b] - q_len;  /* causal offset */
    widen_row(J->q + (r * P->Hq + h) * D, D, qbuf);
    attend(P, qbuf, kvh, J->req_to_token + (int64_t)b * J->r2t_stride, c + i + 1, J->out + it * D);
  } else if (J->kind == JOB_MASKED) {
    int b;
    int64_t i, c;
    if (J->is_decode) {
      b = J->item_row[it];
      i = 0;
      c = (int64_t)J->seq_lens[b] - 1;
      widen_row(J->q + ((int64_t)b * P->Hq + h) * D, D, qbuf);
    } else {
      int64_t r = J->item_row[it];
      b = request_of_row(J->qo_indptr, J->B, r);
      i = r - J->qo_indptr[b];
      c = (int64_t)J->seq_lens[b] - ((int64_t)J->qo_indptr[b + 1] - J->qo_indptr[b]);
      widen_row(J->q + (r * P->Hq + h) * D, D, qbuf);
    }
    const int32_t *row_slots = J->req_to_token + (int64_t)b * J->r2t_stride;
    const uint8_t *mrow = J->mask_dims == 2 ? J->mask + (int64_t)b * J->kv_pitch
                                            : J->mask + ((int64_t)b * J->q_pitch + i) * J->kv_pitch;
    const int64_t n = J->seq_lens[b];
    int32_t *vis = (int32_t *)malloc(sizeof(int32_t) * (size_t)(n > 0 ? n : 1));
    int64_t nv = 0;
    for (int64_t j = 0; j < n; ++j) {
      const int causal_ok = !J->causal || j <= c + i;
      if (causal_ok && mrow[j] != 0) vis[nv++] = row_slots[j];
    }
    attend(P, qbuf, kvh, vis, nv, J->out + it * D);
    free(vis);
  } else if (J->kind == JOB_RANGES) {
    int b = J->item_row[it];
    widen_row(J->q + ((int64_t)b * P->Hq + h) * D, D, qbuf);
    partial(P, qbuf, kvh, J->req_to_token + (int64_t)b * J->r2t_stride, J->item_lo[it], J->item_hi[it],
            J->o_part + it * D, &J->ml_part[2 * it], &J->ml_part[2 * it + 1]);
  } else { /* JOB_PARTIALS: even split of request b's keys into S pieces */
    int b = J->item_row[it];
    widen_row(J->q + ((int64_t)b * P->Hq + h) * D, D, qbuf);
    int64_t n = J->seq_lens[b];
    int64_t chunk = (n + J->S - 1) / J->S;
    const int32_t *slots = J->req_to_token + (int64_t)b * J->r2t_stride;
    for (int s = 0; s < J->S; ++s) {
      int64_t lo = (int64_t)s * chunk, hi = lo + chunk;
      if (lo > n) lo = n;
      if (hi > n) hi = n;
      int64_t base = ((int64_t)b * P->Hq + h) * J->S + s;
      partial(P, qbuf, kvh, slots, lo, hi, J->o_part + base * D, &J->ml_part[2 * base], &J->ml_part[2 * base + 1]);
    }
  }
}

static void *worker(void *arg) {
  targ_t *T = (targ_t *)arg;
  job_t *J = T->J;
  double *qbuf = (double *)malloc(sizeof(double) * (size_t)J->P.D);
  for (int64_t it = T->tid; it < J->n_items; it += J->nthreads) run_item(J, it, qbuf);
  free(qbuf);
  return NULL;
}

static void run_job(job_t *J, int nthreads) {
  if (nthreads < 1) nthreads = 1;
  if (nthreads > 1024) nthreads = 1024;
  if ((int64_t)nthreads > J->n_items) nthreads = J->n_items > 0 ? (int)J->n_items : 1;
  J->nthreads = nthreads;
  pthread_t th[1024];
  targ_t args[1024];
  for (int t = 0; t < nthreads; ++t) {
    args[t].J = J;
    args[t].tid = t;
  }
  for (int t = 1; t < nthreads; ++t) pthread_create(&th[t], NULL, worker, &args[t]);
  worker(&args[0]);
  for (int t = 1; t < nthreads; ++t) pthread_join(th[t], NULL);
}

/* ---------------------------------------------------------------- exported API */

/* Decode attention for the listed (b, h) pairs; out is [n_items, D]. */
void oracle_decode_rows(int B, int Hq, int Hkv, int D, const uint16_t *q, const uint16_t *k_pool,
                        const uint16_t *v_pool, const int32_t *req_to_token, int64_t r2t_stride,
                        const int32_t *seq_lens, double sm_scale, int64_t n_items, const int32_t *item_b,
                        const int32_t *item_h, double *out, int nthreads) {
  job_t J;
  memset(&J, 0, sizeof J);
  J.kind = JOB_DECODE;
  J.P.Hq = Hq; J.P.Hkv = Hkv; J.P.D = D; J.P.k_pool = k_pool; J.P.v_pool = v_pool; J.P.sm_scale = sm_scale;
  J.B = B; J.q = q; J.req_to_token = req_to_token; J.r2t_stride = r2t_stride; J.seq_lens = seq_lens;
  J.n_items = n_items; J.item_row = item_b; J.item_head = item_h; J.out = out;
  run_job(&J, nthreads);
}

/* Prefill/extend attention for the listed (flat query row, h) pairs; out is [n_items, D]. */
void oracle_prefill_rows(int B, int Hq, int Hkv, int D, const uint16_t *q, const int32_t *qo_indptr,
                         const uint16_t *k_pool, const uint16_t *v_pool, const int32_t *req_to_token,
                         int64_t r2t_stride, const int32_t *seq_lens, double sm_scale, int64_t n_items,
                         const int32_t *item_row, const int32_t *item_h, double *out, int nthreads) {
  job_t J;
  memset(&J, 0, sizeof J);
  J.kind = JOB_PREFILL;
  J.P.Hq = Hq; J.P.Hkv = Hkv; J.P.D = D; J.P.k_pool = k_pool; J.P.v_pool = v_pool; J.P.sm_scale = sm_scale;
  J.B = B; J.q = q; J.qo_indptr = qo_indptr; J.req_to_token = req_to_token; J.r2t_stride = r2t_stride;
  J.seq_lens = seq_lens; J.n_items = n_items; J.item_row = item_row; J.item_head = item_h; J.out = out;
  run_job(&J, nthreads);
}

/* Even S-way split partials for every (b, h): o_part [B,Hq,S,D], ml_part [B,Hq,S,2]. */
void oracle_decode_split_partials(int B, int Hq, int Hkv, int D, const uint16_t *q, const uint16_t *k_pool,
                                  const uint16_t *v_pool, const int32_t *req_to_token, int64_t r2t_stride,
                                  const int32_t *seq_lens, double sm_scale, int S, double *o_part,
                                  double *ml_part, int nthreads) {
  job_t J;
  memset(&J, 0, sizeof J);
  J.kind = JOB_PARTIALS;
  J.P.Hq = Hq; J.P.Hkv = Hkv; J.P.D = D; J.P.k_pool = k_pool; J.P.v_pool = v_pool; J.P.sm_scale = sm_scale;
  J.B = B; J.q = q; J.req_to_token = req_to_token; J.r2t_stride = r2t_stride; J.seq_lens = seq_lens;
  J.S = S; J.o_part = o_part; J.ml_part = ml_part;
  int32_t *ib = (int32_t *)malloc(sizeof(int32_t) * (size_t)B * Hq + 1);
  int32_t *ih = (int32_t *)malloc(sizeof(int32_t) * (size_t)B * Hq + 1);
  for (int b = 0; b < B; ++b)
    for (int h = 0; h < Hq; ++h) { ib[b * Hq + h] = b; ih[b * Hq + h] = h; }
  J.n_items = (int64_t)B * Hq; J.item_row = ib; J.item_head = ih;
  run_job(&J, nthreads);
  free(ib);
  free(ih);
}

/* Partials over explicit key ranges: item n is (request b, query head h, keys [lo, hi) of
 * request b, i.e. positions lo .. hi-1 of its req_to_token row); it stores the split's
 * (o, m, l) as described in the header into o_out [n_items, D] and ml_out [n_items, 2].
 * Where the split boundaries lie is the caller's choice: this is the per-split piece of the
 * kernel-rename commit for any one split. */
void oracle_partial_ranges(int B, int Hq, int Hkv, int D, const uint16_t *q, const uint16_t *k_pool,
                           const uint16_t *v_pool, const int32_t *req_to_token, int64_t r2t_stride,
                           double sm_scale, int64_t n_items, const int32_t *item_b, const int32_t *item_h,
                           const int64_t *item_lo, const int64_t *item_hi, double *o_out, double *ml_out,
                           int nthreads) {
  job_t J;
  memset(&J, 0, sizeof J);
  J.kind = JOB_RANGES;
  J.P.Hq = Hq; J.P.Hkv = Hkv; J.P.D = D; J.P.k_pool = k_pool; J.P.v_pool = v_pool; J.P.sm_scale = sm_scale;
  J.B = B; J.q = q; J.req_to_token = req_to_token; J.r2t_stride = r2t_stride;
  J.n_items = n_items; J.item_row = item_b; J.item_head = item_h; J.item_lo = item_lo; J.item_hi = item_hi;
  J.o_part = o_out; J.ml_part = ml_out;
  run_job(&J, nthreads);
}

/* Log-sum-exp combine of the first nsplit[b] partials of each (b, h); out [B,Hq,D]. */
void oracle_combine(int B, int Hq, int S, int D, const double *o_part, const double *ml_part,
                    const int32_t *nsplit, double *out) {
  for (int b = 0; b < B; ++b) {
    int n = nsplit ? nsplit[b] : S;
    for (int h = 0; h < Hq; ++h) {
      int64_t base = ((int64_t)b * Hq + h) * S;
      double *o = out + ((int64_t)b * Hq + h) * D;
      double M = -INFINITY;
      for (int s = 0; s < n; ++s)
        if (ml_part[2 * (base + s)] > M) M = ml_part[2 * (base + s)];
      for (int d = 0; d < D; ++d) o[d] = 0.0;
      if (M == -INFINITY) continue;
      double L = 0.0;
      for (int s = 0; s < n; ++s) {
        double m = ml_part[2 * (base + s)];
        double w = (m == -INFINITY) ? 0.0 : exp(m - M);
        L += w * ml_part[2 * (base + s) + 1];
        for (int d = 0; d < D; ++d) o[d] += w * o_part[(base + s) * D + d];
      }
      for (int d = 0; d < D; ++d) o[d] /= L;
    }
  }
}

/* KV append: copy each new token's K and V rows (all KV heads) into its pool slot.
 * k_new, v_new: [total_q, Hkv, D]; pools are modified in place. */
void oracle_kv_append(int B, int Hkv, int D, const int32_t *qo_indptr, const int32_t *seq_lens,
                      const int32_t *req_to_token, int64_t r2t_stride, const uint16_t *k_new,
                      const uint16_t *v_new, uint16_t *k_pool, uint16_t *v_pool) {
  const int64_t row = (int64_t)Hkv * D;  /* elements of one slot (all KV heads) */
  for (int b = 0; b < B; ++b) {
    const int64_t q_len = (int64_t)qo_indptr[b + 1] - qo_indptr[b];
    const int64_t c = (int64_t)seq_lens[b] - q_len;
    for (int64_t i = 0; i < q_len; ++i) {
      const int64_t src = (int64_t)qo_indptr[b] + i;
      const int32_t slot = req_to_token[(int64_t)b * r2t_stride + c + i];
      memcpy(k_pool + (int64_t)slot * row, k_new + src * row, sizeof(uint16_t) * (size_t)row);
      memcpy(v_pool + (int64_t)slot * row, v_new + src * row, sizeof(uint16_t) * (size_t)row);
    }
  }
}

/* Attention with an explicit mask (and, for prefill, the causal flag) for the listed rows:
 * decode rows are (b, h) pairs (is_decode = 1, qo_indptr unused), prefill rows (flat row, h). */
void oracle_masked_rows(int is_decode, int B, int Hq, int Hkv, int D, const uint16_t *q, const int32_t *qo_indptr,
                        const uint16_t *k_pool, const uint16_t *v_pool, const int32_t *req_to_token,
                        int64_t r2t_stride, const int32_t *seq_lens, double sm_scale, const uint8_t *mask,
                        int mask_dims, int64_t kv_pitch, int64_t q_pitch, int causal, int64_t n_items,
                        const int32_t *item_row, const int32_t *item_h, double *out, int nthreads) {
  job_t J;
  memset(&J, 0, sizeof J);
  J.kind = JOB_MASKED;
  J.P.Hq = Hq; J.P.Hkv = Hkv; J.P.D = D; J.P.k_pool = k_pool; J.P.v_pool = v_pool; J.P.sm_scale = sm_scale;
  J.B = B; J.q = q; J.qo_indptr = qo_indptr; J.req_to_token = req_to_token; J.r2t_stride = r2t_stride;
  J.seq_lens = seq_lens; J.n_items = n_items; J.item_row = item_row; J.item_head = item_h; J.out = out;
  J.mask = mask; J.mask_dims = mask_dims; J.kv_pitch = kv_pitch; J.q_pitch = q_pitch;
  J.is_decode = is_decode; J.causal = causal;
  run_job(&J, nthreads);
}
