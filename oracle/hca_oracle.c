/*
 * hca_oracle.c -- plain, slow, fp64 CPU oracle for Heavily Compressed
 * Attention (HCA).  TEST INFRASTRUCTURE ONLY: it is linked by the tests, by
 * the smoke check and by the CPU-baseline leg of the benchmark, never by the
 * product path.  It shares no code, header or table with the CUDA library.
 *
 * What it computes (the plain definition, evaluated element by element):
 *
 *   For batch row b and query position i with seg[b,i] >= 0, the candidate
 *   key set is the union of
 *     raw rows t      : i-W < t <= i  and  seg[b,t] == seg[b,i]
 *     compressed j    : (j+1)*m <= i+1  and every position x of the window
 *                       [j*m, (j+1)*m-1] has seg[b,x] == seg[b,i]
 *   ("Add HCA Static Compilation for Splash Attention [Deepseek v4]",
 *   Description: the HCA pattern is a local sliding window plus the
 *   compression windows that have completed before the query; segment ids
 *   isolate packed documents.  "DSV4: Route compressed and sliding train
 *   attention onto the splash kernels", review suggestion on the segment
 *   mask: two positions may interact only when their segment ids are equal.)
 *
 *   K = V: the one shared kv tensor (and the compressed ckv tensor) serves as
 *   both key and value for every head ("[DeepSeek-V4] Implement Compressed
 *   Attention Layers", review suggestions on the logits and output einsums:
 *   k and v are both the single-head kv, broadcast over the query heads).
 *
 *   s_k   = scale * <q[b,h,i,:], r_k>         r_k = kv[b,t,:] or ckv[b,j,:]
 *   lse   = log sum_k exp(s_k)                (natural log, scaled logits)
 *   out   = sum_k exp(s_k - lse) r_k
 *
 *   backward for a cotangent dO = d loss / d out:
 *   P_k   = exp(s_k - lse),  dP_k = <dO, r_k>,  Delta = sum_k P_k dP_k
 *   dS_k  = P_k (dP_k - Delta)
 *   dq    = scale * sum_k dS_k r_k
 *   d r_k += scale * dS_k * q + P_k * dO     (summed over heads and queries;
 *                                             the K role plus the V role)
 *
 *   Positions with seg < 0 are padding: they are neither queries nor keys;
 *   their out and dq rows are 0 and their lse is -inf.
 *
 *   Compressed sparse attention (CSA) takes the same two sets, except that a
 *   compressed entry also has to be kept by the indexer's top-k selection for
 *   that query ("Add HCA Static Compilation for Splash Attention [Deepseek
 *   v4]", Description: CSA, compress ratio 4, needs a top-k step and runtime
 *   indexer masks; "DSV4: Route compressed and sliding train attention onto
 *   the splash kernels": the indexer mask keeps or discards a (query,
 *   compressed entry) pair).  The hca_oracle_csa_* entry points take that
 *   selection as a dense keep mask sel[B,S,Sc]; the pages do not define the
 *   indexer, so the selection is an input.  Completion and document rules are
 *   those above (the plainest reading: selection narrows the HCA set).
 *
 * Inputs are read in their stored type (bf16 bits, fp32 or fp64) and widened
 * exactly to double; every result is double.  Parallelism is plain pthreads
 * over independent rows; each output element is produced by one thread in a
 * fixed order, so results are deterministic.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

enum { OR_BF16 = 0, OR_F32 = 1, OR_F64 = 2 };

static double widen(const void *p, int dt, size_t idx) {
  if (dt == OR_BF16) {
    uint32_t u = ((uint32_t)((const uint16_t *)p)[idx]) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
  }
  if (dt == OR_F32) return (double)((const float *)p)[idx];
  return ((const double *)p)[idx];
}

/* ------------------------------------------------------------------ */
/* the visibility predicate, one element at a time                      */
/* ------------------------------------------------------------------ */

typedef struct {
  const int32_t *seg; /* [B,S] or NULL (one segment, id 0)          */
  int B, S, W, m, Sc;
  int32_t *win_id;    /* [B,Sc]: the id shared by all m positions of
                         window j, or INT32_MIN when the window mixes ids,
                         touches padding or runs past S               */
  const uint8_t *sel; /* [B,S,Sc] CSA keep mask (nonzero = the indexer
                         kept entry j for query i); NULL for HCA      */
} vis_t;

static int32_t seg_at(const vis_t *v, int b, int x) {
  return v->seg ? v->seg[(size_t)b * v->S + x] : 0;
}

static int vis_init(vis_t *v, const int32_t *seg, int B, int S, int W, int m) {
  v->seg = seg; v->B = B; v->S = S; v->W = W; v->m = m;
  v->Sc = (S + m - 1) / m;
  v->sel = NULL;
  v->win_id = (int32_t *)malloc(sizeof(int32_t) * (size_t)(B > 0 ? B : 1) * (v->Sc > 0 ? v->Sc : 1));
  if (!v->win_id) return -1;
  for (int b = 0; b < B; ++b)
    for (int j = 0; j < v->Sc; ++j) {
      int32_t id = INT32_MIN;
      if ((long)(j + 1) * m <= S) {
        id = seg_at(v, b, j * m);
        for (int x = j * m; x < (j + 1) * m; ++x)
          if (seg_at(v, b, x) != id) { id = INT32_MIN; break; }
        if (id < 0) id = INT32_MIN;
      }
      v->win_id[(size_t)b * v->Sc + j] = id;
    }
  return 0;
}

/* raw row t visible from query i (both in batch row b) */
static int raw_visible(const vis_t *v, int b, int i, int t) {
  int32_t si = seg_at(v, b, i);
  if (si < 0 || t < 0 || t >= v->S) return 0;
  if (!(i - v->W < t && t <= i)) return 0;
  return seg_at(v, b, t) == si;
}

/* compressed entry j visible from query i */
static int comp_visible(const vis_t *v, int b, int i, int j) {
  int32_t si = seg_at(v, b, i);
  if (si < 0 || j < 0 || j >= v->Sc) return 0;
  if ((long)(j + 1) * v->m > (long)i + 1) return 0;
  if (v->sel && !v->sel[((size_t)b * v->S + i) * v->Sc + j]) return 0;
  return v->win_id[(size_t)b * v->Sc + j] == si;
}

/* ------------------------------------------------------------------ */
/* a tiny work-sharing thread pool                                     */
/* ------------------------------------------------------------------ */

typedef void (*task_fn)(void *ctx, long item, double *scratch);

typedef struct {
  task_fn fn;
  void *ctx;
  long n;
  long next;
  size_t scratch_doubles;
  int failed;
} pool_t;

static void *pool_worker(void *arg) {
  pool_t *p = (pool_t *)arg;
  double *scratch = (double *)malloc(sizeof(double) * (p->scratch_doubles ? p->scratch_doubles : 1));
  if (!scratch) { __atomic_store_n(&p->failed, 1, __ATOMIC_SEQ_CST); return NULL; }
  for (;;) {
    long it = __atomic_fetch_add(&p->next, 1, __ATOMIC_SEQ_CST);
    if (it >= p->n) break;
    p->fn(p->ctx, it, scratch);
  }
  free(scratch);
  return NULL;
}

static int resolve_threads(int nthreads) {
  if (nthreads > 0) return nthreads;
  long n = sysconf(_SC_NPROCESSORS_ONLN);
  return n > 0 ? (int)n : 1;
}

static int run_pool(task_fn fn, void *ctx, long n, size_t scratch_doubles, int nthreads) {
  pool_t p = {fn, ctx, n, 0, scratch_doubles, 0};
  int T = resolve_threads(nthreads);
  if (T > n) T = (int)(n > 0 ? n : 1);
  pthread_t *th = (pthread_t *)malloc(sizeof(pthread_t) * (size_t)T);
  if (!th) return -1;
  int started = 0;
  for (int k = 0; k < T; ++k) {
    if (pthread_create(&th[k], NULL, pool_worker, &p) != 0) break;
    ++started;
  }
  if (started == 0) { pool_worker(&p); }
  for (int k = 0; k < started; ++k) pthread_join(th[k], NULL);
  free(th);
  return p.failed ? -1 : 0;
}

int hca_oracle_num_threads(int nthreads) { return resolve_threads(nthreads); }

/* ------------------------------------------------------------------ */
/* shared problem description                                           */
/* ------------------------------------------------------------------ */

typedef struct {
  vis_t v;
  const void *q, *kv, *ckv, *dout;
  int dt;
  int H, D;
  double scale;
  int row_begin, row_end; /* query positions processed (all batch rows) */
  double *out, *lse, *dq;
  double *lse_all, *delta_all; /* [B,H,S] internal for the key pass      */
  const uint8_t *need;         /* [B,S] queries whose lse/Delta are needed */
  double *dkv, *dckv;
  const int64_t *key_list; /* key pass: flat (b*S+t) or (b*Sc+j) ids      */
  double *key_out;         /* key pass: [n][D]                           */
  int comp_keys;           /* key pass over compressed entries?          */
} prob_t;

/* Gather the visible keys of query (b,i) into rows of K[n][D]; returns n. */
static int gather_keys(const prob_t *P, int b, int i, double *K) {
  const vis_t *v = &P->v;
  int D = P->D, n = 0;
  int t0 = i - v->W + 1;
  if (t0 < 0) t0 = 0;
  for (int t = t0; t <= i; ++t)
    if (raw_visible(v, b, i, t)) {
      for (int d = 0; d < D; ++d) K[(size_t)n * D + d] = widen(P->kv, P->dt, ((size_t)b * v->S + t) * D + d);
      ++n;
    }
  for (int j = 0; j < v->Sc; ++j)
    if (comp_visible(v, b, i, j)) {
      for (int d = 0; d < D; ++d) K[(size_t)n * D + d] = widen(P->ckv, P->dt, ((size_t)b * v->Sc + j) * D + d);
      ++n;
    }
  return n;
}

static size_t keys_scratch(const prob_t *P) {
  /* K[n][D] + logits[n] + q[D] + dO[D] + dP[n] */
  size_t nmax = (size_t)P->v.W + (size_t)P->v.Sc + 1;
  return nmax * (size_t)P->D + 2 * nmax + 2 * (size_t)P->D + 16;
}

/* softmax statistics of one (b,h,i) row: logits s[n], returns lse */
static double row_logits(const prob_t *P, int b, int h, int i, const double *K, int n, double *qrow, double *s) {
  int D = P->D, S = P->v.S;
  for (int d = 0; d < D; ++d) qrow[d] = widen(P->q, P->dt, (((size_t)b * P->H + h) * S + i) * D + d);
  double mx = -INFINITY;
  for (int k = 0; k < n; ++k) {
    double acc = 0.0;
    for (int d = 0; d < D; ++d) acc += qrow[d] * K[(size_t)k * D + d];
    s[k] = P->scale * acc;
    if (s[k] > mx) mx = s[k];
  }
  double sum = 0.0;
  for (int k = 0; k < n; ++k) sum += exp(s[k] - mx);
  return mx + log(sum);
}

/* ------------------------------------------------------------------ */
/* forward                                                              */
/* ------------------------------------------------------------------ */

static void fwd_task(void *ctx, long item, double *scr) {
  const prob_t *P = (const prob_t *)ctx;
  int rows = P->row_end - P->row_begin;
  int b = (int)(item / rows), i = P->row_begin + (int)(item % rows);
  int D = P->D, S = P->v.S, H = P->H;
  size_t nmax = (size_t)P->v.W + P->v.Sc + 1;
  double *K = scr, *s = K + nmax * D, *qrow = s + nmax;
  int n = gather_keys(P, b, i, K);
  for (int h = 0; h < H; ++h) {
    size_t r = ((size_t)b * H + h) * S + i;
    double *o = P->out + r * D;
    if (n == 0) {
      for (int d = 0; d < D; ++d) o[d] = 0.0;
      P->lse[r] = -INFINITY;
      continue;
    }
    double lse = row_logits(P, b, h, i, K, n, qrow, s);
    for (int d = 0; d < D; ++d) o[d] = 0.0;
    for (int k = 0; k < n; ++k) {
      double p = exp(s[k] - lse);
      for (int d = 0; d < D; ++d) o[d] += p * K[(size_t)k * D + d];
    }
    P->lse[r] = lse;
  }
}

static int check_rows(int S, int *rb, int *re) {
  if (*rb < 0) *rb = 0;
  if (*re > S || *re < 0) *re = S;
  return *re >= *rb;
}

/* out[B,H,S,D] and lse[B,H,S] for query positions [row_begin,row_end) of
 * every batch row (other rows are left untouched). */
static int fwd_impl(const void *q, const void *kv, const void *ckv, const int32_t *seg, const uint8_t *sel,
                    int dtype, int B, int H, int S, int D, int W, int m, double scale,
                    int row_begin, int row_end, double *out, double *lse, int nthreads) {
  if (B < 0 || H < 1 || S < 0 || D < 1 || W < 1 || m < 1) return -2;
  if (!check_rows(S, &row_begin, &row_end)) return -2;
  prob_t P;
  memset(&P, 0, sizeof P);
  if (vis_init(&P.v, seg, B, S, W, m)) return -1;
  P.v.sel = sel;
  P.q = q; P.kv = kv; P.ckv = ckv; P.dt = dtype; P.H = H; P.D = D; P.scale = scale;
  P.row_begin = row_begin; P.row_end = row_end; P.out = out; P.lse = lse;
  int rc = run_pool(fwd_task, &P, (long)B * (row_end - row_begin), keys_scratch(&P), nthreads);
  free(P.v.win_id);
  return rc;
}

int hca_oracle_fwd(const void *q, const void *kv, const void *ckv, const int32_t *seg, int dtype,
                   int B, int H, int S, int D, int W, int m, double scale,
                   int row_begin, int row_end, double *out, double *lse, int nthreads) {
  return fwd_impl(q, kv, ckv, seg, NULL, dtype, B, H, S, D, W, m, scale, row_begin, row_end, out, lse, nthreads);
}

/* CSA forward: as hca_oracle_fwd, compressed entries also need sel[b,i,j]. */
int hca_oracle_csa_fwd(const void *q, const void *kv, const void *ckv, const int32_t *seg, const uint8_t *sel,
                       int dtype, int B, int H, int S, int D, int W, int m, double scale,
                       int row_begin, int row_end, double *out, double *lse, int nthreads) {
  if (!sel) return -2;
  return fwd_impl(q, kv, ckv, seg, sel, dtype, B, H, S, D, W, m, scale, row_begin, row_end, out, lse, nthreads);
}

/* ------------------------------------------------------------------ */
/* backward                                                             */
/* ------------------------------------------------------------------ */

/* Query pass: lse, Delta and dq for one (b,i), all heads. */
static void bwd_query_task(void *ctx, long item, double *scr) {
  const prob_t *P = (const prob_t *)ctx;
  int b = (int)(item / P->v.S), i = (int)(item % P->v.S);
  if (P->need && !P->need[(size_t)b * P->v.S + i]) return;
  int D = P->D, S = P->v.S, H = P->H;
  size_t nmax = (size_t)P->v.W + P->v.Sc + 1;
  double *K = scr, *s = K + nmax * D, *qrow = s + nmax, *dP = qrow + D, *dO = dP + nmax;
  int n = gather_keys(P, b, i, K);
  int own_dq = P->dq && i >= P->row_begin && i < P->row_end;
  for (int h = 0; h < H; ++h) {
    size_t r = ((size_t)b * H + h) * S + i;
    if (n == 0) {
      P->lse_all[r] = -INFINITY;
      P->delta_all[r] = 0.0;
      if (own_dq) for (int d = 0; d < D; ++d) P->dq[r * D + d] = 0.0;
      continue;
    }
    double lse = row_logits(P, b, h, i, K, n, qrow, s);
    for (int d = 0; d < D; ++d) dO[d] = widen(P->dout, P->dt, r * D + d);
    double delta = 0.0;
    for (int k = 0; k < n; ++k) {
      double acc = 0.0;
      for (int d = 0; d < D; ++d) acc += dO[d] * K[(size_t)k * D + d];
      dP[k] = acc;
      delta += exp(s[k] - lse) * acc;
    }
    P->lse_all[r] = lse;
    P->delta_all[r] = delta;
    if (own_dq) {
      double *g = P->dq + r * D;
      for (int d = 0; d < D; ++d) g[d] = 0.0;
      for (int k = 0; k < n; ++k) {
        double ds = exp(s[k] - lse) * (dP[k] - delta);
        for (int d = 0; d < D; ++d) g[d] += P->scale * ds * K[(size_t)k * D + d];
      }
    }
  }
}

/* Gradient of one key row r (raw row t or compressed entry j of batch row
 * b) summed over the visible queries in [qlo,qhi) and every head. */
static void key_grad(const prob_t *P, int b, int is_comp, int key, int qlo, int qhi, double *g, double *scr) {
  const vis_t *v = &P->v;
  int D = P->D, S = v->S, H = P->H;
  double *r = scr, *qrow = r + D, *dO = qrow + D;
  for (int d = 0; d < D; ++d)
    r[d] = is_comp ? widen(P->ckv, P->dt, ((size_t)b * v->Sc + key) * D + d)
                   : widen(P->kv, P->dt, ((size_t)b * S + key) * D + d);
  for (int d = 0; d < D; ++d) g[d] = 0.0;
  /* candidates: raw t can be seen only by i in [t, t+W-1]; compressed j
   * only by i >= (j+1)m-1.  The predicate is still checked per element. */
  int lo = is_comp ? (key + 1) * v->m - 1 : key;
  int hi = is_comp ? S : (key + v->W < S ? key + v->W : S);
  if (lo < qlo) lo = qlo;
  if (hi > qhi) hi = qhi;
  for (int i = lo; i < hi; ++i) {
    int vis = is_comp ? comp_visible(v, b, i, key) : raw_visible(v, b, i, key);
    if (!vis) continue;
    for (int h = 0; h < H; ++h) {
      size_t row = ((size_t)b * H + h) * S + i;
      double acc = 0.0, accd = 0.0;
      for (int d = 0; d < D; ++d) {
        qrow[d] = widen(P->q, P->dt, row * D + d);
        dO[d] = widen(P->dout, P->dt, row * D + d);
        acc += qrow[d] * r[d];
        accd += dO[d] * r[d];
      }
      double p = exp(P->scale * acc - P->lse_all[row]);
      double ds = p * (accd - P->delta_all[row]);
      for (int d = 0; d < D; ++d) g[d] += P->scale * ds * qrow[d] + p * dO[d];
    }
  }
}

static void bwd_key_task(void *ctx, long item, double *scr) {
  const prob_t *P = (const prob_t *)ctx;
  const vis_t *v = &P->v;
  long nraw = (long)v->B * v->S;
  if (item < nraw) {
    int b = (int)(item / v->S), t = (int)(item % v->S);
    key_grad(P, b, 0, t, P->row_begin, P->row_end, P->dkv + (size_t)item * P->D, scr);
  } else {
    long c = item - nraw;
    int b = (int)(c / v->Sc), j = (int)(c % v->Sc);
    key_grad(P, b, 1, j, P->row_begin, P->row_end, P->dckv + (size_t)c * P->D, scr);
  }
}

/* dq[B,H,S,D] for query positions [row_begin,row_end) and dkv[B,S,D],
 * dckv[B,Sc,D] holding the contributions of exactly those queries (the
 * full gradient when the range is [0,S)). */
static int bwd_impl(const void *q, const void *kv, const void *ckv, const int32_t *seg, const uint8_t *sel,
                    const void *dout, int dtype, int B, int H, int S, int D, int W, int m, double scale,
                    int row_begin, int row_end, double *dq, double *dkv, double *dckv, int nthreads) {
  if (B < 0 || H < 1 || S < 0 || D < 1 || W < 1 || m < 1) return -2;
  if (!check_rows(S, &row_begin, &row_end)) return -2;
  prob_t P;
  memset(&P, 0, sizeof P);
  if (vis_init(&P.v, seg, B, S, W, m)) return -1;
  P.v.sel = sel;
  P.q = q; P.kv = kv; P.ckv = ckv; P.dout = dout; P.dt = dtype; P.H = H; P.D = D; P.scale = scale;
  P.row_begin = row_begin; P.row_end = row_end; P.dq = dq; P.dkv = dkv; P.dckv = dckv;
  size_t nrow = (size_t)B * H * (S > 0 ? S : 1);
  P.lse_all = (double *)malloc(sizeof(double) * nrow);
  P.delta_all = (double *)malloc(sizeof(double) * nrow);
  uint8_t *need = (uint8_t *)calloc((size_t)B * (S > 0 ? S : 1), 1);
  int rc = -1;
  if (P.lse_all && P.delta_all && need) {
    for (int b = 0; b < B; ++b)
      for (int i = row_begin; i < row_end; ++i) need[(size_t)b * S + i] = 1;
    P.need = need;
    rc = run_pool(bwd_query_task, &P, (long)B * S, keys_scratch(&P), nthreads);
    if (rc == 0)
      rc = run_pool(bwd_key_task, &P, (long)B * S + (long)B * P.v.Sc, 3 * (size_t)D + 16, nthreads);
  }
  free(need);
  free(P.lse_all);
  free(P.delta_all);
  free(P.v.win_id);
  return rc;
}

int hca_oracle_bwd(const void *q, const void *kv, const void *ckv, const int32_t *seg, const void *dout, int dtype,
                   int B, int H, int S, int D, int W, int m, double scale, int row_begin, int row_end,
                   double *dq, double *dkv, double *dckv, int nthreads) {
  return bwd_impl(q, kv, ckv, seg, NULL, dout, dtype, B, H, S, D, W, m, scale, row_begin, row_end, dq, dkv, dckv,
                  nthreads);
}

/* CSA backward: as hca_oracle_bwd, compressed entries also need sel[b,i,j]. */
int hca_oracle_csa_bwd(const void *q, const void *kv, const void *ckv, const int32_t *seg, const uint8_t *sel,
                       const void *dout, int dtype, int B, int H, int S, int D, int W, int m, double scale,
                       int row_begin, int row_end, double *dq, double *dkv, double *dckv, int nthreads) {
  if (!sel) return -2;
  return bwd_impl(q, kv, ckv, seg, sel, dout, dtype, B, H, S, D, W, m, scale, row_begin, row_end, dq, dkv, dckv,
                  nthreads);
}

static void key_list_task(void *ctx, long item, double *scr) {
  const prob_t *P = (const prob_t *)ctx;
  const vis_t *v = &P->v;
  int64_t id = P->key_list[item];
  int per = P->comp_keys ? v->Sc : v->S;
  int b = (int)(id / per), key = (int)(id % per);
  key_grad(P, b, P->comp_keys, key, 0, v->S, P->key_out + (size_t)item * P->D, scr);
}

/* Exact gradient of selected keys over ALL queries: raw rows listed as
 * b*S+t in raw_ids (n_raw of them) into draw[n_raw][D], compressed entries
 * listed as b*Sc+j in comp_ids into dcomp[n_comp][D].  Only the queries that
 * can see a selected key are evaluated. */
int hca_oracle_bwd_keys(const void *q, const void *kv, const void *ckv, const int32_t *seg, const void *dout, int dtype,
                        int B, int H, int S, int D, int W, int m, double scale,
                        const int64_t *raw_ids, int n_raw, const int64_t *comp_ids, int n_comp,
                        double *draw, double *dcomp, int nthreads) {
  if (B < 0 || H < 1 || S < 0 || D < 1 || W < 1 || m < 1 || n_raw < 0 || n_comp < 0) return -2;
  prob_t P;
  memset(&P, 0, sizeof P);
  if (vis_init(&P.v, seg, B, S, W, m)) return -1;
  P.q = q; P.kv = kv; P.ckv = ckv; P.dout = dout; P.dt = dtype; P.H = H; P.D = D; P.scale = scale;
  P.row_begin = 0; P.row_end = S;
  size_t nrow = (size_t)B * H * (S > 0 ? S : 1);
  P.lse_all = (double *)malloc(sizeof(double) * nrow);
  P.delta_all = (double *)malloc(sizeof(double) * nrow);
  uint8_t *need = (uint8_t *)calloc((size_t)B * (S > 0 ? S : 1), 1);
  int rc = -1;
  if (P.lse_all && P.delta_all && need) {
    rc = 0;
    for (int k = 0; k < n_raw && rc == 0; ++k) {
      int64_t id = raw_ids[k];
      if (id < 0 || id >= (int64_t)B * S) { rc = -2; break; }
      int b = (int)(id / S), t = (int)(id % S);
      for (int i = t; i < S && i < t + W; ++i) need[(size_t)b * S + i] = 1;
    }
    for (int k = 0; k < n_comp && rc == 0; ++k) {
      int64_t id = comp_ids[k];
      if (id < 0 || id >= (int64_t)B * P.v.Sc) { rc = -2; break; }
      int b = (int)(id / P.v.Sc), j = (int)(id % P.v.Sc);
      for (int i = (j + 1) * m - 1; i < S; ++i) need[(size_t)b * S + i] = 1;
    }
    if (rc == 0) {
      P.need = need;
      rc = run_pool(bwd_query_task, &P, (long)B * S, keys_scratch(&P), nthreads);
    }
    if (rc == 0 && n_raw > 0) {
      P.key_list = raw_ids; P.key_out = draw; P.comp_keys = 0;
      rc = run_pool(key_list_task, &P, n_raw, 3 * (size_t)D + 16, nthreads);
    }
    if (rc == 0 && n_comp > 0) {
      P.key_list = comp_ids; P.key_out = dcomp; P.comp_keys = 1;
      rc = run_pool(key_list_task, &P, n_comp, 3 * (size_t)D + 16, nthreads);
    }
  }
  free(need);
  free(P.lse_all);
  free(P.delta_all);
  free(P.v.win_id);
  return rc;
}

/* ------------------------------------------------------------------ */
/* visibility enumeration                                               */
/* ------------------------------------------------------------------ */

/* Visible (query, key) pairs of every batch row, per head, counted element
 * by element: raw_pairs[b] over raw rows, comp_pairs[b] over compressed
 * entries. */
static int pairs_impl(const int32_t *seg, const uint8_t *sel, int B, int S, int W, int m, int64_t *raw_pairs,
                      int64_t *comp_pairs) {
  if (B < 0 || S < 0 || W < 1 || m < 1) return -2;
  vis_t v;
  if (vis_init(&v, seg, B, S, W, m)) return -1;
  v.sel = sel;
  for (int b = 0; b < B; ++b) {
    int64_t nr = 0, nc = 0;
    for (int i = 0; i < S; ++i) {
      /* raw t can only satisfy i-W < t <= i: scan exactly that band */
      for (int t = i - W + 1; t <= i; ++t) nr += raw_visible(&v, b, i, t);
      for (int j = 0; j < v.Sc; ++j) nc += comp_visible(&v, b, i, j);
    }
    raw_pairs[b] = nr;
    comp_pairs[b] = nc;
  }
  free(v.win_id);
  return 0;
}

int hca_oracle_visible_pairs(const int32_t *seg, int B, int S, int W, int m, int64_t *raw_pairs, int64_t *comp_pairs) {
  return pairs_impl(seg, NULL, B, S, W, m, raw_pairs, comp_pairs);
}

/* CSA pair counts: compressed pairs also need sel[b,i,j]. */
int hca_oracle_csa_visible_pairs(const int32_t *seg, const uint8_t *sel, int B, int S, int W, int m,
                                 int64_t *raw_pairs, int64_t *comp_pairs) {
  if (!sel) return -2;
  return pairs_impl(seg, sel, B, S, W, m, raw_pairs, comp_pairs);
}

/* For query tiles of Pq consecutive positions, the smallest range of keys
 * that holds every visible pair of the tile:
 *   map[b][tile] = {raw_lo, raw_hi, comp_lo, comp_hi}  (half-open; 0,0 when
 *   the tile sees no key of that kind).  Enumerated element by element. */
int hca_oracle_tile_ranges(const int32_t *seg, int B, int S, int W, int m, int Pq, int32_t *map) {
  if (B < 0 || S < 0 || W < 1 || m < 1 || Pq < 1) return -2;
  vis_t v;
  if (vis_init(&v, seg, B, S, W, m)) return -1;
  int nt = (S + Pq - 1) / Pq;
  for (int b = 0; b < B; ++b)
    for (int tile = 0; tile < nt; ++tile) {
      int rlo = INT32_MAX, rhi = -1, clo = INT32_MAX, chi = -1;
      for (int i = tile * Pq; i < S && i < (tile + 1) * Pq; ++i) {
        for (int t = i - W + 1; t <= i; ++t)
          if (raw_visible(&v, b, i, t)) {
            if (t < rlo) rlo = t;
            if (t > rhi) rhi = t;
          }
        for (int j = 0; j < v.Sc; ++j)
          if (comp_visible(&v, b, i, j)) {
            if (j < clo) clo = j;
            if (j > chi) chi = j;
          }
      }
      int32_t *e = map + ((size_t)b * nt + tile) * 4;
      e[0] = rhi < 0 ? 0 : rlo;
      e[1] = rhi < 0 ? 0 : rhi + 1;
      e[2] = chi < 0 ? 0 : clo;
      e[3] = chi < 0 ? 0 : chi + 1;
    }
  free(v.win_id);
  return 0;
}
