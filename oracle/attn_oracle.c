/*
 * Exact-attention oracle, fp64, CPU only.
 *
 * TEST INFRASTRUCTURE. Only the test suite, the smoke check and the CPU
 * baseline leg of the benchmark load this library. The product path (the
 * CUDA library and its Python binding) never calls it, and it shares no
 * code, header, table or constant with that path.
 *
 * What it computes (per batch b, head h; Q, O, dO, dQ contiguous [B,H,Nq,d],
 * K, V, dK, dV contiguous [B,H,Nk,d]; Nq query rows i, Nk key rows j):
 *
 *   s_ij  = scale * sum_c Q_ic K_jc                       for j in J(i)
 *   m_i   = max_j s_ij,  l_i = sum_j exp(s_ij - m_i)
 *   P_ij  = exp(s_ij - m_i) / l_i
 *   O_ic  = sum_j P_ij V_jc,   LSE_i = m_i + ln l_i
 *
 * following the standard definition S = QK^T, P = softmax(S), O = PV
 * ("FlashAttention" paper notes, section "What Are We Computing?") with the
 * numerically stable softmax m / f / l of section "Tiling: Block-by-Block
 * Softmax", and the 1/sqrt(d) score scale of the numpy attention_naive in
 * "flash attention" (muhibwaqar.com), section "build it from scratch".
 * The scale is an explicit argument; the worked examples use scale = 1.
 *
 * J(i), the keys query i may see (the pages only say that causal masking is
 * applied per tile and that a block-sparse variant exists, so this is a
 * reading): key j is visible iff (!causal || j <= i + Nk - Nq) and, when a
 * block mask is given, mask[(i / tile) * Tk + (j / tile)] != 0 with
 * Tq = ceil(Nq / tile), Tk = ceil(Nk / tile) and the mask laid out [Tq][Tk].
 * With Nq = Nk the causal rule is the pages' j <= i. With Nq != Nk the pages
 * say nothing; the rule aligns the last query with the last key, so the Nq
 * queries are the last Nq positions of a sequence of Nk keys (queries that
 * come before every key, i < Nq - Nk, see nothing).
 * A row with no visible key gets O_i = 0 and LSE_i = -inf.
 *
 * The backward pass is not written out on the pages (the aicassindra page,
 * section "The backward pass: recompute instead of store", defers it to a
 * companion article that is not available). It is the analytic gradient of
 * the definition above for an upstream gradient dO:
 *
 *   dV_j  = sum_i P_ij dO_i
 *   dP_ij = dO_i . V_j
 *   D_i   = sum_j P_ij dP_ij
 *   dS_ij = P_ij (dP_ij - D_i)            (0 for j not in J(i))
 *   dQ_i  = scale * sum_j dS_ij K_j
 *   dK_j  = scale * sum_i dS_ij Q_i
 *
 * evaluated row by row (dQ, LSE, D) and then key by key (dK, dV), so that
 * every output element is owned by one work item and the threads never
 * reduce into shared buffers.
 *
 * The second forward entry point, oracle_forward_tiled, is the online
 * softmax recurrence (running max m, running sum l, unnormalised
 * accumulator, one division at the end) of the numpy flash_attention in
 * "flash attention" (muhibwaqar.com), section "build it from scratch", and
 * of the aicassindra page, section "Rescale and accumulate: the forward pass
 * in one loop". It exists to pin that recurrence against the definition.
 */
#include <math.h>
#include <pthread.h>
#include <stddef.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_OK 0
#define ORACLE_ERR_ARG 1
#define ORACLE_ERR_NOMEM 2

typedef struct {
  int B, H, Nq, Nk, d;
  int causal;
  double scale;
  const unsigned char *mask; /* [Tq][Tk] or NULL */
  int tile;                  /* edge of one mask tile, in rows */
  int Tq, Tk;                /* mask tiles along the queries and along the keys */
} attn_shape;

static int key_visible(const attn_shape *sh, int i, int j) {
  if (sh->causal && (long)j > (long)i + (long)sh->Nk - (long)sh->Nq) return 0;
  if (sh->mask && !sh->mask[(size_t)(i / sh->tile) * (size_t)sh->Tk + (size_t)(j / sh->tile)])
    return 0;
  return 1;
}

static double dot(const double *a, const double *b, int n) {
  double acc = 0.0;
  for (int c = 0; c < n; ++c) acc += a[c] * b[c];
  return acc;
}

/* ------------------------------------------------------------------------ */
/* A small static thread pool: items [0, n) are dealt round-robin.            */

typedef void (*item_fn)(void *ctx, long item, double *scratch);

typedef struct {
  item_fn fn;
  void *ctx;
  long n_items;
  int n_threads;
  int tid;
  size_t scratch_len;
  int failed;
} worker_arg;

static void *worker_main(void *p) {
  worker_arg *w = (worker_arg *)p;
  double *scratch = (double *)malloc(w->scratch_len * sizeof(double) + 1);
  if (!scratch) {
    w->failed = 1;
    return NULL;
  }
  for (long it = w->tid; it < w->n_items; it += w->n_threads) w->fn(w->ctx, it, scratch);
  free(scratch);
  return NULL;
}

static int run_items(item_fn fn, void *ctx, long n_items, int n_threads, size_t scratch_len) {
  if (n_items <= 0) return ORACLE_OK;
  if (n_threads < 1) n_threads = 1;
  if (n_threads > n_items) n_threads = (int)n_items;
  pthread_t *th = (pthread_t *)malloc(sizeof(pthread_t) * (size_t)n_threads);
  worker_arg *args = (worker_arg *)malloc(sizeof(worker_arg) * (size_t)n_threads);
  if (!th || !args) {
    free(th);
    free(args);
    return ORACLE_ERR_NOMEM;
  }
  int failed = 0;
  for (int t = 0; t < n_threads; ++t) {
    args[t].fn = fn;
    args[t].ctx = ctx;
    args[t].n_items = n_items;
    args[t].n_threads = n_threads;
    args[t].tid = t;
    args[t].scratch_len = scratch_len;
    args[t].failed = 0;
  }
  int started = 0;
  for (int t = 1; t < n_threads; ++t) {
    if (pthread_create(&th[t], NULL, worker_main, &args[t]) != 0) break;
    started = t;
  }
  /* Thread 0 runs on the caller; items of threads that failed to start are
   * picked up serially below so that every item still runs exactly once. */
  worker_main(&args[0]);
  for (int t = 1; t <= started; ++t) pthread_join(th[t], NULL);
  for (int t = started + 1; t < n_threads; ++t) worker_main(&args[t]);
  for (int t = 0; t < n_threads; ++t) failed |= args[t].failed;
  free(th);
  free(args);
  return failed ? ORACLE_ERR_NOMEM : ORACLE_OK;
}

static int check_shape(const attn_shape *sh) {
  if (sh->B < 0 || sh->H < 0 || sh->Nq < 0 || sh->Nk < 0 || sh->d <= 0) return ORACLE_ERR_ARG;
  if (sh->mask && sh->tile <= 0) return ORACLE_ERR_ARG;
  return ORACLE_OK;
}

static attn_shape make_shape(int B, int H, int Nq, int Nk, int d, int causal, double scale,
                             const unsigned char *mask, int tile) {
  attn_shape sh;
  sh.B = B;
  sh.H = H;
  sh.Nq = Nq;
  sh.Nk = Nk;
  sh.d = d;
  sh.causal = causal;
  sh.scale = scale;
  sh.mask = mask;
  sh.tile = tile > 0 ? tile : 1;
  sh.Tq = (Nq + sh.tile - 1) / sh.tile;
  sh.Tk = (Nk + sh.tile - 1) / sh.tile;
  return sh;
}

/* ------------------------------------------------------------------------ */
/* Forward, straight from the definition, one query row at a time.           */

typedef struct {
  attn_shape sh;
  const double *Q, *K, *V;
  double *O, *LSE;
  const int *rows; /* query rows to compute; NULL = all */
  int n_rows;
} fwd_ctx;

/* Scores of row i against every visible key: s[j] (unused entries untouched),
 * vis[j] flags; returns the row max (or -inf when no key is visible). */
static double score_row(const attn_shape *sh, const double *Qh, const double *Kh, int i,
                        double *s, unsigned char *vis) {
  const int Nk = sh->Nk, d = sh->d;
  double m = -INFINITY;
  for (int j = 0; j < Nk; ++j) {
    vis[j] = (unsigned char)key_visible(sh, i, j);
    if (!vis[j]) continue;
    s[j] = sh->scale * dot(Qh + (size_t)i * d, Kh + (size_t)j * d, d);
    if (s[j] > m) m = s[j];
  }
  return m;
}

static void fwd_item(void *p, long item, double *scratch) {
  fwd_ctx *c = (fwd_ctx *)p;
  const attn_shape *sh = &c->sh;
  const int Nk = sh->Nk, d = sh->d;
  const long bh = item / c->n_rows;
  const int r = (int)(item % c->n_rows);
  const int i = c->rows ? c->rows[r] : r;
  const double *Qh = c->Q + (size_t)bh * (size_t)sh->Nq * (size_t)d;
  const double *Kh = c->K + (size_t)bh * (size_t)Nk * (size_t)d;
  const double *Vh = c->V + (size_t)bh * (size_t)Nk * (size_t)d;
  double *s = scratch;
  unsigned char *vis = (unsigned char *)(scratch + Nk);
  double *o = c->O + ((size_t)bh * (size_t)c->n_rows + (size_t)r) * (size_t)d;
  double *lse = c->LSE + (size_t)bh * (size_t)c->n_rows + (size_t)r;

  const double m = score_row(sh, Qh, Kh, i, s, vis);
  for (int x = 0; x < d; ++x) o[x] = 0.0;
  if (m == -INFINITY) { /* no visible key */
    *lse = -INFINITY;
    return;
  }
  double l = 0.0;
  for (int j = 0; j < Nk; ++j)
    if (vis[j]) l += exp(s[j] - m);
  for (int j = 0; j < Nk; ++j) {
    if (!vis[j]) continue;
    const double pij = exp(s[j] - m) / l;
    const double *vj = Vh + (size_t)j * d;
    for (int x = 0; x < d; ++x) o[x] += pij * vj[x];
  }
  *lse = m + log(l);
}

/* O and LSE for the query rows `rows` (all Nq rows when rows == NULL), laid
 * out [B,H,n_rows,d] and [B,H,n_rows]. */
int oracle_forward(const double *Q, const double *K, const double *V, double *O, double *LSE,
                   int B, int H, int Nq, int Nk, int d, int causal, double scale,
                   const unsigned char *block_mask, int mask_tile, const int *rows, int n_rows,
                   int n_threads) {
  fwd_ctx c;
  c.sh = make_shape(B, H, Nq, Nk, d, causal, scale, block_mask, mask_tile);
  if (check_shape(&c.sh) != ORACLE_OK) return ORACLE_ERR_ARG;
  c.Q = Q;
  c.K = K;
  c.V = V;
  c.O = O;
  c.LSE = LSE;
  c.rows = rows;
  c.n_rows = rows ? n_rows : Nq;
  if (rows)
    for (int r = 0; r < n_rows; ++r)
      if (rows[r] < 0 || rows[r] >= Nq) return ORACLE_ERR_ARG;
  /* scratch: s[Nk] doubles + vis[Nk] bytes */
  return run_items(fwd_item, &c, (long)B * H * c.n_rows, n_threads,
                   (size_t)Nk + (size_t)Nk / 8 + 2);
}

/* ------------------------------------------------------------------------ */
/* Forward by the online-softmax recurrence over Bq x Bk blocks.             */

typedef struct {
  attn_shape sh;
  const double *Q, *K, *V;
  double *O, *LSE;
  int bq, bk;
  int n_qblocks;
} tiled_ctx;

static void tiled_item(void *p, long item, double *scratch) {
  tiled_ctx *c = (tiled_ctx *)p;
  const attn_shape *sh = &c->sh;
  const int Nq = sh->Nq, Nk = sh->Nk, d = sh->d, bq = c->bq, bk = c->bk;
  const long bh = item / c->n_qblocks;
  const int i0 = (int)(item % c->n_qblocks) * bq;
  const int rows = (i0 + bq <= Nq) ? bq : Nq - i0;
  const size_t qhead = (size_t)bh * (size_t)Nq * (size_t)d;
  const size_t khead = (size_t)bh * (size_t)Nk * (size_t)d;
  const double *Qh = c->Q + qhead, *Kh = c->K + khead, *Vh = c->V + khead;

  double *m = scratch;             /* running max        [bq]     */
  double *l = m + bq;              /* running sum        [bq]     */
  double *acc = l + bq;            /* running output     [bq][d]  */
  double *s = acc + (size_t)bq * d; /* one score tile    [bq][bk] */
  double *pt = s + (size_t)bq * bk; /* its exponentials  [bq][bk] */

  for (int r = 0; r < rows; ++r) {
    m[r] = -INFINITY;
    l[r] = 0.0;
    for (int x = 0; x < d; ++x) acc[(size_t)r * d + x] = 0.0;
  }
  for (int j0 = 0; j0 < Nk; j0 += bk) {
    const int cols = (j0 + bk <= Nk) ? bk : Nk - j0;
    for (int r = 0; r < rows; ++r) {
      const int i = i0 + r;
      /* s = (q @ k.T) * scale on this tile, hidden keys held at -inf */
      double tile_max = -INFINITY;
      for (int cc = 0; cc < cols; ++cc) {
        const int j = j0 + cc;
        double v = -INFINITY;
        if (key_visible(sh, i, j)) v = sh->scale * dot(Qh + (size_t)i * d, Kh + (size_t)j * d, d);
        s[(size_t)r * bk + cc] = v;
        if (v > tile_max) tile_max = v;
      }
      const double m_new = (tile_max > m[r]) ? tile_max : m[r];
      if (m_new == -INFINITY) continue; /* nothing seen yet in this row */
      /* p = exp(s - m_new); a = exp(m - m_new) */
      double psum = 0.0;
      for (int cc = 0; cc < cols; ++cc) {
        const double v = s[(size_t)r * bk + cc];
        const double e = (v == -INFINITY) ? 0.0 : exp(v - m_new);
        pt[(size_t)r * bk + cc] = e;
        psum += e;
      }
      const double a = (m[r] == -INFINITY) ? 0.0 : exp(m[r] - m_new);
      /* l = a*l + rowsum(p); acc = a*acc + p @ v; m = m_new */
      l[r] = a * l[r] + psum;
      for (int x = 0; x < d; ++x) {
        double pv = 0.0;
        for (int cc = 0; cc < cols; ++cc)
          pv += pt[(size_t)r * bk + cc] * Vh[(size_t)(j0 + cc) * d + x];
        acc[(size_t)r * d + x] = a * acc[(size_t)r * d + x] + pv;
      }
      m[r] = m_new;
    }
  }
  for (int r = 0; r < rows; ++r) {
    double *o = c->O + qhead + (size_t)(i0 + r) * d;
    double *lse = c->LSE + (size_t)bh * Nq + (size_t)(i0 + r);
    if (l[r] == 0.0) {
      for (int x = 0; x < d; ++x) o[x] = 0.0;
      *lse = -INFINITY;
      continue;
    }
    for (int x = 0; x < d; ++x) o[x] = acc[(size_t)r * d + x] / l[r]; /* normalise at the end */
    *lse = m[r] + log(l[r]);
  }
}

int oracle_forward_tiled(const double *Q, const double *K, const double *V, double *O,
                         double *LSE, int B, int H, int Nq, int Nk, int d, int causal,
                         double scale, const unsigned char *block_mask, int mask_tile, int bq,
                         int bk, int n_threads) {
  tiled_ctx c;
  c.sh = make_shape(B, H, Nq, Nk, d, causal, scale, block_mask, mask_tile);
  if (check_shape(&c.sh) != ORACLE_OK || bq <= 0 || bk <= 0) return ORACLE_ERR_ARG;
  c.Q = Q;
  c.K = K;
  c.V = V;
  c.O = O;
  c.LSE = LSE;
  c.bq = bq;
  c.bk = bk;
  c.n_qblocks = (Nq + bq - 1) / bq;
  const size_t scratch = (size_t)2 * bq + (size_t)bq * d + (size_t)2 * bq * bk;
  return run_items(tiled_item, &c, (long)B * H * c.n_qblocks, n_threads, scratch);
}

/* ------------------------------------------------------------------------ */
/* Backward: analytic gradients of the definition.                           */

typedef struct {
  attn_shape sh;
  const double *Q, *K, *V, *dO;
  double *dQ, *dK, *dV;
  double *lse_all, *D_all; /* [B*H][Nq] statistics of every query row */
  const int *qrows;
  int n_q;
  const int *kcols;
  int n_k;
} bwd_ctx;

/* Pass 1, one query row: LSE_i and D_i (stored when `store_stats`) and, if
 * dq_out is given, dQ_i. */
static void bwd_row(bwd_ctx *c, long bh, int i, int store_stats, double *dq_out,
                    double *scratch) {
  const attn_shape *sh = &c->sh;
  const int Nq = sh->Nq, Nk = sh->Nk, d = sh->d;
  const size_t qhead = (size_t)bh * (size_t)Nq * (size_t)d;
  const size_t khead = (size_t)bh * (size_t)Nk * (size_t)d;
  const double *Qh = c->Q + qhead, *dOh = c->dO + qhead;
  const double *Kh = c->K + khead, *Vh = c->V + khead;
  double *s = scratch;       /* scores, then P           [Nk] */
  double *dp = scratch + Nk; /* dP                        [Nk] */
  unsigned char *vis = (unsigned char *)(scratch + 2 * (size_t)Nk);

  const double m = score_row(sh, Qh, Kh, i, s, vis);
  double *lse = c->lse_all + (size_t)bh * Nq + i;
  double *Dd = c->D_all + (size_t)bh * Nq + i;
  if (m == -INFINITY) {
    if (store_stats) {
      *lse = -INFINITY;
      *Dd = 0.0;
    }
    if (dq_out)
      for (int x = 0; x < d; ++x) dq_out[x] = 0.0;
    return;
  }
  double l = 0.0;
  for (int j = 0; j < Nk; ++j)
    if (vis[j]) l += exp(s[j] - m);
  double D = 0.0;
  for (int j = 0; j < Nk; ++j) {
    if (!vis[j]) continue;
    s[j] = exp(s[j] - m) / l;                                          /* P_ij  */
    dp[j] = dot(dOh + (size_t)i * d, Vh + (size_t)j * d, d);           /* dP_ij */
    D += s[j] * dp[j];
  }
  if (store_stats) {
    *lse = m + log(l);
    *Dd = D;
  }
  if (!dq_out) return;
  for (int x = 0; x < d; ++x) dq_out[x] = 0.0;
  for (int j = 0; j < Nk; ++j) {
    if (!vis[j]) continue;
    const double ds = s[j] * (dp[j] - D);
    const double *kj = Kh + (size_t)j * d;
    for (int x = 0; x < d; ++x) dq_out[x] += ds * kj[x];
  }
  for (int x = 0; x < d; ++x) dq_out[x] *= sh->scale;
}

static void bwd_stats_item(void *p, long item, double *scratch) {
  bwd_ctx *c = (bwd_ctx *)p;
  const int Nq = c->sh.Nq;
  const long bh = item / Nq;
  const int i = (int)(item % Nq);
  bwd_row(c, bh, i, 1, NULL, scratch);
}

static void bwd_dq_item(void *p, long item, double *scratch) {
  bwd_ctx *c = (bwd_ctx *)p;
  const long bh = item / c->n_q;
  const int r = (int)(item % c->n_q);
  const int i = c->qrows ? c->qrows[r] : r;
  bwd_row(c, bh, i, 0, c->dQ + ((size_t)bh * c->n_q + r) * (size_t)c->sh.d, scratch);
}

/* Pass 2, one key row: dK_j and dV_j from the row statistics of pass 1. */
static void bwd_key_item(void *p, long item, double *scratch) {
  bwd_ctx *c = (bwd_ctx *)p;
  const attn_shape *sh = &c->sh;
  const int Nq = sh->Nq, Nk = sh->Nk, d = sh->d;
  const long bh = item / c->n_k;
  const int r = (int)(item % c->n_k);
  const int j = c->kcols ? c->kcols[r] : r;
  const size_t qhead = (size_t)bh * (size_t)Nq * (size_t)d;
  const size_t khead = (size_t)bh * (size_t)Nk * (size_t)d;
  const double *Qh = c->Q + qhead, *dOh = c->dO + qhead;
  const double *Kh = c->K + khead, *Vh = c->V + khead;
  double *dk = c->dK + ((size_t)bh * c->n_k + r) * (size_t)d;
  double *dv = c->dV + ((size_t)bh * c->n_k + r) * (size_t)d;
  (void)scratch;
  for (int x = 0; x < d; ++x) {
    dk[x] = 0.0;
    dv[x] = 0.0;
  }
  for (int i = 0; i < Nq; ++i) {
    if (!key_visible(sh, i, j)) continue;
    const double lse = c->lse_all[(size_t)bh * Nq + i];
    const double D = c->D_all[(size_t)bh * Nq + i];
    const double pij = exp(sh->scale * dot(Qh + (size_t)i * d, Kh + (size_t)j * d, d) - lse);
    const double dpij = dot(dOh + (size_t)i * d, Vh + (size_t)j * d, d);
    const double ds = pij * (dpij - D);
    const double *qi = Qh + (size_t)i * d, *doi = dOh + (size_t)i * d;
    for (int x = 0; x < d; ++x) {
      dv[x] += pij * doi[x];
      dk[x] += ds * qi[x];
    }
  }
  for (int x = 0; x < d; ++x) dk[x] *= sh->scale;
}

/* dQ for the query rows `qrows` ([B,H,n_q,d]; all Nq rows when qrows == NULL),
 * dK and dV for the key rows `kcols` ([B,H,n_k,d]; all Nk when kcols == NULL),
 * and, when lse_out / D_out are given, LSE_i and D_i of every query row
 * [B,H,Nq]. Set n_q = 0 (with qrows != NULL) or n_k = 0 to skip that part. */
int oracle_backward(const double *Q, const double *K, const double *V, const double *dO,
                    double *dQ, double *dK, double *dV, double *lse_out, double *D_out, int B,
                    int H, int Nq, int Nk, int d, int causal, double scale,
                    const unsigned char *block_mask, int mask_tile, const int *qrows, int n_q,
                    const int *kcols, int n_k, int n_threads) {
  bwd_ctx c;
  c.sh = make_shape(B, H, Nq, Nk, d, causal, scale, block_mask, mask_tile);
  if (check_shape(&c.sh) != ORACLE_OK) return ORACLE_ERR_ARG;
  c.Q = Q;
  c.K = K;
  c.V = V;
  c.dO = dO;
  c.dQ = dQ;
  c.dK = dK;
  c.dV = dV;
  c.qrows = qrows;
  c.n_q = qrows ? n_q : Nq;
  c.kcols = kcols;
  c.n_k = kcols ? n_k : Nk;
  if (qrows)
    for (int r = 0; r < n_q; ++r)
      if (qrows[r] < 0 || qrows[r] >= Nq) return ORACLE_ERR_ARG;
  if (kcols)
    for (int r = 0; r < n_k; ++r)
      if (kcols[r] < 0 || kcols[r] >= Nk) return ORACLE_ERR_ARG;
  const size_t nstat = (size_t)B * H * Nq;
  c.lse_all = lse_out ? lse_out : (double *)malloc(sizeof(double) * (nstat + 1));
  c.D_all = D_out ? D_out : (double *)malloc(sizeof(double) * (nstat + 1));
  int rc = ORACLE_OK;
  if (!c.lse_all || !c.D_all) rc = ORACLE_ERR_NOMEM;
  const size_t row_scratch = 2 * (size_t)Nk + (size_t)Nk / 8 + 2;
  /* statistics of every row are needed by the key pass and by the caller */
  if (rc == ORACLE_OK && (c.n_k > 0 || lse_out || D_out))
    rc = run_items(bwd_stats_item, &c, (long)B * H * Nq, n_threads, row_scratch);
  if (rc == ORACLE_OK && c.n_q > 0)
    rc = run_items(bwd_dq_item, &c, (long)B * H * c.n_q, n_threads, row_scratch);
  if (rc == ORACLE_OK && c.n_k > 0)
    rc = run_items(bwd_key_item, &c, (long)B * H * c.n_k, n_threads, 1);
  if (!lse_out) free(c.lse_all);
  if (!D_out) free(c.D_all);
  return rc;
}
