/*
 * oracle.c -- plain, slow fp64 CPU oracle for prefix-tree attention.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may link, load or
 * call this file; only the tests, the smoke check and the benchmark's CPU
 * baseline do.  It shares no code, header, table or helper with the CUDA
 * library.
 *
 * What it computes (each function cites the passage it follows):
 *
 *  - Labels.  A prefix tree is given as node lengths plus root->leaf sample
 *    paths ("cp=1 shared-prefix prefix-tree attention for rollouts": the fold
 *    emits the tree as (node_lengths, sample_paths) and the mask is built with
 *    AttnMaskSpec.prefix_tree).  Node i's tokens sit contiguously, nodes in id
 *    order.  The segment form (per-token group id and suffix id, -1 on prompt
 *    tokens) is "prefix_grouper_kernel.py", PrefixSegInfo.
 *  - keep(q, kv) = node(kv) is node(q) or one of its ancestors, and kv <= q.
 *    For depth 2 this is the mask_mod of "prefix_grouper_kernel.py"
 *    (_make_mask_mod): a completion sees its whole prompt and itself
 *    causally, prompt tokens are causal, nothing crosses groups.
 *  - Block map: each (q tile, kv block) pair is empty, full or partial by
 *    brute-force counting of kept pairs ("prefix_grouper_kernel.py",
 *    get_block_mask / create_block_mask: masked-out blocks are never
 *    computed).
 *  - Forward: exact softmax attention restricted to kept pairs, scale
 *    1/sqrt(head_dim) by default ("prefix_grouper_kernel.py",
 *    flex_shared_prefix_attention), with grouped-query heads (enable_gqa):
 *    q head h reads kv head h / (Hq/Hkv).
 *  - Backward: the gradients of that function, written out from the
 *    definition of softmax attention (the pages give no formula).
 *
 * Arithmetic is fp64 throughout.  Loops follow the definitions directly; the
 * only parallelism is independent rows (or independent kv columns) spread
 * over threads.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define OR_OK 0
#define OR_EINVAL (-1)
#define OR_ENOMEM (-2)

/* ------------------------------------------------------------------------- */
/* A tiny thread pool: run fn(ctx, i) for i in [0, n) over n_threads threads. */
/* ------------------------------------------------------------------------- */
typedef void (*or_task_fn)(void* ctx, int64_t i);
typedef struct {
  or_task_fn fn;
  void* ctx;
  int64_t n;
  int64_t next; /* shared counter */
} or_pool;

static void* or_worker(void* arg) {
  or_pool* p = (or_pool*)arg;
  for (;;) {
    int64_t i = __atomic_fetch_add(&p->next, 1, __ATOMIC_RELAXED);
    if (i >= p->n) break;
    p->fn(p->ctx, i);
  }
  return NULL;
}

static void or_parallel_for(int64_t n, or_task_fn fn, void* ctx, int n_threads) {
  or_pool p = {fn, ctx, n, 0};
  if (n_threads < 1) n_threads = 1;
  if (n_threads > 256) n_threads = 256;
  if (n_threads == 1 || n < 2) {
    or_worker(&p);
    return;
  }
  pthread_t th[256];
  int started = 0;
  for (int t = 0; t < n_threads - 1; ++t) {
    if (pthread_create(&th[t], NULL, or_worker, &p) != 0) break;
    ++started;
  }
  or_worker(&p);
  for (int t = 0; t < started; ++t) pthread_join(th[t], NULL);
}

/* ------------------------------------------------------------------------- */
/* Labels                                                                     */
/* ------------------------------------------------------------------------- */

/* Tree form.  Validates and fills parent[n_nodes] (-1 for a root) and
 * node_of[T] (T = sum of node lengths, which the caller has sized).
 * Rules (fail loudly on anything else): lengths >= 0; every path non-empty,
 * node ids in range; consecutive path entries (a, b) make a the parent of b,
 * consistently across paths; a path starts at a root; a parent has a smaller
 * id than its child (ancestors precede descendants in the flat layout);
 * every node lies on some path. */
int or_tree_labels(int32_t n_nodes, const int32_t* node_lengths, int32_t n_samples,
                   const int32_t* path_ptr, const int32_t* path_nodes, int32_t* parent,
                   int64_t T, int32_t* node_of) {
  if (n_nodes < 0 || n_samples < 0) return OR_EINVAL;
  int64_t total = 0;
  for (int32_t i = 0; i < n_nodes; ++i) {
    if (node_lengths[i] < 0) return OR_EINVAL;
    total += node_lengths[i];
  }
  if (total != T) return OR_EINVAL;
  /* parent[i] = -2 means "not yet seen on any path" */
  for (int32_t i = 0; i < n_nodes; ++i) parent[i] = -2;
  if (path_ptr[0] != 0) return OR_EINVAL;
  for (int32_t s = 0; s < n_samples; ++s) {
    int32_t b = path_ptr[s], e = path_ptr[s + 1];
    if (e <= b) return OR_EINVAL;
    for (int32_t k = b; k < e; ++k) {
      int32_t node = path_nodes[k];
      if (node < 0 || node >= n_nodes) return OR_EINVAL;
      int32_t want = (k == b) ? -1 : path_nodes[k - 1];
      if (want >= node) return OR_EINVAL; /* parent must precede child */
      if (parent[node] == -2)
        parent[node] = want;
      else if (parent[node] != want)
        return OR_EINVAL; /* inconsistent parents */
    }
  }
  for (int32_t i = 0; i < n_nodes; ++i)
    if (parent[i] == -2) return OR_EINVAL; /* node on no path */
  int64_t t = 0;
  for (int32_t i = 0; i < n_nodes; ++i)
    for (int32_t r = 0; r < node_lengths[i]; ++r) node_of[t++] = i;
  return OR_OK;
}

/* Segment form ("prefix_grouper_kernel.py", PrefixSegInfo): every maximal run
 * of tokens with equal (group_id, suffix_id) is one node, numbered in run
 * order.  A run with suffix_id == -1 is its group's prompt and must be the
 * first run of its group; a completion run's parent is its group's prompt
 * run when the group has one, else it is a root.  Group ids and suffix ids
 * must each form one contiguous run (suffix ids are globally unique).
 * Fills node_of[T], parent[<= T] and *n_nodes. */
int or_seg_labels(int64_t T, const int32_t* group_id, const int32_t* suffix_id,
                  int32_t* node_of, int32_t* parent, int32_t* n_nodes_out) {
  int32_t n = 0;
  int32_t cur_group_prompt = -1; /* node id of current group's prompt run */
  for (int64_t t = 0; t < T; ++t) {
    int new_run = (t == 0) || group_id[t] != group_id[t - 1] || suffix_id[t] != suffix_id[t - 1];
    if (suffix_id[t] < -1 || group_id[t] < 0) return OR_EINVAL;
    if (new_run) {
      int new_group = (t == 0) || group_id[t] != group_id[t - 1];
      /* a group id or suffix id must not reappear after its run ended */
      for (int64_t u = 0; u < t; ++u) {
        if (new_group && group_id[u] == group_id[t]) return OR_EINVAL;
        if (suffix_id[t] >= 0 && suffix_id[u] == suffix_id[t]) return OR_EINVAL;
      }
      if (new_group) cur_group_prompt = -1;
      if (suffix_id[t] == -1) {
        if (!new_group) return OR_EINVAL; /* prompt must open its group */
        cur_group_prompt = n;
        parent[n] = -1;
      } else {
        parent[n] = cur_group_prompt;
      }
      ++n;
    }
    node_of[t] = n - 1;
  }
  *n_nodes_out = n;
  return OR_OK;
}

/* keep(q, kv): node(kv) on the ancestor-or-self chain of node(q), kv <= q. */
static int or_keep(const int32_t* node_of, const int32_t* parent, int64_t q, int64_t kv) {
  if (kv > q) return 0;
  int32_t a = node_of[kv];
  for (int32_t n = node_of[q]; n != -1; n = parent[n])
    if (n == a) return 1;
  return 0;
}

void or_dense_mask(int64_t T, const int32_t* node_of, const int32_t* parent, uint8_t* mask) {
  for (int64_t q = 0; q < T; ++q)
    for (int64_t kv = 0; kv < T; ++kv) mask[q * T + kv] = (uint8_t)or_keep(node_of, parent, q, kv);
}

/* Number of kept (q, kv) pairs, per head. */
typedef struct {
  int64_t T;
  const int32_t* node_of;
  const int32_t* parent;
  int64_t* per_row;
} or_count_ctx;

static void or_count_row(void* c, int64_t q) {
  or_count_ctx* x = (or_count_ctx*)c;
  int64_t s = 0;
  for (int64_t kv = 0; kv <= q; ++kv) s += or_keep(x->node_of, x->parent, q, kv);
  x->per_row[q] = s;
}

int64_t or_count_pairs(int64_t T, const int32_t* node_of, const int32_t* parent, int n_threads) {
  int64_t* per_row = (int64_t*)calloc((size_t)(T > 0 ? T : 1), sizeof(int64_t));
  if (!per_row) return -1;
  or_count_ctx c = {T, node_of, parent, per_row};
  or_parallel_for(T, or_count_row, &c, n_threads);
  int64_t s = 0;
  for (int64_t q = 0; q < T; ++q) s += per_row[q];
  free(per_row);
  return s;
}

/* ------------------------------------------------------------------------- */
/* Block map by brute force                                                   */
/* ------------------------------------------------------------------------- */
typedef struct {
  int64_t T;
  int32_t BM, BN, nk;
  const int32_t* node_of;
  const int32_t* parent;
  uint8_t* kinds; /* [nq * nk] */
} or_bm_ctx;

static void or_bm_row(void* c, int64_t i) {
  or_bm_ctx* x = (or_bm_ctx*)c;
  for (int32_t j = 0; j < x->nk; ++j) {
    int64_t kept = 0;
    int all_in_range = 1;
    for (int64_t r = 0; r < x->BM; ++r) {
      int64_t q = i * x->BM + r;
      for (int64_t cc = 0; cc < x->BN; ++cc) {
        int64_t kv = (int64_t)j * x->BN + cc;
        if (q >= x->T || kv >= x->T) {
          all_in_range = 0;
          continue;
        }
        kept += or_keep(x->node_of, x->parent, q, kv);
      }
    }
    uint8_t kind;
    if (kept == 0)
      kind = 0; /* empty */
    else if (all_in_range && kept == (int64_t)x->BM * x->BN)
      kind = 1; /* full */
    else
      kind = 2; /* partial */
    x->kinds[i * x->nk + j] = kind;
  }
}

/* q-major CSR (q_ptr[nq+1], kv_idx, kind; kv ascending within a row) and its
 * kv-major transpose (k_ptr[nk+1], q_idx, kindT; q ascending).  Output arrays
 * must hold nq*nk entries.  Returns nnz through *nnz_out. */
int or_blockmap(int64_t T, const int32_t* node_of, const int32_t* parent, int32_t BM, int32_t BN,
                int32_t* q_ptr, int32_t* kv_idx, uint8_t* kind, int32_t* k_ptr, int32_t* q_idx,
                uint8_t* kindT, int64_t* nnz_out, int n_threads) {
  if (BM <= 0 || BN <= 0 || T < 0) return OR_EINVAL;
  int32_t nq = (int32_t)((T + BM - 1) / BM), nk = (int32_t)((T + BN - 1) / BN);
  uint8_t* kinds = (uint8_t*)calloc((size_t)nq * nk + 1, 1);
  if (!kinds) return OR_ENOMEM;
  or_bm_ctx c = {T, BM, BN, nk, node_of, parent, kinds};
  or_parallel_for(nq, or_bm_row, &c, n_threads);
  int64_t e = 0;
  q_ptr[0] = 0;
  for (int32_t i = 0; i < nq; ++i) {
    for (int32_t j = 0; j < nk; ++j)
      if (kinds[(int64_t)i * nk + j]) {
        kv_idx[e] = j;
        kind[e] = kinds[(int64_t)i * nk + j];
        ++e;
      }
    q_ptr[i + 1] = (int32_t)e;
  }
  int64_t f = 0;
  k_ptr[0] = 0;
  for (int32_t j = 0; j < nk; ++j) {
    for (int32_t i = 0; i < nq; ++i)
      if (kinds[(int64_t)i * nk + j]) {
        q_idx[f] = i;
        kindT[f] = kinds[(int64_t)i * nk + j];
        ++f;
      }
    k_ptr[j + 1] = (int32_t)f;
  }
  *nnz_out = e;
  free(kinds);
  return OR_OK;
}

/* ------------------------------------------------------------------------- */
/* Forward                                                                    */
/* ------------------------------------------------------------------------- */
/* Q [T,Hq,D], K/V [T,Hkv,D], all fp64, token-major.  For row q and head h:
 *   s_j   = scale * sum_d Q[q,h,d] K[j,hk,d]      over kept j
 *   m     = max_j s_j
 *   l     = sum_j exp(s_j - m)
 *   O     = sum_j exp(s_j - m) V[j,hk,:] / l
 *   LSE   = m + log(l)
 * A row with nothing kept (cannot happen for valid input: the diagonal is
 * always kept) gives O = 0 and LSE = -inf. */
typedef struct {
  int64_t T;
  int32_t Hq, Hkv, D;
  double scale;
  const double *Q, *K, *V;
  const int32_t* node_of;
  const int32_t* parent;
  const int64_t* rows; /* NULL: all rows */
  double* O;           /* [n_rows, Hq, D] */
  double* LSE;         /* [Hq, n_rows] */
  int64_t n_rows;
} or_fwd_ctx;

static void or_fwd_one(const or_fwd_ctx* x, int64_t q, int32_t h, double* o_out, double* lse_out,
                       double* s_buf) {
  int32_t g = x->Hq / x->Hkv, hk = h / g, D = x->D;
  const double* qv = x->Q + ((int64_t)q * x->Hq + h) * D;
  double m = -INFINITY;
  for (int64_t j = 0; j <= q; ++j) {
    s_buf[j] = NAN;
    if (!or_keep(x->node_of, x->parent, q, j)) continue;
    const double* kv = x->K + ((int64_t)j * x->Hkv + hk) * D;
    double s = 0.0;
    for (int32_t d = 0; d < D; ++d) s += qv[d] * kv[d];
    s *= x->scale;
    s_buf[j] = s;
    if (s > m) m = s;
  }
  for (int32_t d = 0; d < D; ++d) o_out[d] = 0.0;
  if (m == -INFINITY) {
    *lse_out = -INFINITY;
    return;
  }
  double l = 0.0;
  for (int64_t j = 0; j <= q; ++j) {
    if (isnan(s_buf[j])) continue;
    double p = exp(s_buf[j] - m);
    l += p;
    const double* vv = x->V + ((int64_t)j * x->Hkv + hk) * D;
    for (int32_t d = 0; d < D; ++d) o_out[d] += p * vv[d];
  }
  for (int32_t d = 0; d < D; ++d) o_out[d] /= l;
  *lse_out = m + log(l);
}

static void or_fwd_row(void* c, int64_t r) {
  or_fwd_ctx* x = (or_fwd_ctx*)c;
  int64_t q = x->rows ? x->rows[r] : r;
  double* s_buf = (double*)malloc(sizeof(double) * (size_t)(q + 1));
  for (int32_t h = 0; h < x->Hq; ++h)
    or_fwd_one(x, q, h, x->O + (r * x->Hq + h) * x->D, x->LSE + (int64_t)h * x->n_rows + r, s_buf);
  free(s_buf);
}

int or_attn_fwd(int64_t T, int32_t Hq, int32_t Hkv, int32_t D, double scale, const double* Q,
                const double* K, const double* V, const int32_t* node_of, const int32_t* parent,
                int64_t n_rows, const int64_t* rows, double* O, double* LSE, int n_threads) {
  if (Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0 || D <= 0) return OR_EINVAL;
  if (!rows) n_rows = T;
  for (int64_t r = 0; rows && r < n_rows; ++r)
    if (rows[r] < 0 || rows[r] >= T) return OR_EINVAL;
  if (scale <= 0.0) scale = 1.0 / sqrt((double)D);
  or_fwd_ctx c = {T, Hq, Hkv, D, scale, Q, K, V, node_of, parent, rows, O, LSE, n_rows};
  or_parallel_for(n_rows, or_fwd_row, &c, n_threads);
  return OR_OK;
}

/* ------------------------------------------------------------------------- */
/* Backward                                                                   */
/* ------------------------------------------------------------------------- */
/* With P_ij = exp(s_ij - LSE_i) over kept pairs, dP_ij = dO_i . V_j,
 * Delta_i = dO_i . O_i and dS_ij = P_ij (dP_ij - Delta_i):
 *   dQ_i = scale * sum_j dS_ij K_j
 *   dK_j = scale * sum_{h in group(hk)} sum_i dS_ij Q_i
 *   dV_j =         sum_{h in group(hk)} sum_i P_ij dO_i
 * O and LSE come from this file's own forward.  Output rows/columns may be a
 * subset; every row that sees a requested column is evaluated. */
typedef struct {
  int64_t T;
  int32_t Hq, Hkv, D;
  double scale;
  const double *Q, *K, *V, *dO;
  const int32_t* node_of;
  const int32_t* parent;
  /* per (row, head) statistics, [T * Hq]; need[T] marks rows to evaluate */
  const uint8_t* need;
  double* lse;
  double* delta;
  /* dQ over requested rows */
  const int64_t* qrows;
  int64_t n_qrows;
  double* dQ;
  /* dK/dV over requested columns */
  const int64_t* kvcols;
  int64_t n_kvcols;
  double* dK;
  double* dV;
} or_bwd_ctx;

static void or_bwd_stats_row(void* c, int64_t q) {
  or_bwd_ctx* x = (or_bwd_ctx*)c;
  if (!x->need[q]) return;
  or_fwd_ctx f = {x->T, x->Hq, x->Hkv, x->D, x->scale, x->Q, x->K, x->V, x->node_of, x->parent, NULL, NULL, NULL, 0};
  double* s_buf = (double*)malloc(sizeof(double) * (size_t)(q + 1));
  double* o = (double*)malloc(sizeof(double) * (size_t)x->D);
  for (int32_t h = 0; h < x->Hq; ++h) {
    double lse;
    or_fwd_one(&f, q, h, o, &lse, s_buf);
    const double* dov = x->dO + (q * x->Hq + h) * x->D;
    double dl = 0.0;
    for (int32_t d = 0; d < x->D; ++d) dl += dov[d] * o[d];
    x->lse[q * x->Hq + h] = lse;
    x->delta[q * x->Hq + h] = dl;
  }
  free(o);
  free(s_buf);
}

static double or_dot(const double* a, const double* b, int32_t D) {
  double s = 0.0;
  for (int32_t d = 0; d < D; ++d) s += a[d] * b[d];
  return s;
}

static void or_bwd_dq_row(void* c, int64_t r) {
  or_bwd_ctx* x = (or_bwd_ctx*)c;
  int64_t i = x->qrows ? x->qrows[r] : r;
  int32_t g = x->Hq / x->Hkv, D = x->D;
  for (int32_t h = 0; h < x->Hq; ++h) {
    int32_t hk = h / g;
    double* out = x->dQ + (r * x->Hq + h) * D;
    for (int32_t d = 0; d < D; ++d) out[d] = 0.0;
    const double* qv = x->Q + (i * x->Hq + h) * D;
    const double* dov = x->dO + (i * x->Hq + h) * D;
    double lse = x->lse[i * x->Hq + h], delta = x->delta[i * x->Hq + h];
    for (int64_t j = 0; j <= i; ++j) {
      if (!or_keep(x->node_of, x->parent, i, j)) continue;
      const double* kv = x->K + (j * x->Hkv + hk) * D;
      const double* vv = x->V + (j * x->Hkv + hk) * D;
      double p = exp(x->scale * or_dot(qv, kv, D) - lse);
      double ds = p * (or_dot(dov, vv, D) - delta);
      for (int32_t d = 0; d < D; ++d) out[d] += x->scale * ds * kv[d];
    }
  }
}

static void or_bwd_dkv_col(void* c, int64_t r) {
  or_bwd_ctx* x = (or_bwd_ctx*)c;
  int64_t j = x->kvcols ? x->kvcols[r] : r;
  int32_t g = x->Hq / x->Hkv, D = x->D;
  for (int32_t hk = 0; hk < x->Hkv; ++hk) {
    double* dk = x->dK + (r * x->Hkv + hk) * D;
    double* dv = x->dV + (r * x->Hkv + hk) * D;
    for (int32_t d = 0; d < D; ++d) dk[d] = dv[d] = 0.0;
    const double* kv = x->K + (j * x->Hkv + hk) * D;
    const double* vv = x->V + (j * x->Hkv + hk) * D;
    for (int32_t h = hk * g; h < (hk + 1) * g; ++h) {
      for (int64_t i = j; i < x->T; ++i) {
        if (!or_keep(x->node_of, x->parent, i, j)) continue;
        const double* qv = x->Q + (i * x->Hq + h) * D;
        const double* dov = x->dO + (i * x->Hq + h) * D;
        double p = exp(x->scale * or_dot(qv, kv, D) - x->lse[i * x->Hq + h]);
        double ds = p * (or_dot(dov, vv, D) - x->delta[i * x->Hq + h]);
        for (int32_t d = 0; d < D; ++d) {
          dv[d] += p * dov[d];
          dk[d] += x->scale * ds * qv[d];
        }
      }
    }
  }
}

int or_attn_bwd(int64_t T, int32_t Hq, int32_t Hkv, int32_t D, double scale, const double* Q,
                const double* K, const double* V, const double* dO, const int32_t* node_of,
                const int32_t* parent, int64_t n_qrows, const int64_t* qrows, double* dQ,
                int64_t n_kvcols, const int64_t* kvcols, double* dK, double* dV, int n_threads) {
  if (Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0 || D <= 0) return OR_EINVAL;
  if (scale <= 0.0) scale = 1.0 / sqrt((double)D);
  if (!qrows) n_qrows = T;
  if (!kvcols) n_kvcols = T;
  for (int64_t r = 0; qrows && r < n_qrows; ++r)
    if (qrows[r] < 0 || qrows[r] >= T) return OR_EINVAL;
  for (int64_t r = 0; kvcols && r < n_kvcols; ++r)
    if (kvcols[r] < 0 || kvcols[r] >= T) return OR_EINVAL;
  uint8_t* need = (uint8_t*)calloc((size_t)(T > 0 ? T : 1), 1);
  double* lse = (double*)malloc(sizeof(double) * (size_t)(T > 0 ? T : 1) * Hq);
  double* delta = (double*)malloc(sizeof(double) * (size_t)(T > 0 ? T : 1) * Hq);
  if (!need || !lse || !delta) {
    free(need);
    free(lse);
    free(delta);
    return OR_ENOMEM;
  }
  /* rows whose statistics are needed: requested dQ rows, and every row that
   * keeps a requested kv column */
  for (int64_t r = 0; r < n_qrows; ++r) need[qrows ? qrows[r] : r] = 1;
  for (int64_t r = 0; r < n_kvcols; ++r) {
    int64_t j = kvcols ? kvcols[r] : r;
    for (int64_t i = j; i < T; ++i)
      if (!need[i] && or_keep(node_of, parent, i, j)) need[i] = 1;
  }
  or_bwd_ctx c = {T, Hq, Hkv, D, scale, Q, K, V, dO, node_of, parent, need, lse, delta,
                  qrows, n_qrows, dQ, kvcols, n_kvcols, dK, dV};
  or_parallel_for(T, or_bwd_stats_row, &c, n_threads);
  if (dQ) or_parallel_for(n_qrows, or_bwd_dq_row, &c, n_threads);
  if (dK && dV) or_parallel_for(n_kvcols, or_bwd_dkv_col, &c, n_threads);
  free(need);
  free(lse);
  free(delta);
  return OR_OK;
}
