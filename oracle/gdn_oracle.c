/*
 * gdn_oracle.c -- plain fp64 CPU oracle for the Gated DeltaNet tail-replay
 * state rebuild and the chunk-operator composition.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may call, link or
 * load this file: only the tests, the smoke check and the CPU-baseline leg of
 * the benchmark use it.  It shares no code, header, table or helper with the
 * CUDA library; the two meet only in the seeded inputs.
 *
 * What it computes (sources, by page and equation):
 *
 *  - "Tail-Replay: Escaping the Curse of Linear Attention in Prefix Caching
 *    for Hybrid LLMs", section 2, Eq. (1): the GDN update
 *        S_i = T_i S_{i-1} + beta_i v_i k_i^T,  T_i = alpha_i (I - beta_i k_i k_i^T),
 *    alpha_i in (0, 1].  Section 3, Eq. (2): the replay starts from a zero
 *    state at the beginning of the tail and applies Eq. (1) to each tail
 *    token; the final state is the rebuilt state.
 *    Reading: the state is stored as S in R^{d_v x d_k} (row-major), and the
 *    update is applied as S_i = S_{i-1} T_i + beta_i v_i k_i^T.  This is Eq. (1)
 *    on the transposed state; the two agree because every T_i is symmetric.
 *    Readout (not on the pages; the plainest reading): o_i = S_i (scale * q_i),
 *    with the post-update state.
 *  - "LinearKV: One Cached State Suffices for Position-Independent Caching in
 *    Hybrid LLMs", the composition passage: a chunk C maps an entering state
 *    S_in to T_C S_in + S_local, with T_C the product of the per-token T_t of
 *    the chunk (latest on the left) and S_local the state the chunk reaches
 *    from an empty start; K chunks compose in closed form as
 *        S_K = T_{C_K} ... T_{C_2} S_local_1 + ... + T_{C_K} S_local_{K-1} + S_local_K
 *    (pages' left form, i.e. on the transposed state here).
 *
 * Optional per-token L2 normalisation of q and k (a flag): x / sqrt(sum x^2 + 1e-6),
 * applied before use, in fp64.
 *
 * Scalar-decay family (a flag): the LinearKV page sets beside GDN the Mamba-2
 * family, whose per-token transition is a scalar, so a chunk's transition is a
 * single scalar decay.  Reading: T_t = alpha_t I, i.e. the same update without
 * the rank-1 projection term,
 *     S_i = alpha_i S_{i-1} + beta_i v_i k_i^T,
 * with the same readout; its chunk transition is (prod alpha_t) I.
 *
 * Everything is fp64; inputs arrive already widened to fp64 by the caller.
 * Threads split independent (sequence, head) problems only; each problem is
 * the plain token loop.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

typedef struct {
  int64_t n_seqs;   /* number of packed sequences (replay tails) */
  int64_t h_k;      /* q/k heads */
  int64_t h_v;      /* v heads; h_v is a multiple of h_k */
  int64_t d_k;      /* key (and query) head dim */
  int64_t d_v;      /* value head dim */
  int32_t l2norm_qk;/* 1: normalise q and k per (token, head) before use */
  int32_t n_threads;/* 0: all online cores */
  double scale;     /* multiplies q in the readout */
  int32_t scalar_decay; /* 1: Mamba-2 family, scalar per-token transition T_t = alpha_t I */
} gdn_oracle_dims;

/* ------------------------------------------------------------------ */
/* a tiny parallel-for over independent items                        */
/* ------------------------------------------------------------------ */
typedef void (*item_fn)(void* ctx, int64_t item);
typedef struct {
  item_fn fn;
  void* ctx;
  int64_t n_items;
  int64_t next;
  pthread_mutex_t mu;
} pool_t;

static void* pool_worker(void* arg) {
  pool_t* p = (pool_t*)arg;
  for (;;) {
    pthread_mutex_lock(&p->mu);
    int64_t it = p->next++;
    pthread_mutex_unlock(&p->mu);
    if (it >= p->n_items) break;
    p->fn(p->ctx, it);
  }
  return NULL;
}

static int resolve_threads(int32_t n) {
  if (n > 0) return n;
  long c = sysconf(_SC_NPROCESSORS_ONLN);
  return c > 0 ? (int)c : 1;
}

static void parallel_for(int n_threads, int64_t n_items, item_fn fn, void* ctx) {
  pool_t p;
  p.fn = fn; p.ctx = ctx; p.n_items = n_items; p.next = 0;
  pthread_mutex_init(&p.mu, NULL);
  if (n_threads > n_items) n_threads = (int)(n_items > 0 ? n_items : 1);
  if (n_threads <= 1) {
    pool_worker(&p);
  } else {
    pthread_t* th = (pthread_t*)malloc(sizeof(pthread_t) * (size_t)n_threads);
    for (int i = 0; i < n_threads; ++i) pthread_create(&th[i], NULL, pool_worker, &p);
    for (int i = 0; i < n_threads; ++i) pthread_join(th[i], NULL);
    free(th);
  }
  pthread_mutex_destroy(&p.mu);
}

int gdn_oracle_num_threads(int32_t requested) { return resolve_threads(requested); }

/* ------------------------------------------------------------------ */
/* the token loop of Eq. (1) / Eq. (2)                                 */
/* ------------------------------------------------------------------ */

/* out = x / sqrt(sum x^2 + 1e-6) */
static void l2_normalise(const double* x, int64_t n, double* out) {
  double ss = 0.0;
  for (int64_t i = 0; i < n; ++i) ss += x[i] * x[i];
  double r = 1.0 / sqrt(ss + 1e-6);
  for (int64_t i = 0; i < n; ++i) out[i] = x[i] * r;
}

/*
 * One (sequence, v-head) replay over tokens [t0, t1).
 *   S (d_v x d_k) starts from S0 (or zero), then for each token t:
 *     alpha = exp(g_t); S <- alpha * S (I - beta k k^T) + beta v k^T
 *   which, with sk = S k (using the state before the update), is
 *     S[i][j] <- alpha * S[i][j] - alpha * beta * sk[i] * k[j] + beta * v[i] * k[j].
 *   If O is given, o_t = S_t (scale * q_t) with the updated state.
 * Layouts: q,k [T][h_k][d_k]; v, O [T][h_v][d_v]; g, beta [T][h_v].
 */
static void replay_one(const gdn_oracle_dims* d, const double* q, const double* k, const double* v,
                       const double* g, const double* beta, int64_t t0, int64_t t1, int64_t hv,
                       const double* S0, double* S, double* O) {
  const int64_t dk = d->d_k, dv = d->d_v;
  const int64_t group = d->h_v / d->h_k;
  const int64_t hk = hv / group;
  double* kt = (double*)malloc(sizeof(double) * (size_t)dk);
  double* qt = (double*)malloc(sizeof(double) * (size_t)dk);
  double* sk = (double*)malloc(sizeof(double) * (size_t)dv);
  if (S0) memcpy(S, S0, sizeof(double) * (size_t)(dv * dk));
  else memset(S, 0, sizeof(double) * (size_t)(dv * dk));
  for (int64_t t = t0; t < t1; ++t) {
    const double* kin = k + (t * d->h_k + hk) * dk;
    const double* qin = q + (t * d->h_k + hk) * dk;
    const double* vt = v + (t * d->h_v + hv) * dv;
    if (d->l2norm_qk) {
      l2_normalise(kin, dk, kt);
      l2_normalise(qin, dk, qt);
    } else {
      memcpy(kt, kin, sizeof(double) * (size_t)dk);
      memcpy(qt, qin, sizeof(double) * (size_t)dk);
    }
    const double alpha = exp(g[t * d->h_v + hv]);
    const double b = beta[t * d->h_v + hv];
    for (int64_t i = 0; i < dv; ++i) {
      double acc = 0.0;
      for (int64_t j = 0; j < dk; ++j) acc += S[i * dk + j] * kt[j];
      sk[i] = acc;
    }
    for (int64_t i = 0; i < dv; ++i) {
      for (int64_t j = 0; j < dk; ++j) {
        S[i * dk + j] = d->scalar_decay ? alpha * S[i * dk + j] + b * vt[i] * kt[j]
                                        : alpha * S[i * dk + j] - alpha * b * sk[i] * kt[j] + b * vt[i] * kt[j];
      }
    }
    if (O) {
      double* ot = O + (t * d->h_v + hv) * dv;
      for (int64_t i = 0; i < dv; ++i) {
        double acc = 0.0;
        for (int64_t j = 0; j < dk; ++j) acc += S[i * dk + j] * (d->scale * qt[j]);
        ot[i] = acc;
      }
    }
  }
  free(kt); free(qt); free(sk);
}

typedef struct {
  const gdn_oracle_dims* d;
  const double *q, *k, *v, *g, *beta, *S0;
  const int64_t* cu;
  double *O, *S_out;
  const int64_t* sel; /* pairs (seq, hv) or NULL */
} replay_ctx;

static void replay_item(void* vctx, int64_t item) {
  replay_ctx* c = (replay_ctx*)vctx;
  int64_t s, hv;
  if (c->sel) { s = c->sel[2 * item]; hv = c->sel[2 * item + 1]; }
  else { s = item / c->d->h_v; hv = item % c->d->h_v; }
  const int64_t st = c->d->d_v * c->d->d_k;
  const double* S0 = c->S0 ? c->S0 + (s * c->d->h_v + hv) * st : NULL;
  replay_one(c->d, c->q, c->k, c->v, c->g, c->beta, c->cu[s], c->cu[s + 1], hv, S0,
             c->S_out + (s * c->d->h_v + hv) * st, c->O);
}

/*
 * Replay every (sequence, v-head) pair, or only the n_sel pairs listed in sel
 * (sel[2i] = sequence, sel[2i+1] = v-head).  O may be NULL (state only); when
 * given, only the rows of the selected pairs are written.  S_out is
 * [n_seqs][h_v][d_v][d_k]; with sel, only the selected blocks are written.
 * Returns 0, or -1 on bad dims.
 */
int gdn_oracle_replay(const gdn_oracle_dims* d, const double* q, const double* k, const double* v,
                      const double* g, const double* beta, const int64_t* cu_seqlens,
                      const double* S0, double* O, double* S_out, const int64_t* sel, int64_t n_sel) {
  if (!d || d->h_k <= 0 || d->h_v <= 0 || d->h_v % d->h_k != 0 || d->d_k <= 0 || d->d_v <= 0) return -1;
  replay_ctx c = {d, q, k, v, g, beta, S0, cu_seqlens, O, S_out, sel};
  int64_t n = sel ? n_sel : d->n_seqs * d->h_v;
  parallel_for(resolve_threads(d->n_threads), n, replay_item, &c);
  return 0;
}

/* ------------------------------------------------------------------ */
/* chunk operator: T_C and S_local of one chunk                        */
/* ------------------------------------------------------------------ */

/*
 * T_C = T_{t_n} ... T_{t_1} for the tokens of one chunk, built by multiplying
 * each new transition onto the left of the running product:
 *   Tc <- T_t Tc,   T_t = alpha_t (I - beta_t k_t k_t^T),
 * where T_t Tc is evaluated from T_t's definition as
 *   alpha_t (Tc - beta_t k_t (k_t^T Tc)).
 * Scalar-decay family: T_t = alpha_t I, so Tc <- alpha_t Tc.
 */
static void transition_product(const gdn_oracle_dims* d, const double* k, const double* g,
                               const double* beta, int64_t t0, int64_t t1, int64_t hv, double* Tc) {
  const int64_t dk = d->d_k;
  const int64_t hk = hv / (d->h_v / d->h_k);
  double* kt = (double*)malloc(sizeof(double) * (size_t)dk);
  double* ktT = (double*)malloc(sizeof(double) * (size_t)dk); /* row vector k^T Tc */
  for (int64_t i = 0; i < dk; ++i)
    for (int64_t j = 0; j < dk; ++j) Tc[i * dk + j] = (i == j) ? 1.0 : 0.0;
  for (int64_t t = t0; t < t1; ++t) {
    const double* kin = k + (t * d->h_k + hk) * dk;
    if (d->l2norm_qk) l2_normalise(kin, dk, kt);
    else memcpy(kt, kin, sizeof(double) * (size_t)dk);
    const double alpha = exp(g[t * d->h_v + hv]);
    const double b = beta[t * d->h_v + hv];
    for (int64_t j = 0; j < dk; ++j) {
      double acc = 0.0;
      for (int64_t i = 0; i < dk; ++i) acc += kt[i] * Tc[i * dk + j];
      ktT[j] = acc;
    }
    for (int64_t i = 0; i < dk; ++i)
      for (int64_t j = 0; j < dk; ++j)
        Tc[i * dk + j] = d->scalar_decay ? alpha * Tc[i * dk + j] : alpha * (Tc[i * dk + j] - b * kt[i] * ktT[j]);
  }
  free(kt); free(ktT);
}

typedef struct {
  const gdn_oracle_dims* d;
  const double *k, *v, *g, *beta;
  const int64_t* cu;
  double *T_out, *Sl_out;
} chunkop_ctx;

static void chunkop_item(void* vctx, int64_t item) {
  chunkop_ctx* c = (chunkop_ctx*)vctx;
  const int64_t s = item / c->d->h_v, hv = item % c->d->h_v;
  const int64_t dk = c->d->d_k, dv = c->d->d_v;
  transition_product(c->d, c->k, c->g, c->beta, c->cu[s], c->cu[s + 1], hv,
                     c->T_out + (s * c->d->h_v + hv) * dk * dk);
  /* S_local: the chunk's state from an empty start (Eq. (2) with S = 0) */
  replay_one(c->d, c->k /* q unused */, c->k, c->v, c->g, c->beta, c->cu[s], c->cu[s + 1], hv, NULL,
             c->Sl_out + (s * c->d->h_v + hv) * dv * dk, NULL);
}

/*
 * For each chunk s (tokens cu[s]..cu[s+1]) and v-head: T_out[s][hv] = T_C
 * (d_k x d_k, row-major, the pages' left operator) and Sl_out[s][hv] = S_local
 * (d_v x d_k, this file's state layout).  Returns 0, or -1 on bad dims.
 */
int gdn_oracle_chunk_operator(const gdn_oracle_dims* d, const double* k, const double* g,
                              const double* beta, const double* v, const int64_t* cu_seqlens,
                              double* T_out, double* Sl_out) {
  if (!d || d->h_k <= 0 || d->h_v <= 0 || d->h_v % d->h_k != 0 || d->d_k <= 0 || d->d_v <= 0) return -1;
  chunkop_ctx c = {d, k, v, g, beta, cu_seqlens, T_out, Sl_out};
  parallel_for(resolve_threads(d->n_threads), d->n_seqs * d->h_v, chunkop_item, &c);
  return 0;
}

/* ------------------------------------------------------------------ */
/* closed-form composition of K chunk operators                        */
/* ------------------------------------------------------------------ */

static void matmul(const double* A, const double* B, double* C, int64_t n, int64_t m, int64_t p) {
  /* C (n x p) = A (n x m) B (m x p) */
  for (int64_t i = 0; i < n; ++i)
    for (int64_t j = 0; j < p; ++j) {
      double acc = 0.0;
      for (int64_t l = 0; l < m; ++l) acc += A[i * m + l] * B[l * p + j];
      C[i * p + j] = acc;
    }
}

typedef struct {
  const gdn_oracle_dims* d;
  int64_t K;
  const double *T, *Sl, *S_in;
  double* S_out;
} compose_ctx;

/*
 * For one head, the closed form on the transposed state:
 *   S_K^T = sum_{j=1..K} (T_K ... T_{j+1}) S_local_j^T  +  (T_K ... T_1) S_in^T.
 * Each carried product is formed from scratch (no Horner sharing), then
 * applied; the result is transposed back to the d_v x d_k layout.
 */
static void compose_item(void* vctx, int64_t hv) {
  compose_ctx* c = (compose_ctx*)vctx;
  const int64_t dk = c->d->d_k, dv = c->d->d_v, H = c->d->h_v, K = c->K;
  double* prod = (double*)malloc(sizeof(double) * (size_t)(dk * dk));
  double* tmp = (double*)malloc(sizeof(double) * (size_t)(dk * dk));
  double* StT = (double*)malloc(sizeof(double) * (size_t)(dk * dv)); /* S_local^T, d_k x d_v */
  double* term = (double*)malloc(sizeof(double) * (size_t)(dk * dv));
  double* acc = (double*)calloc((size_t)(dk * dv), sizeof(double));  /* S_K^T */
  /* j = 0 stands for the entering state S_in (carried by all K transitions) */
  for (int64_t j = (c->S_in ? 0 : 1); j <= K; ++j) {
    for (int64_t i = 0; i < dk; ++i)
      for (int64_t l = 0; l < dk; ++l) prod[i * dk + l] = (i == l) ? 1.0 : 0.0;
    for (int64_t m = K; m > j; --m) { /* prod <- prod * T_m, i.e. T_K ... T_{j+1} */
      const double* Tm = c->T + ((m - 1) * H + hv) * dk * dk;
      matmul(prod, Tm, tmp, dk, dk, dk);
      memcpy(prod, tmp, sizeof(double) * (size_t)(dk * dk));
    }
    const double* Sj = (j == 0) ? c->S_in + hv * dv * dk : c->Sl + ((j - 1) * H + hv) * dv * dk;
    for (int64_t a = 0; a < dv; ++a)
      for (int64_t b = 0; b < dk; ++b) StT[b * dv + a] = Sj[a * dk + b];
    matmul(prod, StT, term, dk, dk, dv);
    for (int64_t i = 0; i < dk * dv; ++i) acc[i] += term[i];
  }
  double* out = c->S_out + hv * dv * dk;
  for (int64_t a = 0; a < dv; ++a)
    for (int64_t b = 0; b < dk; ++b) out[a * dk + b] = acc[b * dv + a];
  free(prod); free(tmp); free(StT); free(term); free(acc);
}

/*
 * T: K blocks of [h_v][d_k][d_k]; Sl: K blocks of [h_v][d_v][d_k];
 * S_in: [h_v][d_v][d_k] or NULL (empty entering state); S_out: [h_v][d_v][d_k].
 * Returns 0, or -1 on bad dims.
 */
int gdn_oracle_compose(const gdn_oracle_dims* d, int64_t K, const double* T, const double* Sl,
                       const double* S_in, double* S_out) {
  if (!d || K < 0 || d->h_v <= 0 || d->d_k <= 0 || d->d_v <= 0) return -1;
  compose_ctx c = {d, K, T, Sl, S_in, S_out};
  parallel_for(resolve_threads(d->n_threads), d->h_v, compose_item, &c);
  return 0;
}
