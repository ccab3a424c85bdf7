/*
 * kda_ref_bwd.c -- plain fp64 CPU reference of the gradient of the KDA
 * forward pass of kda_ref.c (its vector-Jacobian product).
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check and the
 * benchmark's CPU-baseline leg load this file; the GPU library neither links
 * nor calls it, and the two share no code.
 *
 * The forward pass (page "feat(kda): integrate KDA attention with tokamax
 * backend and CP support", section "Delta Rule formulation"; packed runs as
 * in section "Public API") is, per (b, h) and token t of a run,
 *
 *     S' = diag(e^{g_t}) S_{t-1},  r = v_t - S'^T k_t,
 *     S_t = S' + beta_t k_t r^T,   o_t = scale * S_t^T q_t.
 *
 * Given the upstream gradients do_t (of o_t) and dS_final (of final_state),
 * this returns the gradients of L = sum_t <do_t, o_t> + <dS_final,
 * final_state> with respect to q, k, v, g, beta and initial_state, by
 * reverse-mode differentiation of that recurrence, one token at a time from
 * the last to the first, with dS the gradient of S_t:
 *
 *     dS     += scale * q_t do_t^T
 *     dq_t    = scale * S_t do_t
 *     dr      = beta_t * dS^T k_t
 *     dbeta_t = k_t^T dS r
 *     dk_t    = beta_t * dS r - S' dr
 *     dv_t    = dr
 *     dS'     = dS - k_t dr^T
 *     dg_t[i] = sum_j S'[i][j] dS'[i][j]
 *     dS      = diag(e^{g_t}) dS'                (now the gradient of S_{t-1})
 *
 * A run start at which the state was reset to zero stops dS there; the
 * row's first run hands it on to initial_state.  Padding tokens get zero
 * gradients and pass dS through unchanged (they leave the state alone).
 *
 * The states S_{t-1} are recomputed rather than stored: a forward pass keeps
 * the state (and the run bookkeeping) at every CB-th token, and each block of
 * CB tokens is replayed from its checkpoint with the same operations in the
 * same order as kda_ref.c, so the replayed states equal the forward's
 * exactly.  No chunking, blocking or reordering of the arithmetic itself.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

enum { CB = 64 };                   /* tokens per checkpoint block */
enum { TOK_PAD = 0, TOK_IN_RUN = 1, TOK_RESET = 2, TOK_FIRST = 3 };

typedef struct {
  int B, T, H, K, V;
  const double *q, *k, *v, *g, *beta;
  double scale;
  const double *initial_state;
  const int32_t *segment_ids;
  const double *d_o, *d_final;
  double *dq, *dk, *dv, *dg, *dbeta, *d_initial;
  int n_threads, tid;
  int status;
} kda_bwd_job;

typedef struct {
  double *ckpt;        /* nblk x K*V: state entering each block       */
  int *ckpt_seen;      /* nblk: a run has started before the block     */
  int32_t *ckpt_prev;  /* nblk: id of the token before the block       */
  double *blk;         /* CB x K*V: state entering each token (after a reset) */
  int *kind;           /* CB: TOK_*                                    */
  double *S, *Sp, *St, *dS, *dSp, *r, *dr;
} kda_bwd_scratch;

/* One forward token step on S (K x V) in place; r is V scratch. */
static void fwd_step(int K, int V, const double *kt, const double *gt,
                     const double *vt, double bt, double *S, double *r) {
  for (int i = 0; i < K; ++i) {
    const double e = exp(gt[i]);
    double *Si = S + (size_t)i * V;
    for (int j = 0; j < V; ++j) Si[j] *= e;
  }
  for (int j = 0; j < V; ++j) r[j] = vt[j];
  for (int i = 0; i < K; ++i) {
    const double ki = kt[i];
    const double *Si = S + (size_t)i * V;
    for (int j = 0; j < V; ++j) r[j] -= ki * Si[j];
  }
  for (int i = 0; i < K; ++i) {
    const double c = bt * kt[i];
    double *Si = S + (size_t)i * V;
    for (int j = 0; j < V; ++j) Si[j] += c * r[j];
  }
}

/* The run bookkeeping of kda_ref.c for token t: returns TOK_*, resetting S
 * to zero at a run start after an earlier run. */
static int run_step(int32_t s, int *seen, int32_t *prev, double *S, size_t kv) {
  if (s == 0) {
    *prev = 0;
    return TOK_PAD;
  }
  int kind = TOK_IN_RUN;
  if (s != *prev) {
    kind = *seen ? TOK_RESET : TOK_FIRST;
    if (*seen) memset(S, 0, sizeof(double) * kv);
    *seen = 1;
  }
  *prev = s;
  return kind;
}

static void kda_bwd_head(const kda_bwd_job *J, int b, int h, kda_bwd_scratch *W) {
  const int T = J->T, H = J->H, K = J->K, V = J->V;
  const size_t kv = (size_t)K * V;
  const size_t state_off = ((size_t)b * H + h) * kv;
  const int nblk = (T + CB - 1) / CB;

  /* forward pass: checkpoints */
  double *S = W->S;
  if (J->initial_state) memcpy(S, J->initial_state + state_off, sizeof(double) * kv);
  else memset(S, 0, sizeof(double) * kv);
  int seen = 0;
  int32_t prev = 0;
  for (int t = 0; t < T; ++t) {
    if (t % CB == 0) {
      const int bi = t / CB;
      memcpy(W->ckpt + (size_t)bi * kv, S, sizeof(double) * kv);
      W->ckpt_seen[bi] = seen;
      W->ckpt_prev[bi] = prev;
    }
    const int32_t s = J->segment_ids ? J->segment_ids[(size_t)b * T + t] : 1;
    if (run_step(s, &seen, &prev, S, kv) == TOK_PAD) continue;
    const size_t th = (size_t)b * T * H + (size_t)t * H + h;
    fwd_step(K, V, J->k + th * K, J->g + th * K, J->v + th * V, J->beta[th], S, W->r);
  }

  /* backward pass, block by block from the end */
  double *dS = W->dS;
  if (J->d_final) memcpy(dS, J->d_final + state_off, sizeof(double) * kv);
  else memset(dS, 0, sizeof(double) * kv);
  for (int bi = nblk - 1; bi >= 0; --bi) {
    const int t0 = bi * CB, t1 = t0 + CB < T ? t0 + CB : T;
    /* replay the block, keeping the state entering each token */
    memcpy(S, W->ckpt + (size_t)bi * kv, sizeof(double) * kv);
    seen = W->ckpt_seen[bi];
    prev = W->ckpt_prev[bi];
    for (int t = t0; t < t1; ++t) {
      const int32_t s = J->segment_ids ? J->segment_ids[(size_t)b * T + t] : 1;
      const int kind = run_step(s, &seen, &prev, S, kv);
      W->kind[t - t0] = kind;
      if (kind == TOK_PAD) continue;
      memcpy(W->blk + (size_t)(t - t0) * kv, S, sizeof(double) * kv);
      const size_t th = (size_t)b * T * H + (size_t)t * H + h;
      fwd_step(K, V, J->k + th * K, J->g + th * K, J->v + th * V, J->beta[th], S, W->r);
    }
    for (int t = t1 - 1; t >= t0; --t) {
      const size_t th = (size_t)b * T * H + (size_t)t * H + h;
      double *dqt = J->dq + th * K, *dkt = J->dk + th * K, *dgt = J->dg + th * K;
      double *dvt = J->dv + th * V;
      const int kind = W->kind[t - t0];
      if (kind == TOK_PAD) {
        for (int i = 0; i < K; ++i) dqt[i] = dkt[i] = dgt[i] = 0.0;
        for (int j = 0; j < V; ++j) dvt[j] = 0.0;
        J->dbeta[th] = 0.0;
        continue;
      }
      const double *qt = J->q + th * K, *kt = J->k + th * K, *gt = J->g + th * K;
      const double *vt = J->v + th * V, *dot = J->d_o + th * V;
      const double bt = J->beta[th];
      const double *Sb = W->blk + (size_t)(t - t0) * kv;  /* S_{t-1} */
      double *Sp = W->Sp, *St = W->St, *dSp = W->dSp, *r = W->r, *dr = W->dr;
      /* forward quantities of token t */
      for (int i = 0; i < K; ++i) {
        const double e = exp(gt[i]);
        for (int j = 0; j < V; ++j) Sp[(size_t)i * V + j] = Sb[(size_t)i * V + j] * e;
      }
      for (int j = 0; j < V; ++j) r[j] = vt[j];
      for (int i = 0; i < K; ++i)
        for (int j = 0; j < V; ++j) r[j] -= kt[i] * Sp[(size_t)i * V + j];
      for (int i = 0; i < K; ++i)
        for (int j = 0; j < V; ++j)
          St[(size_t)i * V + j] = Sp[(size_t)i * V + j] + bt * kt[i] * r[j];
      /* o_t = scale S_t^T q_t */
      for (int i = 0; i < K; ++i)
        for (int j = 0; j < V; ++j) dS[(size_t)i * V + j] += J->scale * qt[i] * dot[j];
      for (int i = 0; i < K; ++i) {
        double a = 0.0;
        for (int j = 0; j < V; ++j) a += St[(size_t)i * V + j] * dot[j];
        dqt[i] = J->scale * a;
      }
      /* S_t = S' + beta k r^T */
      double db = 0.0;
      for (int j = 0; j < V; ++j) {
        double a = 0.0;
        for (int i = 0; i < K; ++i) a += dS[(size_t)i * V + j] * kt[i];
        dr[j] = bt * a;
        db += a * r[j];
      }
      J->dbeta[th] = db;
      for (int i = 0; i < K; ++i) {
        double a = 0.0, c = 0.0;
        for (int j = 0; j < V; ++j) {
          a += dS[(size_t)i * V + j] * r[j];
          c += Sp[(size_t)i * V + j] * dr[j];
        }
        dkt[i] = bt * a - c;       /* the r^T factor, then r = v - S'^T k */
      }
      for (int j = 0; j < V; ++j) dvt[j] = dr[j];
      for (int i = 0; i < K; ++i)
        for (int j = 0; j < V; ++j)
          dSp[(size_t)i * V + j] = dS[(size_t)i * V + j] - kt[i] * dr[j];
      /* S' = diag(e^g) S_{t-1} */
      for (int i = 0; i < K; ++i) {
        const double e = exp(gt[i]);
        double a = 0.0;
        for (int j = 0; j < V; ++j) {
          a += Sp[(size_t)i * V + j] * dSp[(size_t)i * V + j];
          dS[(size_t)i * V + j] = e * dSp[(size_t)i * V + j];
        }
        dgt[i] = a;
      }
      if (kind == TOK_RESET) memset(dS, 0, sizeof(double) * kv);
    }
  }
  if (J->d_initial) memcpy(J->d_initial + state_off, dS, sizeof(double) * kv);
}

static void *kda_bwd_worker(void *arg) {
  kda_bwd_job *J = (kda_bwd_job *)arg;
  const size_t kv = (size_t)J->K * J->V;
  const int nblk = (J->T + CB - 1) / CB > 0 ? (J->T + CB - 1) / CB : 1;
  kda_bwd_scratch W;
  W.ckpt = (double *)malloc(sizeof(double) * kv * (size_t)nblk);
  W.ckpt_seen = (int *)malloc(sizeof(int) * (size_t)nblk);
  W.ckpt_prev = (int32_t *)malloc(sizeof(int32_t) * (size_t)nblk);
  W.blk = (double *)malloc(sizeof(double) * kv * CB);
  W.kind = (int *)malloc(sizeof(int) * CB);
  W.S = (double *)malloc(sizeof(double) * kv);
  W.Sp = (double *)malloc(sizeof(double) * kv);
  W.St = (double *)malloc(sizeof(double) * kv);
  W.dS = (double *)malloc(sizeof(double) * kv);
  W.dSp = (double *)malloc(sizeof(double) * kv);
  W.r = (double *)malloc(sizeof(double) * (size_t)J->V);
  W.dr = (double *)malloc(sizeof(double) * (size_t)J->V);
  if (!W.ckpt || !W.ckpt_seen || !W.ckpt_prev || !W.blk || !W.kind || !W.S || !W.Sp ||
      !W.St || !W.dS || !W.dSp || !W.r || !W.dr) {
    J->status = -2;
  } else {
    const int pairs = J->B * J->H;
    for (int p = J->tid; p < pairs; p += J->n_threads) kda_bwd_head(J, p / J->H, p % J->H, &W);
  }
  free(W.ckpt); free(W.ckpt_seen); free(W.ckpt_prev); free(W.blk); free(W.kind);
  free(W.S); free(W.Sp); free(W.St); free(W.dS); free(W.dSp); free(W.r); free(W.dr);
  return NULL;
}

/*
 * Layouts as kda_ref_forward: q, k, g, dq, dk, dg [B, T, H, K]; v, d_o, dv
 * [B, T, H, V]; beta, dbeta [B, T, H]; initial_state, d_final, d_initial
 * [B, H, K, V] (initial_state and d_final may be NULL = zeros, d_initial
 * may be NULL = not wanted); segment_ids [B, T] or NULL.  Work is split over
 * (b, h) pairs across n_threads POSIX threads.  Returns 0, -1 on bad
 * arguments, -2 when scratch allocation fails.
 */
int kda_ref_backward(int B, int T, int H, int K, int V, const double *q,
                     const double *k, const double *v, const double *g,
                     const double *beta, double scale, const double *initial_state,
                     const int32_t *segment_ids, const double *d_o,
                     const double *d_final, double *dq, double *dk, double *dv,
                     double *dg, double *dbeta, double *d_initial, int n_threads) {
  if (B < 0 || T < 0 || H < 0 || K <= 0 || V <= 0) return -1;
  if (B == 0 || H == 0) return 0;
  if (T > 0 && (!q || !k || !v || !g || !beta || !d_o || !dq || !dk || !dv || !dg || !dbeta))
    return -1;
  if (n_threads <= 0) n_threads = 1;
  if (n_threads > B * H) n_threads = B * H;
  kda_bwd_job *jobs = (kda_bwd_job *)calloc((size_t)n_threads, sizeof(*jobs));
  pthread_t *th = (pthread_t *)calloc((size_t)n_threads, sizeof(*th));
  if (!jobs || !th) {
    free(jobs);
    free(th);
    return -2;
  }
  for (int i = 0; i < n_threads; ++i) {
    kda_bwd_job *J = &jobs[i];
    J->B = B; J->T = T; J->H = H; J->K = K; J->V = V;
    J->q = q; J->k = k; J->v = v; J->g = g; J->beta = beta;
    J->scale = scale;
    J->initial_state = initial_state;
    J->segment_ids = segment_ids;
    J->d_o = d_o; J->d_final = d_final;
    J->dq = dq; J->dk = dk; J->dv = dv; J->dg = dg; J->dbeta = dbeta;
    J->d_initial = d_initial;
    J->n_threads = n_threads; J->tid = i; J->status = 0;
  }
  int started = 0;
  for (int i = 1; i < n_threads; ++i) {
    if (pthread_create(&th[i], NULL, kda_bwd_worker, &jobs[i]) != 0) break;
    started = i;
  }
  for (int i = started + 1; i < n_threads; ++i) kda_bwd_worker(&jobs[i]);
  kda_bwd_worker(&jobs[0]);
  for (int i = 1; i <= started; ++i) pthread_join(th[i], NULL);
  int status = 0;
  for (int i = 0; i < n_threads; ++i)
    if (jobs[i].status) status = jobs[i].status;
  free(jobs);
  free(th);
  return status;
}
