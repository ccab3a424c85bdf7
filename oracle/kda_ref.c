/*
 * kda_ref.c -- plain fp64 CPU reference of the KDA forward pass.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check and the
 * benchmark's CPU-baseline leg load this file; the GPU library neither links
 * nor calls it, and the two share no code.
 *
 * What it computes (page "feat(kda): integrate KDA attention with tokamax
 * backend and CP support", section "Delta Rule formulation"), per batch row b
 * and head h, one token t at a time, with S a K x V matrix indexed [key][value]:
 *
 *     S'       = S * exp(g_t)            g_t in R^K scales the key rows of S
 *     residual = v_t - k_t^T S'
 *     S        = S' + beta_t * k_t (outer) residual
 *     o_t      = scale * q_t^T S         read after the write
 *
 * Packed sequences (same page, section "Public API": decoder_segment_ids
 * [B,T], 1-based, 0 = padding; section "Motivation": packed variable-length
 * sequences via segment_ids): a run is a maximal span of equal non-zero ids.
 * The state restarts from zero at every run start except the row's first run,
 * which starts from initial_state (zeros when none is given).  Padding tokens
 * give o = 0, leave the state alone and end the current run.  final_state is
 * the state after the row's last non-padding token.
 *
 * The arithmetic is the definition written out: no chunking, no blocking,
 * no reordering; exp() is the C library's.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

typedef struct {
  int B, T, H, K, V;
  const double *q, *k, *v, *g, *beta;
  double scale;
  const double *initial_state;
  const int32_t *segment_ids;
  double *o, *final_state;
  int n_threads, tid;
  int status;
} kda_ref_job;

/* One (b, h) recurrence.  S and r are caller-provided scratch (K*V and V). */
static void kda_ref_head(const kda_ref_job *J, int b, int h, double *S,
                         double *r) {
  const int T = J->T, H = J->H, K = J->K, V = J->V;
  const size_t state_off = ((size_t)b * H + h) * (size_t)K * V;

  if (J->initial_state)
    memcpy(S, J->initial_state + state_off, sizeof(double) * (size_t)K * V);
  else
    memset(S, 0, sizeof(double) * (size_t)K * V);

  int seen_run = 0;
  int32_t prev = 0;
  for (int t = 0; t < T; ++t) {
    const int32_t s = J->segment_ids ? J->segment_ids[(size_t)b * T + t] : 1;
    const size_t th = (size_t)b * T * H + (size_t)t * H + h; /* token-head */
    double *ot = J->o + th * V;
    if (s == 0) { /* padding */
      for (int j = 0; j < V; ++j) ot[j] = 0.0;
      prev = 0;
      continue;
    }
    if (s != prev) { /* a run starts at t */
      if (seen_run) memset(S, 0, sizeof(double) * (size_t)K * V);
      seen_run = 1;
    }
    prev = s;

    const double *qt = J->q + th * K;
    const double *kt = J->k + th * K;
    const double *gt = J->g + th * K;
    const double *vt = J->v + th * V;
    const double bt = J->beta[th];

    /* S' = S * exp(g_t): key row i scaled by exp(g_t[i]). */
    for (int i = 0; i < K; ++i) {
      const double e = exp(gt[i]);
      double *Si = S + (size_t)i * V;
      for (int j = 0; j < V; ++j) Si[j] *= e;
    }
    /* residual = v_t - k_t^T S' */
    for (int j = 0; j < V; ++j) r[j] = vt[j];
    for (int i = 0; i < K; ++i) {
      const double ki = kt[i];
      const double *Si = S + (size_t)i * V;
      for (int j = 0; j < V; ++j) r[j] -= ki * Si[j];
    }
    /* S = S' + beta_t k_t (outer) residual */
    for (int i = 0; i < K; ++i) {
      const double c = bt * kt[i];
      double *Si = S + (size_t)i * V;
      for (int j = 0; j < V; ++j) Si[j] += c * r[j];
    }
    /* o_t = scale * q_t^T S (the updated S) */
    for (int j = 0; j < V; ++j) ot[j] = 0.0;
    for (int i = 0; i < K; ++i) {
      const double qi = qt[i];
      const double *Si = S + (size_t)i * V;
      for (int j = 0; j < V; ++j) ot[j] += qi * Si[j];
    }
    for (int j = 0; j < V; ++j) ot[j] *= J->scale;
  }
  if (J->final_state)
    memcpy(J->final_state + state_off, S, sizeof(double) * (size_t)K * V);
}

static void *kda_ref_worker(void *arg) {
  kda_ref_job *J = (kda_ref_job *)arg;
  double *S = (double *)malloc(sizeof(double) * (size_t)J->K * J->V);
  double *r = (double *)malloc(sizeof(double) * (size_t)J->V);
  if (!S || !r) {
    J->status = -2;
    free(S);
    free(r);
    return NULL;
  }
  const int pairs = J->B * J->H;
  for (int p = J->tid; p < pairs; p += J->n_threads)
    kda_ref_head(J, p / J->H, p % J->H, S, r);
  free(S);
  free(r);
  return NULL;
}

/*
 * Layouts (all contiguous, row-major):
 *   q, k, g : [B, T, H, K]     v, o : [B, T, H, V]     beta : [B, T, H]
 *   initial_state, final_state : [B, H, K, V]  (either may be NULL)
 *   segment_ids : [B, T] int32, NULL means every token has id 1.
 * Work is split over (b, h) pairs across n_threads POSIX threads
 * (n_threads <= 0 means one thread).  Returns 0, -1 on bad arguments,
 * -2 when scratch allocation fails.
 */
int kda_ref_forward(int B, int T, int H, int K, int V, const double *q,
                    const double *k, const double *v, const double *g,
                    const double *beta, double scale,
                    const double *initial_state, const int32_t *segment_ids,
                    double *o, double *final_state, int n_threads) {
  if (B < 0 || T < 0 || H < 0 || K <= 0 || V <= 0) return -1;
  if (B == 0 || H == 0) return 0;
  if (T > 0 && (!q || !k || !v || !g || !beta || !o)) return -1;
  if (n_threads <= 0) n_threads = 1;
  if (n_threads > B * H) n_threads = B * H;

  kda_ref_job *jobs = (kda_ref_job *)calloc((size_t)n_threads, sizeof(*jobs));
  pthread_t *th = (pthread_t *)calloc((size_t)n_threads, sizeof(*th));
  if (!jobs || !th) {
    free(jobs);
    free(th);
    return -2;
  }
  for (int i = 0; i < n_threads; ++i) {
    kda_ref_job *J = &jobs[i];
    J->B = B; J->T = T; J->H = H; J->K = K; J->V = V;
    J->q = q; J->k = k; J->v = v; J->g = g; J->beta = beta;
    J->scale = scale;
    J->initial_state = initial_state;
    J->segment_ids = segment_ids;
    J->o = o; J->final_state = final_state;
    J->n_threads = n_threads; J->tid = i; J->status = 0;
  }
  int status = 0;
  int started = 0;
  for (int i = 1; i < n_threads; ++i) {
    if (pthread_create(&th[i], NULL, kda_ref_worker, &jobs[i]) != 0) break;
    started = i;
  }
  /* Threads that failed to start have their pairs done by the caller. */
  for (int i = started + 1; i < n_threads; ++i) {
    jobs[i].n_threads = n_threads;
    kda_ref_worker(&jobs[i]);
  }
  kda_ref_worker(&jobs[0]);
  for (int i = 1; i <= started; ++i) pthread_join(th[i], NULL);
  for (int i = 0; i < n_threads; ++i)
    if (jobs[i].status) status = jobs[i].status;
  free(jobs);
  free(th);
  return status;
}

/*
 * Causal depthwise convolution of width W (4 on the pages) followed by SiLU,
 * page "feat(kda): ...", section "Layer architecture", step 1 (a short causal
 * depthwise 1D conv with SiLU on each of Q, K, V), made segment-aware as the
 * page's later description requires.  Per channel c of x [B, T, C]:
 *
 *     y_t[c] = SiLU( sum_{i=0}^{W-1} w[c][W-1-i] * x_{t-i}[c] )
 *
 * where a tap x_{t-i} counts only when t-i lies in the same run as t
 * (taps before t = 0 or before the run's first token are zero), the weight
 * w[c][W-1] multiplies the current token (left-padded Conv1d order), and
 * there is no bias.  Padding tokens (id 0) give y = 0.
 * SiLU(z) = z / (1 + exp(-z)).
 */
int kda_ref_short_conv_silu(int B, int T, int C, int W, const double *x,
                            const double *w, const int32_t *segment_ids,
                            double *y) {
  if (B < 0 || T < 0 || C <= 0 || W <= 0 || !x || !w || !y) return -1;
  for (int b = 0; b < B; ++b) {
    int run_start = 0;
    int32_t prev = 0;
    for (int t = 0; t < T; ++t) {
      const int32_t s = segment_ids ? segment_ids[(size_t)b * T + t] : 1;
      double *yt = y + ((size_t)b * T + t) * C;
      if (s == 0) {
        for (int c = 0; c < C; ++c) yt[c] = 0.0;
        prev = 0;
        continue;
      }
      if (s != prev) run_start = t;
      prev = s;
      for (int c = 0; c < C; ++c) {
        double z = 0.0;
        for (int i = 0; i < W; ++i) {
          const int tt = t - i;
          if (tt < run_start) break;
          z += w[(size_t)c * W + (W - 1 - i)] * x[((size_t)b * T + tt) * C + c];
        }
        yt[c] = z / (1.0 + exp(-z));
      }
    }
  }
  return 0;
}

/*
 * Per-(token, head) L2 normalisation with an epsilon inside the root, as the
 * optional in-kernel Q/K normalisation (page "feat(kda): ...", section
 * "Public API", use_qk_l2norm_in_kernel; section "Layer architecture",
 * step 5).  x [N, D] is scaled in place row by row:
 *     x <- x / sqrt(sum x^2 + eps)
 */
int kda_ref_l2norm_rows(long N, int D, double eps, double *x) {
  if (N < 0 || D <= 0 || !x) return -1;
  for (long n = 0; n < N; ++n) {
    double *xr = x + (size_t)n * D;
    double ss = 0.0;
    for (int d = 0; d < D; ++d) ss += xr[d] * xr[d];
    const double inv = 1.0 / sqrt(ss + eps);
    for (int d = 0; d < D; ++d) xr[d] *= inv;
  }
  return 0;
}
