/*
 * KDA oracle -- TEST INFRASTRUCTURE ONLY.
 *
 * A plain, slow, fp64 CPU statement of what the Kimi Delta Attention (KDA) forward pass
 * computes, written token by token from its definition. Only the test-suite, the smoke check
 * and the timed CPU baseline of the benchmark may load this library; the product path never
 * does, and it shares no code, header or table with the CUDA kernels.
 *
 * Definitions followed (Kimi K3 wiki, "Notations mathématiques", table "Attention et KDA"):
 *   alpha_t = exp(g_t)                      per-key-channel retention, g_t in (g_min, 0)^{d_k}
 *   M_t     = (I - beta_t k_t k_t^T) Diag(alpha_t)
 *   S_t     = M_t S_{t-1} + beta_t k_t v_t^T  S in R^{d_k x d_v}
 *   o_t     = S_t^T q_t                       raw output, read from the post-update state
 * The delta rule of the "Glossaire" page (entry "Delta rule") is the alpha == 1 special case.
 *
 * The product (I - beta k k^T) Diag(alpha) S is evaluated as three plain loops, in the order
 * the transition matrix is written: decay each row i of S by alpha_i, then read the current
 * association c = S^T k, then write S += beta k (v - c)^T. Nothing is blocked, fused or
 * reordered beyond that. Independent (batch, head) or (sequence, head) problems are spread
 * over POSIX threads; each problem runs start to finish on one thread, so threading does not
 * change a single rounding.
 *
 * Layouts (all fp64, row-major, contiguous):
 *   q, k, g : [B, T, H, d_k]      v : [B, T, H, d_v]      beta : [B, T, H]
 *   out     : [B, T, H, d_v]      S0, S_final : [B, H, d_k, d_v]   (S0 may be NULL: zeros)
 * Packed variable-length batches use B = 1 and cu_seqlens[0..N] (int32, host) with
 * S0 / S_final shaped [N, H, d_k, d_v].
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

typedef struct {
  const double *q, *k, *v, *g, *beta, *S0;
  double *out, *S_final;
  int B, H, T, dk, dv;
  const int32_t *cu; /* NULL for the dense [B, T, H] layout */
  int n_seq;
  int n_problems;
  int next; /* shared work counter, guarded by mu */
  pthread_mutex_t mu;
} job_t;

/* One token of the recurrence on a single state S[dk][dv] (see the header comment). */
static void kda_token(double *S, const double *q, const double *k, const double *v,
                      const double *g, double beta, double *o, double *c, int dk, int dv) {
  for (int i = 0; i < dk; ++i) {
    double a = exp(g[i]);
    for (int j = 0; j < dv; ++j) S[i * dv + j] *= a;
  }
  for (int j = 0; j < dv; ++j) {
    double s = 0.0;
    for (int i = 0; i < dk; ++i) s += S[i * dv + j] * k[i];
    c[j] = s;
  }
  for (int i = 0; i < dk; ++i) {
    double bk = beta * k[i];
    for (int j = 0; j < dv; ++j) S[i * dv + j] += bk * (v[j] - c[j]);
  }
  if (o) {
    for (int j = 0; j < dv; ++j) {
      double s = 0.0;
      for (int i = 0; i < dk; ++i) s += S[i * dv + j] * q[i];
      o[j] = s;
    }
  }
}

/* Runs problem p (a (batch, head) pair, or a (sequence, head) pair for packed batches). */
static void run_problem(job_t *J, int p, double *S, double *c) {
  const int H = J->H, dk = J->dk, dv = J->dv;
  int b, h, t0, t1;
  if (J->cu) {
    int s = p / H;
    h = p % H;
    b = 0;
    t0 = J->cu[s];
    t1 = J->cu[s + 1];
  } else {
    b = p / H;
    h = p % H;
    t0 = 0;
    t1 = J->T;
  }
  const size_t sidx = (size_t)p * dk * dv; /* [B|N, H, dk, dv] */
  if (J->S0)
    memcpy(S, J->S0 + sidx, sizeof(double) * dk * dv);
  else
    memset(S, 0, sizeof(double) * dk * dv);
  for (int t = t0; t < t1; ++t) {
    const size_t row = ((size_t)b * J->T + t) * H + h;
    kda_token(S, J->q + row * dk, J->k + row * dk, J->v + row * dv, J->g + row * dk,
              J->beta[row], J->out ? J->out + row * dv : NULL, c, dk, dv);
  }
  if (J->S_final) memcpy(J->S_final + sidx, S, sizeof(double) * dk * dv);
}

static void *worker(void *arg) {
  job_t *J = (job_t *)arg;
  double *S = (double *)malloc(sizeof(double) * J->dk * J->dv);
  double *c = (double *)malloc(sizeof(double) * J->dv);
  for (;;) {
    pthread_mutex_lock(&J->mu);
    int p = J->next++;
    pthread_mutex_unlock(&J->mu);
    if (p >= J->n_problems) break;
    run_problem(J, p, S, c);
  }
  free(S);
  free(c);
  return NULL;
}

static int run_job(job_t *J, int nthreads) {
  if (nthreads < 1) nthreads = 1;
  if (nthreads > J->n_problems) nthreads = J->n_problems > 0 ? J->n_problems : 1;
  J->next = 0;
  pthread_mutex_init(&J->mu, NULL);
  pthread_t *th = (pthread_t *)malloc(sizeof(pthread_t) * nthreads);
  int started = 0;
  for (int i = 0; i < nthreads; ++i) {
    if (pthread_create(&th[i], NULL, worker, J) != 0) break;
    ++started;
  }
  if (started == 0) worker(J);
  for (int i = 0; i < started; ++i) pthread_join(th[i], NULL);
  free(th);
  pthread_mutex_destroy(&J->mu);
  return 0;
}

/* Dense batch: B independent sequences of length T. Returns 0 on success, -1 on bad sizes. */
int kda_oracle_recurrent(const double *q, const double *k, const double *v, const double *g,
                         const double *beta, const double *S0, double *out, double *S_final,
                         int B, int H, int T, int dk, int dv, int nthreads) {
  if (B < 0 || H < 1 || T < 0 || dk < 1 || dv < 1) return -1;
  job_t J;
  memset(&J, 0, sizeof(J));
  J.q = q; J.k = k; J.v = v; J.g = g; J.beta = beta; J.S0 = S0;
  J.out = out; J.S_final = S_final;
  J.B = B; J.H = H; J.T = T; J.dk = dk; J.dv = dv;
  J.n_problems = B * H;
  return run_job(&J, nthreads);
}

/* Packed batch: one [1, T_total, H, d] tensor holding N sequences; sequence s covers
 * tokens [cu_seqlens[s], cu_seqlens[s+1]) and starts from S0[s] (zeros when S0 is NULL). */
int kda_oracle_recurrent_varlen(const double *q, const double *k, const double *v,
                                const double *g, const double *beta, const double *S0,
                                double *out, double *S_final, const int32_t *cu_seqlens,
                                int n_seq, int H, int T_total, int dk, int dv, int nthreads) {
  if (n_seq < 0 || H < 1 || dk < 1 || dv < 1) return -1;
  if (n_seq > 0 && (cu_seqlens[0] != 0 || cu_seqlens[n_seq] != T_total)) return -1;
  for (int s = 0; s < n_seq; ++s)
    if (cu_seqlens[s + 1] < cu_seqlens[s]) return -1;
  job_t J;
  memset(&J, 0, sizeof(J));
  J.q = q; J.k = k; J.v = v; J.g = g; J.beta = beta; J.S0 = S0;
  J.out = out; J.S_final = S_final;
  J.B = 1; J.H = H; J.T = T_total; J.dk = dk; J.dv = dv;
  J.cu = cu_seqlens; J.n_seq = n_seq;
  J.n_problems = n_seq * H;
  return run_job(&J, nthreads);
}

/* One decode token for N sequences x H heads: q, k, g [N, H, dk]; v, out [N, H, dv];
 * beta [N, H]; S [N, H, dk, dv] is updated in place. Same token update as above. */
int kda_oracle_decode_step(const double *q, const double *k, const double *v, const double *g,
                           const double *beta, double *S, double *out, int N, int H, int dk,
                           int dv) {
  if (N < 0 || H < 1 || dk < 1 || dv < 1) return -1;
  double *c = (double *)malloc(sizeof(double) * dv);
  for (int p = 0; p < N * H; ++p) {
    kda_token(S + (size_t)p * dk * dv, q + (size_t)p * dk, k + (size_t)p * dk,
              v + (size_t)p * dv, g + (size_t)p * dk, beta[p], out + (size_t)p * dv, c, dk,
              dv);
  }
  free(c);
  return 0;
}
