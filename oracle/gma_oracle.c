/*
 * gma_oracle.c -- plain float64 CPU oracle for the Gaussian Mixture Attention
 * (GMA) forward pass.  TEST INFRASTRUCTURE ONLY: the tests, the package's
 * smoke check and the CPU-baseline leg of the benchmark call it; the product
 * path never does.  It shares no source with the CUDA library.
 *
 * Source: "Gaussian Mixture Attention: Linear-Time Sequence Mixing via
 * Probabilistic Latent Routing" (Huang & Raza, arXiv 2606.18283), as summarised
 * on gist.science (ja / de technical summaries) and in the English abstract on
 * fugumt.com.  Citations below name the page and its section.
 *
 *   [R]  Responsibilities: gist.science summary, "Core mechanism" item 1
 *        (probabilistic latent routing): gamma_{i,k} = p(z = k | x) from the
 *        standard GMM posterior with means mu_k, diagonal covariances Sigma_k and
 *        priors pi_k; queries and keys share one set of components (abstract:
 *        "shared latent routing space").
 *   [W]  Write phase: same section, item 2: Vt = Gamma_K^T V, Z = Gamma_K^T 1.
 *   [Rd] Read phase: same section, item 2: O = Gamma_Q Vt / (Gamma_Q Z + eps).
 *   [C]  Causal variant: "Variants and training" item 3: prefix sums of the
 *        latent memory and the normaliser so that O_i depends on j <= i only.
 *   [B]  Backward pass: "Variants and training" item 3 (the Gaussian
 *        components are parameterised differentiably and learned end to end by
 *        backpropagation through this path): gradients of a loss L with respect
 *        to Q, K, V, mu, sigma2 and log pi given dL/dO, bidirectional form, by
 *        the chain rule through [Rd], [W] and [R] (written out at
 *        gma_oracle_backward_bidir below).
 *   [X]  Cross-attention: gist.science summary, "Significance and claims",
 *        closing paragraph (cross-attention applications named as future work
 *        beyond the self-attention setting): queries of one sequence read
 *        the latent memory written by the keys and values of another, so the
 *        write runs over Nk keys and the read over N queries; nothing else in
 *        [W] / [Rd] changes.
 *
 * Readings where the pages leave a step open:
 *   - The log-density keeps every term of the diagonal Gaussian, including
 *     -1/2 sum_d log sigma2_kd and -(d/2) log(2 pi); the last one cancels in
 *     the posterior but is kept so the formula reads like the textbook one.
 *   - The routing vector x is the head's query / key row itself.
 *   - eps is added once to the scalar denominator of each output row.
 *   - The causal sum is inclusive: position i sees keys j = 0..i.
 *
 * Everything is computed in the centered form sum_d (x_d - mu_kd)^2 / sigma2_kd,
 * with a max-subtracted log-sum-exp over the K components.  Work is split over
 * (batch, head) units across threads; each unit is computed by the plain
 * sequential code below, so threading does not change any arithmetic.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define GMA_ORACLE_LOG_2PI 1.8378770664093454835606594728112

/* sum_d log sigma2_kd for each of the K components of one head (the Gaussian's log-determinant). */
static void log_determinants(int d, int K, const double *sigma2, double *logdet) {
  for (int k = 0; k < K; ++k) {
    double s = 0.0;
    for (int j = 0; j < d; ++j) s += log(sigma2[(size_t)k * d + j]);
    logdet[k] = s;
  }
}

/* [R] posterior responsibilities of one routing vector x (length d) over the
 * K components of one head.  mu, sigma2: [K][d]; logdet: [K] from
 * log_determinants(); log_pi: [K]; out: [K]. */
static void posterior(int d, int K, const double *x, const double *mu, const double *sigma2, const double *logdet,
                      const double *log_pi, double *out) {
  double m = -INFINITY;
  for (int k = 0; k < K; ++k) {
    double quad = 0.0;
    for (int j = 0; j < d; ++j) {
      double diff = x[j] - mu[(size_t)k * d + j];
      quad += diff * diff / sigma2[(size_t)k * d + j];
    }
    /* log pi_k + log N(x; mu_k, diag(sigma2_k)) */
    double l = log_pi[k] - 0.5 * (quad + logdet[k]) - 0.5 * d * GMA_ORACLE_LOG_2PI;
    out[k] = l;
    if (l > m) m = l;
  }
  double s = 0.0;
  for (int k = 0; k < K; ++k) {
    out[k] = exp(out[k] - m);
    s += out[k];
  }
  for (int k = 0; k < K; ++k) out[k] /= s;
}

typedef struct {
  int mode; /* 0 = responsibilities, 1 = bidirectional (or cross), 2 = causal */
  int B, H, N, d, dv, K;
  int Nk; /* keys per unit: N except for cross-attention */
  const double *Q, *Kx, *V, *mu, *sigma2, *log_pi;
  double eps;
  const int64_t *rows; /* sorted ascending, or NULL for every row */
  int64_t nrows;
  double *out;
  int nthreads;
  int next_unit;
  pthread_mutex_t lock;
} job_t;

/* One (b, h) unit. */
static void run_unit(job_t *J, int unit) {
  const int H = J->H, N = J->N, d = J->d, dv = J->dv, K = J->K;
  const int h = unit % H;
  const double *mu = J->mu + (size_t)h * K * d;
  const double *s2 = J->sigma2 + (size_t)h * K * d;
  const double *lp = J->log_pi + (size_t)h * K;
  const int64_t nout = J->rows ? J->nrows : N;
  double *g = (double *)malloc(sizeof(double) * K);
  double *ld = (double *)malloc(sizeof(double) * K);
  log_determinants(d, K, s2, ld);

  if (J->mode == 0) {
    const double *X = J->Q + (size_t)unit * N * d;
    double *G = J->out + (size_t)unit * nout * K;
    for (int64_t r = 0; r < nout; ++r) {
      int64_t i = J->rows ? J->rows[r] : r;
      posterior(d, K, X + i * d, mu, s2, ld, lp, G + r * K);
    }
    free(g);
    free(ld);
    return;
  }

  const int Nk = J->Nk;
  const double *Q = J->Q + (size_t)unit * N * d;
  const double *Kx = J->Kx + (size_t)unit * Nk * d;
  const double *V = J->V + (size_t)unit * Nk * dv;
  double *O = J->out + (size_t)unit * nout * dv;
  double *Vt = (double *)calloc((size_t)K * dv, sizeof(double)); /* latent memory, K x dv */
  double *Z = (double *)calloc((size_t)K, sizeof(double));       /* normaliser, K */

  if (J->mode == 1) {
    /* [W] write phase over all Nk keys */
    for (int j = 0; j < Nk; ++j) {
      posterior(d, K, Kx + (size_t)j * d, mu, s2, ld, lp, g);
      for (int k = 0; k < K; ++k) {
        Z[k] += g[k];
        for (int c = 0; c < dv; ++c) Vt[(size_t)k * dv + c] += g[k] * V[(size_t)j * dv + c];
      }
    }
    /* [Rd] read phase for the requested query rows */
    for (int64_t r = 0; r < nout; ++r) {
      int64_t i = J->rows ? J->rows[r] : r;
      posterior(d, K, Q + i * d, mu, s2, ld, lp, g);
      double den = 0.0;
      for (int k = 0; k < K; ++k) den += g[k] * Z[k];
      den += J->eps;
      for (int c = 0; c < dv; ++c) {
        double num = 0.0;
        for (int k = 0; k < K; ++k) num += g[k] * Vt[(size_t)k * dv + c];
        O[r * dv + c] = num / den;
      }
    }
  } else {
    /* [C] running prefix sums, inclusive of the current position */
    int64_t r = 0;
    for (int64_t i = 0; i < N && r < nout; ++i) {
      posterior(d, K, Kx + i * d, mu, s2, ld, lp, g);
      for (int k = 0; k < K; ++k) {
        Z[k] += g[k];
        for (int c = 0; c < dv; ++c) Vt[(size_t)k * dv + c] += g[k] * V[i * dv + c];
      }
      int64_t want = J->rows ? J->rows[r] : i;
      if (want != i) continue;
      posterior(d, K, Q + i * d, mu, s2, ld, lp, g);
      double den = 0.0;
      for (int k = 0; k < K; ++k) den += g[k] * Z[k];
      den += J->eps;
      for (int c = 0; c < dv; ++c) {
        double num = 0.0;
        for (int k = 0; k < K; ++k) num += g[k] * Vt[(size_t)k * dv + c];
        O[r * dv + c] = num / den;
      }
      ++r;
    }
  }
  free(Vt);
  free(Z);
  free(g);
  free(ld);
}

static void *worker(void *arg) {
  job_t *J = (job_t *)arg;
  for (;;) {
    pthread_mutex_lock(&J->lock);
    int u = J->next_unit++;
    pthread_mutex_unlock(&J->lock);
    if (u >= J->B * J->H) break;
    run_unit(J, u);
  }
  return NULL;
}

static int run_job(job_t *J) {
  int nt = J->nthreads < 1 ? 1 : J->nthreads;
  if (nt > J->B * J->H) nt = J->B * J->H;
  if (nt < 1) return 0;
  J->next_unit = 0;
  pthread_mutex_init(&J->lock, NULL);
  pthread_t *th = (pthread_t *)malloc(sizeof(pthread_t) * nt);
  int started = 0;
  for (int t = 0; t < nt; ++t)
    if (pthread_create(&th[t], NULL, worker, J) == 0) ++started;
  if (started == 0) worker(J);
  for (int t = 0; t < started; ++t) pthread_join(th[t], NULL);
  free(th);
  pthread_mutex_destroy(&J->lock);
  return 0;
}

/* Gamma [B,H,nrows or N,K] of routing vectors X [B,H,N,d]. */
int gma_oracle_responsibilities(int B, int H, int N, int d, int K, const double *X, const double *mu,
                                const double *sigma2, const double *log_pi, const int64_t *rows, int64_t nrows,
                                double *gamma, int nthreads) {
  job_t J;
  memset(&J, 0, sizeof J);
  J.mode = 0; J.B = B; J.H = H; J.N = N; J.d = d; J.dv = 0; J.K = K;
  J.Q = X; J.mu = mu; J.sigma2 = sigma2; J.log_pi = log_pi;
  J.rows = rows; J.nrows = nrows; J.out = gamma; J.nthreads = nthreads;
  return run_job(&J);
}

/* O [B,H,nrows or N,dv]; causal = 0 bidirectional, 1 causal. */
int gma_oracle_forward(int causal, int B, int H, int N, int d, int dv, int K, const double *Q, const double *Kx,
                       const double *V, const double *mu, const double *sigma2, const double *log_pi, double eps,
                       const int64_t *rows, int64_t nrows, double *O, int nthreads) {
  job_t J;
  memset(&J, 0, sizeof J);
  J.mode = causal ? 2 : 1; J.B = B; J.H = H; J.N = N; J.d = d; J.dv = dv; J.K = K; J.Nk = N;
  J.Q = Q; J.Kx = Kx; J.V = V; J.mu = mu; J.sigma2 = sigma2; J.log_pi = log_pi; J.eps = eps;
  J.rows = rows; J.nrows = nrows; J.out = O; J.nthreads = nthreads;
  return run_job(&J);
}

/* [X] O [B,H,nrows or N,dv] for N queries reading the memory written by Nk keys / values per unit. */
int gma_oracle_forward_cross(int B, int H, int N, int Nk, int d, int dv, int K, const double *Q, const double *Kx,
                             const double *V, const double *mu, const double *sigma2, const double *log_pi,
                             double eps, const int64_t *rows, int64_t nrows, double *O, int nthreads) {
  job_t J;
  memset(&J, 0, sizeof J);
  J.mode = 1; J.B = B; J.H = H; J.N = N; J.d = d; J.dv = dv; J.K = K; J.Nk = Nk;
  J.Q = Q; J.Kx = Kx; J.V = V; J.mu = mu; J.sigma2 = sigma2; J.log_pi = log_pi; J.eps = eps;
  J.rows = rows; J.nrows = nrows; J.out = O; J.nthreads = nthreads;
  return run_job(&J);
}

/* [B] Gradients of the bidirectional forward, given G = dL/dO [B,H,N,dv].
 * Per (b, h), with gamma rows from [R], Vt = Gamma_K^T V, Z = Gamma_K^T 1, n_i = gamma_Qi . Vt,
 * den_i = gamma_Qi . Z + eps, O_i = n_i / den_i:
 *   dn_i = G_i / den_i,  dden_i = -(G_i . O_i) / den_i
 *   dgamma_Qi = Vt dn_i + Z dden_i,       dVt = sum_i gamma_Qi dn_i^T,   dZ = sum_i gamma_Qi dden_i
 *   dgamma_Kj = dVt v_j + dZ,             dv_j = dVt^T gamma_Kj
 *   softmax: dl = gamma * (dgamma - gamma . dgamma)
 *   l_k(x) = log pi_k - 1/2 sum_d [(x_d - mu_kd)^2 / sigma2_kd + log sigma2_kd] - (d/2) log 2pi:
 *     dx_d += dl_k (mu_kd - x_d) / sigma2_kd,  dmu_kd += dl_k (x_d - mu_kd) / sigma2_kd,
 *     dsigma2_kd += dl_k (1/2) [(x_d - mu_kd)^2 / sigma2_kd^2 - 1 / sigma2_kd],  dlog_pi_k += dl_k,
 * with the parameter gradients summed over every query and key row of every batch entry of the
 * head.  Sequential over (b, h) units (deterministic sums); small problems only. */
static void softmax_backward(int K, const double *g, const double *dg, double *dl) {
  double dot = 0.0;
  for (int k = 0; k < K; ++k) dot += g[k] * dg[k];
  for (int k = 0; k < K; ++k) dl[k] = g[k] * (dg[k] - dot);
}

static void logdensity_backward(int d, int K, const double *x, const double *mu, const double *sigma2,
                                const double *dl, double *dx, double *dmu, double *ds2, double *dlp) {
  for (int j = 0; j < d; ++j) dx[j] = 0.0;
  for (int k = 0; k < K; ++k) {
    dlp[k] += dl[k];
    for (int j = 0; j < d; ++j) {
      const double s2 = sigma2[(size_t)k * d + j];
      const double diff = x[j] - mu[(size_t)k * d + j];
      dx[j] += dl[k] * (-diff / s2);
      dmu[(size_t)k * d + j] += dl[k] * (diff / s2);
      ds2[(size_t)k * d + j] += dl[k] * 0.5 * (diff * diff / (s2 * s2) - 1.0 / s2);
    }
  }
}

int gma_oracle_backward_bidir(int B, int H, int N, int d, int dv, int K, const double *Q, const double *Kx,
                              const double *V, const double *mu, const double *sigma2, const double *log_pi,
                              double eps, const double *G, double *dQ, double *dK, double *dV, double *dmu,
                              double *dsigma2, double *dlog_pi) {
  double *gq = (double *)malloc(sizeof(double) * (size_t)(N > 0 ? N : 1) * K);
  double *gk = (double *)malloc(sizeof(double) * (size_t)(N > 0 ? N : 1) * K);
  double *ld = (double *)malloc(sizeof(double) * K);
  double *Vt = (double *)malloc(sizeof(double) * (size_t)K * dv), *Z = (double *)malloc(sizeof(double) * K);
  double *dVt = (double *)malloc(sizeof(double) * (size_t)K * dv), *dZ = (double *)malloc(sizeof(double) * K);
  double *dn = (double *)malloc(sizeof(double) * dv), *dg = (double *)malloc(sizeof(double) * K);
  double *dl = (double *)malloc(sizeof(double) * K), *On = (double *)malloc(sizeof(double) * dv);
  memset(dmu, 0, sizeof(double) * (size_t)H * K * d);
  memset(dsigma2, 0, sizeof(double) * (size_t)H * K * d);
  memset(dlog_pi, 0, sizeof(double) * (size_t)H * K);
  for (int u = 0; u < B * H; ++u) {
    const int h = u % H;
    const double *mu_h = mu + (size_t)h * K * d, *s2_h = sigma2 + (size_t)h * K * d, *lp_h = log_pi + (size_t)h * K;
    double *dmu_h = dmu + (size_t)h * K * d, *ds2_h = dsigma2 + (size_t)h * K * d, *dlp_h = dlog_pi + (size_t)h * K;
    const double *q = Q + (size_t)u * N * d, *kx = Kx + (size_t)u * N * d, *v = V + (size_t)u * N * dv;
    const double *g = G + (size_t)u * N * dv;
    log_determinants(d, K, s2_h, ld);
    memset(Vt, 0, sizeof(double) * (size_t)K * dv);
    memset(Z, 0, sizeof(double) * K);
    memset(dVt, 0, sizeof(double) * (size_t)K * dv);
    memset(dZ, 0, sizeof(double) * K);
    for (int j = 0; j < N; ++j) {
      posterior(d, K, kx + (size_t)j * d, mu_h, s2_h, ld, lp_h, gk + (size_t)j * K);
      for (int k = 0; k < K; ++k) {
        Z[k] += gk[(size_t)j * K + k];
        for (int c = 0; c < dv; ++c) Vt[(size_t)k * dv + c] += gk[(size_t)j * K + k] * v[(size_t)j * dv + c];
      }
    }
    /* queries: recompute O_i, push G_i back through the read */
    for (int i = 0; i < N; ++i) {
      const double *gqi = gq + (size_t)i * K;
      posterior(d, K, q + (size_t)i * d, mu_h, s2_h, ld, lp_h, gq + (size_t)i * K);
      double den = eps;
      for (int k = 0; k < K; ++k) den += gqi[k] * Z[k];
      double gdoto = 0.0;
      for (int c = 0; c < dv; ++c) {
        double num = 0.0;
        for (int k = 0; k < K; ++k) num += gqi[k] * Vt[(size_t)k * dv + c];
        On[c] = num / den;
        gdoto += g[(size_t)i * dv + c] * On[c];
      }
      const double dden = -gdoto / den;
      for (int c = 0; c < dv; ++c) dn[c] = g[(size_t)i * dv + c] / den;
      for (int k = 0; k < K; ++k) {
        double s = Z[k] * dden;
        for (int c = 0; c < dv; ++c) s += Vt[(size_t)k * dv + c] * dn[c];
        dg[k] = s;
        dZ[k] += gqi[k] * dden;
        for (int c = 0; c < dv; ++c) dVt[(size_t)k * dv + c] += gqi[k] * dn[c];
      }
      softmax_backward(K, gqi, dg, dl);
      logdensity_backward(d, K, q + (size_t)i * d, mu_h, s2_h, dl, dQ + ((size_t)u * N + i) * d, dmu_h, ds2_h, dlp_h);
    }
    /* keys: push dVt, dZ back through the write */
    for (int j = 0; j < N; ++j) {
      const double *gkj = gk + (size_t)j * K;
      for (int k = 0; k < K; ++k) {
        double s = dZ[k];
        for (int c = 0; c < dv; ++c) s += dVt[(size_t)k * dv + c] * v[(size_t)j * dv + c];
        dg[k] = s;
      }
      for (int c = 0; c < dv; ++c) {
        double s = 0.0;
        for (int k = 0; k < K; ++k) s += gkj[k] * dVt[(size_t)k * dv + c];
        dV[((size_t)u * N + j) * dv + c] = s;
      }
      softmax_backward(K, gkj, dg, dl);
      logdensity_backward(d, K, kx + (size_t)j * d, mu_h, s2_h, dl, dK + ((size_t)u * N + j) * d, dmu_h, ds2_h, dlp_h);
    }
  }
  free(gq); free(gk); free(ld); free(Vt); free(Z); free(dVt); free(dZ); free(dn); free(dg); free(dl); free(On);
  return 0;
}

/* [B] + [C] Gradients of the causal forward, given G = dL/dO.  Per (b, h), with the running state
 * S_i = sum_{j <= i} gamma_Kj [v_j | 1] (latent memory and normaliser after key i), den_i = gamma_Qi . Z_i
 * + eps, O_i = gamma_Qi . Vt_i / den_i, and u_i = [G_i / den_i | -(G_i . O_i) / den_i]:
 *   dgamma_Qi = S_i u_i,
 *   R_j = sum_{i >= j} gamma_Qi u_i^T (the suffix sum of the queries' contributions),
 *   dgamma_Kj = R_j [v_j | 1],   dv_j = R_j[:, :dv]^T gamma_Kj,
 * then the softmax and log-density steps of the bidirectional backward.  Forward over i, then
 * backward over j. */
int gma_oracle_backward_causal(int B, int H, int N, int d, int dv, int K, const double *Q, const double *Kx,
                               const double *V, const double *mu, const double *sigma2, const double *log_pi,
                               double eps, const double *G, double *dQ, double *dK, double *dV, double *dmu,
                               double *dsigma2, double *dlog_pi) {
  const int C = dv + 1;
  double *gq = (double *)malloc(sizeof(double) * (size_t)(N > 0 ? N : 1) * K);
  double *gk = (double *)malloc(sizeof(double) * (size_t)(N > 0 ? N : 1) * K);
  double *u = (double *)malloc(sizeof(double) * (size_t)(N > 0 ? N : 1) * C);
  double *ld = (double *)malloc(sizeof(double) * K);
  double *S = (double *)malloc(sizeof(double) * (size_t)K * C), *R = (double *)malloc(sizeof(double) * (size_t)K * C);
  double *dg = (double *)malloc(sizeof(double) * K), *dl = (double *)malloc(sizeof(double) * K);
  memset(dmu, 0, sizeof(double) * (size_t)H * K * d);
  memset(dsigma2, 0, sizeof(double) * (size_t)H * K * d);
  memset(dlog_pi, 0, sizeof(double) * (size_t)H * K);
  for (int unit = 0; unit < B * H; ++unit) {
    const int h = unit % H;
    const double *mu_h = mu + (size_t)h * K * d, *s2_h = sigma2 + (size_t)h * K * d, *lp_h = log_pi + (size_t)h * K;
    double *dmu_h = dmu + (size_t)h * K * d, *ds2_h = dsigma2 + (size_t)h * K * d, *dlp_h = dlog_pi + (size_t)h * K;
    const double *q = Q + (size_t)unit * N * d, *kx = Kx + (size_t)unit * N * d, *v = V + (size_t)unit * N * dv;
    const double *g = G + (size_t)unit * N * dv;
    log_determinants(d, K, s2_h, ld);
    memset(S, 0, sizeof(double) * (size_t)K * C);
    /* forward over i: running state, output, u_i, dgamma_Q */
    for (int i = 0; i < N; ++i) {
      double *gqi = gq + (size_t)i * K, *gki = gk + (size_t)i * K, *ui = u + (size_t)i * C;
      posterior(d, K, kx + (size_t)i * d, mu_h, s2_h, ld, lp_h, gki);
      for (int k = 0; k < K; ++k) {
        for (int c = 0; c < dv; ++c) S[(size_t)k * C + c] += gki[k] * v[(size_t)i * dv + c];
        S[(size_t)k * C + dv] += gki[k];
      }
      posterior(d, K, q + (size_t)i * d, mu_h, s2_h, ld, lp_h, gqi);
      double den = eps, go = 0.0;
      for (int k = 0; k < K; ++k) den += gqi[k] * S[(size_t)k * C + dv];
      for (int c = 0; c < dv; ++c) {
        double num = 0.0;
        for (int k = 0; k < K; ++k) num += gqi[k] * S[(size_t)k * C + c];
        go += g[(size_t)i * dv + c] * (num / den);
      }
      for (int c = 0; c < dv; ++c) ui[c] = g[(size_t)i * dv + c] / den;
      ui[dv] = -go / den;
      for (int k = 0; k < K; ++k) {
        double s = 0.0;
        for (int c = 0; c < C; ++c) s += S[(size_t)k * C + c] * ui[c];
        dg[k] = s;
      }
      softmax_backward(K, gqi, dg, dl);
      logdensity_backward(d, K, q + (size_t)i * d, mu_h, s2_h, dl, dQ + ((size_t)unit * N + i) * d, dmu_h, ds2_h, dlp_h);
    }
    /* backward over j: suffix sums R_j, dgamma_K and dv */
    memset(R, 0, sizeof(double) * (size_t)K * C);
    for (int j = N - 1; j >= 0; --j) {
      const double *gqj = gq + (size_t)j * K, *gkj = gk + (size_t)j * K, *uj = u + (size_t)j * C;
      for (int k = 0; k < K; ++k)
        for (int c = 0; c < C; ++c) R[(size_t)k * C + c] += gqj[k] * uj[c];
      for (int k = 0; k < K; ++k) {
        double s = R[(size_t)k * C + dv];
        for (int c = 0; c < dv; ++c) s += R[(size_t)k * C + c] * v[(size_t)j * dv + c];
        dg[k] = s;
      }
      for (int c = 0; c < dv; ++c) {
        double s = 0.0;
        for (int k = 0; k < K; ++k) s += gkj[k] * R[(size_t)k * C + c];
        dV[((size_t)unit * N + j) * dv + c] = s;
      }
      softmax_backward(K, gkj, dg, dl);
      logdensity_backward(d, K, kx + (size_t)j * d, mu_h, s2_h, dl, dK + ((size_t)unit * N + j) * d, dmu_h, ds2_h, dlp_h);
    }
  }
  free(gq); free(gk); free(u); free(ld); free(S); free(R); free(dg); free(dl);
  return 0;
}

/* Latent memory Vt [B,H,K,dv] and normaliser Z [B,H,K] over all N keys ([W]). */
int gma_oracle_state(int B, int H, int N, int d, int dv, int K, const double *Kx, const double *V, const double *mu,
                     const double *sigma2, const double *log_pi, double *Vt, double *Z) {
  double *g = (double *)malloc(sizeof(double) * (K > 0 ? K : 1));
  double *ld = (double *)malloc(sizeof(double) * (K > 0 ? K : 1));
  for (int u = 0; u < B * H; ++u) {
    int h = u % H;
    log_determinants(d, K, sigma2 + (size_t)h * K * d, ld);
    double *vt = Vt + (size_t)u * K * dv, *z = Z + (size_t)u * K;
    memset(vt, 0, sizeof(double) * K * dv);
    memset(z, 0, sizeof(double) * K);
    for (int j = 0; j < N; ++j) {
      posterior(d, K, Kx + ((size_t)u * N + j) * d, mu + (size_t)h * K * d, sigma2 + (size_t)h * K * d, ld,
                log_pi + (size_t)h * K, g);
      for (int k = 0; k < K; ++k) {
        z[k] += g[k];
        for (int c = 0; c < dv; ++c) vt[(size_t)k * dv + c] += g[k] * V[((size_t)u * N + j) * dv + c];
      }
    }
  }
  free(g);
  free(ld);
  return 0;
}
