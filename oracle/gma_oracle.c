/*
 * gma_oracle.c -- plain, slow, single-threaded fp64 CPU oracle for the
 * Gaussian Mixture Attention (GMA) forward pass and its gradients.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may link, load or
 * call this file: only the test-suite, the smoke check and the CPU-baseline
 * leg of the benchmark use it.  It shares no code, header, table or constant
 * with the CUDA library.
 *
 * Source of every definition below (cited as [GMA, ...]):
 *   "Gaussian Mixture Attention: Linear-Time Sequence Mixing via
 *    Probabilistic Latent Routing" (arXiv 2606.18283, HTML version),
 *   method section: Gaussian routing components, latent aggregation,
 *   normalized broadcasting, causal variant.
 *
 * Every function works on ONE head: row-major arrays
 *   X, Q, Kx : [N, d_r]      V : [N, d_v]      O : [N, d_v]
 *   mu, sigma2 : [K, d_r]    log_pi : [K]      Gamma : [N, K]
 * No blocking, no fusion, no reordering beyond what the definitions state.
 */
#include <math.h>
#include <stdlib.h>
#include <string.h>

/*
 * GMA_ORACLE_MUTANT (default 0) plants ONE deliberate mistake, so that the
 * test-suite can check that its pins catch it.  Builds with a non-zero value
 * are made only by tests/test_oracle_mutants.py; they are never the oracle.
 *   1: drop the per-component log-determinant term (log sigma2)
 *   2: divide the squared distance by sigma instead of sigma^2
 *   3: exclusive causal prefix (j < i) instead of inclusive (j <= i)
 *   4: eps added to the numerator as well as the denominator
 *   5: write with query responsibilities, read with key responsibilities
 *   6: prior enters with the wrong sign
 *   7: backward: the gradient entering the score is not mean-centred (Eq. 18)
 *   8: backward: the causal key gradient uses prefix (j <= i) instead of suffix sums
 *   9: decode step reads the memory before the new key enters it (exclusive)
 *  10: marginal usage counts hard assignments instead of summing responsibilities
 */
#ifndef GMA_ORACLE_MUTANT
#define GMA_ORACLE_MUTANT 0
#endif

/*
 * Log-density score of routing vector x under component k plus its log prior
 * ([GMA, the density under component k (Eq. 2) and the posterior
 * responsibility p(z_i = k | x_i) (Eq. 3)], and the score form s_{i,k} used
 * before the softmax in the gradient section).  The display equations were
 * lost in extraction; the prose fixes a diagonal-covariance Gaussian density
 * times the prior pi_k.  Written out, up to the constant -(d_r/2) log(2 pi),
 * which is the same for every k and cancels in the softmax:
 *
 *   s_{i,k} = log pi_k - 1/2 sum_j [ (x_ij - mu_kj)^2 / sigma2_kj + log sigma2_kj ]
 *
 * This is the centred form, evaluated term by term.
 */
static double score_one(const double *x, const double *mu_k, const double *s2_k,
                        double log_pi_k, int d_r)
{
    double q = 0.0;
    for (int j = 0; j < d_r; ++j) {
        double diff = x[j] - mu_k[j];
#if GMA_ORACLE_MUTANT == 1
        q += diff * diff / s2_k[j];
#elif GMA_ORACLE_MUTANT == 2
        q += diff * diff / sqrt(s2_k[j]) + log(s2_k[j]);
#else
        q += diff * diff / s2_k[j] + log(s2_k[j]);
#endif
    }
#if GMA_ORACLE_MUTANT == 6
    return -log_pi_k - 0.5 * q;
#else
    return log_pi_k - 0.5 * q;
#endif
}

void gma_oracle_scores(const double *X, int N, int d_r, const double *mu,
                       const double *sigma2, const double *log_pi, int K,
                       double *S)
{
    for (int i = 0; i < N; ++i)
        for (int k = 0; k < K; ++k)
            S[(size_t)i * K + k] = score_one(X + (size_t)i * d_r, mu + (size_t)k * d_r,
                                             sigma2 + (size_t)k * d_r, log_pi[k], d_r);
}

/*
 * Responsibilities ([GMA, Eq. 3]; "each row of Gamma is a probability
 * distribution over the latent Gaussian components"): the posterior is the
 * softmax over k of the scores.  The row maximum is subtracted before the
 * exponential, which changes nothing in exact arithmetic.
 */
void gma_oracle_responsibilities(const double *X, int N, int d_r, const double *mu,
                                 const double *sigma2, const double *log_pi, int K,
                                 double *Gamma)
{
    gma_oracle_scores(X, N, d_r, mu, sigma2, log_pi, K, Gamma);
    for (int i = 0; i < N; ++i) {
        double *g = Gamma + (size_t)i * K;
        double m = g[0];
        for (int k = 1; k < K; ++k)
            if (g[k] > m) m = g[k];
        double z = 0.0;
        for (int k = 0; k < K; ++k) {
            g[k] = exp(g[k] - m);
            z += g[k];
        }
        for (int k = 0; k < K; ++k) g[k] /= z;
    }
}

/*
 * Bidirectional GMA forward ([GMA, Eqs. 5-7 and footnote 4]).
 *   Latent aggregation (Eqs. 5, 6):  Vt_k = sum_j gK_jk V_j,  Z_k = sum_j gK_jk
 *   Normalized broadcasting (Eq. 7): O_i  = (sum_k gQ_ik Vt_k) / (sum_k gQ_ik Z_k + eps)
 * eps is added after the sum over k (footnote 4: d = Gamma^Q Z + eps 1_N).
 */
void gma_oracle_bidir(const double *Q, const double *Kx, const double *V, int N,
                      int d_r, int d_v, const double *mu, const double *sigma2,
                      const double *log_pi, int K, double eps, double *O)
{
    double *GQ = malloc(sizeof(double) * (size_t)N * K);
    double *GK = malloc(sizeof(double) * (size_t)N * K);
    double *Vt = calloc((size_t)K * d_v, sizeof(double));
    double *Z = calloc((size_t)K, sizeof(double));
#if GMA_ORACLE_MUTANT == 5
    gma_oracle_responsibilities(Kx, N, d_r, mu, sigma2, log_pi, K, GQ);
    gma_oracle_responsibilities(Q, N, d_r, mu, sigma2, log_pi, K, GK);
#else
    gma_oracle_responsibilities(Q, N, d_r, mu, sigma2, log_pi, K, GQ);
    gma_oracle_responsibilities(Kx, N, d_r, mu, sigma2, log_pi, K, GK);
#endif

    for (int j = 0; j < N; ++j)
        for (int k = 0; k < K; ++k) {
            double g = GK[(size_t)j * K + k];
            Z[k] += g;
            for (int c = 0; c < d_v; ++c) Vt[(size_t)k * d_v + c] += g * V[(size_t)j * d_v + c];
        }

    for (int i = 0; i < N; ++i) {
        double den = 0.0;
        for (int k = 0; k < K; ++k) den += GQ[(size_t)i * K + k] * Z[k];
        den += eps;
        for (int c = 0; c < d_v; ++c) {
            double num = 0.0;
            for (int k = 0; k < K; ++k) num += GQ[(size_t)i * K + k] * Vt[(size_t)k * d_v + c];
#if GMA_ORACLE_MUTANT == 4
            num += eps;
#endif
            O[(size_t)i * d_v + c] = num / den;
        }
    }
    free(GQ); free(GK); free(Vt); free(Z);
}

/*
 * Causal GMA forward ([GMA, causal variant, Eqs. 8a/8b and the remark that
 * the prefix memories are cumulative sums along the sequence]).
 *   Vt^(i)_k = sum_{j<=i} gK_jk V_j,   Z^(i)_k = sum_{j<=i} gK_jk   (j <= i inclusive)
 *   O_i = (sum_k gQ_ik Vt^(i)_k) / (sum_k gQ_ik Z^(i)_k + eps)
 * The prefix memories are carried as running sums, one position at a time.
 */
void gma_oracle_causal(const double *Q, const double *Kx, const double *V, int N,
                       int d_r, int d_v, const double *mu, const double *sigma2,
                       const double *log_pi, int K, double eps, double *O)
{
    double *GQ = malloc(sizeof(double) * (size_t)N * K);
    double *GK = malloc(sizeof(double) * (size_t)N * K);
    double *Vt = calloc((size_t)K * d_v, sizeof(double));
    double *Z = calloc((size_t)K, sizeof(double));
    gma_oracle_responsibilities(Q, N, d_r, mu, sigma2, log_pi, K, GQ);
    gma_oracle_responsibilities(Kx, N, d_r, mu, sigma2, log_pi, K, GK);

    for (int i = 0; i < N; ++i) {
#if GMA_ORACLE_MUTANT != 3
        /* extend the prefix memory with key/value i */
        for (int k = 0; k < K; ++k) {
            double g = GK[(size_t)i * K + k];
            Z[k] += g;
            for (int c = 0; c < d_v; ++c) Vt[(size_t)k * d_v + c] += g * V[(size_t)i * d_v + c];
        }
#endif
        /* read it with query i */
        double den = 0.0;
        for (int k = 0; k < K; ++k) den += GQ[(size_t)i * K + k] * Z[k];
        den += eps;
        for (int c = 0; c < d_v; ++c) {
            double num = 0.0;
            for (int k = 0; k < K; ++k) num += GQ[(size_t)i * K + k] * Vt[(size_t)k * d_v + c];
#if GMA_ORACLE_MUTANT == 4
            num += eps;
#endif
            O[(size_t)i * d_v + c] = num / den;
        }
#if GMA_ORACLE_MUTANT == 3
        for (int k = 0; k < K; ++k) {
            double g = GK[(size_t)i * K + k];
            Z[k] += g;
            for (int c = 0; c < d_v; ++c) Vt[(size_t)k * d_v + c] += g * V[(size_t)i * d_v + c];
        }
#endif
    }
    free(GQ); free(GK); free(Vt); free(Z);
}

/*
 * Selected output rows, for checks at sizes where the full O is too slow.
 * Bidirectional: the full latent memory is built once (Eqs. 5, 6), then only
 * the requested query rows are read (Eq. 7).  Causal: the running prefix is
 * advanced to each requested row in increasing order (rows must be sorted
 * ascending), reading the query there (Eq. 8b).
 */
void gma_oracle_bidir_rows(const double *Q, const double *Kx, const double *V, int N,
                           int d_r, int d_v, const double *mu, const double *sigma2,
                           const double *log_pi, int K, double eps,
                           const long *rows, int nrows, double *O_rows)
{
    double *gk = malloc(sizeof(double) * (size_t)K);
    double *gq = malloc(sizeof(double) * (size_t)K);
    double *Vt = calloc((size_t)K * d_v, sizeof(double));
    double *Z = calloc((size_t)K, sizeof(double));
    for (int j = 0; j < N; ++j) {
        gma_oracle_responsibilities(Kx + (size_t)j * d_r, 1, d_r, mu, sigma2, log_pi, K, gk);
        for (int k = 0; k < K; ++k) {
            Z[k] += gk[k];
            for (int c = 0; c < d_v; ++c) Vt[(size_t)k * d_v + c] += gk[k] * V[(size_t)j * d_v + c];
        }
    }
    for (int r = 0; r < nrows; ++r) {
        long i = rows[r];
        gma_oracle_responsibilities(Q + (size_t)i * d_r, 1, d_r, mu, sigma2, log_pi, K, gq);
        double den = eps;
        for (int k = 0; k < K; ++k) den += gq[k] * Z[k];
        for (int c = 0; c < d_v; ++c) {
            double num = 0.0;
            for (int k = 0; k < K; ++k) num += gq[k] * Vt[(size_t)k * d_v + c];
            O_rows[(size_t)r * d_v + c] = num / den;
        }
    }
    free(gk); free(gq); free(Vt); free(Z);
}

int gma_oracle_causal_rows(const double *Q, const double *Kx, const double *V, int N,
                           int d_r, int d_v, const double *mu, const double *sigma2,
                           const double *log_pi, int K, double eps,
                           const long *rows, int nrows, double *O_rows)
{
    for (int r = 1; r < nrows; ++r)
        if (rows[r] < rows[r - 1]) return -1;
    if (nrows > 0 && (rows[0] < 0 || rows[nrows - 1] >= N)) return -1;
    double *gk = malloc(sizeof(double) * (size_t)K);
    double *gq = malloc(sizeof(double) * (size_t)K);
    double *Vt = calloc((size_t)K * d_v, sizeof(double));
    double *Z = calloc((size_t)K, sizeof(double));
    long next = 0; /* keys 0..next-1 are already in the prefix */
    for (int r = 0; r < nrows; ++r) {
        long i = rows[r];
        for (; next <= i; ++next) {
            gma_oracle_responsibilities(Kx + (size_t)next * d_r, 1, d_r, mu, sigma2, log_pi, K, gk);
            for (int k = 0; k < K; ++k) {
                Z[k] += gk[k];
                for (int c = 0; c < d_v; ++c) Vt[(size_t)k * d_v + c] += gk[k] * V[(size_t)next * d_v + c];
            }
        }
        gma_oracle_responsibilities(Q + (size_t)i * d_r, 1, d_r, mu, sigma2, log_pi, K, gq);
        double den = eps;
        for (int k = 0; k < K; ++k) den += gq[k] * Z[k];
        for (int c = 0; c < d_v; ++c) {
            double num = 0.0;
            for (int k = 0; k < K; ++k) num += gq[k] * Vt[(size_t)k * d_v + c];
            O_rows[(size_t)r * d_v + c] = num / den;
        }
    }
    free(gk); free(gq); free(Vt); free(Z);
    return 0;
}

/*
 * Brute force through the materialised affinity, for tiny N only
 * ([GMA, Eqs. 9-11 and footnote 4]):
 *   Atilde_ij = <gQ_i, gK_j>          (Eq. 11, un-normalised affinity)
 *   d_i       = sum_l Atilde_il + eps  (row normaliser; equals gQ_i . Z + eps)
 *   O_i       = (sum_j Atilde_ij V_j) / d_i   (Eqs. 9-10: O = A^GMA V_X)
 * causal != 0 applies the lower-triangular (j <= i) mask of the causal
 * variant before the row sums.  Shares only the score routine above.
 */
void gma_oracle_affinity_forward(const double *Q, const double *Kx, const double *V,
                                 int N, int d_r, int d_v, const double *mu,
                                 const double *sigma2, const double *log_pi, int K,
                                 double eps, int causal, double *O)
{
    double *GQ = malloc(sizeof(double) * (size_t)N * K);
    double *GK = malloc(sizeof(double) * (size_t)N * K);
    double *A = malloc(sizeof(double) * (size_t)N * N);
    gma_oracle_responsibilities(Q, N, d_r, mu, sigma2, log_pi, K, GQ);
    gma_oracle_responsibilities(Kx, N, d_r, mu, sigma2, log_pi, K, GK);
    for (int i = 0; i < N; ++i)
        for (int j = 0; j < N; ++j) {
            double a = 0.0;
            if (!causal || j <= i)
                for (int k = 0; k < K; ++k) a += GQ[(size_t)i * K + k] * GK[(size_t)j * K + k];
            A[(size_t)i * N + j] = a;
        }
    for (int i = 0; i < N; ++i) {
        double d = eps;
        for (int j = 0; j < N; ++j) d += A[(size_t)i * N + j];
        for (int c = 0; c < d_v; ++c) {
            double num = 0.0;
            for (int j = 0; j < N; ++j) num += A[(size_t)i * N + j] * V[(size_t)j * d_v + c];
            O[(size_t)i * d_v + c] = num / d;
        }
    }
    free(GQ); free(GK); free(A);
}

/* Materialised un-normalised affinity Atilde = Gamma^Q (Gamma^K)^T ([GMA, Eq. 11]). */
void gma_oracle_affinity(const double *Q, const double *Kx, int N, int d_r,
                         const double *mu, const double *sigma2, const double *log_pi,
                         int K, double *A)
{
    double *GQ = malloc(sizeof(double) * (size_t)N * K);
    double *GK = malloc(sizeof(double) * (size_t)N * K);
    gma_oracle_responsibilities(Q, N, d_r, mu, sigma2, log_pi, K, GQ);
    gma_oracle_responsibilities(Kx, N, d_r, mu, sigma2, log_pi, K, GK);
    for (int i = 0; i < N; ++i)
        for (int j = 0; j < N; ++j) {
            double a = 0.0;
            for (int k = 0; k < K; ++k) a += GQ[(size_t)i * K + k] * GK[(size_t)j * K + k];
            A[(size_t)i * N + j] = a;
        }
    free(GQ); free(GK);
}

/*
 * ---------------------------------------------------------------- gradients
 *
 * Backward pass of one head ([GMA, gradient section]: the upstream gradient
 * g_ik = dL/dgamma_ik arriving at a responsibility row, the softmax Jacobian
 * (Eq. 17) and the gradient entering the score (Eq. 18),
 *   dL/ds_ik = gamma_ik (g_ik - sum_l gamma_il g_il),
 * then the chain rule for every quantity that enters the score).  Through
 *   s_ik = log pi_k - 1/2 sum_m [ (x_im - mu_km)^2 / sigma2_km + log sigma2_km ]
 * the score gradient reaches
 *   dL/dx_im       = sum_k ds_ik (mu_km - x_im) / sigma2_km
 *   dL/dmu_km      = sum_i ds_ik (x_im - mu_km) / sigma2_km
 *   dL/dsigma2_km  = sum_i ds_ik ((x_im - mu_km)^2 / sigma2_km^2 - 1 / sigma2_km) / 2
 *   dL/dlog_pi_k   = sum_i ds_ik
 * for the query rows (x = q) and the key rows (x = k) alike.  dmu, dsigma2 and
 * dlog_pi are ACCUMULATED (the caller zeroes them once and sums every head and
 * batch row that shares the parameters); dX is written.
 */
static void score_backward(const double *X, const double *G, const double *Gup, int N,
                           int d_r, const double *mu, const double *sigma2, int K,
                           double *dX, double *dmu, double *dsigma2, double *dlog_pi)
{
    double *ds = malloc(sizeof(double) * (size_t)K);
    for (int i = 0; i < N; ++i) {
        const double *g = G + (size_t)i * K, *up = Gup + (size_t)i * K;
        const double *x = X + (size_t)i * d_r;
        double mean = 0.0;
        for (int l = 0; l < K; ++l) mean += g[l] * up[l];
        for (int k = 0; k < K; ++k) {
#if GMA_ORACLE_MUTANT == 7
            ds[k] = g[k] * up[k];
#else
            ds[k] = g[k] * (up[k] - mean);
#endif
        }
        for (int m = 0; m < d_r; ++m) {
            double acc = 0.0;
            for (int k = 0; k < K; ++k)
                acc += ds[k] * (mu[(size_t)k * d_r + m] - x[m]) / sigma2[(size_t)k * d_r + m];
            dX[(size_t)i * d_r + m] = acc;
        }
        for (int k = 0; k < K; ++k) {
            dlog_pi[k] += ds[k];
            for (int m = 0; m < d_r; ++m) {
                const double s2 = sigma2[(size_t)k * d_r + m];
                const double diff = x[m] - mu[(size_t)k * d_r + m];
                dmu[(size_t)k * d_r + m] += ds[k] * diff / s2;
                dsigma2[(size_t)k * d_r + m] += ds[k] * 0.5 * (diff * diff / (s2 * s2) - 1.0 / s2);
            }
        }
    }
    free(ds);
}

/*
 * Bidirectional backward ([GMA, Eqs. 5-7] differentiated).  With
 *   num_i = sum_k gQ_ik Vt_k,  den_i = sum_k gQ_ik Z_k + eps,  O_i = num_i / den_i
 * and the upstream dO:
 *   dnum_i = dO_i / den_i,                 dden_i = -(dO_i . O_i) / den_i
 *   dL/dgQ_ik = dnum_i . Vt_k + dden_i Z_k
 *   dVt_k = sum_i gQ_ik dnum_i,            dZ_k = sum_i gQ_ik dden_i
 *   dL/dgK_jk = V_j . dVt_k + dZ_k,        dV_j = sum_k gK_jk dVt_k
 * then score_backward for both sides.
 */
void gma_oracle_bidir_backward(const double *Q, const double *Kx, const double *V, int N,
                               int d_r, int d_v, const double *mu, const double *sigma2,
                               const double *log_pi, int K, double eps, const double *dO,
                               double *dQ, double *dK, double *dV, double *dmu,
                               double *dsigma2, double *dlog_pi)
{
    double *GQ = malloc(sizeof(double) * (size_t)N * K);
    double *GK = malloc(sizeof(double) * (size_t)N * K);
    double *UQ = malloc(sizeof(double) * (size_t)N * K);
    double *UK = malloc(sizeof(double) * (size_t)N * K);
    double *Vt = calloc((size_t)K * d_v, sizeof(double));
    double *Z = calloc((size_t)K, sizeof(double));
    double *dVt = calloc((size_t)K * d_v, sizeof(double));
    double *dZ = calloc((size_t)K, sizeof(double));
    double *dnum = malloc(sizeof(double) * (size_t)d_v);
    gma_oracle_responsibilities(Q, N, d_r, mu, sigma2, log_pi, K, GQ);
    gma_oracle_responsibilities(Kx, N, d_r, mu, sigma2, log_pi, K, GK);
    for (int j = 0; j < N; ++j)
        for (int k = 0; k < K; ++k) {
            double g = GK[(size_t)j * K + k];
            Z[k] += g;
            for (int c = 0; c < d_v; ++c) Vt[(size_t)k * d_v + c] += g * V[(size_t)j * d_v + c];
        }
    for (int i = 0; i < N; ++i) {
        const double *gq = GQ + (size_t)i * K;
        double den = eps;
        for (int k = 0; k < K; ++k) den += gq[k] * Z[k];
        double dot = 0.0;
        for (int c = 0; c < d_v; ++c) {
            double num = 0.0;
            for (int k = 0; k < K; ++k) num += gq[k] * Vt[(size_t)k * d_v + c];
            dot += dO[(size_t)i * d_v + c] * (num / den);
            dnum[c] = dO[(size_t)i * d_v + c] / den;
        }
        const double dden = -dot / den;
        for (int k = 0; k < K; ++k) {
            double u = dden * Z[k];
            for (int c = 0; c < d_v; ++c) u += dnum[c] * Vt[(size_t)k * d_v + c];
            UQ[(size_t)i * K + k] = u;
            dZ[k] += gq[k] * dden;
            for (int c = 0; c < d_v; ++c) dVt[(size_t)k * d_v + c] += gq[k] * dnum[c];
        }
    }
    for (int j = 0; j < N; ++j)
        for (int k = 0; k < K; ++k) {
            double u = dZ[k];
            for (int c = 0; c < d_v; ++c) u += V[(size_t)j * d_v + c] * dVt[(size_t)k * d_v + c];
            UK[(size_t)j * K + k] = u;
        }
    for (int j = 0; j < N; ++j)
        for (int c = 0; c < d_v; ++c) {
            double acc = 0.0;
            for (int k = 0; k < K; ++k) acc += GK[(size_t)j * K + k] * dVt[(size_t)k * d_v + c];
            dV[(size_t)j * d_v + c] = acc;
        }
    score_backward(Q, GQ, UQ, N, d_r, mu, sigma2, K, dQ, dmu, dsigma2, dlog_pi);
    score_backward(Kx, GK, UK, N, d_r, mu, sigma2, K, dK, dmu, dsigma2, dlog_pi);
    free(GQ); free(GK); free(UQ); free(UK); free(Vt); free(Z); free(dVt); free(dZ); free(dnum);
}

/*
 * Causal backward ([GMA, Eq. 8b] differentiated).  The query side is as in the
 * bidirectional case with the prefix memories Vt^(i), Z^(i) (j <= i) in place
 * of the whole-sequence ones; a key j reaches every query i >= j, so its
 * gradient collects the SUFFIX sums
 *   D^(j)_k = sum_{i>=j} gQ_ik dnum_i,     E^(j)_k = sum_{i>=j} gQ_ik dden_i
 *   dL/dgK_jk = V_j . D^(j)_k + E^(j)_k,   dV_j = sum_k gK_jk D^(j)_k
 * The prefix memories are carried forward one position at a time, the suffix
 * sums backward one position at a time.
 */
void gma_oracle_causal_backward(const double *Q, const double *Kx, const double *V, int N,
                                int d_r, int d_v, const double *mu, const double *sigma2,
                                const double *log_pi, int K, double eps, const double *dO,
                                double *dQ, double *dK, double *dV, double *dmu,
                                double *dsigma2, double *dlog_pi)
{
    double *GQ = malloc(sizeof(double) * (size_t)N * K);
    double *GK = malloc(sizeof(double) * (size_t)N * K);
    double *UQ = malloc(sizeof(double) * (size_t)N * K);
    double *UK = malloc(sizeof(double) * (size_t)N * K);
    double *DN = malloc(sizeof(double) * (size_t)N * d_v);   /* dnum_i */
    double *DD = malloc(sizeof(double) * (size_t)N);         /* dden_i */
    double *Vt = calloc((size_t)K * d_v, sizeof(double));
    double *Z = calloc((size_t)K, sizeof(double));
    double *D = calloc((size_t)K * d_v, sizeof(double));
    double *E = calloc((size_t)K, sizeof(double));
    gma_oracle_responsibilities(Q, N, d_r, mu, sigma2, log_pi, K, GQ);
    gma_oracle_responsibilities(Kx, N, d_r, mu, sigma2, log_pi, K, GK);
    for (int i = 0; i < N; ++i) {
        for (int k = 0; k < K; ++k) {
            double g = GK[(size_t)i * K + k];
            Z[k] += g;
            for (int c = 0; c < d_v; ++c) Vt[(size_t)k * d_v + c] += g * V[(size_t)i * d_v + c];
        }
        const double *gq = GQ + (size_t)i * K;
        double den = eps;
        for (int k = 0; k < K; ++k) den += gq[k] * Z[k];
        double dot = 0.0;
        for (int c = 0; c < d_v; ++c) {
            double num = 0.0;
            for (int k = 0; k < K; ++k) num += gq[k] * Vt[(size_t)k * d_v + c];
            dot += dO[(size_t)i * d_v + c] * (num / den);
            DN[(size_t)i * d_v + c] = dO[(size_t)i * d_v + c] / den;
        }
        DD[i] = -dot / den;
        for (int k = 0; k < K; ++k) {
            double u = DD[i] * Z[k];
            for (int c = 0; c < d_v; ++c) u += DN[(size_t)i * d_v + c] * Vt[(size_t)k * d_v + c];
            UQ[(size_t)i * K + k] = u;
        }
    }
#if GMA_ORACLE_MUTANT == 8
    for (int j = 0; j < N; ++j) {
#else
    for (int j = N - 1; j >= 0; --j) {
#endif
        for (int k = 0; k < K; ++k) {
            double g = GQ[(size_t)j * K + k];
            E[k] += g * DD[j];
            for (int c = 0; c < d_v; ++c) D[(size_t)k * d_v + c] += g * DN[(size_t)j * d_v + c];
        }
        for (int k = 0; k < K; ++k) {
            double u = E[k];
            for (int c = 0; c < d_v; ++c) u += V[(size_t)j * d_v + c] * D[(size_t)k * d_v + c];
            UK[(size_t)j * K + k] = u;
        }
        for (int c = 0; c < d_v; ++c) {
            double acc = 0.0;
            for (int k = 0; k < K; ++k) acc += GK[(size_t)j * K + k] * D[(size_t)k * d_v + c];
            dV[(size_t)j * d_v + c] = acc;
        }
    }
    score_backward(Q, GQ, UQ, N, d_r, mu, sigma2, K, dQ, dmu, dsigma2, dlog_pi);
    score_backward(Kx, GK, UK, N, d_r, mu, sigma2, K, dK, dmu, dsigma2, dlog_pi);
    free(GQ); free(GK); free(UQ); free(UK); free(DN); free(DD);
    free(Vt); free(Z); free(D); free(E);
}

/*
 * Latent memory of a key/value sequence ([GMA, Eqs. 5-6], latent aggregation):
 *   Vt_k = sum_j gK_jk V_j,   Z_k = sum_j gK_jk.
 * This is also the causal carried state after the last position ([GMA, causal
 * variant]: the prefix memories at i = N - 1), i.e. what a decoder holds after
 * reading a prompt of N tokens.  Vt [K, d_v], Z [K] are overwritten.
 */
void gma_oracle_latent_memory(const double *Kx, const double *V, int N, int d_r, int d_v,
                              const double *mu, const double *sigma2, const double *log_pi,
                              int K, double *Vt, double *Z)
{
    double *gk = malloc(sizeof(double) * (size_t)K);
    for (int k = 0; k < K; ++k) {
        Z[k] = 0.0;
        for (int c = 0; c < d_v; ++c) Vt[(size_t)k * d_v + c] = 0.0;
    }
    for (int j = 0; j < N; ++j) {
        gma_oracle_responsibilities(Kx + (size_t)j * d_r, 1, d_r, mu, sigma2, log_pi, K, gk);
        for (int k = 0; k < K; ++k) {
            Z[k] += gk[k];
            for (int c = 0; c < d_v; ++c) Vt[(size_t)k * d_v + c] += gk[k] * V[(size_t)j * d_v + c];
        }
    }
    free(gk);
}

/*
 * One autoregressive step of the causal variant ([GMA, causal variant, Eq. 8b]
 * with the prefix memories carried as running sums).  Given the memory of the
 * positions before i (Vt, Z) and the new position's query q, key k and value v:
 *   Vt_k += gK_k v,  Z_k += gK_k          (position i enters its own prefix: j <= i)
 *   o = (sum_k gQ_k Vt_k) / (sum_k gQ_k Z_k + eps)
 * Vt [K, d_v] and Z [K] are updated in place; o [d_v] is written.
 */
void gma_oracle_decode_step(const double *q, const double *kx, const double *v, int d_r, int d_v,
                            const double *mu, const double *sigma2, const double *log_pi, int K,
                            double eps, double *Vt, double *Z, double *o)
{
    double *gk = malloc(sizeof(double) * (size_t)K);
    double *gq = malloc(sizeof(double) * (size_t)K);
    gma_oracle_responsibilities(kx, 1, d_r, mu, sigma2, log_pi, K, gk);
    gma_oracle_responsibilities(q, 1, d_r, mu, sigma2, log_pi, K, gq);
#if GMA_ORACLE_MUTANT != 9
    for (int k = 0; k < K; ++k) {
        Z[k] += gk[k];
        for (int c = 0; c < d_v; ++c) Vt[(size_t)k * d_v + c] += gk[k] * v[c];
    }
#endif
    double den = eps;
    for (int k = 0; k < K; ++k) den += gq[k] * Z[k];
    for (int c = 0; c < d_v; ++c) {
        double num = 0.0;
        for (int k = 0; k < K; ++k) num += gq[k] * Vt[(size_t)k * d_v + c];
        o[c] = num / den;
    }
#if GMA_ORACLE_MUTANT == 9
    for (int k = 0; k < K; ++k) {
        Z[k] += gk[k];
        for (int c = 0; c < d_v; ++c) Vt[(size_t)k * d_v + c] += gk[k] * v[c];
    }
#endif
    free(gk); free(gq);
}

/*
 * Component-usage diagnostics of one head's responsibilities ([GMA,
 * introduction: the marginal usage of the mixture components shows whether
 * the routing space is used broadly or collapses onto a few components, and
 * the hard assignment z_i = argmax_k gamma_ik can be compared with token
 * categories]; the interpretability results quote the number of components
 * used and a usage entropy).
 *   usage_k  = sum_i gamma_ik                       (soft, marginal usage)
 *   z_i      = argmax_k gamma_ik, the smallest such k on ties (hard assignment)
 *   counts_k = #{i : z_i = k}
 *   p_k      = usage_k / N,  H = -sum_{k: p_k > 0} p_k log p_k  (nats)
 *   H_norm   = H / log K  (K >= 2), 1 for K = 1 (one component is trivially uniform)
 *   used     = #{k : counts_k > 0}
 * z may be NULL.  stats[0] = H, stats[1] = H_norm, stats[2] = used.
 */
void gma_oracle_routing_stats(const double *X, int N, int d_r, const double *mu,
                              const double *sigma2, const double *log_pi, int K,
                              double *usage, long *counts, long *z, double *stats)
{
    double *g = malloc(sizeof(double) * (size_t)K);
    for (int k = 0; k < K; ++k) { usage[k] = 0.0; counts[k] = 0; }
    for (int i = 0; i < N; ++i) {
        gma_oracle_responsibilities(X + (size_t)i * d_r, 1, d_r, mu, sigma2, log_pi, K, g);
        int best = 0;
        for (int k = 1; k < K; ++k)
            if (g[k] > g[best]) best = k;
        counts[best] += 1;
        if (z) z[i] = best;
#if GMA_ORACLE_MUTANT == 10
        usage[best] += 1.0;
#else
        for (int k = 0; k < K; ++k) usage[k] += g[k];
#endif
    }
    double H = 0.0;
    long used = 0;
    for (int k = 0; k < K; ++k) {
        double p = usage[k] / (double)N;
        if (p > 0.0) H -= p * log(p);
        if (counts[k] > 0) used += 1;
    }
    stats[0] = H;
    stats[1] = K >= 2 ? H / log((double)K) : 1.0;
    stats[2] = (double)used;
    free(g);
}

/*
 * Normalized broadcasting from a given latent memory ([GMA, Eq. 7], footnote 4):
 *   O_i = (sum_k gQ_ik Vt_k) / (sum_k gQ_ik Z_k + eps)
 * with Vt [K, d_v], Z [K] supplied by the caller (for example the sum of the
 * latent memories of several key/value shards).
 */
void gma_oracle_read_memory(const double *Q, int N, int d_r, int d_v, const double *mu,
                            const double *sigma2, const double *log_pi, int K, double eps,
                            const double *Vt, const double *Z, double *O)
{
    double *gq = malloc(sizeof(double) * (size_t)K);
    for (int i = 0; i < N; ++i) {
        gma_oracle_responsibilities(Q + (size_t)i * d_r, 1, d_r, mu, sigma2, log_pi, K, gq);
        double den = eps;
        for (int k = 0; k < K; ++k) den += gq[k] * Z[k];
        for (int c = 0; c < d_v; ++c) {
            double num = 0.0;
            for (int k = 0; k < K; ++k) num += gq[k] * Vt[(size_t)k * d_v + c];
            O[(size_t)i * d_v + c] = num / den;
        }
    }
    free(gq);
}

/*
 * Reparameterised mixture parameters of one head ([GMA, Eqs. 14-15]):
 *   sigma2_kj = log(1 + exp(omega_kj)) + eps_sigma        (softplus, Eq. 14)
 *   pi_k      = exp(alpha_k) / sum_l exp(alpha_l)          (softmax, Eq. 15)
 * returned as log_pi_k = alpha_k - log sum_l exp(alpha_l).  The softplus is
 * evaluated as max(w, 0) + log1p(exp(-|w|)) and the log-sum-exp with the
 * maximum taken out, which are the same functions without overflow.
 */
void gma_oracle_reparameterize(const double *omega, const double *alpha, int K, int d_r,
                               double eps_sigma, double *sigma2, double *log_pi)
{
    for (int e = 0; e < K * d_r; ++e) {
        double w = omega[e];
        sigma2[e] = (w > 0.0 ? w : 0.0) + log1p(exp(-fabs(w))) + eps_sigma;
    }
    double m = alpha[0];
    for (int k = 1; k < K; ++k)
        if (alpha[k] > m) m = alpha[k];
    double z = 0.0;
    for (int k = 0; k < K; ++k) z += exp(alpha[k] - m);
    double lse = m + log(z);
    for (int k = 0; k < K; ++k) log_pi[k] = alpha[k] - lse;
}

/*
 * Chain rule through the reparameterisations (the gradient appendix's
 * reparameterised means, covariances and prior logits):
 *   d omega_kj = d sigma2_kj * sigmoid(omega_kj)          (d softplus / d w = sigmoid(w))
 *   d alpha_k  = d log_pi_k - pi_k * sum_l d log_pi_l      (Jacobian of log-softmax)
 */
void gma_oracle_reparameterize_backward(const double *omega, const double *alpha, int K, int d_r,
                                        const double *dsigma2, const double *dlog_pi,
                                        double *domega, double *dalpha)
{
    for (int e = 0; e < K * d_r; ++e) {
        double w = omega[e];
        double sg = w >= 0.0 ? 1.0 / (1.0 + exp(-w)) : exp(w) / (1.0 + exp(w));
        domega[e] = dsigma2[e] * sg;
    }
    double m = alpha[0];
    for (int k = 1; k < K; ++k)
        if (alpha[k] > m) m = alpha[k];
    double z = 0.0, g = 0.0;
    for (int k = 0; k < K; ++k) { z += exp(alpha[k] - m); g += dlog_pi[k]; }
    for (int k = 0; k < K; ++k) dalpha[k] = dlog_pi[k] - exp(alpha[k] - m) / z * g;
}

/*
 * Projection of the input rows into the routing and value spaces ([GMA, the
 * projections of Eq. 4]: Q_X, K_X, V_X are linear maps of the layer input X;
 * the display equation was lost in extraction, the plainest reading being
 * Q_X = X W_Q and the like).  Weights are stored [out, in] (one output
 * feature per row):
 *   Y[m, o] = sum_i X[m, i] W[o, i]      X : [M, D]   W : [O, D]   Y : [M, O]
 */
void gma_oracle_project(const double *X, int M, int D, const double *W, int O, double *Y)
{
    for (int m = 0; m < M; ++m)
        for (int o = 0; o < O; ++o) {
            double acc = 0.0;
            for (int i = 0; i < D; ++i) acc += X[(size_t)m * D + i] * W[(size_t)o * D + i];
            Y[(size_t)m * O + o] = acc;
        }
}
