/*
 * gma_oracle.c -- plain, slow, single-threaded fp64 CPU oracle for the
 * Gaussian Mixture Attention (GMA) forward pass.
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
