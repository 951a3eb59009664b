// gma_param.cu -- the reparameterised mixture parameters and the chain rule
// through them.
//
// Paper: "Gaussian Mixture Attention: Linear-Time Sequence Mixing via
// Probabilistic Latent Routing" (arXiv 2606.18283), Eqs. (14)-(15):
//   sigma2_kj = log(1 + exp(omega_kj)) + eps_sigma     (softplus keeps the
//                                                      covariances positive)
//   pi_k      = softmax_k(alpha)                       (priors on the simplex)
// produced as log_pi (what the forward entry points take), and the gradients
//   d omega_kj = d sigma2_kj * sigmoid(omega_kj)
//   d alpha_k  = d log_pi_k - pi_k * sum_l d log_pi_l.
// Grid (element chunks, H): every CTA takes kParamChunk covariance elements of
// its head (many CTAs, so many loads in flight), and the first CTA of each head
// also does the priors, whose log-sum-exp and gradient sum are taken by one
// thread in component order (K <= 128), so results are reproducible.
#include <cmath>

#include "gma_internal.h"

namespace gma {
namespace {

constexpr int kParamThreads = 256;
constexpr int kParamChunk = 4 * kParamThreads;  // covariance elements per CTA

// softplus(w) = max(w, 0) + log1p(exp(-|w|)): no overflow for large |w|
__device__ __forceinline__ float softplus_f(float w) { return fmaxf(w, 0.f) + log1pf(expf(-fabsf(w))); }

// sigmoid(w) without overflow: exp is only taken of a non-positive argument
__device__ __forceinline__ float sigmoid_f(float w) {
    const float e = expf(-fabsf(w));
    return w >= 0.f ? 1.f / (1.f + e) : e / (1.f + e);
}

// Max and sum of exp(alpha - max) over the head's K priors, in component order.
__device__ void prior_lse(const float *a, int K, float *sm) {
    if (threadIdx.x == 0) {
        float m = a[0];
        for (int k = 1; k < K; ++k) m = fmaxf(m, a[k]);
        float z = 0.f;
        for (int k = 0; k < K; ++k) z += expf(a[k] - m);
        sm[0] = m;
        sm[1] = z;
    }
    __syncthreads();
}

__global__ void __launch_bounds__(kParamThreads) reparam_kernel(const float *__restrict__ omega,
                                                                const float *__restrict__ alpha, int K, int d_r,
                                                                float eps_sigma, float *__restrict__ sigma2,
                                                                float *__restrict__ log_pi) {
    __shared__ float sm[2];
    const int h = blockIdx.y;
    const size_t base = (size_t)h * K * d_r;
    const int e1 = min(K * d_r, (int)(blockIdx.x + 1) * kParamChunk);
#pragma unroll 4
    for (int e = blockIdx.x * kParamChunk + threadIdx.x; e < e1; e += kParamThreads)
        sigma2[base + e] = softplus_f(omega[base + e]) + eps_sigma;
    if (blockIdx.x != 0) return;
    const float *a = alpha + (size_t)h * K;
    prior_lse(a, K, sm);
    const float lse = sm[0] + logf(sm[1]);
    for (int k = threadIdx.x; k < K; k += kParamThreads) log_pi[(size_t)h * K + k] = a[k] - lse;
}

__global__ void __launch_bounds__(kParamThreads) reparam_backward_kernel(
    const float *__restrict__ omega, const float *__restrict__ alpha, const float *__restrict__ dsigma2,
    const float *__restrict__ dlog_pi, int K, int d_r, float *__restrict__ domega, float *__restrict__ dalpha) {
    __shared__ float sm[3];
    const int h = blockIdx.y;
    const size_t base = (size_t)h * K * d_r;
    const int e1 = min(K * d_r, (int)(blockIdx.x + 1) * kParamChunk);
#pragma unroll 4
    for (int e = blockIdx.x * kParamChunk + threadIdx.x; e < e1; e += kParamThreads)
        domega[base + e] = dsigma2[base + e] * sigmoid_f(omega[base + e]);
    if (blockIdx.x != 0) return;
    const float *a = alpha + (size_t)h * K, *g = dlog_pi + (size_t)h * K;
    if (threadIdx.x == 0) {
        float gs = 0.f;
        for (int k = 0; k < K; ++k) gs += g[k];
        sm[2] = gs;
    }
    prior_lse(a, K, sm);
    const float m = sm[0], rz = 1.f / sm[1], gs = sm[2];
    for (int k = threadIdx.x; k < K; k += kParamThreads)
        dalpha[(size_t)h * K + k] = g[k] - expf(a[k] - m) * rz * gs;
}

}  // namespace

cudaError_t reparameterize(const float *omega, const float *alpha, int H, int K, int d_r, float eps_sigma,
                           float *sigma2, float *log_pi, cudaStream_t s) {
    const dim3 grid((K * d_r + kParamChunk - 1) / kParamChunk, H);
    reparam_kernel<<<grid, kParamThreads, 0, s>>>(omega, alpha, K, d_r, eps_sigma, sigma2, log_pi);
    return cudaGetLastError();
}

cudaError_t reparameterize_backward(const float *omega, const float *alpha, const float *dsigma2,
                                    const float *dlog_pi, int H, int K, int d_r, float *domega, float *dalpha,
                                    cudaStream_t s) {
    const dim3 grid((K * d_r + kParamChunk - 1) / kParamChunk, H);
    reparam_backward_kernel<<<grid, kParamThreads, 0, s>>>(omega, alpha, dsigma2, dlog_pi, K, d_r, domega, dalpha);
    return cudaGetLastError();
}

}  // namespace gma
