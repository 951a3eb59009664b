// gma_stats.cu -- component-usage diagnostics of the responsibilities,
// computed beside them so that Gamma never reaches HBM.
//
// Paper: "Gaussian Mixture Attention: Linear-Time Sequence Mixing via
// Probabilistic Latent Routing" (arXiv 2606.18283): the introduction names the
// marginal usage of the mixture components (broad use of the routing space
// versus collapse onto a few components) and the hard assignment
// z_i = argmax_k gamma_ik as the diagnostics the responsibilities afford; the
// interpretability results report the number of components used and a usage
// entropy.  Per (b, h):
//   usage_k  = sum_i gamma_ik
//   z_i      = argmax_k s_ik (the smallest k on ties; s is the score of Eq. (3),
//              whose softmax is gamma, so this is the argmax of gamma)
//   counts_k = #{i : z_i = k}
//   entropy  = -sum_k p_k log p_k / log K with p_k = usage_k / N (1 when K = 1)
//
// Stages: prep (1/sigma2, c', validation), rows (one thread per row: scores,
// softmax and argmax, then per-CTA column sums in a fixed order), final
// (fixed-order sum of the CTA partials, entropy).
#include <cuda_bf16.h>

#include <cmath>

#include "gma_internal.h"

namespace gma {
namespace {

__device__ __forceinline__ float to_f32(float x) { return x; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 x) { return __bfloat162float(x); }

__device__ __forceinline__ bool failed(const unsigned *status) {
    return *reinterpret_cast<const volatile unsigned *>(status) != 0u;
}

constexpr int kStatRows = 128;  // rows per CTA, one per thread
constexpr int kStatKC = 32;     // components per parameter stage

struct StatsLayout {
    size_t part_u = 0, part_c = 0, total = 0;
    int nblk = 0;
};

StatsLayout stats_layout(const Problem &p) {
    StatsLayout L;
    size_t off = simt_layout(p, -1, 0).total;
    L.nblk = (p.N + kStatRows - 1) / kStatRows;
    const size_t n = (size_t)p.BH() * L.nblk * p.K;
    L.part_u = off; off = align256(off + sizeof(float) * n);
    L.part_c = off; off = align256(off + sizeof(int) * n);
    L.total = off;
    return L;
}

// grid (nblk, BH), kStatRows threads.  Dynamic shared memory: the parameter
// stage [kStatKC][D_R / 2] float4 {-mu_j, -mu_j+1, 1/sigma2_j, 1/sigma2_j+1}, the
// CTA's scores / responsibilities [kStatRows][K + 1] and the rows' argmax
// [kStatRows].  The score arithmetic runs on packed f32x2 pairs (j, j + 1),
// which round each element as the scalar operations would.
template <int D_R, typename T>
__global__ void __launch_bounds__(kStatRows) stats_rows_kernel(
    const T *__restrict__ X, int H, int N, int K, const float *__restrict__ mu, const float *__restrict__ inv,
    const float *__restrict__ cprime, int nblk, float *__restrict__ part_u, int *__restrict__ part_c,
    int *__restrict__ z, const unsigned *status) {
    if (failed(status)) return;
    extern __shared__ float smem[];
    constexpr int D2 = D_R / 2;
    float4 *sp = reinterpret_cast<float4 *>(smem);  // [kStatKC][D2]
    float *sgam = smem + 2 * kStatKC * D_R;         // [kStatRows][K + 1]
    int *sz = reinterpret_cast<int *>(sgam + kStatRows * (K + 1));
    const int KP = K + 1;
    const int blk = blockIdx.x, bh = blockIdx.y, h = bh % H;
    const int r = threadIdx.x, i = blk * kStatRows + r;
    const bool valid = i < N;
    const int nvalid = min(kStatRows, N - blk * kStatRows);

    float2 x[D2];
    const T *xr = X + ((size_t)bh * N + (valid ? i : 0)) * D_R;
#pragma unroll
    for (int j2 = 0; j2 < D2; ++j2) x[j2] = make_float2(to_f32(xr[2 * j2]), to_f32(xr[2 * j2 + 1]));
    const float *muh = mu + (size_t)h * K * D_R, *invh = inv + (size_t)h * K * D_R;
    const float *ch = cprime + (size_t)h * K;
    float *row = sgam + r * KP;

    float m = -INFINITY;
    int best = 0;
    for (int k0 = 0; k0 < K; k0 += kStatKC) {
        const int nk = min(kStatKC, K - k0);
        __syncthreads();
        for (int e = threadIdx.x; e < nk * D2; e += kStatRows) {
            const size_t o = (size_t)k0 * D_R + 2 * (size_t)e;
            sp[e] = make_float4(-muh[o], -muh[o + 1], invh[o], invh[o + 1]);
        }
        __syncthreads();
        if (!valid) continue;
        for (int kk = 0; kk < nk; ++kk) {
            // centred form, eight partial sums (j mod 8, two per packed
            // register) combined exactly (TwoSum)
            float2 acc[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) acc[u] = make_float2(0.f, 0.f);
#pragma unroll
            for (int j2 = 0; j2 < D2; ++j2) {
                const float4 pv = sp[kk * D2 + j2];
                const float2 d = __fadd2_rn(x[j2], make_float2(pv.x, pv.y));
                acc[j2 & 3] = __ffma2_rn(__fmul2_rn(d, d), make_float2(pv.z, pv.w), acc[j2 & 3]);
            }
            const float q8[8] = {acc[0].x, acc[0].y, acc[1].x, acc[1].y, acc[2].x, acc[2].y, acc[3].x, acc[3].y};
            float hi = q8[0], lo = 0.f;
#pragma unroll
            for (int u = 1; u < 8; ++u) {
                const float t = hi + q8[u], bb = t - hi;
                lo += (hi - (t - bb)) + (q8[u] - bb);
                hi = t;
            }
            const int k = k0 + kk;
            const float s = (__ldg(ch + k) - 0.5f * hi) - 0.5f * lo;
            row[k] = s;
            if (s > m) {
                m = s;
                best = k;
            }
        }
    }
    if (valid) {
        float zsum = 0.f;
        for (int k = 0; k < K; ++k) {
            const float e = expf(row[k] - m);
            row[k] = e;
            zsum += e;
        }
        const float rz = 1.0f / zsum;
        for (int k = 0; k < K; ++k) row[k] *= rz;
        sz[r] = best;
        if (z) z[(size_t)bh * N + i] = best;
    }
    __syncthreads();
    // column sums over the CTA's rows, in row order
    for (int k = threadIdx.x; k < K; k += kStatRows) {
        float u = 0.f;
        int c = 0;
        for (int t = 0; t < nvalid; ++t) {
            u += sgam[t * KP + k];
            c += sz[t] == k;
        }
        part_u[((size_t)bh * nblk + blk) * K + k] = u;
        part_c[((size_t)bh * nblk + blk) * K + k] = c;
    }
}

// grid BH, 128 threads (K <= 128): fixed-order sums of the CTA partials, then
// the normalised usage entropy.
__global__ void __launch_bounds__(128) stats_final_kernel(const float *__restrict__ part_u,
                                                          const int *__restrict__ part_c, int nblk, int K, int N,
                                                          float *__restrict__ usage, int *__restrict__ counts,
                                                          float *__restrict__ entropy, const unsigned *status) {
    if (failed(status)) return;
    __shared__ float sh[128];
    const int bh = blockIdx.x, k = threadIdx.x;
    float u = 0.f;
    if (k < K) {
        int c = 0;
        for (int b = 0; b < nblk; ++b) {
            u += part_u[((size_t)bh * nblk + b) * K + k];
            c += part_c[((size_t)bh * nblk + b) * K + k];
        }
        usage[(size_t)bh * K + k] = u;
        counts[(size_t)bh * K + k] = c;
    }
    if (!entropy) return;
    const float pk = u / (float)N;
    sh[k] = (k < K && pk > 0.f) ? -pk * logf(pk) : 0.f;
    __syncthreads();
    if (k == 0) {
        float hsum = 0.f;
        for (int t = 0; t < K; ++t) hsum += sh[t];
        entropy[bh] = K >= 2 ? hsum / logf((float)K) : 1.0f;
    }
}

template <int D_R, typename T>
cudaError_t launch_rows(const Problem &p, const StatsLayout &L, const float *inv, const float *cprime,
                        float *part_u, int *part_c, int *z, const unsigned *status, cudaStream_t s) {
    const size_t smem = sizeof(float) * (2 * kStatKC * D_R + (size_t)kStatRows * (p.K + 1)) + sizeof(int) * kStatRows;
    auto kern = stats_rows_kernel<D_R, T>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    kern<<<dim3(L.nblk, p.BH()), kStatRows, smem, s>>>(static_cast<const T *>(p.Q), p.H, p.N, p.K, p.mu, inv,
                                                       cprime, L.nblk, part_u, part_c, z, status);
    return cudaGetLastError();
}

template <typename T>
cudaError_t launch_rows_t(const Problem &p, const StatsLayout &L, const float *inv, const float *cprime,
                          float *part_u, int *part_c, int *z, const unsigned *status, cudaStream_t s) {
    switch (p.d_r) {
        case 16: return launch_rows<16, T>(p, L, inv, cprime, part_u, part_c, z, status, s);
        case 32: return launch_rows<32, T>(p, L, inv, cprime, part_u, part_c, z, status, s);
        case 64: return launch_rows<64, T>(p, L, inv, cprime, part_u, part_c, z, status, s);
        case 128: return launch_rows<128, T>(p, L, inv, cprime, part_u, part_c, z, status, s);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace

size_t stats_workspace(const Problem &p) { return stats_layout(p).total; }

cudaError_t simt_routing_stats(const Problem &p, const StatsArgs &a, void *ws, cudaStream_t s, StageClock &clk) {
    const SimtLayout S = simt_layout(p, -1, 0);
    const StatsLayout L = stats_layout(p);
    char *b = static_cast<char *>(ws);
    const unsigned *status = reinterpret_cast<const unsigned *>(b);
    const float *inv = reinterpret_cast<const float *>(b + S.inv_s2);
    const float *cprime = reinterpret_cast<const float *>(b + S.cprime);
    float *part_u = reinterpret_cast<float *>(b + L.part_u);
    int *part_c = reinterpret_cast<int *>(b + L.part_c);
    clk.mark();
    cudaError_t e = simt_prep(p, ws, s);
    if (e != cudaSuccess) return e;
    clk.mark();
    e = p.dtype == GMA_F32 ? launch_rows_t<float>(p, L, inv, cprime, part_u, part_c, a.z, status, s)
                           : launch_rows_t<__nv_bfloat16>(p, L, inv, cprime, part_u, part_c, a.z, status, s);
    if (e != cudaSuccess) return e;
    clk.mark();
    stats_final_kernel<<<p.BH(), 128, 0, s>>>(part_u, part_c, L.nblk, p.K, p.N, a.usage, a.counts, a.entropy,
                                              status);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    clk.mark();
    return cudaSuccess;
}

}  // namespace gma
