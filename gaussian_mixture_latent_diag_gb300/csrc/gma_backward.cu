// gma_backward.cu -- fp32 CUDA-core kernels for the gradients of the
// bidirectional and the causal GMA forward.
//
// Paper: "Gaussian Mixture Attention: Linear-Time Sequence Mixing via
// Probabilistic Latent Routing" (arXiv 2606.18283), gradient section: the
// upstream gradient g_ik = dL/dgamma_ik of a responsibility row, the softmax
// Jacobian (Eq. (17)) and the gradient entering the score (Eq. (18)),
//   ds_ik = gamma_ik (g_ik - sum_l gamma_il g_il),
// then the chain rule for everything that enters the score.  Differentiating
// Eqs. (5)-(7) with num_i = Gamma^Q_i Vt, den_i = Gamma^Q_i Z + eps:
//   dnum_i = dO_i / den_i,  dden_i = -(dO_i . O_i) / den_i
//   g^Q_ik = dnum_i . Vt_k + dden_i Z_k
//   dVt_k = sum_i gQ_ik dnum_i,  dZ_k = sum_i gQ_ik dden_i
//   g^K_jk = V_j . dVt_k + dZ_k,  dV_j = sum_k gK_jk dVt_k
// and through s_ik = c'_k - 1/2 sum_m (x_im - mu_km)^2 / sigma2_km:
//   dx_im = sum_k ds_ik (mu_km - x_im) / sigma2_km
//   dmu_km = sum_i ds_ik (x_im - mu_km) / sigma2_km
//   dsigma2_km = 1/2 sum_i ds_ik ((x_im - mu_km)^2 / sigma2_km^2 - 1 / sigma2_km)
//   dlog_pi_k = sum_i ds_ik
// summed over the query and the key rows of every batch row of the head.
//
// Causal variant ([GMA, Eq. (8b)] differentiated): the query side reads the
// prefix memories Vt^(i), Z^(i) (j <= i) instead, and a key j collects the
// SUFFIX sums over the queries i >= j:
//   g^K_jk = V_j . D^(j)_k + E^(j)_k,  dV_j = sum_k gK_jk D^(j)_k,
//   D^(j)_k = sum_{i>=j} gQ_ik dnum_i,  E^(j)_k = sum_{i>=j} gQ_ik dden_i,
// computed in chunks of kSimtCausalChunk tokens: the sums over earlier (later)
// chunks come from an exclusive prefix (suffix) over per-chunk aggregates, the
// rest inside the chunk.
//
// Steps (each materialises its result in the workspace; fixed summation
// orders throughout, so results are bitwise reproducible):
//   state    : the forward up to the latent memory (simt_bidir_state)
//   upstream : dnum | dden per query row
//   ds_q     : query score gradients
//   dmem     : [dVt | dZ] = Gamma^Q^T [dnum | dden], split over N, fixed-order sum
//   ds_k     : key score gradients;  dV = Gamma^K dVt
//   dx       : dQ, dK
//   params   : sum ds, sum ds (x - mu), sum ds (x - mu)^2 per split, then per head
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

// The thread-per-row kernels read Gamma / ds rows [K][N] with a stride of N, one
// value per component: they load kLoadBatch components before using them, so
// that many HBM round trips overlap (summation order unchanged).
constexpr int kLoadBatch = 4;

// upstream: one thread per query row.  mem [K][D_V + 1] = [Vt | Z] of the head.
// dn[i] = [dnum_i (D_V) | dden_i].
template <int D_V>
__global__ void __launch_bounds__(128) bwd_upstream_kernel(const float *__restrict__ gqt,
                                                           const float *__restrict__ mem,
                                                           const float *__restrict__ dO, int N, int K,
                                                           float eps, float *__restrict__ dn,
                                                           const unsigned *status) {
    if (failed(status)) return;
    extern __shared__ float smem[];
    constexpr int W = D_V + 1;
    const int bh = blockIdx.y;
    for (int e = threadIdx.x; e < K * W; e += blockDim.x) smem[e] = mem[(size_t)bh * K * W + e];
    __syncthreads();
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= N) return;
    float num[D_V];
#pragma unroll
    for (int c = 0; c < D_V; ++c) num[c] = 0.f;
    float den = 0.f;
    const float *g = gqt + (size_t)bh * K * N + i;
    for (int k0 = 0; k0 < K; k0 += kLoadBatch) {
        float gv[kLoadBatch];
#pragma unroll
        for (int u = 0; u < kLoadBatch; ++u) gv[u] = k0 + u < K ? g[(size_t)(k0 + u) * N] : 0.f;
#pragma unroll
        for (int u = 0; u < kLoadBatch; ++u) {
            if (k0 + u >= K) break;
            const float *row = smem + (k0 + u) * W;
#pragma unroll
            for (int c = 0; c < D_V; ++c) num[c] = fmaf(gv[u], row[c], num[c]);
            den = fmaf(gv[u], row[D_V], den);
        }
    }
    den += eps;
    const float r = 1.0f / den;
    const float *go = dO + ((size_t)bh * N + i) * D_V;
    float *out = dn + ((size_t)bh * N + i) * W;
    float dot = 0.f;
#pragma unroll
    for (int c = 0; c < D_V; ++c) {
        const float d = go[c];
        dot = fmaf(d, num[c] * r, dot);
        out[c] = d * r;
    }
    out[D_V] = -dot * r;
}

// Score gradients of one side, one thread per row ([GMA, Eq. (18)]):
//   u_ik = a_i . M_k[0:D_V] + beta_i M_k[D_V],   ds_ik = gamma_ik (u_ik - sum_l gamma_il u_il)
// a_i is row i of A (lda elements apart); beta_i = A[i][D_V] (query side: dden) or 1
// (key side).  ds [K][N] (component-major, like gamma).
template <int D_V, bool BETA_IN_A, typename TA>
__global__ void __launch_bounds__(128) bwd_score_grad_kernel(const float *__restrict__ gt,
                                                             const TA *__restrict__ A, int lda,
                                                             const float *__restrict__ M, int N, int K,
                                                             float *__restrict__ ds, const unsigned *status) {
    if (failed(status)) return;
    extern __shared__ float smem[];
    constexpr int W = D_V + 1;
    const int bh = blockIdx.y;
    for (int e = threadIdx.x; e < K * W; e += blockDim.x) smem[e] = M[(size_t)bh * K * W + e];
    __syncthreads();
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= N) return;
    float a[D_V];
    const TA *ar = A + ((size_t)bh * N + i) * lda;
#pragma unroll
    for (int c = 0; c < D_V; ++c) a[c] = to_f32(ar[c]);
    const float beta = BETA_IN_A ? to_f32(ar[D_V]) : 1.0f;
    const float *g = gt + (size_t)bh * K * N + i;
    float *d = ds + (size_t)bh * K * N + i;
    float mean = 0.f;
    for (int k0 = 0; k0 < K; k0 += kLoadBatch) {
        float gv[kLoadBatch];
#pragma unroll
        for (int u = 0; u < kLoadBatch; ++u) gv[u] = k0 + u < K ? g[(size_t)(k0 + u) * N] : 0.f;
#pragma unroll
        for (int v = 0; v < kLoadBatch; ++v) {
            if (k0 + v >= K) break;
            const float *row = smem + (k0 + v) * W;
            float u = beta * row[D_V];
#pragma unroll
            for (int c = 0; c < D_V; ++c) u = fmaf(a[c], row[c], u);
            d[(size_t)(k0 + v) * N] = u;
            mean = fmaf(gv[v], u, mean);
        }
    }
    for (int k0 = 0; k0 < K; k0 += kLoadBatch) {
        float gv[kLoadBatch], uv[kLoadBatch];
#pragma unroll
        for (int u = 0; u < kLoadBatch; ++u) {
            gv[u] = k0 + u < K ? g[(size_t)(k0 + u) * N] : 0.f;
            uv[u] = k0 + u < K ? d[(size_t)(k0 + u) * N] : 0.f;
        }
#pragma unroll
        for (int u = 0; u < kLoadBatch; ++u)
            if (k0 + u < K) d[(size_t)(k0 + u) * N] = gv[u] * (uv[u] - mean);
    }
}

// Column sums over a range of rows: part[bh][split][k][c] = sum_{i in split} G[k][i] B[i][c]
// for c in [64 z, 64 z + 64) and c < ncol; the last block also takes column
// 64 (z + 1) when that is the last column (ncol = 64 m + 1: the [dnum | dden]
// rows), so the lone column needs no block of its own.  G [K][N]
// (component-major), B rows of ldb floats.  Block: 256 threads, each 4
// components (k) x 8 columns (c, taken interleaved, c = tc + 8 b, so a warp
// reads consecutive columns; the extra column by the tc = 0 threads); rows
// staged 32 at a time in shared memory; fixed summation order.
constexpr int kCT = 32;
__global__ void __launch_bounds__(256) bwd_colsum_kernel(const float *__restrict__ Gt,
                                                         const float *__restrict__ B, int ldb, int ncol,
                                                         int N, int K, int rows_per_split, int nsplit,
                                                         float *__restrict__ part, const unsigned *status) {
    if (failed(status)) return;
    __shared__ float sg[128][kCT + 1];
    __shared__ float sb[kCT][64 + 4];
    const int split = blockIdx.x, bh = blockIdx.y, c0 = 64 * blockIdx.z;
    const int r0 = split * rows_per_split, r1 = min(N, r0 + rows_per_split);
    const int tk = threadIdx.x >> 3, tc = threadIdx.x & 7;  // k tile (4 rows), c tile (8 columns)
    const bool active = 4 * tk < K;
    const bool extra = c0 + 64 == ncol - 1;  // the lone last column rides with this block
    const int sc = extra ? 65 : 64;          // staged columns
    float acc[4][8], ex[4];
#pragma unroll
    for (int a = 0; a < 4; ++a) {
        ex[a] = 0.f;
#pragma unroll
        for (int b = 0; b < 8; ++b) acc[a][b] = 0.f;
    }
    const float *g = Gt + (size_t)bh * K * N;
    const float *bb = B + (size_t)bh * N * ldb;
    for (int base = r0; base < r1; base += kCT) {
        const int n = min(kCT, r1 - base);
        __syncthreads();
        for (int e = threadIdx.x; e < K * kCT; e += blockDim.x) {
            const int k = e / kCT, t = e % kCT;
            sg[k][t] = t < n ? g[(size_t)k * N + base + t] : 0.f;
        }
        for (int e = threadIdx.x; e < kCT * sc; e += blockDim.x) {
            const int t = e / sc, c = e % sc;
            sb[t][c] = (t < n && c0 + c < ncol) ? bb[(size_t)(base + t) * ldb + c0 + c] : 0.f;
        }
        __syncthreads();
        if (active) {
            for (int t = 0; t < n; ++t) {
                float ga[4], vb[8];
#pragma unroll
                for (int a = 0; a < 4; ++a) ga[a] = 4 * tk + a < K ? sg[4 * tk + a][t] : 0.f;
#pragma unroll
                for (int b = 0; b < 8; ++b) vb[b] = sb[t][tc + 8 * b];  // interleaved: no bank conflicts
#pragma unroll
                for (int a = 0; a < 4; ++a)
#pragma unroll
                    for (int b = 0; b < 8; ++b) acc[a][b] = fmaf(ga[a], vb[b], acc[a][b]);
                if (extra && tc == 0) {
                    const float ve = sb[t][64];
#pragma unroll
                    for (int a = 0; a < 4; ++a) ex[a] = fmaf(ga[a], ve, ex[a]);
                }
            }
        }
    }
    if (!active) return;
    float *p = part + ((size_t)bh * nsplit + split) * K * ncol;
#pragma unroll
    for (int a = 0; a < 4; ++a) {
        const int k = 4 * tk + a;
        if (k >= K) continue;
#pragma unroll
        for (int b = 0; b < 8; ++b) {
            const int c = c0 + tc + 8 * b;
            if (c < ncol) p[(size_t)k * ncol + c] = acc[a][b];
        }
        if (extra && tc == 0) p[(size_t)k * ncol + c0 + 64] = ex[a];
    }
}

// Column blocks of bwd_colsum_kernel for ncol columns: 64 each, a lone last column
// taken by the block before it.
inline int colsum_blocks(int ncol) { return ncol > 64 && ncol % 64 == 1 ? ncol / 64 : (ncol + 63) / 64; }

// Fixed-order sum of split partials: out[bh][e] = sum_s part[bh][s][e].
__global__ void bwd_reduce_kernel(const float *__restrict__ part, int nsplit, int E, float *__restrict__ out,
                                  const unsigned *status) {
    if (failed(status)) return;
    const int bh = blockIdx.y;
    const int e = blockIdx.x * blockDim.x + threadIdx.x;
    if (e >= E) return;
    const float *p = part + (size_t)bh * nsplit * E + e;
    float acc = 0.f;
    for (int s = 0; s < nsplit; ++s) acc += p[(size_t)s * E];
    out[(size_t)bh * E + e] = acc;
}

// dV_j = sum_k gK_jk dVt_k, one thread per key row.  dmem [K][D_V + 1].
template <int D_V>
__global__ void __launch_bounds__(128) bwd_dv_kernel(const float *__restrict__ gkt, const float *__restrict__ dmem,
                                                     int N, int K, float *__restrict__ dV,
                                                     const unsigned *status) {
    if (failed(status)) return;
    extern __shared__ float smem[];
    constexpr int W = D_V + 1;
    const int bh = blockIdx.y;
    for (int e = threadIdx.x; e < K * W; e += blockDim.x) smem[e] = dmem[(size_t)bh * K * W + e];
    __syncthreads();
    const int j = blockIdx.x * blockDim.x + threadIdx.x;
    if (j >= N) return;
    float acc[D_V];
#pragma unroll
    for (int c = 0; c < D_V; ++c) acc[c] = 0.f;
    const float *g = gkt + (size_t)bh * K * N + j;
    for (int k0 = 0; k0 < K; k0 += kLoadBatch) {
        float gv[kLoadBatch];
#pragma unroll
        for (int u = 0; u < kLoadBatch; ++u) gv[u] = k0 + u < K ? g[(size_t)(k0 + u) * N] : 0.f;
#pragma unroll
        for (int u = 0; u < kLoadBatch; ++u) {
            if (k0 + u >= K) break;
            const float *row = smem + (k0 + u) * W;
#pragma unroll
            for (int c = 0; c < D_V; ++c) acc[c] = fmaf(gv[u], row[c], acc[c]);
        }
    }
    float *o = dV + ((size_t)bh * N + j) * D_V;
#pragma unroll
    for (int c = 0; c < D_V; ++c) o[c] = acc[c];
}

// dx_im = sum_k ds_ik (mu_km - x_im) / sigma2_km, computed as dx_im = SB_im - x_im SA_im with
// SA_im = sum_k ds_ik / sigma2_km and SB_im = sum_k ds_ik mu_km / sigma2_km, two
// [N x K] x [K x d_r] products.  Block: 64 rows x 64 columns of one head, 256
// threads each 4 rows x 4 columns (every staged value feeds 4 or 8 products);
// components staged kDxKC at a time: ds [kDxKC][64 rows], 1/sigma2 and mu/sigma2
// [kDxKC][64 columns].  Components are summed in order.  The two sums share no
// large cancelling terms beyond those of the centred form (sum_k ds_ik = 0 per
// row keeps SA and SB of the size of dx), and the fp32 result is checked
// against the fp64 oracle like every gradient.
constexpr int kDxKC = 32;
template <typename T>
__global__ void __launch_bounds__(256) bwd_dx_tiled_kernel(const T *__restrict__ X, const float *__restrict__ ds,
                                                           const float *__restrict__ mu,
                                                           const float *__restrict__ inv, int H, int N, int K,
                                                           int d_r, float *__restrict__ dX,
                                                           const unsigned *status) {
    if (failed(status)) return;
    __shared__ __align__(16) float sd[kDxKC][64 + 4];
    __shared__ __align__(16) float sa[kDxKC][64 + 4];
    __shared__ __align__(16) float sb[kDxKC][64 + 4];
    const int bh = blockIdx.y, h = bh % H;
    const int r0 = 64 * blockIdx.x, c0 = 64 * blockIdx.z;
    const int tr = threadIdx.x / 16, tc = threadIdx.x % 16;
    float acc_a[4][4], acc_b[4][4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc_a[i][j] = acc_b[i][j] = 0.f;
    const float *dsb = ds + (size_t)bh * K * N;
    for (int k0 = 0; k0 < K; k0 += kDxKC) {
        __syncthreads();
        for (int e = threadIdx.x; e < kDxKC * 64; e += 256) {
            const int k = e / 64, c = e % 64, kk = k0 + k;
            const int row = r0 + c, col = c0 + c;
            sd[k][c] = (kk < K && row < N) ? dsb[(size_t)kk * N + row] : 0.f;
            const size_t o = ((size_t)h * K + kk) * d_r + col;
            const float iv = (kk < K && col < d_r) ? inv[o] : 0.f;
            sa[k][c] = iv;
            sb[k][c] = (kk < K && col < d_r) ? mu[o] * iv : 0.f;
        }
        __syncthreads();
        const int nk = min(kDxKC, K - k0);
        for (int k = 0; k < nk; ++k) {
            const float4 d = *reinterpret_cast<const float4 *>(&sd[k][4 * tr]);
            const float4 a = *reinterpret_cast<const float4 *>(&sa[k][4 * tc]);
            const float4 b = *reinterpret_cast<const float4 *>(&sb[k][4 * tc]);
            const float dv[4] = {d.x, d.y, d.z, d.w}, av[4] = {a.x, a.y, a.z, a.w}, bv[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    acc_a[i][j] = fmaf(dv[i], av[j], acc_a[i][j]);
                    acc_b[i][j] = fmaf(dv[i], bv[j], acc_b[i][j]);
                }
        }
    }
    const int col = c0 + 4 * tc;
    if (col >= d_r) return;  // d_r is a multiple of 16, so a thread's 4 columns are all in or all out
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int row = r0 + 4 * tr + i;
        if (row >= N) break;
        const T *xr = X + ((size_t)bh * N + row) * d_r + col;
        float4 o;
        o.x = fmaf(-to_f32(xr[0]), acc_a[i][0], acc_b[i][0]);
        o.y = fmaf(-to_f32(xr[1]), acc_a[i][1], acc_b[i][1]);
        o.z = fmaf(-to_f32(xr[2]), acc_a[i][2], acc_b[i][2]);
        o.w = fmaf(-to_f32(xr[3]), acc_a[i][3], acc_b[i][3]);
        *reinterpret_cast<float4 *>(dX + ((size_t)bh * N + row) * d_r + col) = o;
    }
}

// Parameter statistics of one side over a range of rows, columns
// [4 TM z, 4 TM (z + 1)):
//   st[k][0] = sum ds_ik,  st[k][1 + m] = sum ds_ik (x_im - mu_km),
//   st[k][1 + d_r + m] = sum ds_ik (x_im - mu_km)^2
// (centred on mu_km, so no cancellation).  Block: 256 threads, each a 4 (k) x 4 (m)
// tile, TM threads across the columns and 256 / TM down the components (TM = 16
// for K <= 64, so no thread is idle at K = d_r = 64); rows staged kCT at a time in
// shared memory.  The column pairs use packed f32x2 arithmetic, which rounds each
// element as the scalar operations do, so every sum has the same bits as a
// thread-per-element loop over the rows in order.
template <typename T, int TM>
__global__ void __launch_bounds__(256) bwd_param_stats_kernel(const T *__restrict__ X, const float *__restrict__ ds,
                                                              const float *__restrict__ mu, int H, int N, int K,
                                                              int d_r, int rows_per_split, int nsplit, int side,
                                                              float *__restrict__ st, const unsigned *status) {
    if (failed(status)) return;
    constexpr int TK = 256 / TM, MC = 4 * TM, KC = 4 * TK;
    __shared__ float sd[KC][kCT + 1];
    __shared__ __align__(16) float sx[kCT][MC + 4];
    const int split = blockIdx.x, bh = blockIdx.y, h = bh % H;
    const int m0 = MC * blockIdx.z;
    const int r0 = split * rows_per_split, r1 = min(N, r0 + rows_per_split);
    const int tk = threadIdx.x / TM, tm = threadIdx.x % TM;
    const bool active = 4 * tk < K;
    float2 a1[4][2], a2[4][2], nm[4][2];
    float a0[4];
#pragma unroll
    for (int a = 0; a < 4; ++a) {
        a0[a] = 0.f;
#pragma unroll
        for (int b = 0; b < 2; ++b) {
            a1[a][b] = a2[a][b] = make_float2(0.f, 0.f);
            const int k = 4 * tk + a, m = m0 + 4 * tm + 2 * b;
            const float *mk = mu + ((size_t)h * K + k) * d_r + m;
            nm[a][b] = make_float2((k < K && m < d_r) ? -mk[0] : 0.f, (k < K && m + 1 < d_r) ? -mk[1] : 0.f);
        }
    }
    const float *dsb = ds + (size_t)bh * K * N;
    const T *xb = X + (size_t)bh * N * d_r;
    // The next stage's rows are loaded into registers while this stage computes
    // (the loads of a stage are in flight under the previous stage's arithmetic).
    constexpr int ND = KC * kCT / 256, NX = kCT * MC / 256;
    float rd[ND], rx[NX];
    auto load_stage = [&](int base) {
        const int n = min(kCT, r1 - base);
#pragma unroll
        for (int u = 0; u < ND; ++u) {
            const int e = threadIdx.x + 256 * u, k = e / kCT, t = e % kCT;
            rd[u] = (k < K && t < n) ? dsb[(size_t)k * N + base + t] : 0.f;
        }
#pragma unroll
        for (int u = 0; u < NX; ++u) {
            const int e = threadIdx.x + 256 * u, t = e / MC, m = e % MC;
            rx[u] = (t < n && m0 + m < d_r) ? to_f32(xb[(size_t)(base + t) * d_r + m0 + m]) : 0.f;
        }
    };
    if (r0 < r1) load_stage(r0);
    for (int base = r0; base < r1; base += kCT) {
        const int n = min(kCT, r1 - base);
        __syncthreads();
#pragma unroll
        for (int u = 0; u < ND; ++u) {
            const int e = threadIdx.x + 256 * u;
            sd[e / kCT][e % kCT] = rd[u];
        }
#pragma unroll
        for (int u = 0; u < NX; ++u) {
            const int e = threadIdx.x + 256 * u;
            sx[e / MC][e % MC] = rx[u];
        }
        __syncthreads();
        if (base + kCT < r1) load_stage(base + kCT);
        if (active) {
            for (int t = 0; t < n; ++t) {
                const float4 xv = *reinterpret_cast<const float4 *>(&sx[t][4 * tm]);
                const float2 x2[2] = {make_float2(xv.x, xv.y), make_float2(xv.z, xv.w)};
#pragma unroll
                for (int a = 0; a < 4; ++a) {
                    const float d = 4 * tk + a < K ? sd[4 * tk + a][t] : 0.f;
                    a0[a] += d;
                    const float2 dd = make_float2(d, d);
#pragma unroll
                    for (int b = 0; b < 2; ++b) {
                        const float2 diff = __fadd2_rn(x2[b], nm[a][b]);
                        const float2 p = __fmul2_rn(dd, diff);
                        a1[a][b] = __fadd2_rn(a1[a][b], p);
                        a2[a][b] = __ffma2_rn(p, diff, a2[a][b]);
                    }
                }
            }
        }
    }
    if (!active) return;
    const int E = 1 + 2 * d_r;
    float *p = st + (((size_t)bh * 2 + side) * nsplit + split) * K * E;
#pragma unroll
    for (int a = 0; a < 4; ++a) {
        const int k = 4 * tk + a;
        if (k >= K) continue;
        if (m0 == 0 && tm == 0) p[(size_t)k * E] = a0[a];
#pragma unroll
        for (int b = 0; b < 4; ++b) {
            const int m = m0 + 4 * tm + b;
            if (m < d_r) {
                p[(size_t)k * E + 1 + m] = b & 1 ? a1[a][b >> 1].y : a1[a][b >> 1].x;
                p[(size_t)k * E + 1 + d_r + m] = b & 1 ? a2[a][b >> 1].y : a2[a][b >> 1].x;
            }
        }
    }
}

// Per head: the statistics of every batch row, side and split summed in that
// order, then dlog_pi, dmu, dsigma2.  One thread per (k, m) (and per k for dlog_pi).
__global__ void bwd_param_final_kernel(const float *__restrict__ st, const float *__restrict__ inv, int B, int H,
                                       int K, int d_r, int nsplit, float *__restrict__ dmu,
                                       float *__restrict__ dsigma2, float *__restrict__ dlog_pi,
                                       const unsigned *status) {
    if (failed(status)) return;
    const int h = blockIdx.y;
    const int e = blockIdx.x * blockDim.x + threadIdx.x;
    if (e >= K * d_r) return;
    const int k = e / d_r, m = e % d_r;
    const int E = 1 + 2 * d_r;
    float s0 = 0.f, s1 = 0.f, s2 = 0.f;
    for (int b = 0; b < B; ++b)
        for (int side = 0; side < 2; ++side)
            for (int s = 0; s < nsplit; ++s) {
                const float *p = st + ((((size_t)(b * H + h) * 2 + side) * nsplit + s) * K + k) * E;
                s0 += p[0];
                s1 += p[1 + m];
                s2 += p[1 + d_r + m];
            }
    const float v = inv[((size_t)h * K + k) * d_r + m];
    dmu[((size_t)h * K + k) * d_r + m] = v * s1;
    dsigma2[((size_t)h * K + k) * d_r + m] = 0.5f * (v * v * s2 - v * s0);
    if (m == 0) dlog_pi[(size_t)h * K + k] = s0;
}

// The causal chunk kernels give each row kBwdParts threads (a quad of adjacent
// lanes): a thread holds the value columns c = kBwdParts q + l (l its lane in
// the quad), splits the sums over components and over the rows of the chunk
// the same way, and the quad adds its partial sums with two xor shuffles.  The
// shuffle pattern gives every lane of the quad the same bits (each step adds
// the same two values), so the lanes agree on every shared result.
constexpr int kBwdParts = 4;
// Row strides (floats) of the staged Gamma rows and of the b rows: 8 and 4
// banks apart per component / row, so the four lanes of a quad and the eight
// quads of a warp hit 32 different banks.
constexpr int kBwdGS = kSimtCausalChunk + 8;
constexpr int kBwdBS = kSimtCausalChunk + 4;

__device__ __forceinline__ float quad_sum(float v, unsigned mask) {
    v += __shfl_xor_sync(mask, v, 1);
    v += __shfl_xor_sync(mask, v, 2);
    return v;
}

// Causal query rows, one block per chunk of C tokens, one quad per query row i:
// num_i, den_i from the chunk's exclusive prefix (S, Z) plus the intra-chunk
// terms j <= i; dnum_i, dden_i (written to dn); then
//   u_ik = dnum_i . S_k + dden_i Z_k + sum_{t0<=j<=i} gK_jk (dnum_i . V_j + dden_i)
// and ds^Q_ik = gQ_ik (u_ik - sum_l gQ_il u_il) ([GMA, Eq. (18)]).
template <int D_V, typename T>
__global__ void __launch_bounds__(kSimtCausalChunk * kBwdParts, 2) bwd_causal_query_kernel(
    const float *__restrict__ gqt, const float *__restrict__ gkt, const T *__restrict__ V,
    const float *__restrict__ prefix, const float *__restrict__ dO, int N, int K, int nchunk, float eps,
    float *__restrict__ dn, float *__restrict__ dsq, const unsigned *status) {
    if (failed(status)) return;
    constexpr int C = kSimtCausalChunk, P = kBwdParts, CQ = D_V / P, GS = kBwdGS, BS = kBwdBS;
    constexpr int W = D_V + 1;
    extern __shared__ float smem[];
    float *sgq = smem;              // [K][GS]
    float *sgk = sgq + K * GS;      // [K][GS]
    float *sv = sgk + K * GS;       // [C][D_V]
    float *ss = sv + C * D_V;       // [K][W]
    float *sb = ss + K * W;         // [C][BS]: b_ij of query row i
    const int chunk = blockIdx.x, bh = blockIdx.y;
    const int t0 = chunk * C;
    const int n = min(C, N - t0);
    const float *gq = gqt + (size_t)bh * K * N, *gk = gkt + (size_t)bh * K * N;
    for (int e = threadIdx.x; e < K * C; e += blockDim.x) {
        const int k = e / C, t = e % C;
        sgq[k * GS + t] = t < n ? gq[(size_t)k * N + t0 + t] : 0.f;
        sgk[k * GS + t] = t < n ? gk[(size_t)k * N + t0 + t] : 0.f;
    }
    const T *v = V + ((size_t)bh * N + t0) * D_V;
    for (int e = threadIdx.x; e < C * D_V; e += blockDim.x) sv[e] = e < n * D_V ? to_f32(v[e]) : 0.f;
    const float *pre = prefix + ((size_t)bh * nchunk + chunk) * K * W;
    for (int e = threadIdx.x; e < K * W; e += blockDim.x) ss[e] = pre[e];
    __syncthreads();
    const int i = threadIdx.x / P, l = threadIdx.x % P;
    if (i >= n) return;  // whole quads leave together
    const unsigned qm = 0xfu << (threadIdx.x & 28);
    float acc[CQ];
#pragma unroll
    for (int q = 0; q < CQ; ++q) acc[q] = 0.f;
    float den = 0.f;  // the same in every lane of the quad
    for (int k = 0; k < K; ++k) {
        const float g = sgq[k * GS + i];
        const float *row = ss + k * W + l;
#pragma unroll
        for (int q = 0; q < CQ; ++q) acc[q] = fmaf(g, row[P * q], acc[q]);
        den = fmaf(g, ss[k * W + D_V], den);
    }
    // Rows j in pairs: two independent dot / shuffle chains per iteration; the
    // accumulations still run in j order.
    int j = 0;
    for (; j + 1 <= i; j += 2) {
        float a0 = 0.f, a1 = 0.f;
        for (int k = l; k < K; k += P) {
            const float gqk = sgq[k * GS + i];
            a0 = fmaf(gqk, sgk[k * GS + j], a0);
            a1 = fmaf(gqk, sgk[k * GS + j + 1], a1);
        }
        a0 = quad_sum(a0, qm);
        a1 = quad_sum(a1, qm);
        den += a0;
        den += a1;
        const float *v0 = sv + j * D_V + l, *v1 = v0 + D_V;
#pragma unroll
        for (int q = 0; q < CQ; ++q) acc[q] = fmaf(a1, v1[P * q], fmaf(a0, v0[P * q], acc[q]));
    }
    if (j == i) {
        float a = 0.f;
        for (int k = l; k < K; k += P) a = fmaf(sgq[k * GS + i], sgk[k * GS + j], a);
        a = quad_sum(a, qm);
        den += a;
        const float *vr = sv + j * D_V + l;
#pragma unroll
        for (int q = 0; q < CQ; ++q) acc[q] = fmaf(a, vr[P * q], acc[q]);
    }
    den += eps;
    const float r = 1.0f / den;
    const float *go = dO + ((size_t)bh * N + t0 + i) * D_V + l;
    float *out = dn + ((size_t)bh * N + t0 + i) * W;
    float dot = 0.f;
#pragma unroll
    for (int q = 0; q < CQ; ++q) {
        const float d = go[P * q];
        dot = fmaf(d, acc[q] * r, dot);
        acc[q] = d * r;  // dnum
        out[P * q + l] = acc[q];
    }
    const float dden = -quad_sum(dot, qm) * r;
    if (l == 0) out[D_V] = dden;
    float *bi = sb + i * BS;
    for (j = 0; j + 1 <= i; j += 2) {
        const float *v0 = sv + j * D_V + l, *v1 = v0 + D_V;
        float b0 = 0.f, b1 = 0.f;
#pragma unroll
        for (int q = 0; q < CQ; ++q) {
            b0 = fmaf(acc[q], v0[P * q], b0);
            b1 = fmaf(acc[q], v1[P * q], b1);
        }
        b0 = quad_sum(b0, qm) + dden;
        b1 = quad_sum(b1, qm) + dden;
        if ((j & (P - 1)) == l) bi[j] = b0;  // read back by this lane only
        if (((j + 1) & (P - 1)) == l) bi[j + 1] = b1;
    }
    if (j == i) {
        const float *vr = sv + j * D_V + l;
        float b = 0.f;
#pragma unroll
        for (int q = 0; q < CQ; ++q) b = fmaf(acc[q], vr[P * q], b);
        b = quad_sum(b, qm) + dden;
        if ((j & (P - 1)) == l) bi[j] = b;
    }
    float *d = dsq + (size_t)bh * K * N + t0 + i;
    float mean = 0.f;
    int k = 0;
    for (; k + 1 < K; k += 2) {  // components in pairs, accumulated in k order
        const float *r0 = ss + k * W + l, *r1 = r0 + W;
        float u0 = 0.f, u1 = 0.f;
#pragma unroll
        for (int q = 0; q < CQ; ++q) {
            u0 = fmaf(acc[q], r0[P * q], u0);
            u1 = fmaf(acc[q], r1[P * q], u1);
        }
        for (int jj = l; jj <= i; jj += P) {
            const float bj = bi[jj];
            u0 = fmaf(sgk[k * GS + jj], bj, u0);
            u1 = fmaf(sgk[(k + 1) * GS + jj], bj, u1);
        }
        u0 = quad_sum(u0, qm) + dden * ss[k * W + D_V];
        u1 = quad_sum(u1, qm) + dden * ss[(k + 1) * W + D_V];
        if ((k & (P - 1)) == l) d[(size_t)k * N] = u0;
        if (((k + 1) & (P - 1)) == l) d[(size_t)(k + 1) * N] = u1;
        mean = fmaf(sgq[k * GS + i], u0, mean);
        mean = fmaf(sgq[(k + 1) * GS + i], u1, mean);
    }
    if (k < K) {
        const float *row = ss + k * W + l;
        float u = 0.f;
#pragma unroll
        for (int q = 0; q < CQ; ++q) u = fmaf(acc[q], row[P * q], u);
        for (int jj = l; jj <= i; jj += P) u = fmaf(sgk[k * GS + jj], bi[jj], u);
        u = quad_sum(u, qm) + dden * ss[k * W + D_V];
        if ((k & (P - 1)) == l) d[(size_t)k * N] = u;
        mean = fmaf(sgq[k * GS + i], u, mean);
    }
    for (int k = l; k < K; k += P) d[(size_t)k * N] = sgq[k * GS + i] * (d[(size_t)k * N] - mean);
}

// In-place exclusive suffix over the chunk aggregates of each head, in reverse
// chunk order: part[c] <- sum_{c' > c} part[c'].
__global__ void bwd_suffix_scan_kernel(float *__restrict__ part, int nchunk, int E, const unsigned *status) {
    if (failed(status)) return;
    const int bh = blockIdx.y;
    const int e = blockIdx.x * blockDim.x + threadIdx.x;
    if (e >= E) return;
    float *p = part + (size_t)bh * nchunk * E + e;
    float run = 0.f;
    int c = nchunk - 1;
    // eight loads before their sums, so eight memory round trips overlap; the
    // summation order is the reverse chunk order
    for (; c >= 7; c -= 8) {
        float cur[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) cur[u] = p[(size_t)(c - u) * E];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            p[(size_t)(c - u) * E] = run;
            run += cur[u];
        }
    }
    for (; c >= 0; --c) {
        const float cur = p[(size_t)c * E];
        p[(size_t)c * E] = run;
        run += cur;
    }
}

// Causal key rows, one block per chunk, one quad per key row j: with (D, E)
// the suffix over the later chunks (suf) plus the intra-chunk queries i >= j,
//   u_jk = V_j . D_k + E_k,   ds^K_jk = gK_jk (u_jk - sum_l gK_jl u_jl),
//   dV_j = sum_k gK_jk D_k = gK_j . suf + sum_{i>=j} <gK_j, gQ_i> dnum_i.
// The loops over the chunk's queries run from the last row down, so the quads
// of a warp (consecutive j) visit the same row i at the same time.
template <int D_V, typename T>
__global__ void __launch_bounds__(kSimtCausalChunk * kBwdParts, 2) bwd_causal_key_kernel(
    const float *__restrict__ gqt, const float *__restrict__ gkt, const T *__restrict__ V,
    const float *__restrict__ dn, const float *__restrict__ suf, int N, int K, int nchunk,
    float *__restrict__ dsk, float *__restrict__ dV, const unsigned *status) {
    if (failed(status)) return;
    constexpr int C = kSimtCausalChunk, P = kBwdParts, CQ = D_V / P, GS = kBwdGS, BS = kBwdBS;
    constexpr int W = D_V + 1;
    extern __shared__ float smem[];
    float *sgq = smem;              // [K][GS]
    float *sgk = sgq + K * GS;      // [K][GS]
    float *sdn = sgk + K * GS;      // [C][W]: dnum | dden of the chunk's queries
    float *ss = sdn + C * W;        // [K][W]: suffix over the later chunks
    float *sb = ss + K * W;         // [C][BS]: b_ji of key row j
    const int chunk = blockIdx.x, bh = blockIdx.y;
    const int t0 = chunk * C;
    const int n = min(C, N - t0);
    const float *gq = gqt + (size_t)bh * K * N, *gk = gkt + (size_t)bh * K * N;
    for (int e = threadIdx.x; e < K * C; e += blockDim.x) {
        const int k = e / C, t = e % C;
        sgq[k * GS + t] = t < n ? gq[(size_t)k * N + t0 + t] : 0.f;
        sgk[k * GS + t] = t < n ? gk[(size_t)k * N + t0 + t] : 0.f;
    }
    const float *dnc = dn + ((size_t)bh * N + t0) * W;
    for (int e = threadIdx.x; e < C * W; e += blockDim.x) sdn[e] = e < n * W ? dnc[e] : 0.f;
    const float *sp = suf + ((size_t)bh * nchunk + chunk) * K * W;
    for (int e = threadIdx.x; e < K * W; e += blockDim.x) ss[e] = sp[e];
    __syncthreads();
    const int j = threadIdx.x / P, l = threadIdx.x % P;
    if (j >= n) return;  // whole quads leave together
    const unsigned qm = 0xfu << (threadIdx.x & 28);
    float *bj = sb + j * BS;
    float *d = dsk + (size_t)bh * K * N + t0 + j;
    {
        float v[CQ];
        const T *vr = V + ((size_t)bh * N + t0 + j) * D_V + l;
#pragma unroll
        for (int q = 0; q < CQ; ++q) v[q] = to_f32(vr[P * q]);
        int i = n - 1;
        for (; i - 1 >= j; i -= 2) {  // rows in pairs: two independent shuffle chains
            const float *d0 = sdn + i * W + l, *d1 = d0 - W;
            float b0 = 0.f, b1 = 0.f;
#pragma unroll
            for (int q = 0; q < CQ; ++q) {
                b0 = fmaf(v[q], d0[P * q], b0);
                b1 = fmaf(v[q], d1[P * q], b1);
            }
            b0 = quad_sum(b0, qm) + sdn[i * W + D_V];
            b1 = quad_sum(b1, qm) + sdn[(i - 1) * W + D_V];
            if ((i & (P - 1)) == l) bj[i] = b0;  // read back by this lane only
            if (((i - 1) & (P - 1)) == l) bj[i - 1] = b1;
        }
        if (i == j) {
            const float *dr = sdn + i * W + l;
            float b = 0.f;
#pragma unroll
            for (int q = 0; q < CQ; ++q) b = fmaf(v[q], dr[P * q], b);
            b = quad_sum(b, qm) + sdn[i * W + D_V];
            if ((i & (P - 1)) == l) bj[i] = b;
        }
        const int i0 = (j & ~(P - 1)) + l;  // first row of this lane's share (rows below j skipped)
        float mean = 0.f;
        int k = 0;
        for (; k + 1 < K; k += 2) {  // components in pairs, accumulated in k order
            const float *r0 = ss + k * W + l, *r1 = r0 + W;
            float u0 = 0.f, u1 = 0.f;
#pragma unroll
            for (int q = 0; q < CQ; ++q) {
                u0 = fmaf(v[q], r0[P * q], u0);
                u1 = fmaf(v[q], r1[P * q], u1);
            }
            for (int ii = i0; ii < n; ii += P)
                if (ii >= j) {
                    const float b = bj[ii];
                    u0 = fmaf(sgq[k * GS + ii], b, u0);
                    u1 = fmaf(sgq[(k + 1) * GS + ii], b, u1);
                }
            u0 = quad_sum(u0, qm) + ss[k * W + D_V];
            u1 = quad_sum(u1, qm) + ss[(k + 1) * W + D_V];
            if ((k & (P - 1)) == l) d[(size_t)k * N] = u0;
            if (((k + 1) & (P - 1)) == l) d[(size_t)(k + 1) * N] = u1;
            mean = fmaf(sgk[k * GS + j], u0, mean);
            mean = fmaf(sgk[(k + 1) * GS + j], u1, mean);
        }
        if (k < K) {
            const float *row = ss + k * W + l;
            float u = 0.f;
#pragma unroll
            for (int q = 0; q < CQ; ++q) u = fmaf(v[q], row[P * q], u);
            for (int ii = i0; ii < n; ii += P)
                if (ii >= j) u = fmaf(sgq[k * GS + ii], bj[ii], u);
            u = quad_sum(u, qm) + ss[k * W + D_V];
            if ((k & (P - 1)) == l) d[(size_t)k * N] = u;
            mean = fmaf(sgk[k * GS + j], u, mean);
        }
        for (int k = l; k < K; k += P) d[(size_t)k * N] = sgk[k * GS + j] * (d[(size_t)k * N] - mean);
    }
    float acc[CQ];
#pragma unroll
    for (int q = 0; q < CQ; ++q) acc[q] = 0.f;
    for (int k = 0; k < K; ++k) {
        const float g = sgk[k * GS + j];
        const float *row = ss + k * W + l;
#pragma unroll
        for (int q = 0; q < CQ; ++q) acc[q] = fmaf(g, row[P * q], acc[q]);
    }
    int i = n - 1;
    for (; i - 1 >= j; i -= 2) {  // rows in pairs, accumulated in the same (descending) order
        float w0 = 0.f, w1 = 0.f;
        for (int k = l; k < K; k += P) {
            const float gkj = sgk[k * GS + j];
            w0 = fmaf(gkj, sgq[k * GS + i], w0);
            w1 = fmaf(gkj, sgq[k * GS + i - 1], w1);
        }
        w0 = quad_sum(w0, qm);
        w1 = quad_sum(w1, qm);
        const float *d0 = sdn + i * W + l, *d1 = d0 - W;
#pragma unroll
        for (int q = 0; q < CQ; ++q) acc[q] = fmaf(w1, d1[P * q], fmaf(w0, d0[P * q], acc[q]));
    }
    if (i == j) {
        float w = 0.f;
        for (int k = l; k < K; k += P) w = fmaf(sgk[k * GS + j], sgq[k * GS + i], w);
        w = quad_sum(w, qm);
        const float *dr = sdn + i * W + l;
#pragma unroll
        for (int q = 0; q < CQ; ++q) acc[q] = fmaf(w, dr[P * q], acc[q]);
    }
    float *o = dV + ((size_t)bh * N + t0 + j) * D_V + l;
#pragma unroll
    for (int q = 0; q < CQ; ++q) o[P * q] = acc[q];
}

struct BwdLayout {
    SimtLayout F;     // the forward's regions (status, 1/sigma2, c', Gamma^Q, Gamma^K, partials, memory)
    size_t dn = 0;    // [BH][N][d_v + 1]
    size_t dsq = 0, dsk = 0;  // [BH][K][N]
    size_t dpart = 0; // [BH][nsplit][K][d_v + 1] (causal: per chunk, then the suffixes)
    size_t dmem = 0;  // [BH][K][d_v + 1] (bidirectional)
    size_t st = 0;    // [BH][2][sn][K][1 + 2 d_r]
    int sn = 0, srows = 0;  // row splits of the parameter statistics
    size_t total = 0;
};

BwdLayout bwd_layout(const Problem &p, int causal, int splits) {
    BwdLayout L;
    L.F = simt_layout(p, causal, causal ? 0 : splits);
    if (causal || splits <= 0) {
        // 512 rows per block of the parameter statistics: twice the blocks of the
        // write's 1024-row splits, so the last wave of the grid is not mostly empty
        L.srows = 512;
        L.sn = (p.N + L.srows - 1) / L.srows;
    } else {
        L.srows = L.F.tokens_per_split;
        L.sn = L.F.nsplit;
    }
    size_t off = L.F.total;
    const size_t W = (size_t)p.d_v + 1, BH = p.BH();
    L.dn = off; off = align256(off + sizeof(float) * BH * p.N * W);
    L.dsq = off; off = align256(off + sizeof(float) * BH * p.K * p.N);
    L.dsk = off; off = align256(off + sizeof(float) * BH * p.K * p.N);
    L.dpart = off; off = align256(off + sizeof(float) * BH * L.F.nsplit * p.K * W);
    if (!causal) { L.dmem = off; off = align256(off + sizeof(float) * BH * p.K * W); }
    L.st = off; off = align256(off + sizeof(float) * BH * 2 * L.sn * p.K * (1 + 2 * (size_t)p.d_r));
    L.total = off;
    return L;
}

#define GMA_TRY(x)                              \
    do {                                        \
        cudaError_t err_ = (x);                 \
        if (err_ != cudaSuccess) return err_;   \
    } while (0)

template <int D_V>
cudaError_t launch_rows(const Problem &p, const BwdLayout &L, const BackwardArgs &g, char *b, cudaStream_t s,
                        StageClock &clk) {
    const unsigned *status = reinterpret_cast<const unsigned *>(b);
    const float *gq = reinterpret_cast<const float *>(b + L.F.gq), *gk = reinterpret_cast<const float *>(b + L.F.gk);
    const float *mem = reinterpret_cast<const float *>(b + L.F.mem);
    float *dn = reinterpret_cast<float *>(b + L.dn), *dsq = reinterpret_cast<float *>(b + L.dsq);
    float *dsk = reinterpret_cast<float *>(b + L.dsk), *dpart = reinterpret_cast<float *>(b + L.dpart);
    float *dmem = reinterpret_cast<float *>(b + L.dmem);
    const dim3 grid((p.N + 127) / 128, p.BH());
    const size_t sm = sizeof(float) * (size_t)p.K * (D_V + 1);
    auto big = [&](const void *k) {
        return cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm);
    };
    GMA_TRY(big((const void *)bwd_upstream_kernel<D_V>));
    bwd_upstream_kernel<D_V><<<grid, 128, sm, s>>>(gq, mem, g.dO, p.N, p.K, p.eps, dn, status);
    GMA_TRY(cudaGetLastError());
    clk.mark();
    GMA_TRY(big((const void *)bwd_score_grad_kernel<D_V, true, float>));
    bwd_score_grad_kernel<D_V, true, float><<<grid, 128, sm, s>>>(gq, dn, D_V + 1, mem, p.N, p.K, dsq, status);
    GMA_TRY(cudaGetLastError());
    clk.mark();
    const int W = D_V + 1;
    bwd_colsum_kernel<<<dim3(L.F.nsplit, p.BH(), colsum_blocks(W)), 256, 0, s>>>(gq, dn, W, W, p.N, p.K,
                                                                             L.F.tokens_per_split, L.F.nsplit,
                                                                             dpart, status);
    GMA_TRY(cudaGetLastError());
    bwd_reduce_kernel<<<dim3((p.K * W + 255) / 256, p.BH()), 256, 0, s>>>(dpart, L.F.nsplit, p.K * W, dmem, status);
    GMA_TRY(cudaGetLastError());
    clk.mark();
    if (p.dtype == GMA_F32) {
        GMA_TRY(big((const void *)bwd_score_grad_kernel<D_V, false, float>));
        bwd_score_grad_kernel<D_V, false, float><<<grid, 128, sm, s>>>(gk, static_cast<const float *>(p.V), D_V,
                                                                       dmem, p.N, p.K, dsk, status);
    } else {
        GMA_TRY(big((const void *)bwd_score_grad_kernel<D_V, false, __nv_bfloat16>));
        bwd_score_grad_kernel<D_V, false, __nv_bfloat16><<<grid, 128, sm, s>>>(
            gk, static_cast<const __nv_bfloat16 *>(p.V), D_V, dmem, p.N, p.K, dsk, status);
    }
    GMA_TRY(cudaGetLastError());
    GMA_TRY(big((const void *)bwd_dv_kernel<D_V>));
    bwd_dv_kernel<D_V><<<grid, 128, sm, s>>>(gk, dmem, p.N, p.K, g.dV, status);
    GMA_TRY(cudaGetLastError());
    clk.mark();
    return cudaSuccess;
}

template <typename T>
cudaError_t launch_inputs(const Problem &p, const BwdLayout &L, const BackwardArgs &g, char *b, cudaStream_t s,
                          StageClock &clk) {
    const unsigned *status = reinterpret_cast<const unsigned *>(b);
    const float *inv = reinterpret_cast<const float *>(b + L.F.inv_s2);
    const float *dsq = reinterpret_cast<const float *>(b + L.dsq), *dsk = reinterpret_cast<const float *>(b + L.dsk);
    float *st = reinterpret_cast<float *>(b + L.st);
    const T *Q = static_cast<const T *>(p.Q), *Kx = static_cast<const T *>(p.Kx);
    const dim3 gx((p.N + 63) / 64, p.BH(), (p.d_r + 63) / 64);
    bwd_dx_tiled_kernel<T><<<gx, 256, 0, s>>>(Q, dsq, p.mu, inv, p.H, p.N, p.K, p.d_r, g.dQ, status);
    GMA_TRY(cudaGetLastError());
    bwd_dx_tiled_kernel<T><<<gx, 256, 0, s>>>(Kx, dsk, p.mu, inv, p.H, p.N, p.K, p.d_r, g.dK, status);
    GMA_TRY(cudaGetLastError());
    clk.mark();
    // 64 columns x 64 components per block when K <= 64 and d_r >= 64, else 32 x 128
    const bool wide = p.K <= 64 && p.d_r >= 64;
    const dim3 gs(L.sn, p.BH(), (p.d_r + (wide ? 63 : 31)) / (wide ? 64 : 32));  // z: column block of d_r
    for (int side = 0; side < 2; ++side) {
        const T *X = side ? Kx : Q;
        const float *dss = side ? dsk : dsq;
        if (wide)
            bwd_param_stats_kernel<T, 16><<<gs, 256, 0, s>>>(X, dss, p.mu, p.H, p.N, p.K, p.d_r, L.srows, L.sn,
                                                            side, st, status);
        else
            bwd_param_stats_kernel<T, 8><<<gs, 256, 0, s>>>(X, dss, p.mu, p.H, p.N, p.K, p.d_r, L.srows, L.sn,
                                                           side, st, status);
        GMA_TRY(cudaGetLastError());
    }
    bwd_param_final_kernel<<<dim3((p.K * p.d_r + 127) / 128, p.H), 128, 0, s>>>(
        st, inv, p.B, p.H, p.K, p.d_r, L.sn, g.dmu, g.dsigma2, g.dlog_pi, status);
    GMA_TRY(cudaGetLastError());
    clk.mark();
    return cudaSuccess;
}

template <int D_V, typename T>
cudaError_t launch_causal_rows(const Problem &p, const BwdLayout &L, const BackwardArgs &g, char *b,
                               cudaStream_t s, StageClock &clk) {
    constexpr int C = kSimtCausalChunk, W = D_V + 1;
    const unsigned *status = reinterpret_cast<const unsigned *>(b);
    const float *gq = reinterpret_cast<const float *>(b + L.F.gq), *gk = reinterpret_cast<const float *>(b + L.F.gk);
    const float *prefix = reinterpret_cast<const float *>(b + L.F.partial);
    float *dn = reinterpret_cast<float *>(b + L.dn), *dsq = reinterpret_cast<float *>(b + L.dsq);
    float *dsk = reinterpret_cast<float *>(b + L.dsk), *dpart = reinterpret_cast<float *>(b + L.dpart);
    const T *V = static_cast<const T *>(p.V);
    const int nchunk = L.F.nsplit;
    const dim3 grid(nchunk, p.BH());
    constexpr int GS = kBwdGS, BS = kBwdBS, NT = C * kBwdParts;
    const size_t smq = sizeof(float) * ((size_t)2 * p.K * GS + (size_t)C * D_V + (size_t)p.K * W + (size_t)C * BS);
    const size_t smk = sizeof(float) * ((size_t)2 * p.K * GS + (size_t)C * W + (size_t)p.K * W + (size_t)C * BS);
    GMA_TRY(cudaFuncSetAttribute(bwd_causal_query_kernel<D_V, T>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)smq));
    bwd_causal_query_kernel<D_V, T><<<grid, NT, smq, s>>>(gq, gk, V, prefix, g.dO, p.N, p.K, nchunk, p.eps, dn, dsq,
                                                         status);
    GMA_TRY(cudaGetLastError());
    clk.mark();
    bwd_colsum_kernel<<<dim3(nchunk, p.BH(), colsum_blocks(W)), 256, 0, s>>>(gq, dn, W, W, p.N, p.K, C, nchunk, dpart,
                                                                         status);
    GMA_TRY(cudaGetLastError());
    bwd_suffix_scan_kernel<<<dim3((p.K * W + 255) / 256, p.BH()), 256, 0, s>>>(dpart, nchunk, p.K * W, status);
    GMA_TRY(cudaGetLastError());
    clk.mark();
    GMA_TRY(cudaFuncSetAttribute(bwd_causal_key_kernel<D_V, T>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)smk));
    bwd_causal_key_kernel<D_V, T><<<grid, NT, smk, s>>>(gq, gk, V, dn, dpart, p.N, p.K, nchunk, dsk, g.dV, status);
    GMA_TRY(cudaGetLastError());
    clk.mark();
    return cudaSuccess;
}

template <typename T>
cudaError_t causal_rows(const Problem &p, const BwdLayout &L, const BackwardArgs &g, char *b, cudaStream_t s,
                        StageClock &clk) {
    switch (p.d_v) {
        case 16: return launch_causal_rows<16, T>(p, L, g, b, s, clk);
        case 32: return launch_causal_rows<32, T>(p, L, g, b, s, clk);
        case 64: return launch_causal_rows<64, T>(p, L, g, b, s, clk);
        case 128: return launch_causal_rows<128, T>(p, L, g, b, s, clk);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace

const char *const kBackwardStages[2][8] = {
    {"state", "upstream", "ds_q", "dmem", "ds_k_dv", "dx", "params", nullptr},
    {"state", "query", "suffix", "key", "dx", "params", nullptr},
};

size_t backward_workspace(const Problem &p, int causal, int splits) {
    return bwd_layout(p, causal, splits).total;
}

cudaError_t simt_backward_causal(const Problem &p, const BackwardArgs &g, void *ws, cudaStream_t s,
                                 StageClock &clk) {
    const BwdLayout L = bwd_layout(p, 1, 0);
    char *b = static_cast<char *>(ws);
    clk.mark();
    GMA_TRY(simt_causal_state(p, ws, s));
    clk.mark();
    if (p.dtype == GMA_F32) {
        GMA_TRY(causal_rows<float>(p, L, g, b, s, clk));
        GMA_TRY(launch_inputs<float>(p, L, g, b, s, clk));
    } else {
        GMA_TRY(causal_rows<__nv_bfloat16>(p, L, g, b, s, clk));
        GMA_TRY(launch_inputs<__nv_bfloat16>(p, L, g, b, s, clk));
    }
    return cudaSuccess;
}

cudaError_t simt_backward_bidir(const Problem &p, const BackwardArgs &g, int splits, void *ws, cudaStream_t s,
                                StageClock &clk) {
    const BwdLayout L = bwd_layout(p, 0, splits);
    char *b = static_cast<char *>(ws);
    clk.mark();
    GMA_TRY(simt_bidir_state(p, splits, ws, s));
    clk.mark();
    switch (p.d_v) {
        case 16: GMA_TRY(launch_rows<16>(p, L, g, b, s, clk)); break;
        case 32: GMA_TRY(launch_rows<32>(p, L, g, b, s, clk)); break;
        case 64: GMA_TRY(launch_rows<64>(p, L, g, b, s, clk)); break;
        case 128: GMA_TRY(launch_rows<128>(p, L, g, b, s, clk)); break;
        default: return cudaErrorInvalidValue;
    }
    if (p.dtype == GMA_F32) GMA_TRY(launch_inputs<float>(p, L, g, b, s, clk));
    else GMA_TRY(launch_inputs<__nv_bfloat16>(p, L, g, b, s, clk));
    return cudaSuccess;
}

}  // namespace gma
