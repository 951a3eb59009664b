// gma_simt.cu -- fp32 CUDA-core kernels for the GMA forward pass.
//
// This family serves fp32 inputs and every supported size; it evaluates the
// log-density in centred form in fp32, which is accurate enough for the
// fp32 tolerance.  Each step materialises its result in the workspace:
//   prep   : 1/sigma2 and c'_k = log pi_k - 1/2 sum_j log sigma2_kj per head
//   resp   : Gamma^Q, Gamma^K, component-major [BH][K][N]
//   write  : per-split (or per-chunk) partial latent memories [K][d_v + 1]
//   reduce : fixed-order sum of the splits (bidirectional) /
//   scan   : fixed-order exclusive prefix over chunks (causal)
//   read   : O rows (bidirectional) / chunked causal outputs
//
// Paper: "Gaussian Mixture Attention: Linear-Time Sequence Mixing via
// Probabilistic Latent Routing" (arXiv 2606.18283), cited [GMA, ...].
#include <cuda_bf16.h>

#include <cmath>

#include "gma_internal.h"

namespace gma {
namespace {

// Every kernel of this family starts with dep_wait, so it may be launched with
// programmatic stream serialisation (launch_dep): it begins launching while
// the previous kernel of the stream is still running, and waits, before any
// memory access, until that kernel has completed and its writes are visible.
// The launch latency of the next kernel then overlaps this one, which is most
// of the time of a small call.  dep_trigger lets the next kernel launch as
// soon as every CTA of this one has started (it waits the same way).
__device__ __forceinline__ void dep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void dep_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// Launch with programmatic stream serialisation; a launch error is left for
// the caller's cudaGetLastError, as with <<< >>>.
template <typename... KArgs, typename... Args>
void launch_dep(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s, Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    (void)cudaLaunchKernelEx(&cfg, kern, static_cast<KArgs>(args)...);
}

__device__ __forceinline__ float to_f32(float x) { return x; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 x) { return __bfloat162float(x); }
template <typename T> __device__ __forceinline__ T from_f32(float x);
template <> __device__ __forceinline__ float from_f32<float>(float x) { return x; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float x) {
    return __float2bfloat16_rn(x);
}

__device__ __forceinline__ bool failed(const unsigned *status) {
    return *reinterpret_cast<const volatile unsigned *>(status) != 0u;
}

// Records the first device-side error of a call (later ones are dropped).
__device__ __forceinline__ void set_status(unsigned *status, unsigned code) {
    atomicCAS(status, 0u, code);
}

// Per-head constants of the centred log-density ([GMA, Eqs. (2)-(3)]):
//   s_ik = c'_k - 1/2 sum_j (x_j - mu_kj)^2 * inv_kj,
//   inv_kj = 1 / sigma2_kj,  c'_k = log pi_k - 1/2 sum_j log sigma2_kj.
// Also validates the parameter values.  The logs are taken in the coalesced
// pass over the elements and kept in shared memory (rows padded to d_r + 1
// floats, so the threads, one per component, read distinct banks); thread k
// then sums its component's log-determinant in fp32 as hi + lo, carrying every
// rounding error in lo (TwoSum, Knuth): a plain fp32 sum of up to 128 terms
// would lose the fp32 tolerance, and fp64 arithmetic is slow on this GPU.
constexpr int kPrepThreads = 512;  // many loads in flight: only H CTAs run

__global__ void __launch_bounds__(kPrepThreads) prep_simt_kernel(const float *__restrict__ mu, const float *__restrict__ sigma2,
                                 const float *__restrict__ log_pi, int K, int d_r,
                                 float *__restrict__ inv, float *__restrict__ cprime,
                                 unsigned *status) {
    dep_wait();
    dep_trigger();
    extern __shared__ float slog[];  // [K][d_r + 1]
    const int h = blockIdx.x;
    const size_t base = (size_t)h * K * d_r;
#pragma unroll 4
    for (int e = threadIdx.x; e < K * d_r; e += blockDim.x) {
        float s2 = sigma2[base + e], m = mu[base + e];
        if (!(s2 > 0.f) || !isfinite(s2) || !isfinite(m)) set_status(status, GMA_ERR_NONFINITE_PARAM);
        inv[base + e] = 1.0f / s2;
        slog[(e / d_r) * (d_r + 1) + e % d_r] = logf(s2);
    }
    __syncthreads();
    for (int k = threadIdx.x; k < K; k += blockDim.x) {
        float hi = 0.f, lo = 0.f;
        for (int j = 0; j < d_r; ++j) {
            const float y = slog[k * (d_r + 1) + j];
            const float t = hi + y, bb = t - hi;
            lo += (hi - (t - bb)) + (y - bb);
            hi = t;
        }
        float lp = log_pi[(size_t)h * K + k];
        if (!isfinite(lp)) set_status(status, GMA_ERR_NONFINITE_PARAM);
        cprime[(size_t)h * K + k] = (lp - 0.5f * hi) - 0.5f * lo;
    }
}

// One thread per row: scores, then a max-subtracted softmax over k
// ([GMA, Eq. (3)]).  The row is written three times to `out` (scores,
// exponentials, normalised values); each thread only touches its own row.
// The head's parameters are staged in shared memory 32 components at a time as
// float4 {-mu_j, -mu_j+1, 1/sigma2_j, 1/sigma2_j+1}; every thread of the block
// takes part in the staging.  The score arithmetic runs on packed f32x2 pairs
// (j, j + 1), which round each element as the scalar operations would.
constexpr int kRespKC = 32;
template <int D_R, typename T>
__global__ void __launch_bounds__(128) resp_simt_kernel(
    const T *__restrict__ X, int H, int N, int K, const float *__restrict__ mu,
    const float *__restrict__ inv, const float *__restrict__ cprime, float *out,
    long long out_bh_stride, long long out_stride_n, long long out_stride_k,
    const unsigned *status) {
    dep_wait();
    dep_trigger();
    if (failed(status)) return;
    constexpr int D2 = D_R / 2;
    __shared__ float4 sp[kRespKC][D2];
    const int bh = blockIdx.y, h = bh % H;
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    const bool valid = i < N;
    float2 x[D2];
    const T *xr = X + ((size_t)bh * N + (valid ? i : 0)) * D_R;
#pragma unroll
    for (int j2 = 0; j2 < D2; ++j2) x[j2] = make_float2(to_f32(xr[2 * j2]), to_f32(xr[2 * j2 + 1]));
    const float *muh = mu + (size_t)h * K * D_R;
    const float *invh = inv + (size_t)h * K * D_R;
    const float *ch = cprime + (size_t)h * K;
    float *o = out + (size_t)bh * out_bh_stride + (size_t)(valid ? i : 0) * out_stride_n;

    float m = -INFINITY;
    for (int k0 = 0; k0 < K; k0 += kRespKC) {
        const int nk = min(kRespKC, K - k0);
        __syncthreads();
        for (int e = threadIdx.x; e < nk * D2; e += blockDim.x) {
            const size_t o2 = (size_t)k0 * D_R + 2 * (size_t)e;
            sp[e / D2][e % D2] = make_float4(-muh[o2], -muh[o2 + 1], invh[o2], invh[o2 + 1]);
        }
        __syncthreads();
        if (!valid) continue;
        for (int kk = 0; kk < nk; ++kk) {
            // Eight interleaved partial sums (j mod 8, two per packed register),
            // combined without rounding error into hi + lo (TwoSum, Knuth): the
            // terms are positive and the total reaches several hundred at
            // d_r = 128, where one sequential fp32 sum loses the fp32 tolerance.
            float2 acc[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) acc[u] = make_float2(0.f, 0.f);
#pragma unroll
            for (int j2 = 0; j2 < D2; ++j2) {
                const float4 pv = sp[kk][j2];
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
            float s = (__ldg(ch + k) - 0.5f * hi) - 0.5f * lo;
            o[(size_t)k * out_stride_k] = s;
            m = fmaxf(m, s);
        }
    }
    if (!valid) return;
    // The row goes through global memory twice more (exponentials, then the
    // scale).  Eight components are loaded before any of them is stored back, so
    // eight round trips overlap (the stores would otherwise order every load
    // behind the previous store); the sum runs in component order as before.
    constexpr int KB = 8;
    float z = 0.f;
    for (int k0 = 0; k0 < K; k0 += KB) {
        float e[KB];
#pragma unroll
        for (int u = 0; u < KB; ++u) e[u] = k0 + u < K ? o[(size_t)(k0 + u) * out_stride_k] : 0.f;
#pragma unroll
        for (int u = 0; u < KB; ++u) {
            if (k0 + u >= K) break;
            e[u] = expf(e[u] - m);
            z += e[u];
        }
#pragma unroll
        for (int u = 0; u < KB; ++u)
            if (k0 + u < K) o[(size_t)(k0 + u) * out_stride_k] = e[u];
    }
    const float rz = 1.0f / z;
    for (int k0 = 0; k0 < K; k0 += KB) {
        float e[KB];
#pragma unroll
        for (int u = 0; u < KB; ++u) e[u] = k0 + u < K ? o[(size_t)(k0 + u) * out_stride_k] : 0.f;
#pragma unroll
        for (int u = 0; u < KB; ++u)
            if (k0 + u < K) o[(size_t)(k0 + u) * out_stride_k] = e[u] * rz;
    }
}

// Latent aggregation over one range of keys ([GMA, Eqs. (5)-(6)]):
//   part[k][c] = sum_{j in range} gK_jk V_jc (c < d_v),  part[k][d_v] = sum gK_jk.
// Block: 256 threads, each owns TA components k = TA tk + a and TB value columns
// c = tc + b * tiles_c (interleaved, so the threads of a warp read consecutive
// columns of a staged key row: no bank conflicts); keys staged 32 at a time in
// shared memory.  4 x 4 tiles when 256 of them cover K x d_v, else 8 x 8 (at
// K = d_v = 64 an 8 x 8 tiling leaves three quarters of the threads idle).
// Every element sums its keys in order, whatever the tile: fixed summation order.
constexpr int kWT = 32;  // keys per shared-memory stage
template <typename T, int TA, int TB>
__global__ void __launch_bounds__(256) write_simt_kernel(
    const float *__restrict__ gkt, const T *__restrict__ V, int N, int K, int d_v,
    int tokens_per_split, int nsplit, float *__restrict__ part, const unsigned *status) {
    dep_wait();
    dep_trigger();
    if (failed(status)) return;
    __shared__ float sg[128][kWT + 1];
    __shared__ float sv[kWT][128 + 4];
    const int split = blockIdx.x, bh = blockIdx.y;
    const int t0 = split * tokens_per_split;
    const int t1 = min(N, t0 + tokens_per_split);
    const int tiles_c = (d_v + TB - 1) / TB, tiles_k = (K + TA - 1) / TA;
    const int tk = threadIdx.x / tiles_c, tc = threadIdx.x % tiles_c;
    const bool active = tk < tiles_k;
    float acc[TA][TB];
    float zacc[TA];
#pragma unroll
    for (int a = 0; a < TA; ++a) {
        zacc[a] = 0.f;
#pragma unroll
        for (int b = 0; b < TB; ++b) acc[a][b] = 0.f;
    }
    const float *g = gkt + (size_t)bh * K * N;
    const T *v = V + (size_t)bh * N * d_v;
    for (int base = t0; base < t1; base += kWT) {
        const int n = min(kWT, t1 - base);
        __syncthreads();
        for (int e = threadIdx.x; e < K * kWT; e += blockDim.x) {
            int k = e / kWT, t = e % kWT;
            sg[k][t] = t < n ? g[(size_t)k * N + base + t] : 0.f;
        }
        for (int e = threadIdx.x; e < kWT * d_v; e += blockDim.x) {
            int t = e / d_v, c = e % d_v;
            sv[t][c] = t < n ? to_f32(v[(size_t)(base + t) * d_v + c]) : 0.f;
        }
        __syncthreads();
        if (active) {
            for (int t = 0; t < n; ++t) {
                float ga[TA], vb[TB];
#pragma unroll
                for (int a = 0; a < TA; ++a) {
                    int k = tk * TA + a;
                    ga[a] = k < K ? sg[k][t] : 0.f;
                }
#pragma unroll
                for (int b = 0; b < TB; ++b) {
                    int c = tc + b * tiles_c;
                    vb[b] = c < d_v ? sv[t][c] : 0.f;
                }
#pragma unroll
                for (int a = 0; a < TA; ++a) {
                    zacc[a] += ga[a];
#pragma unroll
                    for (int b = 0; b < TB; ++b) acc[a][b] = fmaf(ga[a], vb[b], acc[a][b]);
                }
            }
        }
    }
    if (!active) return;
    const int W = d_v + 1;
    float *p = part + ((size_t)bh * nsplit + split) * K * W;
#pragma unroll
    for (int a = 0; a < TA; ++a) {
        int k = tk * TA + a;
        if (k >= K) continue;
#pragma unroll
        for (int b = 0; b < TB; ++b) {
            int c = tc + b * tiles_c;
            if (c < d_v) p[(size_t)k * W + c] = acc[a][b];
        }
        if (tc == 0) p[(size_t)k * W + d_v] = zacc[a];
    }
}

// Fixed-order sum of the split partials: mem[bh] = sum_s part[bh][s].
__global__ void reduce_splits_kernel(const float *__restrict__ part, int nsplit, int E,
                                     float *__restrict__ mem, const unsigned *status) {
    dep_wait();
    dep_trigger();
    if (failed(status)) return;
    const int bh = blockIdx.y;
    const int e = blockIdx.x * blockDim.x + threadIdx.x;
    if (e >= E) return;
    const float *p = part + (size_t)bh * nsplit * E + e;
    float acc = 0.f;
    for (int s = 0; s < nsplit; ++s) acc += p[(size_t)s * E];
    mem[(size_t)bh * E + e] = acc;
}

// Fixed-order sum of the split partials into the caller's latent memory:
// Vt[bh][k][c] = sum_s part[bh][s][k][c] (c < d_v), Z[bh][k] = sum_s part[bh][s][k][d_v].
__global__ void reduce_to_memory_kernel(const float *__restrict__ part, int nsplit, int K, int d_v,
                                        float *__restrict__ Vt, float *__restrict__ Z,
                                        const unsigned *status) {
    dep_wait();
    dep_trigger();
    if (failed(status)) return;
    const int bh = blockIdx.y, W = d_v + 1, E = K * W;
    const int e = blockIdx.x * blockDim.x + threadIdx.x;
    if (e >= E) return;
    const float *p = part + (size_t)bh * nsplit * E + e;
    float acc = 0.f;
    for (int s = 0; s < nsplit; ++s) acc += p[(size_t)s * E];
    const int k = e / W, c = e % W;
    if (c < d_v) Vt[((size_t)bh * K + k) * d_v + c] = acc;
    else Z[(size_t)bh * K + k] = acc;
}

// In-place exclusive prefix of p[0], p[E], p[2E], ... (n terms) starting from
// `run`, which returns the total.  Eight loads are issued before their sums, so
// eight memory round trips overlap; the summation order is the chunk order.
__device__ __forceinline__ void exclusive_prefix_strided(float *p, int n, int E, float &run) {
    int c = 0;
    for (; c + 8 <= n; c += 8) {
        float cur[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) cur[u] = p[(size_t)(c + u) * E];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            p[(size_t)(c + u) * E] = run;
            run += cur[u];
        }
    }
    for (; c < n; ++c) {
        const float cur = p[(size_t)c * E];
        p[(size_t)c * E] = run;
        run += cur;
    }
}

// Packs a caller's latent memory into the read kernel's layout:
// mem[bh][k] = [Vt[bh][k][0..d_v) | Z[bh][k]].
__global__ void pack_memory_kernel(const float *__restrict__ Vt, const float *__restrict__ Z, int K, int d_v,
                                   float *__restrict__ mem, const unsigned *status) {
    dep_wait();
    dep_trigger();
    if (failed(status)) return;
    const int bh = blockIdx.y, W = d_v + 1, E = K * W;
    const int e = blockIdx.x * blockDim.x + threadIdx.x;
    if (e >= E) return;
    const int k = e / W, c = e % W;
    mem[(size_t)bh * E + e] = c < d_v ? Vt[((size_t)bh * K + k) * d_v + c] : Z[(size_t)bh * K + k];
}

// As scan_chunks_kernel, with the prefix starting from a carried-in memory
// (Vt_in, Z_in; zero when null) instead of zero, and the total after the last
// chunk -- the prefix memory after position N - 1 -- written to (Vt_out, Z_out)
// when given.
__global__ void scan_chunks_carry_kernel(float *__restrict__ part, int nchunk, int K, int d_v,
                                         const float *__restrict__ Vt_in, const float *__restrict__ Z_in,
                                         float *__restrict__ Vt_out, float *__restrict__ Z_out,
                                         const unsigned *status) {
    dep_wait();
    dep_trigger();
    if (failed(status)) return;
    const int bh = blockIdx.y, W = d_v + 1, E = K * W;
    const int e = blockIdx.x * blockDim.x + threadIdx.x;
    if (e >= E) return;
    const int k = e / W, c = e % W;
    float run = 0.f;
    if (Vt_in) run = c < d_v ? Vt_in[((size_t)bh * K + k) * d_v + c] : Z_in[(size_t)bh * K + k];
    float *p = part + (size_t)bh * nchunk * E + e;
    exclusive_prefix_strided(p, nchunk, E, run);
    if (Vt_out) {
        if (c < d_v) Vt_out[((size_t)bh * K + k) * d_v + c] = run;
        else Z_out[(size_t)bh * K + k] = run;
    }
}

// In-place exclusive prefix over the chunk partials of each head, in chunk
// order: part[c] <- sum_{c' < c} part[c'] (the causal prefix memory at the
// start of chunk c, [GMA, causal variant, cumulative sums]).
__global__ void scan_chunks_kernel(float *__restrict__ part, int nchunk, int E,
                                   const unsigned *status) {
    dep_wait();
    dep_trigger();
    if (failed(status)) return;
    const int bh = blockIdx.y;
    const int e = blockIdx.x * blockDim.x + threadIdx.x;
    if (e >= E) return;
    float *p = part + (size_t)bh * nchunk * E + e;
    float run = 0.f;
    exclusive_prefix_strided(p, nchunk, E, run);
}

// Normalised broadcasting ([GMA, Eq. (7)]): one thread per query row,
// O_i = (sum_k gQ_ik Vt_k) / (sum_k gQ_ik Z_k + eps).
template <int D_V, typename TO>
__global__ void __launch_bounds__(128) read_simt_kernel(
    const float *__restrict__ gqt, const float *__restrict__ mem, int N, int K, float eps,
    TO *__restrict__ O, const unsigned *status) {
    dep_wait();
    dep_trigger();
    if (failed(status)) return;
    extern __shared__ float smem[];
    const int W = D_V + 1;
    const int bh = blockIdx.y;
    for (int e = threadIdx.x; e < K * W; e += blockDim.x) smem[e] = mem[(size_t)bh * K * W + e];
    __syncthreads();
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= N) return;
    float acc[D_V];
#pragma unroll
    for (int c = 0; c < D_V; ++c) acc[c] = 0.f;
    float den = 0.f;
    const float *g = gqt + (size_t)bh * K * N + i;
    // Gamma^Q is read with a stride of N: four components are loaded before
    // their use, so four round trips overlap (component order unchanged)
    constexpr int KB = 4;
    for (int k0 = 0; k0 < K; k0 += KB) {
        float gv[KB];
#pragma unroll
        for (int u = 0; u < KB; ++u) gv[u] = k0 + u < K ? g[(size_t)(k0 + u) * N] : 0.f;
#pragma unroll
        for (int u = 0; u < KB; ++u) {
            if (k0 + u >= K) break;
            const float *row = smem + (k0 + u) * W;
#pragma unroll
            for (int c = 0; c < D_V; ++c) acc[c] = fmaf(gv[u], row[c], acc[c]);
            den = fmaf(gv[u], row[D_V], den);
        }
    }
    const float r = 1.0f / (den + eps);
    TO *o = O + ((size_t)bh * N + i) * D_V;
#pragma unroll
    for (int c = 0; c < D_V; ++c) o[c] = from_f32<TO>(acc[c] * r);
}

// Causal outputs of one chunk of C = 64 queries ([GMA, Eq. (8b)]), given the
// exclusive prefix memory (S, Z) at the chunk start:
//   O_i = (gQ_i S + sum_{t0<=j<=i} <gQ_i, gK_j> V_j)
//         / (gQ_i Z + sum_{t0<=j<=i} <gQ_i, gK_j> + eps).
// Four threads per query row (kCausalParts), each owning a quarter of the
// output columns.  The intra-chunk dots <gQ_i, gK_j> are split over j: part q
// computes them for j = 4m + q and the four parts exchange them by shuffles,
// so the Gamma reads are broadcasts: the chunk's Gamma^Q and Gamma^K are staged
// token-major ([C][KS], components zero-padded to a multiple of 4, rows 16 bytes
// apart modulo 128) and the dots read four components per 16-byte load.  The
// prefix rows are staged kCausalKT at a time, each row as four column quarters
// padded to a multiple of 4 floats, then Z, and V likewise, so the four parts
// read distinct banks with 16-byte loads.
// Summation orders are those of the definition: k for the prefix, then j (the
// zero padding adds exact zeros).
constexpr int kCausalParts = 4;
constexpr int kCausalKT = 16;
template <int D_V>
struct CausalSmem {
    static constexpr int P = kCausalParts, CW = D_V / P, SQ = CW + 4, SR = P * SQ + 4;
    __host__ __device__ static int ks(int K) { return ((K + 3) & ~3) + 4; }  // floats per staged Gamma row
    static size_t floats(int K) {
        return (size_t)2 * ks(K) * kSimtCausalChunk + (size_t)kSimtCausalChunk * P * SQ + (size_t)kCausalKT * SR;
    }
};
template <int D_V, typename T, typename TO>
__global__ void __launch_bounds__(kSimtCausalChunk * kCausalParts) causal_simt_kernel(
    const float *__restrict__ gqt, const float *__restrict__ gkt, const T *__restrict__ V,
    const float *__restrict__ prefix, int N, int K, int nchunk, float eps, TO *__restrict__ O,
    const unsigned *status) {
    dep_wait();
    dep_trigger();
    if (failed(status)) return;
    constexpr int C = kSimtCausalChunk;
    constexpr int W = D_V + 1;
    using L = CausalSmem<D_V>;
    constexpr int P = L::P, CW = L::CW, SQ = L::SQ, SR = L::SR;
    extern __shared__ __align__(16) float smem[];
    const int KS = L::ks(K), K4 = (K + 3) / 4;
    float *sgq = smem;              // [C][KS]: token-major Gamma^Q of the chunk
    float *sgk = sgq + C * KS;      // [C][KS]
    float *sv = sgk + C * KS;       // [C][P * SQ]: V rows in padded quarters
    float *ss = sv + C * P * SQ;    // [kCausalKT][SR]: prefix rows in padded quarters, then Z
    const int chunk = blockIdx.x, bh = blockIdx.y;
    const int t0 = chunk * C;
    const int n = min(C, N - t0);
    const float *gq = gqt + (size_t)bh * K * N, *gk = gkt + (size_t)bh * K * N;
    for (int e = threadIdx.x; e < 4 * K4 * C; e += blockDim.x) {
        const int k = e / C, t = e % C;
        const bool in = t < n && k < K;
        sgq[t * KS + k] = in ? gq[(size_t)k * N + t0 + t] : 0.f;
        sgk[t * KS + k] = in ? gk[(size_t)k * N + t0 + t] : 0.f;
    }
    const T *v = V + ((size_t)bh * N + t0) * D_V;
    for (int e = threadIdx.x; e < C * D_V; e += blockDim.x) {
        const int t = e / D_V, c = e % D_V;
        sv[t * P * SQ + (c / CW) * SQ + c % CW] = t < n ? to_f32(v[e]) : 0.f;
    }
    const int i = threadIdx.x / P, q = threadIdx.x % P, lane = threadIdx.x & 31;
    float acc[CW];
#pragma unroll
    for (int c = 0; c < CW; ++c) acc[c] = 0.f;
    float den = 0.f;
    const float *pre = prefix + ((size_t)bh * nchunk + chunk) * K * W;
    for (int k0 = 0; k0 < K; k0 += kCausalKT) {
        const int nk = min(kCausalKT, K - k0);
        __syncthreads();  // the previous stage is consumed (the first time: sgq, sgk, sv are staged)
        for (int e = threadIdx.x; e < nk * W; e += blockDim.x) {
            const int kk = e / W, c = e % W;
            ss[kk * SR + (c < D_V ? (c / CW) * SQ + c % CW : P * SQ)] = pre[(size_t)k0 * W + e];
        }
        __syncthreads();
        for (int kk = 0; kk < nk; ++kk) {
            const float g = sgq[i * KS + k0 + kk];
            const float4 *row = reinterpret_cast<const float4 *>(ss + kk * SR + q * SQ);
#pragma unroll
            for (int c4 = 0; c4 < CW / 4; ++c4) {
                const float4 r = row[c4];
                acc[4 * c4 + 0] = fmaf(g, r.x, acc[4 * c4 + 0]);
                acc[4 * c4 + 1] = fmaf(g, r.y, acc[4 * c4 + 1]);
                acc[4 * c4 + 2] = fmaf(g, r.z, acc[4 * c4 + 2]);
                acc[4 * c4 + 3] = fmaf(g, r.w, acc[4 * c4 + 3]);
            }
            den = fmaf(g, ss[kk * SR + P * SQ], den);
        }
    }
    // intra-chunk terms j <= i; the loop runs to the warp's last row, so every
    // lane of the warp takes part in every shuffle
    // Two groups of P rows per iteration: each lane runs two independent dot
    // chains (rows j0 + q and j0 + P + q, each in component order), and the
    // groups are accumulated in row order.
    const int wlast = min(n - 1, (threadIdx.x / 32) * (32 / P) + (32 / P) - 1);
    for (int j0 = 0; j0 <= wlast; j0 += 2 * P) {
        const int ja = j0 + q, jb = j0 + P + q;
        float ab[2] = {0.f, 0.f};
        const float4 *gi = reinterpret_cast<const float4 *>(sgq + i * KS);
        const float4 *ga = reinterpret_cast<const float4 *>(sgk + min(ja, C - 1) * KS);
        const float4 *gb = reinterpret_cast<const float4 *>(sgk + min(jb, C - 1) * KS);
        if (jb <= wlast) {
            for (int k4 = 0; k4 < K4; ++k4) {
                const float4 g = gi[k4], x = ga[k4], y = gb[k4];
                ab[0] = fmaf(g.w, x.w, fmaf(g.z, x.z, fmaf(g.y, x.y, fmaf(g.x, x.x, ab[0]))));
                ab[1] = fmaf(g.w, y.w, fmaf(g.z, y.z, fmaf(g.y, y.y, fmaf(g.x, y.x, ab[1]))));
            }
        } else if (ja <= wlast) {
            for (int k4 = 0; k4 < K4; ++k4) {
                const float4 g = gi[k4], x = ga[k4];
                ab[0] = fmaf(g.w, x.w, fmaf(g.z, x.z, fmaf(g.y, x.y, fmaf(g.x, x.x, ab[0]))));
            }
        }
#pragma unroll
        for (int gsel = 0; gsel < 2; ++gsel) {
            if (j0 + gsel * P > wlast) break;  // the same for the whole warp
#pragma unroll
            for (int p2 = 0; p2 < P; ++p2) {
                const float ap = __shfl_sync(0xffffffffu, ab[gsel], (lane & ~(P - 1)) | p2);
                const int jj = j0 + gsel * P + p2;
                if (jj <= i) {
                    den += ap;
                    const float4 *vr = reinterpret_cast<const float4 *>(sv + jj * P * SQ + q * SQ);
#pragma unroll
                    for (int c4 = 0; c4 < CW / 4; ++c4) {
                        const float4 r = vr[c4];
                        acc[4 * c4 + 0] = fmaf(ap, r.x, acc[4 * c4 + 0]);
                        acc[4 * c4 + 1] = fmaf(ap, r.y, acc[4 * c4 + 1]);
                        acc[4 * c4 + 2] = fmaf(ap, r.z, acc[4 * c4 + 2]);
                        acc[4 * c4 + 3] = fmaf(ap, r.w, acc[4 * c4 + 3]);
                    }
                }
            }
        }
    }
    if (i >= n) return;
    const float r = 1.0f / (den + eps);
    TO *o = O + ((size_t)bh * N + t0 + i) * D_V + q * CW;
#pragma unroll
    for (int c = 0; c < CW; ++c) o[c] = from_f32<TO>(acc[c] * r);
}

// ------------------------------------------------------------------ launchers

template <typename T>
cudaError_t launch_resp(const Problem &p, const void *X, const float *inv, const float *cprime,
                        float *out, long long bh_stride, long long sn, long long sk,
                        const unsigned *status, cudaStream_t s) {
    dim3 grid((p.N + 127) / 128, p.BH());
    const T *x = static_cast<const T *>(X);
    switch (p.d_r) {
        case 16: launch_dep(resp_simt_kernel<16, T>, grid, 128, 0, s, x, p.H, p.N, p.K, p.mu, inv, cprime, out, bh_stride, sn, sk, status); break;
        case 32: launch_dep(resp_simt_kernel<32, T>, grid, 128, 0, s, x, p.H, p.N, p.K, p.mu, inv, cprime, out, bh_stride, sn, sk, status); break;
        case 64: launch_dep(resp_simt_kernel<64, T>, grid, 128, 0, s, x, p.H, p.N, p.K, p.mu, inv, cprime, out, bh_stride, sn, sk, status); break;
        case 128: launch_dep(resp_simt_kernel<128, T>, grid, 128, 0, s, x, p.H, p.N, p.K, p.mu, inv, cprime, out, bh_stride, sn, sk, status); break;
        default: return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
}

template <int D_V, typename TO>
cudaError_t launch_read_dv(const Problem &p, const float *gq, const float *mem,
                           const unsigned *status, cudaStream_t s) {
    size_t smem = (size_t)p.K * (D_V + 1) * sizeof(float);
    auto kern = read_simt_kernel<D_V, TO>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    dim3 grid((p.N + 127) / 128, p.BH());
    launch_dep(kern, grid, 128, smem, s, gq, mem, p.N, p.K, p.eps, static_cast<TO *>(p.O), status);
    return cudaGetLastError();
}

template <typename TO>
cudaError_t launch_read(const Problem &p, const float *gq, const float *mem,
                        const unsigned *status, cudaStream_t s) {
    switch (p.d_v) {
        case 16: return launch_read_dv<16, TO>(p, gq, mem, status, s);
        case 32: return launch_read_dv<32, TO>(p, gq, mem, status, s);
        case 64: return launch_read_dv<64, TO>(p, gq, mem, status, s);
        case 128: return launch_read_dv<128, TO>(p, gq, mem, status, s);
        default: return cudaErrorInvalidValue;
    }
}

template <int D_V, typename T, typename TO>
cudaError_t launch_causal_dv(const Problem &p, const float *gq, const float *gk,
                             const float *prefix, int nchunk, const unsigned *status,
                             cudaStream_t s) {
    constexpr int C = kSimtCausalChunk;
    const size_t smem = CausalSmem<D_V>::floats(p.K) * sizeof(float);
    auto kern = causal_simt_kernel<D_V, T, TO>;
    if (smem > 48 * 1024) {  // above the default limit only: the call costs host time
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
    }
    dim3 grid(nchunk, p.BH());
    launch_dep(kern, grid, C * kCausalParts, smem, s, gq, gk, static_cast<const T *>(p.V), prefix, p.N, p.K, nchunk,
                                              p.eps, static_cast<TO *>(p.O), status);
    return cudaGetLastError();
}

template <typename T, typename TO>
cudaError_t launch_causal(const Problem &p, const float *gq, const float *gk,
                          const float *prefix, int nchunk, const unsigned *status,
                          cudaStream_t s) {
    switch (p.d_v) {
        case 16: return launch_causal_dv<16, T, TO>(p, gq, gk, prefix, nchunk, status, s);
        case 32: return launch_causal_dv<32, T, TO>(p, gq, gk, prefix, nchunk, status, s);
        case 64: return launch_causal_dv<64, T, TO>(p, gq, gk, prefix, nchunk, status, s);
        case 128: return launch_causal_dv<128, T, TO>(p, gq, gk, prefix, nchunk, status, s);
        default: return cudaErrorInvalidValue;
    }
}

#define GMA_TRY(x)                              \
    do {                                        \
        cudaError_t err_ = (x);                 \
        if (err_ != cudaSuccess) return err_;   \
    } while (0)

struct Ptrs {
    unsigned *status;
    float *inv, *cprime, *gq, *gk, *part, *mem;
};

Ptrs ptrs(const SimtLayout &L, void *ws) {
    char *b = static_cast<char *>(ws);
    return {reinterpret_cast<unsigned *>(b), reinterpret_cast<float *>(b + L.inv_s2),
            reinterpret_cast<float *>(b + L.cprime), reinterpret_cast<float *>(b + L.gq),
            reinterpret_cast<float *>(b + L.gk), reinterpret_cast<float *>(b + L.partial),
            reinterpret_cast<float *>(b + L.mem)};
}

cudaError_t prep(const Problem &p, const Ptrs &P, cudaStream_t s) {
    GMA_TRY(cudaMemsetAsync(P.status, 0, sizeof(unsigned), s));
    const size_t smem = sizeof(float) * (size_t)p.K * (p.d_r + 1);
    if (smem > 48 * 1024)  // above the default limit only: the call costs host time
        GMA_TRY(cudaFuncSetAttribute(prep_simt_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem));
    launch_dep(prep_simt_kernel, p.H, kPrepThreads, smem, s, p.mu, p.sigma2, p.log_pi, p.K, p.d_r, P.inv, P.cprime, P.status);
    return cudaGetLastError();
}

cudaError_t resp_both(const Problem &p, const Ptrs &P, cudaStream_t s, StageClock &clk) {
    const long long bhs = (long long)p.K * p.N;
    if (p.dtype == GMA_F32) {
        GMA_TRY(launch_resp<float>(p, p.Q, P.inv, P.cprime, P.gq, bhs, 1, p.N, P.status, s));
        clk.mark();
        GMA_TRY(launch_resp<float>(p, p.Kx, P.inv, P.cprime, P.gk, bhs, 1, p.N, P.status, s));
    } else {
        GMA_TRY(launch_resp<__nv_bfloat16>(p, p.Q, P.inv, P.cprime, P.gq, bhs, 1, p.N, P.status, s));
        clk.mark();
        GMA_TRY(launch_resp<__nv_bfloat16>(p, p.Kx, P.inv, P.cprime, P.gk, bhs, 1, p.N, P.status, s));
    }
    clk.mark();
    return cudaSuccess;
}

cudaError_t write_parts(const Problem &p, const SimtLayout &L, const Ptrs &P, cudaStream_t s) {
    dim3 grid(L.nsplit, p.BH());
    // 4 x 4 tiles when they cover K x d_v with the block's 256 threads, else 8 x 8
    // (which always do: K, d_v <= 128)
    const bool big = ((p.K + 3) / 4) * ((p.d_v + 3) / 4) > 256;
    if (p.dtype == GMA_F32) {
        const float *V = static_cast<const float *>(p.V);
        if (big)
            launch_dep(write_simt_kernel<float, 8, 8>, grid, 256, 0, s, P.gk, V, p.N, p.K, p.d_v, L.tokens_per_split,
                                                                L.nsplit, P.part, P.status);
        else
            launch_dep(write_simt_kernel<float, 4, 4>, grid, 256, 0, s, P.gk, V, p.N, p.K, p.d_v, L.tokens_per_split,
                                                                L.nsplit, P.part, P.status);
    } else {
        const __nv_bfloat16 *V = static_cast<const __nv_bfloat16 *>(p.V);
        if (big)
            launch_dep(write_simt_kernel<__nv_bfloat16, 8, 8>, grid, 256, 0, s, P.gk, V, p.N, p.K, p.d_v,
                                                                        L.tokens_per_split, L.nsplit, P.part,
                                                                        P.status);
        else
            launch_dep(write_simt_kernel<__nv_bfloat16, 4, 4>, grid, 256, 0, s, P.gk, V, p.N, p.K, p.d_v,
                                                                        L.tokens_per_split, L.nsplit, P.part,
                                                                        P.status);
    }
    return cudaGetLastError();
}

}  // namespace

SimtLayout simt_layout(const Problem &p, int mode, int splits) {
    SimtLayout L;
    size_t off = kStatusBytes;
    L.inv_s2 = off; off = align256(off + sizeof(float) * (size_t)p.H * p.K * p.d_r);
    L.cprime = off; off = align256(off + sizeof(float) * (size_t)p.H * p.K);
    if (mode == 3) {  // read from a given memory: Gamma^Q and the packed [Vt | Z]
        L.gq = off; off = align256(off + sizeof(float) * (size_t)p.BH() * p.K * p.N);
        L.mem = off; off = align256(off + sizeof(float) * (size_t)p.BH() * p.K * ((size_t)p.d_v + 1));
    } else if (mode >= 0) {
        const size_t g = sizeof(float) * (size_t)p.BH() * p.K * p.N;
        if (mode != 2) { L.gq = off; off = align256(off + g); }
        L.gk = off; off = align256(off + g);
        if (mode == 0 || mode == 2) {
            int ns = splits > 0 ? splits : (p.N + 1023) / 1024;
            ns = ns < 1 ? 1 : (ns > p.N ? p.N : ns);
            L.tokens_per_split = (p.N + ns - 1) / ns;
            L.nsplit = (p.N + L.tokens_per_split - 1) / L.tokens_per_split;
        } else {
            L.tokens_per_split = kSimtCausalChunk;
            L.nsplit = (p.N + kSimtCausalChunk - 1) / kSimtCausalChunk;
        }
        const size_t W = (size_t)p.d_v + 1;
        L.partial = off; off = align256(off + sizeof(float) * (size_t)p.BH() * L.nsplit * p.K * W);
        if (mode == 0) { L.mem = off; off = align256(off + sizeof(float) * (size_t)p.BH() * p.K * W); }
    }
    L.total = off;
    return L;
}

const char *const kSimtStages[3][8] = {
    {"prep", "resp", nullptr},
    {"prep", "resp_q", "resp_k", "write", "reduce", "read", nullptr},
    {"prep", "resp_q", "resp_k", "write", "scan", "causal", nullptr},
};

cudaError_t simt_responsibilities(const Problem &p, void *ws, cudaStream_t s, StageClock &clk) {
    SimtLayout L = simt_layout(p, -1, 0);
    Ptrs P = ptrs(L, ws);
    clk.mark();
    GMA_TRY(prep(p, P, s));
    clk.mark();
    float *G = static_cast<float *>(p.O);
    const long long bhs = (long long)p.N * p.K;
    if (p.dtype == GMA_F32) GMA_TRY(launch_resp<float>(p, p.Q, P.inv, P.cprime, G, bhs, p.K, 1, P.status, s));
    else GMA_TRY(launch_resp<__nv_bfloat16>(p, p.Q, P.inv, P.cprime, G, bhs, p.K, 1, P.status, s));
    clk.mark();
    return cudaSuccess;
}

cudaError_t simt_bidir(const Problem &p, int splits, void *ws, cudaStream_t s, StageClock &clk) {
    SimtLayout L = simt_layout(p, 0, splits);
    Ptrs P = ptrs(L, ws);
    clk.mark();
    GMA_TRY(prep(p, P, s));
    clk.mark();
    GMA_TRY(resp_both(p, P, s, clk));
    GMA_TRY(write_parts(p, L, P, s));
    clk.mark();
    const int E = p.K * (p.d_v + 1);
    launch_dep(reduce_splits_kernel, dim3((E + 255) / 256, p.BH()), 256, 0, s, P.part, L.nsplit, E, P.mem, P.status);
    GMA_TRY(cudaGetLastError());
    clk.mark();
    if (p.o_bf16) GMA_TRY(launch_read<__nv_bfloat16>(p, P.gq, P.mem, P.status, s));
    else GMA_TRY(launch_read<float>(p, P.gq, P.mem, P.status, s));
    clk.mark();
    return cudaSuccess;
}

cudaError_t simt_bidir_state(const Problem &p, int splits, void *ws, cudaStream_t s) {
    SimtLayout L = simt_layout(p, 0, splits);
    Ptrs P = ptrs(L, ws);
    StageClock none;
    none.stream = s;
    GMA_TRY(prep(p, P, s));
    GMA_TRY(resp_both(p, P, s, none));
    GMA_TRY(write_parts(p, L, P, s));
    const int E = p.K * (p.d_v + 1);
    launch_dep(reduce_splits_kernel, dim3((E + 255) / 256, p.BH()), 256, 0, s, P.part, L.nsplit, E, P.mem, P.status);
    return cudaGetLastError();
}

cudaError_t simt_causal_state(const Problem &p, void *ws, cudaStream_t s) {
    SimtLayout L = simt_layout(p, 1, 0);
    Ptrs P = ptrs(L, ws);
    StageClock none;
    none.stream = s;
    GMA_TRY(prep(p, P, s));
    GMA_TRY(resp_both(p, P, s, none));
    GMA_TRY(write_parts(p, L, P, s));
    const int E = p.K * (p.d_v + 1);
    launch_dep(scan_chunks_kernel, dim3((E + 255) / 256, p.BH()), 256, 0, s, P.part, L.nsplit, E, P.status);
    return cudaGetLastError();
}

cudaError_t simt_causal(const Problem &p, void *ws, cudaStream_t s, StageClock &clk) {
    SimtLayout L = simt_layout(p, 1, 0);
    Ptrs P = ptrs(L, ws);
    clk.mark();
    GMA_TRY(prep(p, P, s));
    clk.mark();
    GMA_TRY(resp_both(p, P, s, clk));
    GMA_TRY(write_parts(p, L, P, s));
    clk.mark();
    const int E = p.K * (p.d_v + 1);
    launch_dep(scan_chunks_kernel, dim3((E + 255) / 256, p.BH()), 256, 0, s, P.part, L.nsplit, E, P.status);
    GMA_TRY(cudaGetLastError());
    clk.mark();
    if (p.dtype == GMA_F32 && !p.o_bf16)
        GMA_TRY((launch_causal<float, float>(p, P.gq, P.gk, P.part, L.nsplit, P.status, s)));
    else if (p.dtype == GMA_F32)
        GMA_TRY((launch_causal<float, __nv_bfloat16>(p, P.gq, P.gk, P.part, L.nsplit, P.status, s)));
    else if (!p.o_bf16)
        GMA_TRY((launch_causal<__nv_bfloat16, float>(p, P.gq, P.gk, P.part, L.nsplit, P.status, s)));
    else
        GMA_TRY((launch_causal<__nv_bfloat16, __nv_bfloat16>(p, P.gq, P.gk, P.part, L.nsplit, P.status, s)));
    clk.mark();
    return cudaSuccess;
}

cudaError_t simt_read_memory(const Problem &p, const float *Vt, const float *Z, void *ws, cudaStream_t s,
                             StageClock &clk) {
    SimtLayout L = simt_layout(p, 3, 0);
    Ptrs P = ptrs(L, ws);
    clk.mark();
    GMA_TRY(prep(p, P, s));
    clk.mark();
    const long long bhs = (long long)p.K * p.N;
    if (p.dtype == GMA_F32) GMA_TRY(launch_resp<float>(p, p.Q, P.inv, P.cprime, P.gq, bhs, 1, p.N, P.status, s));
    else GMA_TRY(launch_resp<__nv_bfloat16>(p, p.Q, P.inv, P.cprime, P.gq, bhs, 1, p.N, P.status, s));
    clk.mark();
    const int E = p.K * (p.d_v + 1);
    launch_dep(pack_memory_kernel, dim3((E + 255) / 256, p.BH()), 256, 0, s, Vt, Z, p.K, p.d_v, P.mem, P.status);
    GMA_TRY(cudaGetLastError());
    clk.mark();
    if (p.o_bf16) GMA_TRY(launch_read<__nv_bfloat16>(p, P.gq, P.mem, P.status, s));
    else GMA_TRY(launch_read<float>(p, P.gq, P.mem, P.status, s));
    clk.mark();
    return cudaSuccess;
}

cudaError_t simt_causal_carry(const Problem &p, const float *Vt_in, const float *Z_in, float *Vt_out, float *Z_out,
                              void *ws, cudaStream_t s, StageClock &clk) {
    SimtLayout L = simt_layout(p, 1, 0);
    Ptrs P = ptrs(L, ws);
    clk.mark();
    GMA_TRY(prep(p, P, s));
    clk.mark();
    GMA_TRY(resp_both(p, P, s, clk));
    GMA_TRY(write_parts(p, L, P, s));
    clk.mark();
    const int E = p.K * (p.d_v + 1);
    launch_dep(scan_chunks_carry_kernel, dim3((E + 255) / 256, p.BH()), 256, 0, s, P.part, L.nsplit, p.K, p.d_v, Vt_in, Z_in,
                                                                           Vt_out, Z_out, P.status);
    GMA_TRY(cudaGetLastError());
    clk.mark();
    if (p.dtype == GMA_F32 && !p.o_bf16)
        GMA_TRY((launch_causal<float, float>(p, P.gq, P.gk, P.part, L.nsplit, P.status, s)));
    else if (p.dtype == GMA_F32)
        GMA_TRY((launch_causal<float, __nv_bfloat16>(p, P.gq, P.gk, P.part, L.nsplit, P.status, s)));
    else if (!p.o_bf16)
        GMA_TRY((launch_causal<__nv_bfloat16, float>(p, P.gq, P.gk, P.part, L.nsplit, P.status, s)));
    else
        GMA_TRY((launch_causal<__nv_bfloat16, __nv_bfloat16>(p, P.gq, P.gk, P.part, L.nsplit, P.status, s)));
    clk.mark();
    return cudaSuccess;
}

cudaError_t simt_prep(const Problem &p, void *ws, cudaStream_t s) {
    return prep(p, ptrs(simt_layout(p, -1, 0), ws), s);
}

cudaError_t simt_latent_memory(const Problem &p, int splits, float *Vt, float *Z, void *ws, cudaStream_t s,
                               StageClock &clk) {
    SimtLayout L = simt_layout(p, 2, splits);
    Ptrs P = ptrs(L, ws);
    clk.mark();
    GMA_TRY(prep(p, P, s));
    clk.mark();
    const long long bhs = (long long)p.K * p.N;
    if (p.dtype == GMA_F32) GMA_TRY(launch_resp<float>(p, p.Kx, P.inv, P.cprime, P.gk, bhs, 1, p.N, P.status, s));
    else GMA_TRY(launch_resp<__nv_bfloat16>(p, p.Kx, P.inv, P.cprime, P.gk, bhs, 1, p.N, P.status, s));
    clk.mark();
    GMA_TRY(write_parts(p, L, P, s));
    clk.mark();
    const int E = p.K * (p.d_v + 1);
    launch_dep(reduce_to_memory_kernel, dim3((E + 255) / 256, p.BH()), 256, 0, s, P.part, L.nsplit, p.K, p.d_v, Vt, Z,
                                                                          P.status);
    GMA_TRY(cudaGetLastError());
    clk.mark();
    return cudaSuccess;
}

}  // namespace gma
