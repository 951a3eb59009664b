// gma_decode.cu -- one autoregressive position of the causal GMA for every
// (batch row, head): the carried latent memory is extended with the new key
// and then read with the new query.
//
// Paper: "Gaussian Mixture Attention: Linear-Time Sequence Mixing via
// Probabilistic Latent Routing" (arXiv 2606.18283), causal variant, Eq. (8b),
// with the prefix memories carried as running sums:
//   Vt^(i) = Vt^(i-1) + gamma^K_i v_i,   Z^(i) = Z^(i-1) + gamma^K_i   (j <= i: the new
//   position enters its own prefix before it is read)
//   o_i    = gamma^Q_i Vt^(i) / (gamma^Q_i Z^(i) + eps).
//
// Cost per (b, h): the state is read and written once (2 K (d_v + 1) fp32,
// 33 KB at K = d_v = 64) against a few hundred bytes of q, k, v and o, so the
// step is bound by HBM bandwidth on the state.  One CTA serves kDecRows batch
// rows of one head: the head's (mu, 1/sigma2, c') are derived and staged in
// shared memory once for all of them (no separate preparation launch), each
// thread keeps all of its state rows' loads in flight before it uses any of
// them, and the next row's loads are issued before the current row is updated.
#include <cuda_bf16.h>

#include <cmath>

#include "gma_internal.h"

namespace gma {
namespace {

__device__ __forceinline__ float to_f32(float x) { return x; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 x) { return __bfloat162float(x); }

// Records the first device-side error of a call (later ones are dropped).
__device__ __forceinline__ void set_status(unsigned *status, unsigned code) { atomicCAS(status, 0u, code); }

constexpr int kDecRows = 8;       // batch rows per CTA
constexpr int kDecThreads = 512;  // 16 warps: one query or key row each in the score phase

template <int D_V>
struct DecodeSmem {
    static constexpr int C4 = D_V / 4;              // float4 columns of a state row
    static constexpr int KS = kDecThreads / C4;     // state-row slices (threads per column)
    static constexpr int KPT = (128 + KS - 1) / KS; // state rows per thread at K = 128
    // Offsets (in floats) of the shared-memory regions, each rounded up to 4
    // floats so that every region starts on a 16-byte boundary.  Parameter rows
    // are padded to d_r + 1 floats, so the lanes (consecutive k) read distinct
    // banks.
    __host__ __device__ static int up4(int x) { return (x + 3) & ~3; }
    __host__ __device__ static int o_inv(int K, int d_r) { return up4(K * (d_r + 1)); }
    __host__ __device__ static int o_c(int K, int d_r) { return o_inv(K, d_r) + up4(K * (d_r + 1)); }
    __host__ __device__ static int o_x(int K, int d_r) { return o_c(K, d_r) + up4(K); }
    __host__ __device__ static int o_g(int K, int d_r) { return o_x(K, d_r) + 2 * kDecRows * d_r; }
    __host__ __device__ static int o_v(int K, int d_r) { return o_g(K, d_r) + up4(2 * kDecRows * K); }
    __host__ __device__ static int o_red(int K, int d_r) { return o_v(K, d_r) + kDecRows * D_V; }
    static size_t floats(int K, int d_r) { return (size_t)o_red(K, d_r) + (size_t)KS * (D_V + 1); }
};

// Loads the state rows a thread owns (column c4 of rows ks, ks + KS, ...) of one (b, h).
template <int C4, int KS, int KPT>
__device__ __forceinline__ void load_state(const float4 *S4, const float *Zb, int K, int ks, int c4, float4 (&st)[KPT],
                                           float (&zz)[KPT]) {
#pragma unroll
    for (int u = 0; u < KPT; ++u) {
        const int k = ks + u * KS;
        if (k < K) {
            st[u] = S4[(size_t)k * C4 + c4];
            zz[u] = c4 == 0 ? Zb[k] : 0.f;
        }
    }
}

// grid (ceil(B / kDecRows), H), kDecThreads threads; d_r a multiple of 8.
//   q, kx : [B][H][d_r]   v : [B][H][D_V]   Vt : [B][H][K][D_V]   Z : [B][H][K]   O : [B][H][D_V]
//   mu, sigma2 : [H][K][d_r]   log_pi : [H][K]
// The CTA validates its head's parameters and derives 1/sigma2 and
// c'_k = log pi_k - 1/2 sum_j log sigma2_kj itself; a head with an invalid
// parameter value records GMA_ERR_NONFINITE_PARAM and leaves its rows untouched.
template <int D_V, typename T>
__global__ void __launch_bounds__(kDecThreads, D_V <= 64 ? 2 : 1) decode_step_kernel(
    const T *__restrict__ q, const T *__restrict__ kx, const T *__restrict__ v,
    const float *__restrict__ mu, const float *__restrict__ sigma2, const float *__restrict__ log_pi,
    int B, int H, int K, int d_r, float eps, float *__restrict__ Vt, float *__restrict__ Z,
    float *__restrict__ O, unsigned *status) {
    using L = DecodeSmem<D_V>;
    constexpr int G = kDecRows, C4 = L::C4, KS = L::KS, KPT = L::KPT;
    const int PR = d_r + 1;
    extern __shared__ float smem[];
    float *smu = smem;                      // [K][PR]
    float *sinv = smem + L::o_inv(K, d_r);  // [K][PR]
    float *sc = smem + L::o_c(K, d_r);      // [K]
    float *sx = smem + L::o_x(K, d_r);      // [2G][d_r]: query rows, then key rows
    float *sg = smem + L::o_g(K, d_r);      // [2G][K]: gamma^Q rows, then gamma^K rows
    float *sv = smem + L::o_v(K, d_r);      // [G][D_V], read as float4
    float *red = smem + L::o_red(K, d_r);   // [KS][D_V + 1]

    const int h = blockIdx.y, b0 = blockIdx.x * G;
    const int nrow = min(G, B - b0);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    constexpr int NW = kDecThreads / 32;

    // Parameters of head h ([GMA, Eqs. (2)-(3)]), validated on the way in.
    bool bad = false;
    const float *muh = mu + (size_t)h * K * d_r, *s2h = sigma2 + (size_t)h * K * d_r;
    for (int e = tid; e < K * d_r; e += kDecThreads) {
        const int k = e / d_r, j = e % d_r;
        const float m = muh[e], s2 = s2h[e];
        bad |= !(s2 > 0.f) || !isfinite(s2) || !isfinite(m);
        smu[k * PR + j] = m;
        sinv[k * PR + j] = 1.0f / s2;
    }
    // c'_k: warp w takes k = w, w + NW, ...; the log-determinant is summed in
    // fp64 (a fixed butterfly over the lanes), where an fp32 sum of up to 128
    // terms would lose the fp32 tolerance.
    for (int k = warp; k < K; k += NW) {
        double acc = 0.0;
        for (int j = lane; j < d_r; j += 32) acc += (double)logf(s2h[(size_t)k * d_r + j]);
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
        if (lane == 0) {
            const float lp = log_pi[(size_t)h * K + k];
            bad |= !isfinite(lp);
            sc[k] = (float)((double)lp - 0.5 * acc);
        }
    }
    for (int e = tid; e < G * d_r; e += kDecThreads) {
        const int g = e / d_r, j = e % d_r;
        float xq = 0.f, xk = 0.f;
        if (g < nrow) {
            const size_t off = ((size_t)(b0 + g) * H + h) * d_r + j;
            xq = to_f32(q[off]);
            xk = to_f32(kx[off]);
        }
        sx[g * d_r + j] = xq;
        sx[(G + g) * d_r + j] = xk;
    }
    for (int e = tid; e < G * D_V; e += kDecThreads) {
        const int g = e / D_V, c = e % D_V;
        sv[e] = g < nrow ? to_f32(v[((size_t)(b0 + g) * H + h) * D_V + c]) : 0.f;
    }
    if (__syncthreads_or(bad)) {
        if (tid == 0) set_status(status, GMA_ERR_NONFINITE_PARAM);
        return;
    }

    // The first row's state loads go out before the scores are computed.
    const int c4 = tid % C4, ks = tid / C4;
    float4 st[KPT];
    float zz[KPT];
    load_state<C4, KS, KPT>(reinterpret_cast<const float4 *>(Vt + ((size_t)b0 * H + h) * K * D_V),
                            Z + ((size_t)b0 * H + h) * K, K, ks, c4, st, zz);

    // Responsibilities: warp w scores row w (rows 0..G-1 are queries, G..2G-1
    // keys); lane l takes components l, l + 32, ...  Centred form
    //   s_k = c'_k - 1/2 sum_j (x_j - mu_kj)^2 / sigma2_kj
    // with eight interleaved partial sums (j mod 8) combined exactly (TwoSum)
    // into hi + lo, then a max-subtracted softmax over k.  Each lane reads and
    // writes only its own entries of sg.
    for (int r = warp; r < 2 * G; r += NW) {
        if (r % G >= nrow) continue;  // warp-uniform
        const float *x = sx + r * d_r;
        float *sr = sg + r * K;
        float m = -INFINITY;
#pragma unroll 1
        for (int k = lane; k < K; k += 32) {
            const float *mk = smu + k * PR, *ik = sinv + k * PR;
            float q8[8];
#pragma unroll
            for (int w = 0; w < 8; ++w) q8[w] = 0.f;
            for (int j0 = 0; j0 < d_r; j0 += 8) {
#pragma unroll
                for (int w = 0; w < 8; ++w) {
                    const float d = x[j0 + w] - mk[j0 + w];
                    q8[w] = fmaf(d * d, ik[j0 + w], q8[w]);
                }
            }
            float hi = q8[0], lo = 0.f;
#pragma unroll
            for (int w = 1; w < 8; ++w) {
                const float t = hi + q8[w], bb = t - hi;
                lo += (hi - (t - bb)) + (q8[w] - bb);
                hi = t;
            }
            const float sk = (sc[k] - 0.5f * hi) - 0.5f * lo;
            sr[k] = sk;
            m = fmaxf(m, sk);
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
        float z = 0.f;
        for (int k = lane; k < K; k += 32) {
            const float e = expf(sr[k] - m);
            sr[k] = e;
            z += e;
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) z += __shfl_xor_sync(0xffffffffu, z, off);
        const float rz = 1.0f / z;
        for (int k = lane; k < K; k += 32) sr[k] *= rz;
    }
    __syncthreads();

    // State update and read, one batch row at a time, the next row's state
    // loads in flight while the current row is updated.  Thread (ks, c4) owns
    // the float4 column c4 of state rows ks, ks + KS, ...; the c4 == 0 threads
    // also own Z.  The read's sums over k are finished across the KS slices in
    // a fixed order.
    for (int g = 0; g < nrow; ++g) {
        const size_t bh = (size_t)(b0 + g) * H + h;
        float4 *S4 = reinterpret_cast<float4 *>(Vt + bh * K * D_V);
        float *Zb = Z + bh * K;
        float4 cur[KPT];
        float zc[KPT];
#pragma unroll
        for (int u = 0; u < KPT; ++u) {
            cur[u] = st[u];
            zc[u] = zz[u];
        }
        if (g + 1 < nrow)
            load_state<C4, KS, KPT>(reinterpret_cast<const float4 *>(Vt + (bh + H) * K * D_V), Z + (bh + H) * K, K,
                                    ks, c4, st, zz);
        const float *gq = sg + g * K, *gk = sg + (G + g) * K;
        const float4 vv = reinterpret_cast<const float4 *>(sv + g * D_V)[c4];
        float4 num = make_float4(0.f, 0.f, 0.f, 0.f);
        float den = 0.f;
#pragma unroll
        for (int u = 0; u < KPT; ++u) {
            const int k = ks + u * KS;
            if (k < K) {
                const float a = gk[k], bq = gq[k];
                float4 x = cur[u];
                x.x = fmaf(a, vv.x, x.x);
                x.y = fmaf(a, vv.y, x.y);
                x.z = fmaf(a, vv.z, x.z);
                x.w = fmaf(a, vv.w, x.w);
                S4[(size_t)k * C4 + c4] = x;
                num.x = fmaf(bq, x.x, num.x);
                num.y = fmaf(bq, x.y, num.y);
                num.z = fmaf(bq, x.z, num.z);
                num.w = fmaf(bq, x.w, num.w);
                if (c4 == 0) {
                    const float zn = zc[u] + a;
                    Zb[k] = zn;
                    den = fmaf(bq, zn, den);
                }
            }
        }
        float *rr = red + ks * (D_V + 1);
        rr[4 * c4 + 0] = num.x;
        rr[4 * c4 + 1] = num.y;
        rr[4 * c4 + 2] = num.z;
        rr[4 * c4 + 3] = num.w;
        if (c4 == 0) rr[D_V] = den;
        __syncthreads();
        if (tid < D_V) {
            float acc = 0.f, d = 0.f;
            for (int t = 0; t < KS; ++t) {
                acc += red[t * (D_V + 1) + tid];
                d += red[t * (D_V + 1) + D_V];
            }
            O[bh * D_V + tid] = acc / (d + eps);
        }
        __syncthreads();
    }
}

template <int D_V, typename T>
cudaError_t launch_decode_v(const Problem &p, float *Vt, float *Z, unsigned *status, cudaStream_t s) {
    const size_t smem = DecodeSmem<D_V>::floats(p.K, p.d_r) * sizeof(float);
    auto kern = decode_step_kernel<D_V, T>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    dim3 grid((p.B + kDecRows - 1) / kDecRows, p.H);
    kern<<<grid, kDecThreads, smem, s>>>(static_cast<const T *>(p.Q), static_cast<const T *>(p.Kx),
                                         static_cast<const T *>(p.V), p.mu, p.sigma2, p.log_pi, p.B, p.H, p.K,
                                         p.d_r, p.eps, Vt, Z, static_cast<float *>(p.O), status);
    return cudaGetLastError();
}

template <typename T>
cudaError_t launch_decode(const Problem &p, float *Vt, float *Z, unsigned *status, cudaStream_t s) {
    switch (p.d_v) {
        case 16: return launch_decode_v<16, T>(p, Vt, Z, status, s);
        case 32: return launch_decode_v<32, T>(p, Vt, Z, status, s);
        case 64: return launch_decode_v<64, T>(p, Vt, Z, status, s);
        case 128: return launch_decode_v<128, T>(p, Vt, Z, status, s);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace

size_t decode_workspace() { return kStatusBytes; }

cudaError_t simt_decode_step(const Problem &p, float *Vt, float *Z, void *ws, cudaStream_t s, StageClock &clk) {
    unsigned *status = static_cast<unsigned *>(ws);
    clk.mark();
    cudaError_t e = cudaMemsetAsync(status, 0, sizeof(unsigned), s);
    if (e != cudaSuccess) return e;
    clk.mark();
    e = p.dtype == GMA_F32 ? launch_decode<float>(p, Vt, Z, status, s)
                           : launch_decode<__nv_bfloat16>(p, Vt, Z, status, s);
    if (e != cudaSuccess) return e;
    clk.mark();
    return cudaSuccess;
}

const char *const kAuxStages[5][8] = {
    {"prep", "resp_k", "write", "reduce", nullptr},
    {"reset", "step", nullptr},
    {"prep", "rows", "final", nullptr},
    {"prep", "resp_q", "pack", "read", nullptr},
    {"prep", "resp_q", "resp_k", "write", "scan", "causal", nullptr},
};

}  // namespace gma
