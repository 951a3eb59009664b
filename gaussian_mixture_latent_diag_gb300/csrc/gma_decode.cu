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
// step is bound by HBM bandwidth on the state.  A small preparation kernel
// derives the per-head constants of the log-density once per call; then one
// CTA serves kDecRows batch rows of one head, with the head's constants staged
// in shared memory once for all of them, and each warp serves one row on its
// own, streaming the state through registers in batches of kDecBatch float4
// per lane.  Many resident warps, each with a batch of loads in flight, keep
// enough bytes in flight to cover HBM latency.
#include <cuda_bf16.h>

#include <cmath>

#include "gma_internal.h"

namespace gma {
namespace {

__device__ __forceinline__ float to_f32(float x) { return x; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 x) { return __bfloat162float(x); }

// Records the first device-side error of a call (later ones are dropped).
__device__ __forceinline__ void set_status(unsigned *status, unsigned code) { atomicCAS(status, 0u, code); }

constexpr int kDecRows = 8;                 // batch rows per CTA, one per warp
constexpr int kDecThreads = 32 * kDecRows;
constexpr int kDecBatch = 8;                // state float4 loads in flight per lane

// Workspace: [status word | -mu [H][K][d_r] | 1/sigma2 [H][K][d_r] | c' [H][K] |
// per-head flag [H]], 256-byte aligned regions.
struct DecodeWs {
    size_t negmu, inv, c, flag, total;
    DecodeWs(int H, int K, int d_r) {
        const size_t e = (size_t)H * K * d_r;
        negmu = kStatusBytes;
        inv = align256(negmu + 4 * e);
        c = align256(inv + 4 * e);
        flag = align256(c + 4 * (size_t)H * K);
        total = align256(flag + 4 * (size_t)H);
    }
};

// Per-head constants of the centred log-density ([GMA, Eqs. (2)-(3)]), with
// parameter validation: -mu, 1/sigma2 and c'_k = log pi_k - 1/2 sum_j log sigma2_kj.
// One CTA per head.  The logs are taken in the coalesced pass over the
// elements and kept in shared memory (rows padded to d_r + 1 floats, so the
// threads, one per component, read distinct banks); thread k then sums its
// component's log-determinant in fp32 as hi + lo, carrying every rounding
// error in lo (TwoSum, Knuth): a plain fp32 sum of up to 128 terms would lose
// the fp32 tolerance, and fp64 arithmetic is slow on this GPU.
constexpr int kPrepThreads = 512;  // many loads in flight: only H CTAs run

__global__ void __launch_bounds__(kPrepThreads) decode_prep_kernel(const float *__restrict__ mu,
                                                          const float *__restrict__ sigma2,
                                                          const float *__restrict__ log_pi, int K, int d_r,
                                                          float *__restrict__ negmu, float *__restrict__ inv,
                                                          float *__restrict__ cprime, unsigned *flag,
                                                          unsigned *status) {
    extern __shared__ float slog[];  // [K][d_r + 1]
    const int h = blockIdx.x;
    // Nothing else touches the call's status word until the step kernel, which
    // runs after this one: the first block clears it here.
    if (h == 0 && threadIdx.x == 0) *status = 0u;
    const size_t base = (size_t)h * K * d_r;
    bool bad = false;
#pragma unroll 4
    for (int e = threadIdx.x; e < K * d_r; e += blockDim.x) {
        const float m = mu[base + e], s2 = sigma2[base + e];
        bad |= !(s2 > 0.f) || !isfinite(s2) || !isfinite(m);
        negmu[base + e] = -m;
        inv[base + e] = __frcp_rn(s2);
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
        const float lp = log_pi[(size_t)h * K + k];
        bad |= !isfinite(lp);
        cprime[(size_t)h * K + k] = (lp - 0.5f * hi) - 0.5f * lo;
    }
    // every call writes every head's flag, so no clearing is needed
    if (__syncthreads_or(bad)) {
        if (threadIdx.x == 0) flag[h] = GMA_ERR_NONFINITE_PARAM;
    } else if (threadIdx.x == 0) {
        flag[h] = 0u;
    }
}

// Shared memory of one CTA, in floats, each region starting on a 16-byte
// boundary: -mu and 1/sigma2 rows padded to d_r + 4 floats (read as float4;
// eight consecutive k of a quarter-warp fall on distinct banks), c', the rows'
// q and k, and each warp's gamma^Q | gamma^K.
struct DecodeSmem {
    __host__ __device__ static int up4(int x) { return (x + 3) & ~3; }
    __host__ __device__ static int pr(int d_r) { return d_r + 4; }
    __host__ __device__ static int o_inv(int K, int d_r) { return K * pr(d_r); }
    __host__ __device__ static int o_c(int K, int d_r) { return 2 * K * pr(d_r); }
    __host__ __device__ static int o_x(int K, int d_r) { return o_c(K, d_r) + up4(K); }
    __host__ __device__ static int o_g(int K, int d_r) { return o_x(K, d_r) + 2 * kDecRows * d_r; }
    static size_t floats(int K, int d_r) { return (size_t)o_g(K, d_r) + 2 * kDecRows * up4(K); }
};

// grid (ceil(B / kDecRows), H), kDecThreads threads; d_r a multiple of 8.
//   q, kx : [B][H][d_r]   v : [B][H][D_V]   Vt : [B][H][K][D_V]   Z : [B][H][K]   O : [B][H][D_V]
//   negmu, inv : [H][K][d_r]   cprime : [H][K]   flag : [H]   (decode_prep_kernel)
// A head whose flag is set (an invalid parameter value) is left untouched and
// its first CTA records the flag in the call's status word.  After the head's
// constants are staged, warp w serves batch row b0 + w on its own: its two
// responsibility rows, then its state in batches of kDecBatch float4 per lane,
// with warp-level reductions only.
template <int D_V, typename T>
__global__ void __launch_bounds__(kDecThreads, 4) decode_step_kernel(
    const T *__restrict__ q, const T *__restrict__ kx, const T *__restrict__ v,
    const float *__restrict__ negmu, const float *__restrict__ inv, const float *__restrict__ cprime,
    int B, int H, int K, int d_r, float eps, float *__restrict__ Vt, float *__restrict__ Z,
    float *__restrict__ O, const unsigned *flag, unsigned *status) {
    {
        const unsigned f = flag[blockIdx.y];
        if (f != 0u) {
            if (blockIdx.x == 0 && threadIdx.x == 0) set_status(status, f);
            return;
        }
    }
    using L = DecodeSmem;
    constexpr int C4 = D_V / 4;    // float4 columns of a state row
    constexpr int RPL = 32 / C4;   // state rows one warp-wide float4 access covers
    const int PR = L::pr(d_r), KP = L::up4(K);
    extern __shared__ __align__(16) float smem[];
    float *snm = smem;                      // [K][PR]  -mu
    float *sinv = smem + L::o_inv(K, d_r);  // [K][PR]  1/sigma2
    float *sc = smem + L::o_c(K, d_r);      // [K]
    float *sx = smem + L::o_x(K, d_r);      // [2G][d_r]: query rows, then key rows
    float *sgam = smem + L::o_g(K, d_r);    // [G][2][KP]: gamma^Q | gamma^K of each warp's row

    const int h = blockIdx.y, b0 = blockIdx.x * kDecRows;
    const int nrow = min(kDecRows, B - b0);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

    const int dq = d_r / 4;
    const float4 *nm4 = reinterpret_cast<const float4 *>(negmu + (size_t)h * K * d_r);
    const float4 *iv4 = reinterpret_cast<const float4 *>(inv + (size_t)h * K * d_r);
    for (int e = tid; e < K * dq; e += kDecThreads) {
        const int k = e / dq, j4 = e % dq;
        reinterpret_cast<float4 *>(snm + k * PR)[j4] = nm4[e];
        reinterpret_cast<float4 *>(sinv + k * PR)[j4] = iv4[e];
    }
    for (int k = tid; k < K; k += kDecThreads) sc[k] = cprime[(size_t)h * K + k];
    for (int e = tid; e < kDecRows * d_r; e += kDecThreads) {
        const int g = e / d_r, j = e % d_r;
        float xq = 0.f, xk = 0.f;
        if (g < nrow) {
            const size_t off = ((size_t)(b0 + g) * H + h) * d_r + j;
            xq = to_f32(q[off]);
            xk = to_f32(kx[off]);
        }
        sx[g * d_r + j] = xq;
        sx[(kDecRows + g) * d_r + j] = xk;
    }
    __syncthreads();
    if (warp >= nrow) return;  // no barrier follows

    const size_t bh = (size_t)(b0 + warp) * H + h;
    float4 *S4 = reinterpret_cast<float4 *>(Vt + bh * K * D_V);
    float *Zb = Z + bh * K;
    const int c4 = lane % C4, kk = lane / C4;
    const int nper = (K - kk + RPL - 1) / RPL;  // state rows k = kk + RPL * i this lane owns

    // Responsibilities of the row's query and key ([GMA, Eqs. (2)-(3)]); lane l
    // takes components l, l + 32, ...  Centred form
    //   s_k = c'_k - 1/2 sum_j (x_j - mu_kj)^2 / sigma2_kj
    // with eight interleaved partial sums (j mod 8, two per packed f32x2
    // register) combined exactly (TwoSum) into hi + lo, then a max-subtracted
    // softmax over k.  The packed operations round each element as the scalar
    // ones would.
    float *gam = sgam + warp * 2 * KP;  // [gamma^Q | gamma^K]
    for (int side = 0; side < 2; ++side) {
        const float4 *x4 = reinterpret_cast<const float4 *>(sx + (side * kDecRows + warp) * d_r);
        float *sr = gam + side * KP;
        float m = -INFINITY;
#pragma unroll 1
        for (int k = lane; k < K; k += 32) {
            const float4 *mk = reinterpret_cast<const float4 *>(snm + k * PR);
            const float4 *ik = reinterpret_cast<const float4 *>(sinv + k * PR);
            float2 acc[4];
#pragma unroll
            for (int w = 0; w < 4; ++w) acc[w] = make_float2(0.f, 0.f);
            for (int j4 = 0; j4 < dq; j4 += 2) {
#pragma unroll
                for (int hh = 0; hh < 2; ++hh) {
                    const float4 xv = x4[j4 + hh], mv = mk[j4 + hh], iv = ik[j4 + hh];
                    const float2 d0 = __fadd2_rn(make_float2(xv.x, xv.y), make_float2(mv.x, mv.y));
                    const float2 d1 = __fadd2_rn(make_float2(xv.z, xv.w), make_float2(mv.z, mv.w));
                    acc[2 * hh] = __ffma2_rn(__fmul2_rn(d0, d0), make_float2(iv.x, iv.y), acc[2 * hh]);
                    acc[2 * hh + 1] = __ffma2_rn(__fmul2_rn(d1, d1), make_float2(iv.z, iv.w), acc[2 * hh + 1]);
                }
            }
            const float q8[8] = {acc[0].x, acc[0].y, acc[1].x, acc[1].y, acc[2].x, acc[2].y, acc[3].x, acc[3].y};
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
        float zs = 0.f;
        for (int k = lane; k < K; k += 32) {
            const float e = expf(sr[k] - m);
            sr[k] = e;
            zs += e;
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) zs += __shfl_xor_sync(0xffffffffu, zs, off);
        const float rz = 1.0f / zs;
        for (int k = lane; k < K; k += 32) sr[k] *= rz;
    }
    __syncwarp();
    const float *gq = gam, *gk = gam + KP;

    // Z and den: lane l takes components l, l + 32, ...
    float den = 0.f;
    for (int k = lane; k < K; k += 32) {
        const float zn = Zb[k] + gk[k];
        Zb[k] = zn;
        den = fmaf(gq[k], zn, den);
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) den += __shfl_xor_sync(0xffffffffu, den, off);

    // Vt rows: Vt_k += gamma^K_k v, num += gamma^Q_k Vt_k (the updated row).
    const float4 vv = make_float4(to_f32(v[bh * D_V + 4 * c4 + 0]), to_f32(v[bh * D_V + 4 * c4 + 1]),
                                  to_f32(v[bh * D_V + 4 * c4 + 2]), to_f32(v[bh * D_V + 4 * c4 + 3]));
    float4 num = make_float4(0.f, 0.f, 0.f, 0.f);
    float4 st[kDecBatch];
    for (int i0 = 0; i0 < nper; i0 += kDecBatch) {
#pragma unroll
        for (int u = 0; u < kDecBatch; ++u)
            if (i0 + u < nper) st[u] = S4[(size_t)(kk + RPL * (i0 + u)) * C4 + c4];
#pragma unroll
        for (int u = 0; u < kDecBatch; ++u) {
            if (i0 + u < nper) {
                const int k = kk + RPL * (i0 + u);
                const float a = gk[k], bq = gq[k];
                float4 x = st[u];
                x.x = fmaf(a, vv.x, x.x);
                x.y = fmaf(a, vv.y, x.y);
                x.z = fmaf(a, vv.z, x.z);
                x.w = fmaf(a, vv.w, x.w);
                S4[(size_t)k * C4 + c4] = x;
                num.x = fmaf(bq, x.x, num.x);
                num.y = fmaf(bq, x.y, num.y);
                num.z = fmaf(bq, x.z, num.z);
                num.w = fmaf(bq, x.w, num.w);
            }
        }
    }
    // sum over the lanes that share column c4 (a fixed butterfly)
#pragma unroll
    for (int off = C4; off < 32; off <<= 1) {
        num.x += __shfl_xor_sync(0xffffffffu, num.x, off);
        num.y += __shfl_xor_sync(0xffffffffu, num.y, off);
        num.z += __shfl_xor_sync(0xffffffffu, num.z, off);
        num.w += __shfl_xor_sync(0xffffffffu, num.w, off);
    }
    if (kk == 0) {
        const float d = den + eps;
        reinterpret_cast<float4 *>(O + bh * D_V)[c4] = make_float4(num.x / d, num.y / d, num.z / d, num.w / d);
    }
}

template <int D_V, typename T>
cudaError_t launch_decode_v(const Problem &p, const DecodeWs &W, char *ws, float *Vt, float *Z, cudaStream_t s) {
    const size_t smem = DecodeSmem::floats(p.K, p.d_r) * sizeof(float);
    auto kern = decode_step_kernel<D_V, T>;
    if (smem > 48 * 1024) {  // above the default limit only: the call costs host time
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
    }
    dim3 grid((p.B + kDecRows - 1) / kDecRows, p.H);
    kern<<<grid, kDecThreads, smem, s>>>(static_cast<const T *>(p.Q), static_cast<const T *>(p.Kx),
                                         static_cast<const T *>(p.V), reinterpret_cast<const float *>(ws + W.negmu),
                                         reinterpret_cast<const float *>(ws + W.inv),
                                         reinterpret_cast<const float *>(ws + W.c), p.B, p.H, p.K, p.d_r, p.eps, Vt,
                                         Z, static_cast<float *>(p.O), reinterpret_cast<const unsigned *>(ws + W.flag),
                                         reinterpret_cast<unsigned *>(ws));
    return cudaGetLastError();
}

template <typename T>
cudaError_t launch_decode(const Problem &p, const DecodeWs &W, char *ws, float *Vt, float *Z, cudaStream_t s) {
    switch (p.d_v) {
        case 16: return launch_decode_v<16, T>(p, W, ws, Vt, Z, s);
        case 32: return launch_decode_v<32, T>(p, W, ws, Vt, Z, s);
        case 64: return launch_decode_v<64, T>(p, W, ws, Vt, Z, s);
        case 128: return launch_decode_v<128, T>(p, W, ws, Vt, Z, s);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace

size_t decode_workspace(int H, int K, int d_r) { return DecodeWs(H, K, d_r).total; }

cudaError_t simt_decode_step(const Problem &p, float *Vt, float *Z, void *ws, cudaStream_t s, StageClock &clk) {
    const DecodeWs W(p.H, p.K, p.d_r);
    char *b = static_cast<char *>(ws);
    clk.mark();
    const size_t prep_smem = sizeof(float) * (size_t)p.K * (p.d_r + 1);
    cudaError_t e;
    if (prep_smem > 48 * 1024) {
        e = cudaFuncSetAttribute(decode_prep_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)prep_smem);
        if (e != cudaSuccess) return e;
    }
    decode_prep_kernel<<<p.H, kPrepThreads, prep_smem, s>>>(p.mu, p.sigma2, p.log_pi, p.K, p.d_r,
                                                   reinterpret_cast<float *>(b + W.negmu),
                                                   reinterpret_cast<float *>(b + W.inv),
                                                   reinterpret_cast<float *>(b + W.c),
                                                   reinterpret_cast<unsigned *>(b + W.flag),
                                                   reinterpret_cast<unsigned *>(b));
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    clk.mark();
    e = p.dtype == GMA_F32 ? launch_decode<float>(p, W, b, Vt, Z, s) : launch_decode<__nv_bfloat16>(p, W, b, Vt, Z, s);
    if (e != cudaSuccess) return e;
    clk.mark();
    return cudaSuccess;
}

const char *const kAuxStages[5][8] = {
    {"prep", "resp_k", "write", "reduce", nullptr},
    {"prep", "step", nullptr},
    {"prep", "rows", "final", nullptr},
    {"prep", "resp_q", "pack", "read", nullptr},
    {"prep", "resp_q", "resp_k", "write", "scan", "causal", nullptr},
};

}  // namespace gma
