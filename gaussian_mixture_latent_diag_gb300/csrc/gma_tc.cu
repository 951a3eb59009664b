// gma_tc.cu -- tcgen05 tensor-core kernels for the GMA forward pass (bf16
// inputs, d_r = 64, K <= 64, d_v in {64, 128}).
//
// Responsibilities ([GMA, Eqs. (2)-(3)]) are computed as a GEMM on the
// expanded quadratic,
//   s_ik * log2(e) = sum_j x_ij^2 a_kj + x_ij b_kj + c_k,
//   a = -log2(e) / (2 sigma2),  b = log2(e) mu / sigma2,
//   c = log2(e) (log pi_k - 1/2 sum_j (mu^2 / sigma2 + log sigma2)),
// with every operand split into a bf16 high part and a bf16 low part so that
// the five products x2hi*ahi + x2hi*alo + x2lo*ahi + x*bhi + x*blo carry
// ~16 significant bits (x is bf16, so x^2 is exactly x2hi + x2lo).  The
// softmax over k runs in fp32 on the TMEM accumulator rows.  Gamma is split
// into bf16 hi + lo again for the value contractions:
//   write (Eqs. (5)-(6)):  [Vt | Z] += [Ghi ; Glo]^T [V | 1]     (per key tile)
//   read  (Eq. (7)):       [num | den] = Ghi [Vhi|Zhi] + Glo [Vhi|Zhi] + Ghi [Vlo|Zlo]
// and O = num / (den + eps * r) with r the un-normalised query row sum.
//
// Paper: "Gaussian Mixture Attention: Linear-Time Sequence Mixing via
// Probabilistic Latent Routing" (arXiv 2606.18283), cited [GMA, ...].
#include <cuda.h>
#include <cuda_bf16.h>
#include <cudaTypedefs.h>

#include <cmath>
#include <mutex>

#include "gma_internal.h"
#include "tc_ptx.cuh"

namespace gma {
namespace {

using namespace ptx;

constexpr int kTile = 128;         // tokens per tile (UMMA M)
constexpr int kDR = 64;            // routing dimension handled here
constexpr int kKP = 64;            // padded number of components
constexpr int kTileBytes = kTile * 128;                  // one [128 x 64] bf16 SW128 tile
constexpr int kCoefMatBytes = kKP * kDR * 2;             // one coefficient matrix [KP x d_r] bf16
constexpr int kCoefBytes = 4 * kCoefMatBytes + kKP * 4;  // a_hi | a_lo | b_hi | b_lo | c
constexpr size_t kCoefStride = (kCoefBytes + 1023) & ~1023;
constexpr int kGS = 2 * (kKP / 64) * 1024;               // Gamma buffer: bytes per 8-token group
constexpr float kLog2e = 1.4426950408889634f;

__device__ __forceinline__ bool failed(const unsigned *status) {
    return *reinterpret_cast<const volatile unsigned *>(status) != 0u;
}
__device__ __forceinline__ void set_status(unsigned *status, unsigned code) { atomicCAS(status, 0u, code); }

// Byte offset of element (row, col) of a K-major SW128 tile whose rows are
// 128 bytes (64 bf16) and whose 8-row groups are `group_stride` bytes apart.
__host__ __device__ __forceinline__ uint32_t sw128_offset(int row, int col, int group_stride) {
    return (uint32_t)((row >> 3) * group_stride + (row & 7) * 128 + ((((col >> 3) ^ (row & 7)) & 7) << 4) +
                      (col & 7) * 2);
}

// ------------------------------------------------------------------ coefficient prep
// One block per head.  Writes the four bf16 coefficient matrices in the
// K-major SW128 byte image the score MMA reads (rows = components, 128 B of
// d_r per row), plus c_k (fp32, -inf for padded components).  Validates the
// parameters.
__global__ void coef_prep_tc_kernel(const float *__restrict__ mu, const float *__restrict__ sigma2,
                                    const float *__restrict__ log_pi, int K, uint8_t *__restrict__ img,
                                    unsigned *status) {
    const int h = blockIdx.x;
    uint8_t *base = img + (size_t)h * kCoefStride;
    __nv_bfloat16 *ahi = reinterpret_cast<__nv_bfloat16 *>(base);
    for (int e = threadIdx.x; e < kKP * kDR; e += blockDim.x) {
        const int k = e / kDR, j = e % kDR;
        float a = 0.f, b = 0.f;
        if (k < K) {
            const float s2 = sigma2[((size_t)h * K + k) * kDR + j], m = mu[((size_t)h * K + k) * kDR + j];
            if (!(s2 > 0.f) || !isfinite(s2) || !isfinite(m)) set_status(status, GMA_ERR_NONFINITE_PARAM);
            a = -0.5f * kLog2e / s2;
            b = kLog2e * m / s2;
        }
        const __nv_bfloat16 ah = __float2bfloat16_rn(a), bh = __float2bfloat16_rn(b);
        const uint32_t off = sw128_offset(k, j, 1024) / 2;  // in bf16 elements
        ahi[off] = ah;
        ahi[kCoefMatBytes / 2 + off] = __float2bfloat16_rn(a - __bfloat162float(ah));
        ahi[2 * kCoefMatBytes / 2 + off] = bh;
        ahi[3 * kCoefMatBytes / 2 + off] = __float2bfloat16_rn(b - __bfloat162float(bh));
    }
    // c_k: one warp per component, lanes over j, fp32 terms summed in fp64.
    float *cvec = reinterpret_cast<float *>(base + 4 * kCoefMatBytes);
    const int lane = threadIdx.x & 31, nwarps = blockDim.x >> 5;
    for (int k = threadIdx.x >> 5; k < kKP; k += nwarps) {
        double acc = 0.0;
        if (k < K)
            for (int j = lane; j < kDR; j += 32) {
                const float s2 = sigma2[((size_t)h * K + k) * kDR + j], m = mu[((size_t)h * K + k) * kDR + j];
                acc += (double)(m * m / s2) + (double)logf(s2);
            }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
        if (lane == 0) {
            if (k < K) {
                const float lp = log_pi[(size_t)h * K + k];
                if (!isfinite(lp)) set_status(status, GMA_ERR_NONFINITE_PARAM);
                cvec[k] = (float)((double)kLog2e * ((double)lp - 0.5 * acc));
            } else {
                cvec[k] = -INFINITY;
            }
        }
    }
}

// ------------------------------------------------------------------ shared pieces

// x^2 split: for every bf16 x of a tile, x2hi = rn(x*x), x2lo = x*x - x2hi
// (exact, since x*x has at most 16 significant bits).  Position-preserving on
// the swizzled tile, so the outputs share the tile's layout.
__device__ __forceinline__ void prep_x2(const uint8_t *x, uint8_t *x2h, uint8_t *x2l, int bytes, int tid,
                                        int nthreads) {
    const uint4 *src = reinterpret_cast<const uint4 *>(x);
    uint4 *dh = reinterpret_cast<uint4 *>(x2h);
    uint4 *dl = reinterpret_cast<uint4 *>(x2l);
    for (int i = tid; i < bytes / 16; i += nthreads) {
        const uint4 v = src[i];
        uint4 h, l;
        h.x = bf2_fma(v.x, v.x, 0x80008000u); l.x = bf2_fma(v.x, v.x, h.x ^ 0x80008000u);
        h.y = bf2_fma(v.y, v.y, 0x80008000u); l.y = bf2_fma(v.y, v.y, h.y ^ 0x80008000u);
        h.z = bf2_fma(v.z, v.z, 0x80008000u); l.z = bf2_fma(v.z, v.z, h.z ^ 0x80008000u);
        h.w = bf2_fma(v.w, v.w, 0x80008000u); l.w = bf2_fma(v.w, v.w, h.w ^ 0x80008000u);
        dh[i] = h;
        dl[i] = l;
    }
}

// The 20 score MMAs of one 128-token tile: D[128 x KP] = x2hi*ahi + x2hi*alo +
// x2lo*ahi + x*bhi + x*blo, each over d_r = 64 in four K-steps of 16.
__device__ __forceinline__ void issue_scores(uint32_t d_tmem, const uint8_t *x, const uint8_t *x2h,
                                             const uint8_t *x2l, const uint8_t *coef) {
    constexpr uint32_t idesc = idesc_bf16(kTile, kKP, false, false);
    const uint32_t sx = smem_u32(x), sh = smem_u32(x2h), sl = smem_u32(x2l), sc = smem_u32(coef);
#pragma unroll
    for (int kk = 0; kk < kDR / 16; ++kk) {
        const uint32_t o = kk * 32;
        const uint64_t ax = sdesc_sw128(sx + o, 16, 1024), ah = sdesc_sw128(sh + o, 16, 1024),
                       al = sdesc_sw128(sl + o, 16, 1024);
        const uint64_t bah = sdesc_sw128(sc + o, 16, 1024), bal = sdesc_sw128(sc + kCoefMatBytes + o, 16, 1024),
                       bbh = sdesc_sw128(sc + 2 * kCoefMatBytes + o, 16, 1024),
                       bbl = sdesc_sw128(sc + 3 * kCoefMatBytes + o, 16, 1024);
        umma_bf16(d_tmem, ah, bah, idesc, kk > 0 ? 1u : 0u);
        umma_bf16(d_tmem, ah, bal, idesc, 1u);
        umma_bf16(d_tmem, al, bah, idesc, 1u);
        umma_bf16(d_tmem, ax, bbh, idesc, 1u);
        umma_bf16(d_tmem, ax, bbl, idesc, 1u);
    }
}

// Loads this thread's score row (KP columns) and turns it into exponentials
// e_k = 2^(s_k + c_k - max) (un-normalised responsibilities, max e = 1).
// Returns the row sum r.
__device__ __forceinline__ float score_row_exp(uint32_t taddr, const float *cvec, float (&e)[kKP]) {
    uint32_t r0[32], r1[32];
    tmem_ld32(taddr, r0);
    tmem_ld32(taddr + 32, r1);
    tmem_wait_ld();
    float m = -INFINITY;
#pragma unroll
    for (int k = 0; k < 32; ++k) {
        e[k] = __uint_as_float(r0[k]) + cvec[k];
        e[k + 32] = __uint_as_float(r1[k]) + cvec[k + 32];
        m = fmaxf(m, fmaxf(e[k], e[k + 32]));
    }
    float r = 0.f;
#pragma unroll
    for (int k = 0; k < kKP; ++k) {
        e[k] = ex2(e[k] - m);
        r += e[k];
    }
    return r;
}

// Writes one responsibility row (scaled by `scale`) as bf16 hi and lo parts
// into the Gamma buffer: 8-token groups of kGS bytes, hi rows at +0, lo rows
// at +1024 within a group, 16-byte chunks swizzled by (row % 8).
__device__ __forceinline__ void store_gamma_row(uint8_t *gbuf, int t, const float (&e)[kKP], float scale) {
    uint8_t *hi = gbuf + (t >> 3) * kGS + (t & 7) * 128;
    uint8_t *lo = hi + 1024;
#pragma unroll
    for (int c = 0; c < kKP / 8; ++c) {
        uint32_t wh[4], wl[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const float g0 = e[c * 8 + 2 * q] * scale, g1 = e[c * 8 + 2 * q + 1] * scale;
            wh[q] = pack_bf2(g0, g1);
            wl[q] = pack_bf2(g0 - bf_lo(wh[q]), g1 - bf_hi(wh[q]));
        }
        const uint32_t sw = (uint32_t)((c ^ (t & 7)) << 4);
        *reinterpret_cast<uint4 *>(hi + sw) = make_uint4(wh[0], wh[1], wh[2], wh[3]);
        *reinterpret_cast<uint4 *>(lo + sw) = make_uint4(wl[0], wl[1], wl[2], wl[3]);
    }
}

// Aborts the CTA's work on a timed-out wait: records the status once.
__device__ __forceinline__ void note_timeout(unsigned *status, int *abort_flag) {
    set_status(status, GMA_ERR_TIMEOUT);
    *reinterpret_cast<volatile int *>(abort_flag) = 1;
}

// ------------------------------------------------------------------ write kernel
// Latent aggregation over one split of the keys of one head ([GMA, Eqs. (5)-(6)]):
// part[k][c] = sum_{j in split} gamma^K_jk V_jc, part[k][d_v] = sum gamma^K_jk.
// Grid (nsplit, B*H); 128 threads; thread t owns TMEM lane / tile row t.
template <int D_V>
struct WriteSmem {
    static constexpr int kX = 0;                                  // K_X tile (16 KB)
    static constexpr int kX2 = kX + kTileBytes;                   // x2hi | x2lo (32 KB), then Gamma
    static constexpr int kV = kX2 + 2 * kTileBytes;               // V tile(s): D_V/64 boxes of 16 KB
    static constexpr int kCoef = kV + (D_V / 64) * kTileBytes;    // 32 KB + c
    static constexpr int kOnes = kCoef + ((kCoefBytes + 1023) & ~1023);  // 2 KB of bf16 1.0
    static constexpr int kBars = kOnes + 2048;
    static constexpr int kBytes = kBars + 64;
    static constexpr int kAlloc = kBytes + 1024;                  // slack for 1 KB alignment
};

template <int D_V>
__global__ void __launch_bounds__(128, 1) tc_write_kernel(const __grid_constant__ CUtensorMap tmK,
                                                           const __grid_constant__ CUtensorMap tmV,
                                                           const uint8_t *__restrict__ coef_img, int H, int N,
                                                           int tiles_per_split, int nsplit,
                                                           float *__restrict__ part, unsigned *status) {
    using L = WriteSmem<D_V>;
    constexpr int kTmemCols = 256;
    constexpr int kAccV = kKP, kAccZ = kKP + D_V;  // TMEM columns
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t *xk = smem + L::kX, *x2 = smem + L::kX2, *vt = smem + L::kV, *coef = smem + L::kCoef,
            *ones = smem + L::kOnes;
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + L::kBars);  // [0] TMA, [1] MMA
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + 2);
    int *abort_flag = reinterpret_cast<int *>(bars + 3);
    const float *cvec = reinterpret_cast<const float *>(coef + 4 * kCoefMatBytes);

    const int tid = threadIdx.x, warp = tid >> 5;
    const int split = blockIdx.x, bh = blockIdx.y, h = bh % H;
    const int ntiles = (N + kTile - 1) / kTile;
    const int tile0 = split * tiles_per_split, tile1 = min(ntiles, tile0 + tiles_per_split);
    if (failed(status)) return;

    if (warp == 0) {
        tmem_alloc(tmem_slot, kTmemCols);
        tmem_relinquish();
    }
    if (tid == 0) {
        mbar_init(&bars[0], 1);
        mbar_init(&bars[1], 1);
        *abort_flag = 0;
        fence_mbar_init();
        tma_prefetch_desc(&tmK);
        tma_prefetch_desc(&tmV);
    }
    {
        const uint4 *src = reinterpret_cast<const uint4 *>(coef_img + (size_t)h * kCoefStride);
        uint4 *dst = reinterpret_cast<uint4 *>(coef);
        for (int i = tid; i < kCoefBytes / 16; i += blockDim.x) dst[i] = src[i];
        uint4 one4 = make_uint4(0x3F803F80u, 0x3F803F80u, 0x3F803F80u, 0x3F803F80u);
        for (int i = tid; i < 2048 / 16; i += blockDim.x) reinterpret_cast<uint4 *>(ones)[i] = one4;
    }
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
    constexpr uint32_t kTxBytes = kTileBytes * (1 + D_V / 64);

    if (tid == 0 && tile0 < tile1) {
        mbar_arrive_expect_tx(&bars[0], kTxBytes);
        tma_load_3d(xk, &tmK, 0, tile0 * kTile, bh, &bars[0]);
#pragma unroll
        for (int vb = 0; vb < D_V / 64; ++vb) tma_load_3d(vt + vb * kTileBytes, &tmV, vb * 64, tile0 * kTile, bh, &bars[0]);
    }
    uint32_t ph_tma = 0, ph_mma = 0;
    constexpr uint32_t idesc_v = idesc_bf16(kTile, 64, true, true);
    constexpr uint32_t idesc_z = idesc_bf16(kTile, 16, true, false);

    for (int tile = tile0; tile < tile1; ++tile) {
        if (!mbar_wait(&bars[0], ph_tma)) note_timeout(status, abort_flag);
        ph_tma ^= 1;
        prep_x2(xk, x2, x2 + kTileBytes, kTileBytes, tid, blockDim.x);
        fence_proxy_async_smem();
        __syncthreads();
        if (*reinterpret_cast<volatile int *>(abort_flag)) break;
        if (tid == 0) {
            tc_fence_after();
            issue_scores(tmem, xk, x2, x2 + kTileBytes, coef);
            umma_commit(&bars[1]);
        }
        if (!mbar_wait(&bars[1], ph_mma)) note_timeout(status, abort_flag);
        ph_mma ^= 1;
        tc_fence_after();
        {
            float e[kKP];
            const float r = score_row_exp(tmem + lane_base, cvec, e);
            const int tok = tile * kTile + tid;
            const float scale = tok < N ? 1.0f / r : 0.0f;  // rows past N contribute nothing
            store_gamma_row(x2, tid, e, scale);
        }
        tc_fence_before();
        fence_proxy_async_smem();
        __syncthreads();
        if (*reinterpret_cast<volatile int *>(abort_flag)) break;
        if (tid == 0) {
            tc_fence_after();
            const uint32_t sg = smem_u32(x2), sv = smem_u32(vt), so = smem_u32(ones);
            const uint64_t bz = sdesc_sw128(so, 16, 1024);
#pragma unroll
            for (int kk = 0; kk < kTile / 16; ++kk) {
                const uint32_t acc = (tile > tile0 || kk > 0) ? 1u : 0u;
                const uint64_t a = sdesc_sw128(sg + kk * 2 * kGS, 1024, kGS);
#pragma unroll
                for (int vb = 0; vb < D_V / 64; ++vb) {
                    const uint64_t b = sdesc_sw128(sv + vb * kTileBytes + kk * 2048, 16, 1024);
                    umma_bf16(tmem + kAccV + vb * 64, a, b, idesc_v, acc);
                }
                umma_bf16(tmem + kAccZ, a, bz, idesc_z, acc);
            }
            umma_commit(&bars[1]);
        }
        if (!mbar_wait(&bars[1], ph_mma)) note_timeout(status, abort_flag);
        ph_mma ^= 1;
        __syncthreads();
        if (*reinterpret_cast<volatile int *>(abort_flag)) break;
        if (tid == 0 && tile + 1 < tile1) {
            mbar_arrive_expect_tx(&bars[0], kTxBytes);
            tma_load_3d(xk, &tmK, 0, (tile + 1) * kTile, bh, &bars[0]);
#pragma unroll
            for (int vb = 0; vb < D_V / 64; ++vb)
                tma_load_3d(vt + vb * kTileBytes, &tmV, vb * 64, (tile + 1) * kTile, bh, &bars[0]);
        }
    }

    // Partial memory: rows 0..63 of the accumulator hold the hi-weighted sums,
    // rows 64..127 the lo-weighted ones; add them and write [KP][D_V + 1].
    const bool ok = !*reinterpret_cast<volatile int *>(abort_flag);
    if (ok && tile0 < tile1) {
        tc_fence_after();
        float *red = reinterpret_cast<float *>(smem);  // [128][D_V + 1] fp32, over the tiles region
        constexpr int W = D_V + 1;
#pragma unroll
        for (int cb = 0; cb < D_V / 32; ++cb) {
            uint32_t v[32];
            tmem_ld32(tmem + lane_base + kAccV + cb * 32, v);
            tmem_wait_ld();
#pragma unroll
            for (int q = 0; q < 32; ++q) red[tid * W + cb * 32 + q] = __uint_as_float(v[q]);
        }
        {
            uint32_t z[16];
            tmem_ld16(tmem + lane_base + kAccZ, z);
            tmem_wait_ld();
            red[tid * W + D_V] = __uint_as_float(z[0]);
        }
        __syncthreads();
        float *out = part + ((size_t)bh * nsplit + split) * kKP * W;
        for (int e = tid; e < kKP * W; e += blockDim.x) out[e] = red[e] + red[kKP * W + e];
    } else if (ok) {  // a split without tiles contributes zeros
        float *out = part + ((size_t)bh * nsplit + split) * kKP * (D_V + 1);
        for (int e = tid; e < kKP * (D_V + 1); e += blockDim.x) out[e] = 0.f;
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, kTmemCols);
}

// ------------------------------------------------------------------ causal
// Exclusive prefix over the segment aggregates of each head, in segment
// order, in place: part[s] <- sum_{s' < s} part[s'] ([GMA, causal variant:
// the prefix memories are cumulative sums along the sequence]).
__global__ void scan_segments_kernel(float *__restrict__ part, int nseg, int E, const unsigned *status) {
    if (failed(status)) return;
    const int bh = blockIdx.y;
    const int e = blockIdx.x * blockDim.x + threadIdx.x;
    if (e >= E) return;
    float *p = part + (size_t)bh * nseg * E + e;
    float run = 0.f;
    for (int s = 0; s < nseg; ++s) {
        const float cur = p[(size_t)s * E];
        p[(size_t)s * E] = run;
        run += cur;
    }
}

// Writes the state B operand [NB x KP] (bf16 hi at `bop`, lo at bop + NB*128)
// from the fp32 state S[k][n] (row n < D_V: S[:, n]; row D_V: Z; rows above: 0).
template <int D_V>
__device__ __forceinline__ void build_state_operand(const float *S, uint8_t *bop, int tid, int nthreads) {
    constexpr int NB = D_V + 16, W = D_V + 1;
    __nv_bfloat16 *bhi = reinterpret_cast<__nv_bfloat16 *>(bop);
    __nv_bfloat16 *blo = reinterpret_cast<__nv_bfloat16 *>(bop + NB * 128);
    for (int e = tid; e < NB * kKP; e += nthreads) {
        const int n = e / kKP, k = e % kKP;
        const float v = n <= D_V ? S[k * W + n] : 0.f;
        const __nv_bfloat16 vh = __float2bfloat16_rn(v);
        const uint32_t off = sw128_offset(n, k, 1024) / 2;
        bhi[off] = vh;
        blo[off] = __float2bfloat16_rn(v - __bfloat162float(vh));
    }
}

// Causal GMA over one segment of one head ([GMA, Eq. (8b)]), in chunks of
// C = 128 tokens.  With (S, Z) the prefix memory before the chunk and
// P = mask_{j <= i}(Gamma^Q_c Gamma^K_c^T) the intra-chunk affinity:
//   O_i = (sum_j P_ij V_j + gQ_i S) / (sum_j P_ij + gQ_i Z + eps r_i),
// (gQ un-normalised, r_i its row sum), then S += Gamma^K_c^T V_c, Z += Gamma^K_c^T 1.
// The segment's starting prefix comes from scan_segments_kernel.
struct CausalSmem {
    static constexpr int D_V = 64, NB = D_V + 16, W = D_V + 1;
    static constexpr int kA = 0;                      // xq | xk | x2q (x2hi|x2lo) -> gq -> P (64 KB)
    static constexpr int kXQ = kA, kXK = kA + kTileBytes, kX2Q = kA + 2 * kTileBytes;
    static constexpr int kB = kA + 4 * kTileBytes;    // x2k (x2hi|x2lo) -> gk (32 KB)
    static constexpr int kV = kB + 2 * kTileBytes;    // V tile (16 KB)
    static constexpr int kCoef = kV + kTileBytes;
    static constexpr int kBop = kCoef + ((kCoefBytes + 1023) & ~1023);  // state operand hi | lo
    static constexpr int kOnes = kBop + 2 * NB * 128;
    static constexpr int kS = kOnes + 2048;           // fp32 state [KP][W]
    static constexpr int kBars = kS + ((kKP * W * 4 + 1023) & ~1023);
    static constexpr int kBytes = kBars + 64;
    static constexpr int kAlloc = kBytes + 1024;
};
constexpr int kGSP = 4096;  // P buffer: bytes per 8-query group (128 keys, hi | lo)

__global__ void __launch_bounds__(128, 1) tc_causal_kernel(const __grid_constant__ CUtensorMap tmQ,
                                                            const __grid_constant__ CUtensorMap tmK,
                                                            const __grid_constant__ CUtensorMap tmV,
                                                            const uint8_t *__restrict__ coef_img,
                                                            const float *__restrict__ prefix, int H, int N,
                                                            int tiles_per_seg, int nseg, float eps,
                                                            void *__restrict__ O, int o_bf16, unsigned *status) {
    using L = CausalSmem;
    constexpr int D_V = L::D_V, NB = L::NB, W = L::W;
    constexpr int kTmemCols = 256;
    constexpr int kSQ = 0, kSK = kKP, kP = 0, kSc = 0, kO = 128;  // TMEM columns
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t *xq = smem + L::kXQ, *xk = smem + L::kXK, *x2q = smem + L::kX2Q, *pbuf = smem + L::kA;
    uint8_t *x2k = smem + L::kB, *vt = smem + L::kV, *coef = smem + L::kCoef, *bop = smem + L::kBop,
            *ones = smem + L::kOnes;
    float *S = reinterpret_cast<float *>(smem + L::kS);
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + L::kBars);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + 2);
    int *abort_flag = reinterpret_cast<int *>(bars + 3);
    const float *cvec = reinterpret_cast<const float *>(coef + 4 * kCoefMatBytes);

    const int tid = threadIdx.x, warp = tid >> 5;
    const int seg = blockIdx.x, bh = blockIdx.y, h = bh % H;
    const int ntiles = (N + kTile - 1) / kTile;
    const int tile0 = seg * tiles_per_seg, tile1 = min(ntiles, tile0 + tiles_per_seg);
    if (failed(status) || tile0 >= tile1) return;

    if (warp == 0) {
        tmem_alloc(tmem_slot, kTmemCols);
        tmem_relinquish();
    }
    constexpr uint32_t kTx = 3 * kTileBytes;
    if (tid == 0) {
        mbar_init(&bars[0], 1);
        mbar_init(&bars[1], 1);
        *abort_flag = 0;
        fence_mbar_init();
        tma_prefetch_desc(&tmQ);
        tma_prefetch_desc(&tmK);
        tma_prefetch_desc(&tmV);
        mbar_arrive_expect_tx(&bars[0], kTx);
        tma_load_3d(xq, &tmQ, 0, tile0 * kTile, bh, &bars[0]);
        tma_load_3d(xk, &tmK, 0, tile0 * kTile, bh, &bars[0]);
        tma_load_3d(vt, &tmV, 0, tile0 * kTile, bh, &bars[0]);
    }
    {
        const uint4 *src = reinterpret_cast<const uint4 *>(coef_img + (size_t)h * kCoefStride);
        uint4 *dst = reinterpret_cast<uint4 *>(coef);
        for (int i = tid; i < kCoefBytes / 16; i += blockDim.x) dst[i] = src[i];
        const uint4 one4 = make_uint4(0x3F803F80u, 0x3F803F80u, 0x3F803F80u, 0x3F803F80u);
        for (int i = tid; i < 2048 / 16; i += blockDim.x) reinterpret_cast<uint4 *>(ones)[i] = one4;
        const float *pre = prefix + ((size_t)bh * nseg + seg) * kKP * W;
        for (int e = tid; e < kKP * W; e += blockDim.x) S[e] = pre[e];
    }
    __syncthreads();
    build_state_operand<D_V>(S, bop, tid, blockDim.x);
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
    constexpr uint32_t idesc_p = idesc_bf16(kTile, kTile, false, false);
    constexpr uint32_t idesc_o = idesc_bf16(kTile, NB, false, false);
    constexpr uint32_t idesc_v = idesc_bf16(kTile, 64, false, true);   // A K-major (P), B MN-major (V)
    constexpr uint32_t idesc_z = idesc_bf16(kTile, 16, false, false);
    constexpr uint32_t idesc_sv = idesc_bf16(kTile, 64, true, true);   // A MN-major (Gamma^K^T), B MN-major
    constexpr uint32_t idesc_sz = idesc_bf16(kTile, 16, true, false);
    uint32_t ph_tma = 0, ph_mma = 0;

    for (int tile = tile0; tile < tile1; ++tile) {
        const int tok = tile * kTile + tid;
        if (!mbar_wait(&bars[0], ph_tma)) note_timeout(status, abort_flag);
        ph_tma ^= 1;
        prep_x2(xq, x2q, x2q + kTileBytes, kTileBytes, tid, blockDim.x);
        prep_x2(xk, x2k, x2k + kTileBytes, kTileBytes, tid, blockDim.x);
        fence_proxy_async_smem();
        __syncthreads();
        if (*reinterpret_cast<volatile int *>(abort_flag)) break;
        if (tid == 0) {
            tc_fence_after();
            issue_scores(tmem + kSQ, xq, x2q, x2q + kTileBytes, coef);
            issue_scores(tmem + kSK, xk, x2k, x2k + kTileBytes, coef);
            umma_commit(&bars[1]);
        }
        if (!mbar_wait(&bars[1], ph_mma)) note_timeout(status, abort_flag);
        ph_mma ^= 1;
        tc_fence_after();
        float rq;
        {
            float e[kKP];
            rq = score_row_exp(tmem + lane_base + kSQ, cvec, e);
            store_gamma_row(x2q, tid, e, 1.0f);
            const float rk = score_row_exp(tmem + lane_base + kSK, cvec, e);
            store_gamma_row(x2k, tid, e, tok < N ? 1.0f / rk : 0.0f);
        }
        tc_fence_before();
        fence_proxy_async_smem();
        __syncthreads();
        if (*reinterpret_cast<volatile int *>(abort_flag)) break;
        if (tid == 0) {
            tc_fence_after();
            const uint32_t sq = smem_u32(x2q), sk = smem_u32(x2k), sb = smem_u32(bop);
#pragma unroll
            for (int kk = 0; kk < kKP / 16; ++kk) {
                const uint64_t qh = sdesc_sw128(sq + kk * 32, 16, kGS), ql = sdesc_sw128(sq + 1024 + kk * 32, 16, kGS);
                const uint64_t kh = sdesc_sw128(sk + kk * 32, 16, kGS), kl = sdesc_sw128(sk + 1024 + kk * 32, 16, kGS);
                const uint64_t bh_ = sdesc_sw128(sb + kk * 32, 16, 1024), bl_ = sdesc_sw128(sb + NB * 128 + kk * 32, 16, 1024);
                const uint32_t acc = kk > 0 ? 1u : 0u;
                umma_bf16(tmem + kP, qh, kh, idesc_p, acc);   // P = gQ gK^T (3 split terms)
                umma_bf16(tmem + kP, ql, kh, idesc_p, 1u);
                umma_bf16(tmem + kP, qh, kl, idesc_p, 1u);
                umma_bf16(tmem + kO, qh, bh_, idesc_o, acc);  // [num | den] = gQ [S | Z]
                umma_bf16(tmem + kO, ql, bh_, idesc_o, 1u);
                umma_bf16(tmem + kO, qh, bl_, idesc_o, 1u);
            }
            umma_commit(&bars[1]);
        }
        if (!mbar_wait(&bars[1], ph_mma)) note_timeout(status, abort_flag);
        ph_mma ^= 1;
        tc_fence_after();
        // Masked intra-chunk affinity row i = tid: keep keys j <= i, split hi / lo.
        {
            uint8_t *hi = pbuf + (tid >> 3) * kGSP + (tid & 7) * 128;
            uint8_t *lo = hi + 2048;
#pragma unroll
            for (int cb = 0; cb < kTile / 32; ++cb) {
                uint32_t v[32];
                tmem_ld32(tmem + lane_base + kP + cb * 32, v);
                tmem_wait_ld();
#pragma unroll
                for (int c4 = 0; c4 < 4; ++c4) {
                    uint32_t wh[4], wl[4];
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const int j0 = cb * 32 + c4 * 8 + 2 * q;
                        const float p0 = j0 <= tid ? __uint_as_float(v[c4 * 8 + 2 * q]) : 0.f;
                        const float p1 = j0 + 1 <= tid ? __uint_as_float(v[c4 * 8 + 2 * q + 1]) : 0.f;
                        wh[q] = pack_bf2(p0, p1);
                        wl[q] = pack_bf2(p0 - bf_lo(wh[q]), p1 - bf_hi(wh[q]));
                    }
                    const int chunk = (cb * 32 + c4 * 8) >> 3;        // 16-byte chunk over 128 keys
                    const int blk = chunk >> 3, c = chunk & 7;
                    const uint32_t sw = (uint32_t)(blk * 1024 + ((c ^ (tid & 7)) << 4));
                    *reinterpret_cast<uint4 *>(hi + sw) = make_uint4(wh[0], wh[1], wh[2], wh[3]);
                    *reinterpret_cast<uint4 *>(lo + sw) = make_uint4(wl[0], wl[1], wl[2], wl[3]);
                }
            }
        }
        tc_fence_before();
        fence_proxy_async_smem();
        __syncthreads();
        if (*reinterpret_cast<volatile int *>(abort_flag)) break;
        if (tid == 0) {
            tc_fence_after();
            const uint32_t sp = smem_u32(pbuf), sv = smem_u32(vt), sk = smem_u32(x2k), so = smem_u32(ones);
            const uint64_t bz = sdesc_sw128(so, 16, 1024);
#pragma unroll
            for (int kk = 0; kk < kTile / 16; ++kk) {
                const uint32_t ao = (kk >> 2) * 1024 + (kk & 3) * 32;
                const uint64_t ph = sdesc_sw128(sp + ao, 16, kGSP), pl = sdesc_sw128(sp + 2048 + ao, 16, kGSP);
                const uint64_t bv = sdesc_sw128(sv + kk * 2048, 16, 1024);
                umma_bf16(tmem + kO, ph, bv, idesc_v, 1u);          // num += P V
                umma_bf16(tmem + kO, pl, bv, idesc_v, 1u);
                umma_bf16(tmem + kO + D_V, ph, bz, idesc_z, 1u);    // den += P 1
                umma_bf16(tmem + kO + D_V, pl, bz, idesc_z, 1u);
                const uint64_t ag = sdesc_sw128(sk + kk * 2 * kGS, 1024, kGS);  // [gK_hi ; gK_lo]^T
                const uint32_t acc = kk > 0 ? 1u : 0u;
                umma_bf16(tmem + kSc, ag, bv, idesc_sv, acc);       // chunk state: gK^T V
                umma_bf16(tmem + kSc + D_V, ag, bz, idesc_sz, acc); //              gK^T 1
            }
            umma_commit(&bars[1]);
        }
        if (!mbar_wait(&bars[1], ph_mma)) note_timeout(status, abort_flag);
        ph_mma ^= 1;
        tc_fence_after();
        __syncthreads();
        if (*reinterpret_cast<volatile int *>(abort_flag)) break;
        if (tid == 0 && tile + 1 < tile1) {  // every tile buffer is free: fetch the next chunk
            mbar_arrive_expect_tx(&bars[0], kTx);
            tma_load_3d(xq, &tmQ, 0, (tile + 1) * kTile, bh, &bars[0]);
            tma_load_3d(xk, &tmK, 0, (tile + 1) * kTile, bh, &bars[0]);
            tma_load_3d(vt, &tmV, 0, (tile + 1) * kTile, bh, &bars[0]);
        }
        // Outputs of the chunk.
        {
            uint32_t dz[16];
            tmem_ld16(tmem + lane_base + kO + D_V, dz);
            tmem_wait_ld();
            const float inv = 1.0f / (__uint_as_float(dz[0]) + eps * rq);
            const size_t row = (size_t)bh * N + tok;
#pragma unroll
            for (int cb = 0; cb < D_V / 32; ++cb) {
                uint32_t v[32];
                tmem_ld32(tmem + lane_base + kO + cb * 32, v);
                tmem_wait_ld();
                if (tok < N) {
                    if (o_bf16) {
                        uint4 *o = reinterpret_cast<uint4 *>(static_cast<__nv_bfloat16 *>(O) + row * D_V + cb * 32);
#pragma unroll
                        for (int q = 0; q < 4; ++q)
                            o[q] = make_uint4(pack_bf2(__uint_as_float(v[8 * q]) * inv, __uint_as_float(v[8 * q + 1]) * inv),
                                              pack_bf2(__uint_as_float(v[8 * q + 2]) * inv, __uint_as_float(v[8 * q + 3]) * inv),
                                              pack_bf2(__uint_as_float(v[8 * q + 4]) * inv, __uint_as_float(v[8 * q + 5]) * inv),
                                              pack_bf2(__uint_as_float(v[8 * q + 6]) * inv, __uint_as_float(v[8 * q + 7]) * inv));
                    } else {
                        float4 *o = reinterpret_cast<float4 *>(static_cast<float *>(O) + row * D_V + cb * 32);
#pragma unroll
                        for (int q = 0; q < 8; ++q)
                            o[q] = make_float4(__uint_as_float(v[4 * q]) * inv, __uint_as_float(v[4 * q + 1]) * inv,
                                               __uint_as_float(v[4 * q + 2]) * inv, __uint_as_float(v[4 * q + 3]) * inv);
                    }
                }
            }
        }
        // Carry: S += (hi rows 0..63) + (lo rows 64..127) of the chunk state.
        if (tile + 1 < tile1) {
            // the gq area is free again (its MMAs are done and the next chunk's TMA
            // writes only xq / xk): [64][W] fp32 = 16.6 KB
            float *tmp = reinterpret_cast<float *>(x2q);
            uint32_t v[32];
            float row[W];
#pragma unroll
            for (int cb = 0; cb < D_V / 32; ++cb) {
                tmem_ld32(tmem + lane_base + kSc + cb * 32, v);
                tmem_wait_ld();
#pragma unroll
                for (int q = 0; q < 32; ++q) row[cb * 32 + q] = __uint_as_float(v[q]);
            }
            {
                uint32_t z[16];
                tmem_ld16(tmem + lane_base + kSc + D_V, z);
                tmem_wait_ld();
                row[D_V] = __uint_as_float(z[0]);
            }
            if (tid >= kKP)
#pragma unroll
                for (int c = 0; c < W; ++c) tmp[(tid - kKP) * W + c] = row[c];
            __syncthreads();
            if (tid < kKP)
#pragma unroll
                for (int c = 0; c < W; ++c) S[tid * W + c] += row[c] + tmp[tid * W + c];
            __syncthreads();
            build_state_operand<D_V>(S, bop, tid, blockDim.x);
            fence_proxy_async_smem();
        }
        tc_fence_before();
        __syncthreads();
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, kTmemCols);
}

// ------------------------------------------------------------------ persistent pipelined kernels
//
// Work partition: the B*H*ntiles key/query tiles, in (head, tile) order, are
// cut into one contiguous range per CTA (one CTA per SM).  A range that
// crosses a head boundary is processed as one "job" per head.  Each CTA runs
// 10 warps:
//   warp 0      TMA producer (lane 0): tile loads into a ring of stages
//   warp 1      MMA issuer (lane 0): tcgen05.mma + tcgen05.commit
//   warps 2..5  epilogue group 0 \  alternate tiles (ping-pong): x^2 split,
//   warps 6..9  epilogue group 1 /  softmax, Gamma split, outputs
// Group g owns Gamma buffer g and TMEM score / output buffer g, so group g
// handles every tile whose running index has parity g.
constexpr int kThreads2 = 320;
constexpr int kStages = 2;

struct Part {
    int ntiles;  // tiles per head
    int total;   // B*H*ntiles
    int tpc;     // tiles per CTA
    int slots;   // partial slots per CTA (jobs per CTA, upper bound)
};

__host__ __device__ inline int first_cta_of_head(const Part &P, int bh) { return (bh * P.ntiles) / P.tpc; }
__host__ __device__ inline int last_cta_of_head(const Part &P, int bh) {
    return ((bh + 1) * P.ntiles - 1) / P.tpc;
}
// Slot of head bh's job inside CTA c (CTA c's range starts in head (c*tpc)/ntiles).
__host__ __device__ inline int slot_of(const Part &P, int c, int bh) { return bh - (c * P.tpc) / P.ntiles; }

// Coefficient image of head h built directly in shared memory (same layout
// as coef_prep_tc_kernel writes), by every thread of the CTA.
__device__ void build_coef_smem(const float *__restrict__ mu, const float *__restrict__ sigma2,
                                const float *__restrict__ log_pi, int h, int K, uint8_t *coef, unsigned *status,
                                int tid, int nthreads) {
    __nv_bfloat16 *m16 = reinterpret_cast<__nv_bfloat16 *>(coef);
    for (int e = tid; e < kKP * kDR; e += nthreads) {
        const int k = e / kDR, j = e % kDR;
        float a = 0.f, b = 0.f;
        if (k < K) {
            const float s2 = sigma2[((size_t)h * K + k) * kDR + j], m = mu[((size_t)h * K + k) * kDR + j];
            if (!(s2 > 0.f) || !isfinite(s2) || !isfinite(m)) set_status(status, GMA_ERR_NONFINITE_PARAM);
            a = -0.5f * kLog2e / s2;
            b = kLog2e * m / s2;
        }
        const __nv_bfloat16 ah = __float2bfloat16_rn(a), bh = __float2bfloat16_rn(b);
        const uint32_t off = sw128_offset(k, j, 1024) / 2;
        m16[off] = ah;
        m16[kCoefMatBytes / 2 + off] = __float2bfloat16_rn(a - __bfloat162float(ah));
        m16[kCoefMatBytes + off] = bh;
        m16[3 * kCoefMatBytes / 2 + off] = __float2bfloat16_rn(b - __bfloat162float(bh));
    }
    float *cvec = reinterpret_cast<float *>(coef + 4 * kCoefMatBytes);
    const int lane = tid & 31, nwarps = nthreads >> 5;
    for (int k = tid >> 5; k < kKP; k += nwarps) {
        double acc = 0.0;
        if (k < K)
            for (int j = lane; j < kDR; j += 32) {
                const float s2 = sigma2[((size_t)h * K + k) * kDR + j], m = mu[((size_t)h * K + k) * kDR + j];
                acc += (double)(m * m / s2) + (double)logf(s2);
            }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
        if (lane == 0) {
            if (k < K) {
                const float lp = log_pi[(size_t)h * K + k];
                if (!isfinite(lp)) set_status(status, GMA_ERR_NONFINITE_PARAM);
                cvec[k] = (float)((double)kLog2e * ((double)lp - 0.5 * acc));
            } else {
                cvec[k] = -INFINITY;
            }
        }
    }
}

// Bounded polling: tick(progressed) returns false once kWaitLimitNs pass
// without progress (or another role aborted).
struct Stall {
    uint64_t t0 = 0;
    int spins = 0;
    __device__ __forceinline__ bool tick(bool progressed, const int *abort_flag) {
        if (progressed) {
            spins = 0;
            t0 = 0;
            return true;
        }
        if (++spins < 256) return true;
        spins = 0;
        if (*reinterpret_cast<const volatile int *>(abort_flag)) return false;
        const uint64_t now = globaltimer();
        if (t0 == 0) t0 = now;
        return now - t0 <= kWaitLimitNs;
    }
};

__device__ __forceinline__ bool wait_or_abort(uint64_t *bar, uint32_t parity, unsigned *status, int *abort_flag) {
    if (mbar_wait(bar, parity)) return true;
    note_timeout(status, abort_flag);
    return false;
}
__device__ __forceinline__ bool aborted(const int *abort_flag) {
    return *reinterpret_cast<const volatile int *>(abort_flag) != 0;
}

// Row of the tile / TMEM lane handled by an epilogue thread (warp w may only
// read TMEM lanes 32*(w%4) .. 32*(w%4)+31).
__device__ __forceinline__ int epi_row(int warp, int lane) { return 32 * (warp & 3) + lane; }

// Writes one bf16 hi / lo B-operand image [NB rows x KP] for the read of the
// latent memory: row n < D_V holds Vt[:, n], row D_V holds Z, other rows 0.
template <int D_V>
__device__ __forceinline__ void store_memory_operand(const float *S, int ldS, uint8_t *dst, int tid, int nthreads) {
    constexpr int NB = D_V + 16;
    __nv_bfloat16 *bhi = reinterpret_cast<__nv_bfloat16 *>(dst);
    __nv_bfloat16 *blo = reinterpret_cast<__nv_bfloat16 *>(dst + NB * 128);
    for (int e = tid; e < NB * kKP; e += nthreads) {
        const int n = e / kKP, k = e % kKP;
        const float v = n <= D_V ? S[k * ldS + n] : 0.f;
        const __nv_bfloat16 vh = __float2bfloat16_rn(v);
        const uint32_t off = sw128_offset(n, k, 1024) / 2;
        bhi[off] = vh;
        blo[off] = __float2bfloat16_rn(v - __bfloat162float(vh));
    }
}

template <int D_V>
struct Write2Smem {
    static constexpr int W = D_V + 1;
    static constexpr int kKst = 0;                                    // K stages
    static constexpr int kVst = kKst + kStages * kTileBytes;          // V stages
    static constexpr int kXG = kVst + kStages * (D_V / 64) * kTileBytes;  // x2 / Gamma buffers [2][32 KB]
    static constexpr int kCoef = kXG + 2 * 2 * kTileBytes;
    static constexpr int kOnes = kCoef + ((kCoefBytes + 1023) & ~1023);
    static constexpr int kBars = kOnes + 2048;
    static constexpr int kBytes = kBars + 256;
    static constexpr int kAlloc = kBytes + 1024;
    static_assert(128 * W * 4 <= kCoef, "reduction buffer must fit over the tile buffers");
};

// Latent aggregation ([GMA, Eqs. (5)-(6)]) over each job's keys:
//   part[job][k][c] = sum_j gamma^K_jk V_jc,  part[job][k][d_v] = sum_j gamma^K_jk.
// The last job of each head to finish combines the head's jobs in CTA order:
//   mode 0: the bf16 hi / lo read operand of the whole-sequence memory (bidirectional),
//   mode 1: in place, the exclusive prefix of each job (causal carry-in).
template <int D_V>
__global__ void __launch_bounds__(kThreads2, 1) tc_write2_kernel(
    const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
    const float *__restrict__ mu, const float *__restrict__ sigma2, const float *__restrict__ log_pi, int K,
    int H, int N, Part P, float *__restrict__ part, unsigned *__restrict__ counters, uint8_t *__restrict__ mem_img,
    size_t mem_img_stride, int mode, unsigned *status) {
    using L = Write2Smem<D_V>;
    constexpr int W = L::W;
    constexpr int kTmemCols = D_V == 64 ? 256 : 512;
    constexpr int kAccV = 2 * kKP, kAccZ = 2 * kKP + D_V;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t *kst = smem + L::kKst, *vst = smem + L::kVst, *xg = smem + L::kXG, *coef = smem + L::kCoef,
            *ones = smem + L::kOnes;
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + L::kBars);
    uint64_t *kvfull = bars, *kvempty = bars + 2, *xready = bars + 4, *sfull = bars + 6, *gready = bars + 8,
             *wdone = bars + 10, *accfull = bars + 12;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + 14);
    int *abort_flag = reinterpret_cast<int *>(bars + 15);
    int *last_flag = abort_flag + 1;
    const float *cvec = reinterpret_cast<const float *>(coef + 4 * kCoefMatBytes);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int c = blockIdx.x;
    const int g0 = c * P.tpc, gend = min(P.total, g0 + P.tpc);
    if (failed(status) || g0 >= gend) return;

    if (warp == 0) {
        tmem_alloc(tmem_slot, kTmemCols);
        tmem_relinquish();
    }
    if (tid == 32) {
        for (int i = 0; i < 2; ++i) {
            mbar_init(&kvfull[i], 1);
            mbar_init(&kvempty[i], 1);
            mbar_init(&xready[i], 4);
            mbar_init(&sfull[i], 1);
            mbar_init(&gready[i], 4);
            mbar_init(&wdone[i], 1);
        }
        mbar_init(accfull, 1);
        *abort_flag = 0;
        fence_mbar_init();
        tma_prefetch_desc(&tmK);
        tma_prefetch_desc(&tmV);
    }
    {
        const uint4 one4 = make_uint4(0x3F803F80u, 0x3F803F80u, 0x3F803F80u, 0x3F803F80u);
        for (int i = tid; i < 2048 / 16; i += kThreads2) reinterpret_cast<uint4 *>(ones)[i] = one4;
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    constexpr uint32_t kTx = kTileBytes * (1 + D_V / 64);
    constexpr uint32_t idesc_v = idesc_bf16(kTile, 64, true, true);
    constexpr uint32_t idesc_z = idesc_bf16(kTile, 16, true, false);

    int rbase = 0;   // running tile index of the CTA (barrier phases)
    int njob = 0;
    for (int g = g0; g < gend; ++njob) {
        const int bh = g / P.ntiles, t0 = g % P.ntiles;
        const int n = min(P.ntiles - t0, gend - g);
        const int h = bh % H;
        __syncthreads();
        build_coef_smem(mu, sigma2, log_pi, h, K, coef, status, tid, kThreads2);
        fence_proxy_async_smem();
        __syncthreads();

        if (warp == 0) {
            if (lane == 0)
                for (int i = 0; i < n; ++i) {
                    const int r = rbase + i, s = r % kStages;
                    if (!wait_or_abort(&kvempty[s], ((r / kStages) & 1) ^ 1, status, abort_flag)) break;
                    mbar_arrive_expect_tx(&kvfull[s], kTx);
                    tma_load_3d(kst + s * kTileBytes, &tmK, 0, (t0 + i) * kTile, bh, &kvfull[s]);
#pragma unroll
                    for (int vb = 0; vb < D_V / 64; ++vb)
                        tma_load_3d(vst + (s * (D_V / 64) + vb) * kTileBytes, &tmV, vb * 64, (t0 + i) * kTile, bh,
                                    &kvfull[s]);
                }
        } else if (warp == 1) {
            if (lane == 0) {
                // Poll both queues so that neither kind of MMA waits behind the other.
                int ns = 0, nw = 0;
                Stall st;
                while (nw < n) {
                    bool prog = false;
                    if (ns < n) {
                        const int r = rbase + ns, gb = r & 1, s = r % kStages;
                        if (mbar_test(&xready[gb], (r >> 1) & 1)) {
                            tc_fence_after();
                            issue_scores(tmem + gb * kKP, kst + s * kTileBytes, xg + gb * 2 * kTileBytes,
                                         xg + gb * 2 * kTileBytes + kTileBytes, coef);
                            umma_commit(&sfull[gb]);
                            ++ns;
                            prog = true;
                        }
                    }
                    if (nw < ns) {
                        const int r = rbase + nw, gb = r & 1, s = r % kStages;
                        if (mbar_test(&gready[gb], (r >> 1) & 1)) {
                            tc_fence_after();
                            const uint32_t sg = smem_u32(xg + gb * 2 * kTileBytes),
                                           sv = smem_u32(vst + s * (D_V / 64) * kTileBytes);
                            const uint64_t bz = sdesc_sw128(smem_u32(ones), 16, 1024);
#pragma unroll
                            for (int kk = 0; kk < kTile / 16; ++kk) {
                                const uint32_t acc = (nw > 0 || kk > 0) ? 1u : 0u;
                                const uint64_t a = sdesc_sw128(sg + kk * 2 * kGS, 1024, kGS);
#pragma unroll
                                for (int vb = 0; vb < D_V / 64; ++vb)
                                    umma_bf16(tmem + kAccV + vb * 64, a,
                                              sdesc_sw128(sv + vb * kTileBytes + kk * 2048, 16, 1024), idesc_v, acc);
                                umma_bf16(tmem + kAccZ, a, bz, idesc_z, acc);
                            }
                            umma_commit(&kvempty[s]);
                            umma_commit(&wdone[gb]);
                            ++nw;
                            prog = true;
                        }
                    }
                    if (!st.tick(prog, abort_flag)) {
                        note_timeout(status, abort_flag);
                        break;
                    }
                }
                umma_commit(accfull);
            }
        } else {
            const int grp = (warp - 2) >> 2;  // 0 or 1
            const int row = epi_row(warp, lane);
            const uint32_t lane_base = (uint32_t)(32 * (warp & 3)) << 16;
            for (int i = ((rbase & 1) == grp ? 0 : 1); i < n; i += 2) {
                const int r = rbase + i, s = r % kStages;
                uint8_t *gbuf = xg + grp * 2 * kTileBytes;
                if (r >= 2 && !wait_or_abort(&wdone[grp], ((r - 2) >> 1) & 1, status, abort_flag)) break;
                if (!wait_or_abort(&kvfull[s], (r / kStages) & 1, status, abort_flag)) break;
                prep_x2(kst + s * kTileBytes, gbuf, gbuf + kTileBytes, kTileBytes, tid - 64 - 128 * grp, 128);
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(&xready[grp]);
                if (!wait_or_abort(&sfull[grp], (r >> 1) & 1, status, abort_flag)) break;
                tc_fence_after();
                float e[kKP];
                const float rs = score_row_exp(tmem + lane_base + grp * kKP, cvec, e);
                tc_fence_before();
                const int tok = (t0 + i) * kTile + row;
                store_gamma_row(gbuf, row, e, tok < N ? 1.0f / rs : 0.0f);
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(&gready[grp]);
            }
        }
        // ---- job end: the accumulated memory -> partial of this job
        __syncthreads();
        const bool ok = !aborted(abort_flag);
        float *red = reinterpret_cast<float *>(smem);  // [128][W] over the (now idle) tile buffers
        if (ok && warp >= 2 && warp < 6) {
            if (wait_or_abort(accfull, njob & 1, status, abort_flag)) {
                tc_fence_after();
                const int row = epi_row(warp, lane);
                const uint32_t lb = (uint32_t)(32 * (warp & 3)) << 16;
#pragma unroll
                for (int cb = 0; cb < D_V / 32; ++cb) {
                    uint32_t v[32];
                    tmem_ld32(tmem + lb + kAccV + cb * 32, v);
                    tmem_wait_ld();
#pragma unroll
                    for (int q = 0; q < 32; ++q) red[row * W + cb * 32 + q] = __uint_as_float(v[q]);
                }
                uint32_t z[16];
                tmem_ld16(tmem + lb + kAccZ, z);
                tmem_wait_ld();
                red[row * W + D_V] = __uint_as_float(z[0]);
                tc_fence_before();
            }
        }
        __syncthreads();
        if (!aborted(abort_flag)) {
            const int slot = slot_of(P, c, bh);
            float *out = part + ((size_t)c * P.slots + slot) * kKP * W;
            for (int e = tid; e < kKP * W; e += kThreads2) out[e] = red[e] + red[kKP * W + e];
            __threadfence();
            __syncthreads();
            if (tid == 0) {
                const int njobs = last_cta_of_head(P, bh) - first_cta_of_head(P, bh) + 1;
                const unsigned old = atomicAdd(&counters[bh], 1u);
                *last_flag = (old == (unsigned)(njobs - 1));
            }
            __syncthreads();
            if (*last_flag) {
                __threadfence();
                const int cf = first_cta_of_head(P, bh), cl = last_cta_of_head(P, bh);
                if (mode == 0) {
                    for (int e = tid; e < kKP * W; e += kThreads2) {
                        float v = 0.f;
                        for (int cc = cf; cc <= cl; ++cc)
                            v += __ldcg(part + ((size_t)cc * P.slots + slot_of(P, cc, bh)) * kKP * W + e);
                        red[e] = v;
                    }
                    __syncthreads();
                    store_memory_operand<D_V>(red, W, mem_img + (size_t)bh * mem_img_stride, tid, kThreads2);
                } else {
                    for (int e = tid; e < kKP * W; e += kThreads2) {
                        float run = 0.f;
                        for (int cc = cf; cc <= cl; ++cc) {
                            float *pp = part + ((size_t)cc * P.slots + slot_of(P, cc, bh)) * kKP * W + e;
                            const float cur = __ldcg(pp);
                            *pp = run;
                            run += cur;
                        }
                    }
                }
                if (tid == 0) counters[bh] = 0u;  // ready for the next call
            }
        }
        rbase += n;
        g += n;
        if (aborted(abort_flag)) break;
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, kTmemCols);
}

template <int D_V>
struct Read2Smem {
    static constexpr int NB = D_V + 16;
    static constexpr int kQS = 3;
    static constexpr int kQst = 0;
    static constexpr int kXG = kQst + kQS * kTileBytes;
    static constexpr int kCoef = kXG + 2 * 2 * kTileBytes;
    static constexpr int kB = kCoef + ((kCoefBytes + 1023) & ~1023);
    static constexpr int kBars = kB + ((2 * NB * 128 + 1023) & ~1023);
    static constexpr int kBytes = kBars + 256;
    static constexpr int kAlloc = kBytes + 1024;
};

// Normalised broadcasting ([GMA, Eq. (7)]) over each job's query tiles.
template <int D_V>
__global__ void __launch_bounds__(kThreads2, 1) tc_read2_kernel(
    const __grid_constant__ CUtensorMap tmQ, const float *__restrict__ mu, const float *__restrict__ sigma2,
    const float *__restrict__ log_pi, int K, int H, int N, Part P, const uint8_t *__restrict__ mem_img,
    size_t mem_img_stride, float eps, void *__restrict__ O, int o_bf16, unsigned *status) {
    using L = Read2Smem<D_V>;
    constexpr int NB = L::NB, QS = L::kQS;
    constexpr int kTmemCols = 512;
    constexpr int kAccO = 2 * kKP;  // O buffer g at kAccO + g * NB
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t *qst = smem + L::kQst, *xg = smem + L::kXG, *coef = smem + L::kCoef, *bop = smem + L::kB;
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + L::kBars);
    uint64_t *qfull = bars, *qempty = bars + QS, *xready = bars + 2 * QS, *sfull = xready + 2, *gready = sfull + 2,
             *ofull = gready + 2;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(ofull + 2);
    int *abort_flag = reinterpret_cast<int *>(ofull + 3);
    const float *cvec = reinterpret_cast<const float *>(coef + 4 * kCoefMatBytes);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int c = blockIdx.x;
    const int g0 = c * P.tpc, gend = min(P.total, g0 + P.tpc);
    if (failed(status) || g0 >= gend) return;

    if (warp == 0) {
        tmem_alloc(tmem_slot, kTmemCols);
        tmem_relinquish();
    }
    if (tid == 32) {
        for (int i = 0; i < QS; ++i) {
            mbar_init(&qfull[i], 1);
            mbar_init(&qempty[i], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&xready[i], 4);
            mbar_init(&sfull[i], 1);
            mbar_init(&gready[i], 4);
            mbar_init(&ofull[i], 1);
        }
        *abort_flag = 0;
        fence_mbar_init();
        tma_prefetch_desc(&tmQ);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    constexpr uint32_t idesc_o = idesc_bf16(kTile, NB, false, false);

    int rbase = 0;
    for (int g = g0; g < gend;) {
        const int bh = g / P.ntiles, t0 = g % P.ntiles;
        const int n = min(P.ntiles - t0, gend - g);
        const int h = bh % H;
        __syncthreads();
        build_coef_smem(mu, sigma2, log_pi, h, K, coef, status, tid, kThreads2);
        {
            const uint4 *src = reinterpret_cast<const uint4 *>(mem_img + (size_t)bh * mem_img_stride);
            for (int i = tid; i < 2 * NB * 128 / 16; i += kThreads2) reinterpret_cast<uint4 *>(bop)[i] = __ldcg(src + i);
        }
        fence_proxy_async_smem();
        __syncthreads();

        if (warp == 0) {
            if (lane == 0)
                for (int i = 0; i < n; ++i) {
                    const int r = rbase + i, s = r % QS;
                    if (!wait_or_abort(&qempty[s], ((r / QS) & 1) ^ 1, status, abort_flag)) break;
                    mbar_arrive_expect_tx(&qfull[s], kTileBytes);
                    tma_load_3d(qst + s * kTileBytes, &tmQ, 0, (t0 + i) * kTile, bh, &qfull[s]);
                }
        } else if (warp == 1) {
            if (lane == 0) {
                // Poll both queues so that neither kind of MMA waits behind the other.
                int ns = 0, nr = 0;
                Stall st;
                while (nr < n) {
                    bool prog = false;
                    if (ns < n) {
                        const int r = rbase + ns, gb = r & 1, s = r % QS;
                        if (mbar_test(&xready[gb], (r >> 1) & 1)) {
                            tc_fence_after();
                            issue_scores(tmem + gb * kKP, qst + s * kTileBytes, xg + gb * 2 * kTileBytes,
                                         xg + gb * 2 * kTileBytes + kTileBytes, coef);
                            umma_commit(&sfull[gb]);
                            umma_commit(&qempty[s]);
                            ++ns;
                            prog = true;
                        }
                    }
                    if (nr < ns) {
                        const int r = rbase + nr, gb = r & 1;
                        if (mbar_test(&gready[gb], (r >> 1) & 1)) {
                            tc_fence_after();
                            const uint32_t sg = smem_u32(xg + gb * 2 * kTileBytes), sb = smem_u32(bop);
                            const uint32_t d = tmem + kAccO + gb * NB;
#pragma unroll
                            for (int kk = 0; kk < kKP / 16; ++kk) {
                                const uint64_t ahi = sdesc_sw128(sg + kk * 32, 16, kGS),
                                               alo = sdesc_sw128(sg + 1024 + kk * 32, 16, kGS);
                                const uint64_t bhi = sdesc_sw128(sb + kk * 32, 16, 1024),
                                               blo = sdesc_sw128(sb + NB * 128 + kk * 32, 16, 1024);
                                umma_bf16(d, ahi, bhi, idesc_o, kk > 0 ? 1u : 0u);
                                umma_bf16(d, alo, bhi, idesc_o, 1u);
                                umma_bf16(d, ahi, blo, idesc_o, 1u);
                            }
                            umma_commit(&ofull[gb]);
                            ++nr;
                            prog = true;
                        }
                    }
                    if (!st.tick(prog, abort_flag)) {
                        note_timeout(status, abort_flag);
                        break;
                    }
                }
            }
        } else {
            const int grp = (warp - 2) >> 2;
            const int row = epi_row(warp, lane);
            const uint32_t lane_base = (uint32_t)(32 * (warp & 3)) << 16;
            for (int i = ((rbase & 1) == grp ? 0 : 1); i < n; i += 2) {
                const int r = rbase + i, s = r % QS;
                uint8_t *gbuf = xg + grp * 2 * kTileBytes;
                if (!wait_or_abort(&qfull[s], (r / QS) & 1, status, abort_flag)) break;
                prep_x2(qst + s * kTileBytes, gbuf, gbuf + kTileBytes, kTileBytes, tid - 64 - 128 * grp, 128);
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(&xready[grp]);
                if (!wait_or_abort(&sfull[grp], (r >> 1) & 1, status, abort_flag)) break;
                tc_fence_after();
                float rs;
                {
                    float e[kKP];
                    rs = score_row_exp(tmem + lane_base + grp * kKP, cvec, e);
                    tc_fence_before();
                    store_gamma_row(gbuf, row, e, 1.0f);
                }
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(&gready[grp]);
                if (!wait_or_abort(&ofull[grp], (r >> 1) & 1, status, abort_flag)) break;
                tc_fence_after();
                const uint32_t ob = tmem + lane_base + kAccO + grp * NB;
                uint32_t dz[16];
                tmem_ld16(ob + D_V, dz);
                tmem_wait_ld();
                const float inv = 1.0f / (__uint_as_float(dz[0]) + eps * rs);
                const int tok = (t0 + i) * kTile + row;
                const size_t orow = (size_t)bh * N + tok;
#pragma unroll
                for (int cb = 0; cb < D_V / 32; ++cb) {
                    uint32_t v[32];
                    tmem_ld32(ob + cb * 32, v);
                    tmem_wait_ld();
                    if (tok < N) {
                        if (o_bf16) {
                            uint4 *o = reinterpret_cast<uint4 *>(static_cast<__nv_bfloat16 *>(O) + orow * D_V + cb * 32);
#pragma unroll
                            for (int q = 0; q < 4; ++q)
                                o[q] = make_uint4(pack_bf2(__uint_as_float(v[8 * q]) * inv, __uint_as_float(v[8 * q + 1]) * inv),
                                                  pack_bf2(__uint_as_float(v[8 * q + 2]) * inv, __uint_as_float(v[8 * q + 3]) * inv),
                                                  pack_bf2(__uint_as_float(v[8 * q + 4]) * inv, __uint_as_float(v[8 * q + 5]) * inv),
                                                  pack_bf2(__uint_as_float(v[8 * q + 6]) * inv, __uint_as_float(v[8 * q + 7]) * inv));
                        } else {
                            float4 *o = reinterpret_cast<float4 *>(static_cast<float *>(O) + orow * D_V + cb * 32);
#pragma unroll
                            for (int q = 0; q < 8; ++q)
                                o[q] = make_float4(__uint_as_float(v[4 * q]) * inv, __uint_as_float(v[4 * q + 1]) * inv,
                                                   __uint_as_float(v[4 * q + 2]) * inv, __uint_as_float(v[4 * q + 3]) * inv);
                        }
                    }
                }
                tc_fence_before();
            }
        }
        rbase += n;
        g += n;
        __syncthreads();
        if (aborted(abort_flag)) break;
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, kTmemCols);
}

// ------------------------------------------------------------------ host side

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

// [BH][N][d] bf16 tensor, boxes of 64 columns x 128 rows x 1 head, 128-byte
// swizzle; rows past N read as zero.
bool make_map(CUtensorMap *map, const void *base, int BH, int N, int d) {
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)N, (cuuint64_t)BH};
    cuuint64_t strides[2] = {(cuuint64_t)d * 2, (cuuint64_t)N * d * 2};
    cuuint32_t box[3] = {64, (cuuint32_t)kTile, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

struct TcLayout {
    size_t coef = 0, part = 0, total = 0;
    int nsplit = 0, tiles_per_split = 0;
};

constexpr int kTargetCtas = 2 * 152;

constexpr int kCausalSegTiles = 8;  // default causal segment: 1024 tokens

TcLayout tc_layout(const Problem &p, int causal, int splits) {
    TcLayout L;
    const int ntiles = (p.N + kTile - 1) / kTile;
    int ns = splits > 0 ? splits
                        : causal ? (ntiles + kCausalSegTiles - 1) / kCausalSegTiles
                                 : (kTargetCtas + p.BH() - 1) / p.BH();
    ns = ns < 1 ? 1 : (ns > ntiles ? ntiles : ns);
    L.tiles_per_split = (ntiles + ns - 1) / ns;
    L.nsplit = (ntiles + L.tiles_per_split - 1) / L.tiles_per_split;
    size_t off = kStatusBytes;
    L.coef = off;
    off = align256(off + kCoefStride * p.H);
    L.part = off;
    off = align256(off + sizeof(float) * (size_t)p.BH() * L.nsplit * kKP * (p.d_v + 1));
    L.total = off;
    return L;
}

template <typename KernelT>
cudaError_t set_smem(KernelT kern, int bytes) {
    return cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
}

#define GMA_TRY(x)                            \
    do {                                      \
        cudaError_t err_ = (x);               \
        if (err_ != cudaSuccess) return err_; \
    } while (0)

int num_sms() {
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) {
        (void)cudaGetLastError();
        return 152;
    }
    return n;
}

// Workspace of the persistent kernels: status | per-head counters | job
// partials [ctas][slots][KP][d_v + 1] | per-head read operand images.
struct TcLayout2 {
    Part P;
    int nctas = 0;
    size_t counters = 0, part = 0, mem = 0, mem_stride = 0, total = 0, reset_bytes = 0;
};

TcLayout2 tc_layout2(const Problem &p, int splits) {
    TcLayout2 L;
    const int ntiles = (p.N + kTile - 1) / kTile;
    const int total = p.BH() * ntiles;
    int nct = splits > 0 ? splits : num_sms();
    nct = nct < 1 ? 1 : (nct > total ? total : nct);
    const int tpc = (total + nct - 1) / nct;
    L.nctas = (total + tpc - 1) / tpc;
    L.P = Part{ntiles, total, tpc, tpc / ntiles + 2};
    size_t off = kStatusBytes;
    L.counters = off;
    off = align256(off + sizeof(unsigned) * (size_t)p.BH());
    L.reset_bytes = off;
    L.part = off;
    off = align256(off + sizeof(float) * (size_t)L.nctas * L.P.slots * kKP * (p.d_v + 1));
    L.mem_stride = ((size_t)2 * (p.d_v + 16) * 128 + 1023) & ~size_t(1023);
    L.mem = off;
    off = align256(off + L.mem_stride * p.BH());
    L.total = off;
    return L;
}

template <int D_V>
cudaError_t run_bidir2(const Problem &p, const TcLayout2 &L, uint8_t *ws, cudaStream_t s, StageClock &clk) {
    unsigned *status = reinterpret_cast<unsigned *>(ws);
    unsigned *counters = reinterpret_cast<unsigned *>(ws + L.counters);
    float *part = reinterpret_cast<float *>(ws + L.part);
    uint8_t *mem = ws + L.mem;
    CUtensorMap tq, tk, tv;
    if (!make_map(&tq, p.Q, p.BH(), p.N, p.d_r) || !make_map(&tk, p.Kx, p.BH(), p.N, p.d_r) ||
        !make_map(&tv, p.V, p.BH(), p.N, D_V))
        return cudaErrorInvalidValue;
    clk.mark();
    GMA_TRY(cudaMemsetAsync(ws, 0, L.reset_bytes, s));
    clk.mark();
    GMA_TRY(set_smem(tc_write2_kernel<D_V>, Write2Smem<D_V>::kAlloc));
    tc_write2_kernel<D_V><<<L.nctas, kThreads2, Write2Smem<D_V>::kAlloc, s>>>(
        tk, tv, p.mu, p.sigma2, p.log_pi, p.K, p.H, p.N, L.P, part, counters, mem, L.mem_stride, 0, status);
    GMA_TRY(cudaGetLastError());
    clk.mark();
    GMA_TRY(set_smem(tc_read2_kernel<D_V>, Read2Smem<D_V>::kAlloc));
    tc_read2_kernel<D_V><<<L.nctas, kThreads2, Read2Smem<D_V>::kAlloc, s>>>(
        tq, p.mu, p.sigma2, p.log_pi, p.K, p.H, p.N, L.P, mem, L.mem_stride, p.eps, p.O, p.o_bf16 ? 1 : 0, status);
    GMA_TRY(cudaGetLastError());
    clk.mark();
    return cudaSuccess;
}

cudaError_t run_causal(const Problem &p, const TcLayout &L, uint8_t *ws, cudaStream_t s, StageClock &clk) {
    constexpr int D_V = CausalSmem::D_V;
    unsigned *status = reinterpret_cast<unsigned *>(ws);
    uint8_t *coef = ws + L.coef;
    float *part = reinterpret_cast<float *>(ws + L.part);
    CUtensorMap tq, tk, tv;
    if (!make_map(&tq, p.Q, p.BH(), p.N, p.d_r) || !make_map(&tk, p.Kx, p.BH(), p.N, p.d_r) ||
        !make_map(&tv, p.V, p.BH(), p.N, D_V))
        return cudaErrorInvalidValue;
    clk.mark();
    GMA_TRY(cudaMemsetAsync(status, 0, sizeof(unsigned), s));
    coef_prep_tc_kernel<<<p.H, 256, 0, s>>>(p.mu, p.sigma2, p.log_pi, p.K, coef, status);
    GMA_TRY(cudaGetLastError());
    clk.mark();
    GMA_TRY(set_smem(tc_write_kernel<D_V>, WriteSmem<D_V>::kAlloc));
    tc_write_kernel<D_V><<<dim3(L.nsplit, p.BH()), 128, WriteSmem<D_V>::kAlloc, s>>>(
        tk, tv, coef, p.H, p.N, L.tiles_per_split, L.nsplit, part, status);
    GMA_TRY(cudaGetLastError());
    clk.mark();
    const int E = kKP * (D_V + 1);
    scan_segments_kernel<<<dim3((E + 255) / 256, p.BH()), 256, 0, s>>>(part, L.nsplit, E, status);
    GMA_TRY(cudaGetLastError());
    clk.mark();
    GMA_TRY(set_smem(tc_causal_kernel, CausalSmem::kAlloc));
    tc_causal_kernel<<<dim3(L.nsplit, p.BH()), 128, CausalSmem::kAlloc, s>>>(
        tq, tk, tv, coef, part, p.H, p.N, L.tiles_per_split, L.nsplit, p.eps, p.O, p.o_bf16 ? 1 : 0, status);
    GMA_TRY(cudaGetLastError());
    clk.mark();
    return cudaSuccess;
}

}  // namespace

const char *const kTcStages[3][8] = {
    {nullptr},
    {"reset", "tc_write", "tc_read", nullptr},
    {"prep", "tc_aggregate", "scan", "tc_causal", nullptr},
};

bool tc_supported(const Problem &p, int causal) {
    if (p.dtype != GMA_BF16 || p.d_r != kDR || p.K > kKP) return false;
    if (causal == 0) return p.d_v == 64 || p.d_v == 128;
    return causal == 1 && p.d_v == CausalSmem::D_V;
}

size_t tc_workspace(const Problem &p, int causal, int splits) {
    return causal ? tc_layout(p, causal, splits).total : tc_layout2(p, splits).total;
}

cudaError_t tc_bidir(const Problem &p, int splits, void *ws, cudaStream_t s, StageClock &clk) {
    TcLayout2 L = tc_layout2(p, splits);
    uint8_t *w = static_cast<uint8_t *>(ws);
    if (p.d_v == 64) return run_bidir2<64>(p, L, w, s, clk);
    return run_bidir2<128>(p, L, w, s, clk);
}

cudaError_t tc_causal(const Problem &p, int splits, void *ws, cudaStream_t s, StageClock &clk) {
    TcLayout L = tc_layout(p, 1, splits);
    return run_causal(p, L, static_cast<uint8_t *>(ws), s, clk);
}

}  // namespace gma
