// gma_tc.cu -- tcgen05 tensor-core kernels for the GMA forward pass (bf16
// inputs, d_r = 32 or 64 (32 runs zero-padded to 64), d_v = 64, K <= 64).
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
// into bf16 hi + lo again for the value contractions (write: Gamma^K^T [V | 1];
// read: Gamma^Q [Vt | Z] with the memory split too; causal: the masked
// intra-chunk Gamma^Q Gamma^K^T times [V | 1] plus Gamma^Q times the carried
// prefix).  O = num / (den + eps * r) with r the un-normalised query row sum.
//
// Kernels:  coef_prep_tc_kernel (per-head split coefficients), then the
// persistent, warp-specialised tc_write2_kernel (key side: latent memory per
// job, combined per head by the last job), tc_read3_kernel (bidirectional
// query side) and tc_causal2_kernel (causal chunked scan).
//
// Paper: "Gaussian Mixture Attention: Linear-Time Sequence Mixing via
// Probabilistic Latent Routing" (arXiv 2606.18283), cited [GMA, ...].
#include <cuda.h>
#include <cuda_bf16.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <cmath>
#include <mutex>

#include "gma_internal.h"
#include "tc_common.cuh"
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
// Row stride (floats) of a job partial / causal state [KP][kW]: 64 values of
// Gamma^T V, then Z = Gamma^T 1, then 3 zero pads (rows stay 16-byte aligned).
constexpr int kW = 68;



// ------------------------------------------------------------------ coefficient prep
// Grid (KP / 8, H): block (b, h) writes components 8b .. 8b + 7 of head h's
// coefficient image -- the four bf16 matrices in the K-major SW128 byte image
// the score MMA reads (rows = components, 64 routing columns per row, zero past
// d_r) and c_k (fp32, -inf for padded components) -- and validates their parameters into its
// error word err[h * (KP / 8) + b].  Each thread handles four consecutive j of
// one component; the 16 threads of a component (one half-warp) also sum its
// log-determinant terms.  Being the first kernel of a call, it also clears the
// call's status word and the per-head job counters.
constexpr int kPrepBlocks = kKP / 8;

__global__ void __launch_bounds__(128) coef_prep_tc_kernel(const float *__restrict__ mu,
                                                           const float *__restrict__ sigma2,
                                                           const float *__restrict__ log_pi, int K, int DR,
                                                           uint8_t *__restrict__ img, unsigned *status,
                                                           unsigned *head_err, unsigned *counters, int BH) {
    const int tid = threadIdx.x, h = blockIdx.y;
    const int gt = (blockIdx.y * gridDim.x + blockIdx.x) * blockDim.x + tid;
    uint8_t *coef = img + (size_t)h * kCoefStride;
    const int k = blockIdx.x * 8 + (tid >> 4), j = (tid & 15) * 4;
    const bool realk = k < K;
    const bool real = realk && j < DR;  // d_r < 64: columns DR .. 63 are zero padding
    // The previous call's kernels may still read the status, counters and images,
    // and the kernel before this one may have written the parameters: they are read
    // only after the dependency wait.  Their lines are brought into L2 meanwhile (a
    // prefetch returns nothing, and L2 is where that kernel's writes land).
    if (real) {
        prefetch_l2(sigma2 + ((size_t)h * K + k) * DR + j);
        prefetch_l2(mu + ((size_t)h * K + k) * DR + j);
    }
    if (realk && j == 0) prefetch_l2(log_pi + (size_t)h * K + k);
    pdl_wait();
    pdl_trigger();
    if (gt == 0) *status = 0u;
    for (int i = gt; i < BH; i += gridDim.x * gridDim.y * blockDim.x) counters[i] = 0u;
    float4 s4 = make_float4(1.f, 1.f, 1.f, 1.f), m4 = make_float4(0.f, 0.f, 0.f, 0.f);
    float lp = 0.f;
    if (real) {
        s4 = *reinterpret_cast<const float4 *>(sigma2 + ((size_t)h * K + k) * DR + j);
        m4 = *reinterpret_cast<const float4 *>(mu + ((size_t)h * K + k) * DR + j);
    }
    if (realk) lp = log_pi[(size_t)h * K + k];
    const float sv[4] = {s4.x, s4.y, s4.z, s4.w}, mv[4] = {m4.x, m4.y, m4.z, m4.w};
    bool bad = false;
    uint32_t ah[2], al[2], bh[2], bl[2];
    float det = 0.f;
#pragma unroll
    for (int u = 0; u < 2; ++u) {
        float a[2], b[2];
#pragma unroll
        for (int v = 0; v < 2; ++v) {
            const float s2 = sv[2 * u + v], m = mv[2 * u + v];
            if (real && (!(s2 > 0.f) || !isfinite(s2) || !isfinite(m))) bad = true;
            const float inv = real ? __frcp_rn(s2) : 0.f;
            a[v] = (-0.5f * kLog2e) * inv;
            b[v] = (kLog2e * m) * inv;
            det += real ? m * m * inv + __logf(s2) : 0.f;
        }
        ah[u] = pack_bf2(a[0], a[1]);
        al[u] = pack_bf2(a[0] - bf_lo(ah[u]), a[1] - bf_hi(ah[u]));
        bh[u] = pack_bf2(b[0], b[1]);
        bl[u] = pack_bf2(b[0] - bf_lo(bh[u]), b[1] - bf_hi(bh[u]));
    }
#pragma unroll
    for (int o = 8; o > 0; o >>= 1) det += __shfl_xor_sync(0xffffffffu, det, o);
    if (j == 0 && realk && !isfinite(lp)) bad = true;
    const int any = __syncthreads_or(bad ? 1 : 0);
    const uint32_t off = sw128_offset(k, j, 1024);  // 8-byte aligned (j % 4 == 0)
    *reinterpret_cast<uint2 *>(coef + off) = make_uint2(ah[0], ah[1]);
    *reinterpret_cast<uint2 *>(coef + kCoefMatBytes + off) = make_uint2(al[0], al[1]);
    *reinterpret_cast<uint2 *>(coef + 2 * kCoefMatBytes + off) = make_uint2(bh[0], bh[1]);
    *reinterpret_cast<uint2 *>(coef + 3 * kCoefMatBytes + off) = make_uint2(bl[0], bl[1]);
    if (j == 0) reinterpret_cast<float *>(coef + 4 * kCoefMatBytes)[k] = realk ? kLog2e * (lp - 0.5f * det) : -INFINITY;
    if (tid == 0) head_err[h * kPrepBlocks + blockIdx.x] = any ? (unsigned)GMA_ERR_NONFINITE_PARAM : 0u;
}

// ------------------------------------------------------------------ shared pieces



// ------------------------------------------------------------------ persistent pipelined kernels
//
// Work partition: the B*H*ntiles key/query tiles, in (head, tile) order, are
// cut into one contiguous range per CTA (one CTA per SM).  A range that
// crosses a head boundary is processed as one "job" per head.  Each CTA runs
// 2 + 4 NG warps:
//   warp 0            TMA producer (lane 0): tile loads into NG stages
//   warp 1            MMA issuer (lane 0): tcgen05.mma + tcgen05.commit,
//                     polling every queue so no MMA waits behind another
//   warps 2+4g..5+4g  epilogue group g: x^2 split, softmax, Gamma split,
//                     outputs of every tile whose running index is g mod NG
// Group g owns stage g, its Gamma buffer and its TMEM score / output area,
// so NG tiles are in flight and their dependent MMA chains overlap.
constexpr int kNG = 2;                       // epilogue groups (tiles in flight)
constexpr int kThreadsG = 64 + 128 * kNG;    // TMA warp, MMA warp, NG x 4 epilogue warps

// The tiles in (head, tile) order cut into one contiguous range per CTA: CTA c
// takes [start[c], start[c + 1]).  The cuts balance the CTAs' time, not their
// tile counts: a range that crosses a head boundary pays a job end and a job
// start (the accumulator drained, the next head's coefficients and first tiles
// loaded behind a CTA-wide barrier), so such a range gets kSwitchTiles fewer
// tiles (part_cuts).  Traces put a job switch near four tiles of work; six
// measured fastest (3, 4 and 6 compared), as those ranges also tend to hold the
// CTA that combines a head.
constexpr int kMaxPartCtas = 320;
constexpr int kSwitchTiles = 6;
struct Part {
    int ntiles;  // tiles per head
    int total;   // B*H*ntiles
    int nctas;   // ranges (CTAs)
    int slots;   // partial slots per CTA (jobs per CTA, upper bound)
    int start[kMaxPartCtas + 1];
};

// CTA whose range holds tile x (ranges are non-empty and in order).
__host__ __device__ inline int cta_of_tile(const Part &P, int x) {
    int lo = 0, hi = P.nctas - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (P.start[mid] <= x) lo = mid; else hi = mid - 1;
    }
    return lo;
}
__host__ __device__ inline int first_cta_of_head(const Part &P, int bh) { return cta_of_tile(P, bh * P.ntiles); }
__host__ __device__ inline int last_cta_of_head(const Part &P, int bh) {
    return cta_of_tile(P, (bh + 1) * P.ntiles - 1);
}
// Slot of head bh's job inside CTA c (CTA c's range starts in head start[c] / ntiles).
__host__ __device__ inline int slot_of(const Part &P, int c, int bh) { return bh - P.start[c] / P.ntiles; }


// Parameter-error check of the first persistent kernel of a call, by one
// whole warp: any coefficient-prep block that failed validation fails the
// call.  Returns the OR of the error words (all of them carry the same code).
__device__ __forceinline__ unsigned head_error_warp(const unsigned *head_err, int H, int lane) {
    unsigned e = 0u;
    for (int i = lane; i < H * kPrepBlocks; i += 32) e |= __ldcg(head_err + i);
    return __reduce_or_sync(0xffffffffu, e);
}


// x^2 split of this thread's row of a swizzled [128 x 64] bf16 tile, written
// to tensor memory as an MMA A operand: x2hi at columns [0, 32), x2lo at
// [32, 64) of `taddr` (this thread's lane).
__device__ __forceinline__ void prep_x2_row_tmem(const uint8_t *x, int row, uint32_t taddr) {
    uint32_t h[32], l[32];
    const uint8_t *rp = x + row * 128;
#pragma unroll
    for (int c = 0; c < 8; ++c) {
        const uint4 v = *reinterpret_cast<const uint4 *>(rp + ((c ^ (row & 7)) << 4));
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            h[4 * c + q] = bf2_fma(w[q], w[q], 0x80008000u);
            l[4 * c + q] = bf2_fma(w[q], w[q], h[4 * c + q] ^ 0x80008000u);
        }
    }
    tmem_st32(taddr, h);
    tmem_st32(taddr + 32, l);
    tmem_wait_st();
}

// Score MMAs of one tile, 12 instructions (4 K-steps x 3): the coefficient
// image holds [a_hi ; a_lo] and [b_hi ; b_lo] as two N = 128 operands, so
//   D[:, 0:128]  = x2hi [a_hi | a_lo] + x [b_hi | b_lo]   (N = 128)
//   D[:, 0:64]  += x2lo a_hi                               (N = 64)
// and the score of component k is D[:, k] + D[:, 64 + k] (+ c_k).
// The x^2 operands come from tensor memory (a_tmem: x2hi +0, x2lo +32), x from
// shared memory (descriptor dx), coefficients from shared memory (dc).
__device__ __forceinline__ void issue_scores_tA(uint32_t d_tmem, uint32_t a_tmem, uint64_t dx, uint64_t dc) {
    constexpr uint32_t i128 = idesc_bf16(kTile, 128, false, false);
    constexpr uint32_t i64 = idesc_bf16(kTile, 64, false, false);
#pragma unroll
    for (int kk = 0; kk < kDR / 16; ++kk) {
        const uint32_t o = kk * 32;
        umma_bf16_tA(d_tmem, a_tmem + kk * 8, dadd(dc, o), i128, kk > 0 ? 1u : 0u);
        umma_bf16(d_tmem, dadd(dx, o), dadd(dc, 2 * kCoefMatBytes + o), i128, 1u);
        umma_bf16_tA(d_tmem, a_tmem + 32 + kk * 8, dadd(dc, o), i64, 1u);
    }
}

__device__ __noinline__ void issue_scores_ool(uint32_t d_tmem, uint32_t a_tmem, uint64_t dx, uint64_t dc) {
    issue_scores_tA(d_tmem, a_tmem, dx, dc);
}

// Score row (two 64-column halves in TMEM) -> exponentials e_k = 2^(s_k - max);
// returns the row sum.
__device__ __forceinline__ float score_row_exp128(uint32_t taddr, const float *cvec, float (&e)[kKP]) {
    uint32_t r0[32], r1[32], r2[32], r3[32];
    tmem_ld32(taddr, r0);
    tmem_ld32(taddr + 32, r1);
    tmem_ld32(taddr + 64, r2);
    tmem_ld32(taddr + 96, r3);
    tmem_wait_ld();
    const float4 *c4 = reinterpret_cast<const float4 *>(cvec);
    float m0 = -INFINITY, m1 = -INFINITY;
#pragma unroll
    for (int q = 0; q < 8; ++q) {
        const float4 ca = c4[q], cb = c4[q + 8];
#define GMA_U(r, i) __uint_as_float(r[i])
        const float2 a0 = f2_add(f2_add(make_float2(GMA_U(r0, 4 * q), GMA_U(r0, 4 * q + 1)),
                                        make_float2(GMA_U(r2, 4 * q), GMA_U(r2, 4 * q + 1))), make_float2(ca.x, ca.y));
        const float2 a1 = f2_add(f2_add(make_float2(GMA_U(r0, 4 * q + 2), GMA_U(r0, 4 * q + 3)),
                                        make_float2(GMA_U(r2, 4 * q + 2), GMA_U(r2, 4 * q + 3))), make_float2(ca.z, ca.w));
        const float2 b0 = f2_add(f2_add(make_float2(GMA_U(r1, 4 * q), GMA_U(r1, 4 * q + 1)),
                                        make_float2(GMA_U(r3, 4 * q), GMA_U(r3, 4 * q + 1))), make_float2(cb.x, cb.y));
        const float2 b1 = f2_add(f2_add(make_float2(GMA_U(r1, 4 * q + 2), GMA_U(r1, 4 * q + 3)),
                                        make_float2(GMA_U(r3, 4 * q + 2), GMA_U(r3, 4 * q + 3))), make_float2(cb.z, cb.w));
#undef GMA_U
        e[4 * q] = a0.x; e[4 * q + 1] = a0.y; e[4 * q + 2] = a1.x; e[4 * q + 3] = a1.y;
        e[32 + 4 * q] = b0.x; e[32 + 4 * q + 1] = b0.y; e[32 + 4 * q + 2] = b1.x; e[32 + 4 * q + 3] = b1.y;
        m0 = fmaxf(m0, fmaxf(fmaxf(a0.x, a0.y), fmaxf(a1.x, a1.y)));
        m1 = fmaxf(m1, fmaxf(fmaxf(b0.x, b0.y), fmaxf(b1.x, b1.y)));
    }
    const float m = fmaxf(m0, m1);
    const float2 mm = make_float2(m, m);
    float2 s0 = make_float2(0.f, 0.f), s1 = make_float2(0.f, 0.f);
#pragma unroll
    for (int k = 0; k < kKP; k += 4) {
        const float2 d0 = f2_sub(make_float2(e[k], e[k + 1]), mm), d1 = f2_sub(make_float2(e[k + 2], e[k + 3]), mm);
        e[k] = ex2(d0.x); e[k + 1] = ex2(d0.y); e[k + 2] = ex2(d1.x); e[k + 3] = ex2(d1.y);
        s0 = f2_add(s0, make_float2(e[k], e[k + 1]));
        s1 = f2_add(s1, make_float2(e[k + 2], e[k + 3]));
    }
    return (s0.x + s0.y) + (s1.x + s1.y);
}

// bf16 hi / lo words of a responsibility row scaled by `scale`.
__device__ __forceinline__ void split_row(const float (&e)[kKP], float scale, uint32_t (&wh)[32], uint32_t (&wl)[32]) {
    const float2 sc = make_float2(scale, scale);
#pragma unroll
    for (int q = 0; q < 32; ++q) {
        const float2 g = f2_mul(make_float2(e[2 * q], e[2 * q + 1]), sc);
        wh[q] = pack_bf2(g.x, g.y);
        const float2 r = f2_sub(g, make_float2(bf_lo(wh[q]), bf_hi(wh[q])));
        wl[q] = pack_bf2(r.x, r.y);
    }
}

// Same row written as the MN-major / K-major SMEM layout of a Gamma buffer.
__device__ __forceinline__ void store_gamma_words(uint8_t *gbuf, int t, const uint32_t (&wh)[32],
                                                  const uint32_t (&wl)[32]) {
    uint8_t *hi = gbuf + (t >> 3) * kGS + (t & 7) * 128;
    uint8_t *lo = hi + 1024;
#pragma unroll
    for (int c = 0; c < 8; ++c) {
        const uint32_t sw = (uint32_t)((c ^ (t & 7)) << 4);
        *reinterpret_cast<uint4 *>(hi + sw) = make_uint4(wh[4 * c], wh[4 * c + 1], wh[4 * c + 2], wh[4 * c + 3]);
        *reinterpret_cast<uint4 *>(lo + sw) = make_uint4(wl[4 * c], wl[4 * c + 1], wl[4 * c + 2], wl[4 * c + 3]);
    }
}

// Optional fp32 inputs and outputs of the per-head combine (caller buffers,
// or null):
//   mode 0: out = the head's memory [Vt | Z], the sum of every job's partial;
//   mode 1: the running prefix starts at carry instead of zero, and out = the
//           prefix after the head's last job.
// Vt [BH][K][64], Z [BH][K] fp32; K <= KP (components past K are not touched).
struct CombineIO {
    const float *carry_vt, *carry_z;
    float *out_vt, *out_z;
    int K;
};

// Element (k, n0 .. n0 + 3) of a [KP][kW] partial from / to the caller's
// [Vt | Z]: n < 64 is Vt[k][n], n = 64 is Z[k], n > 64 is padding (zero).
__device__ __forceinline__ float4 io_load(const CombineIO &io, int bh, int k, int n0) {
    float v[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const int n = n0 + j;
        v[j] = k >= io.K ? 0.f
               : n < 64  ? io.carry_vt[((size_t)bh * io.K + k) * 64 + n]
               : n == 64 ? io.carry_z[(size_t)bh * io.K + k]
                         : 0.f;
    }
    return make_float4(v[0], v[1], v[2], v[3]);
}
__device__ __forceinline__ void io_store(const CombineIO &io, int bh, int k, int n0, float4 a) {
    if (k >= io.K) return;
    const float v[4] = {a.x, a.y, a.z, a.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const int n = n0 + j;
        if (n < 64) io.out_vt[((size_t)bh * io.K + k) * 64 + n] = v[j];
        else if (n == 64) io.out_z[(size_t)bh * io.K + k] = v[j];
    }
}

// Combines the job partials ([KP][kW] fp32 each) of head bh in CTA order, so
// the result does not depend on which job finished last:
//   mode 0: img (shared memory) = the sum of the partials as the bf16 hi | lo
//           read operand [NB = 80 rows x KP], K-major, 128-byte swizzled: row
//           n < 64 Vt[:, n], row 64 Z, rows 65 .. 67 the partials' zero padding,
//           rows 68 .. 79 zero;
//   mode 1: each partial replaced in place by the sum of the ones before it.
// Each thread owns four float4 slots of the [KP][kW] layout and keeps the loads
// of six CTAs for all of them in flight (one round for up to six jobs).
__device__ void combine_partials(float *__restrict__ part, const Part &P, int bh, int mode, uint8_t *img, int tid,
                                 int nthreads, const CombineIO &io) {
    constexpr int kRow4 = kW / 4, kE4 = kKP * kRow4, NQ = 4, NB = 6;
    constexpr size_t kPS4 = (size_t)kKP * kRow4;
    const int cf = first_cta_of_head(P, bh), cl = last_cta_of_head(P, bh);
    float4 acc[NQ];
#pragma unroll
    for (int q = 0; q < NQ; ++q) {
        const int e4 = tid + q * nthreads;
        acc[q] = (mode == 1 && io.carry_vt && e4 < kE4) ? io_load(io, bh, e4 / kRow4, 4 * (e4 % kRow4))
                                                         : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    for (int cb = cf; cb <= cl; cb += NB) {
        float4 v[NB][NQ];
#pragma unroll
        for (int u = 0; u < NB; ++u) {
            const int cc = cb + u;
            const float4 *src = reinterpret_cast<const float4 *>(part) +
                                ((size_t)cc * P.slots + (cc <= cl ? slot_of(P, cc, bh) : 0)) * kPS4;
#pragma unroll
            for (int q = 0; q < NQ; ++q) {
                const int e4 = tid + q * nthreads;
                v[u][q] = (cc <= cl && e4 < kE4) ? __ldcg(src + e4) : make_float4(0.f, 0.f, 0.f, 0.f);
            }
        }
#pragma unroll
        for (int u = 0; u < NB; ++u) {
            const int cc = cb + u;
            if (cc > cl) break;
            float4 *dst = reinterpret_cast<float4 *>(part) + ((size_t)cc * P.slots + slot_of(P, cc, bh)) * kPS4;
#pragma unroll
            for (int q = 0; q < NQ; ++q) {
                const int e4 = tid + q * nthreads;
                if (e4 >= kE4) continue;
                if (mode == 1) __stcg(dst + e4, acc[q]);
                acc[q].x += v[u][q].x;
                acc[q].y += v[u][q].y;
                acc[q].z += v[u][q].z;
                acc[q].w += v[u][q].w;
            }
        }
    }
    if (io.out_vt) {
#pragma unroll
        for (int q = 0; q < NQ; ++q) {
            const int e4 = tid + q * nthreads;
            if (e4 < kE4) io_store(io, bh, e4 / kRow4, 4 * (e4 % kRow4), acc[q]);
        }
    }
    if (mode == 0) {
        constexpr int NBR = 64 + 16;
        __nv_bfloat16 *bhi = reinterpret_cast<__nv_bfloat16 *>(img);
        __nv_bfloat16 *blo = reinterpret_cast<__nv_bfloat16 *>(img + NBR * 128);
#pragma unroll
        for (int q = 0; q < NQ; ++q) {
            const int e4 = tid + q * nthreads;
            if (e4 >= kE4) continue;
            const int k = e4 / kRow4, n0 = 4 * (e4 % kRow4);
            const float v[4] = {acc[q].x, acc[q].y, acc[q].z, acc[q].w};
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const __nv_bfloat16 vh = __float2bfloat16_rn(v[j]);
                const uint32_t off = sw128_offset(n0 + j, k, 1024) / 2;
                bhi[off] = vh;
                blo[off] = __float2bfloat16_rn(v[j] - __bfloat162float(vh));
            }
        }
        // rows 4 kRow4 .. NBR - 1 (never a partial's column): zero, in both images
        constexpr int kZ0 = 4 * kRow4 * 128, kZ16 = (NBR * 128 - kZ0) / 16;
        for (int i = tid; i < 2 * kZ16; i += nthreads)
            *reinterpret_cast<uint4 *>(img + (i / kZ16) * NBR * 128 + kZ0 + (i % kZ16) * 16) = make_uint4(0, 0, 0, 0);
    }
}

// Write kernel stages.  K tiles are freed once their score MMAs complete, V
// tiles once their write MMA completes, so the two rings are separate and the
// loads run ahead of the epilogue groups.  The Z column comes from a constant
// chunk of ones read as the second MN chunk of the V operand: each V stage's
// descriptor sets its chunk stride (LBO) to the distance from that stage to
// the ones chunk, so one N = 80 MMA gives Gamma^T V (columns 0..63) and
// Gamma^T 1 (column 64).
struct Write2Smem {
    static constexpr int W = kW;
    static constexpr int kKS = 4, kVS = 3;                      // K / V ring depths
    static constexpr int kKst = 0;                              // K stages
    static constexpr int kVst = kKst + kKS * kTileBytes;        // V stages
    static constexpr int kOnes = kVst + kVS * kTileBytes;       // chunk of ones (MN-major, 128 x 64)
    static constexpr int kXG = kOnes + kTileBytes;              // Gamma^K buffers [NG][32 KB]
    static constexpr int kCoef = kXG + kNG * 2 * kTileBytes;
    static constexpr int kBars = kCoef + ((kCoefBytes + 1023) & ~1023);
    static constexpr int kBytes = kBars + 256;
    static constexpr int kAlloc = kBytes + 1024;
    static_assert(128 * W * 4 <= kVst, "reduction buffer must fit over the K stages");
    static_assert(kAlloc <= 232448, "shared memory budget");
};

// Latent aggregation ([GMA, Eqs. (5)-(6)]) over each job's keys (d_v = 64):
//   part[job][k][c] = sum_j gamma^K_jk V_jc,  part[job][k][64] = sum_j gamma^K_jk.
// The last job of each head to finish combines the head's jobs in CTA order:
//   mode 0: the bf16 hi / lo read operand of the whole-sequence memory (bidirectional),
//   mode 1: in place, the exclusive prefix of each job (causal carry-in).
// TMEM: scores of group g at [128 g, +128); x^2 operand of group g at
// [128 NG + 64 g, +64); accumulator [Vt | Z] (N = 80) at 192 NG.
__global__ void __launch_bounds__(kThreadsG, 1) tc_write2_kernel(
    const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
    const uint8_t *__restrict__ coef_img, const unsigned *__restrict__ head_err, int H, int N, const __grid_constant__ Part P,
    float *__restrict__ part, unsigned *__restrict__ counters, uint8_t *__restrict__ mem_img, size_t mem_img_stride,
    uint8_t *__restrict__ gk_out, int mode, int stall, CombineIO io, unsigned *status) {
    using L = Write2Smem;
    constexpr int D_V = 64, W = L::W;
    constexpr int kTmemCols = 512;
    constexpr int kA = 2 * kNG * kKP, kAcc = 3 * kNG * kKP;
    static_assert(kAcc + 80 <= kTmemCols, "TMEM budget");
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    constexpr int KS = L::kKS, VS = L::kVS;
    uint8_t *kst = smem + L::kKst, *vst = smem + L::kVst, *xg = smem + L::kXG, *coef = smem + L::kCoef;
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + L::kBars);
    uint64_t *kfull = bars, *kempty = kfull + KS, *vfull = kempty + KS, *vempty = vfull + VS;
    uint64_t *xready = vempty + VS, *sfull = xready + kNG, *gready = sfull + kNG, *wdone = gready + kNG,
             *accfull = wdone + kNG, *cfull = accfull + 1;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(cfull + 1);
    int *abort_flag = reinterpret_cast<int *>(cfull + 2);
    int *last_flag = abort_flag + 1;
    static_assert((2 * KS + 2 * VS + 4 * kNG + 4) * 8 <= 256, "barrier area");
    const float *cvec = reinterpret_cast<const float *>(coef + 4 * kCoefMatBytes);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int c = blockIdx.x;
    const int g0 = P.start[c], gend = P.start[c + 1];
    if (g0 >= gend) return;

    if (warp == 0) {
        tmem_alloc(tmem_slot, kTmemCols);
        tmem_relinquish();
    }
    if (tid == 32) {
        for (int i = 0; i < KS; ++i) {
            mbar_init(&kfull[i], 1);
            mbar_init(&kempty[i], 1);
        }
        for (int i = 0; i < VS; ++i) {
            mbar_init(&vfull[i], 1);
            mbar_init(&vempty[i], 1);
        }
        for (int i = 0; i < kNG; ++i) {
            mbar_init(&xready[i], 4);
            mbar_init(&sfull[i], 1);
            mbar_init(&gready[i], 4);
            mbar_init(&wdone[i], 1);
        }
        mbar_init(accfull, 1);
        mbar_init(cfull, 1);
        *abort_flag = 0;
        fence_mbar_init();
        tma_prefetch_desc(&tmK);
        tma_prefetch_desc(&tmV);
    }
    {   // the constant ones chunk
        const uint4 one4 = make_uint4(0x3F803F80u, 0x3F803F80u, 0x3F803F80u, 0x3F803F80u);
        for (int i = tid; i < kTileBytes / 16; i += kThreadsG) reinterpret_cast<uint4 *>(smem + L::kOnes)[i] = one4;
    }
    // Everything below reads the coefficient prep's output (and the workspace the
    // previous call's kernels used): wait for it, then let the next kernel launch.
    pdl_wait();
    pdl_trigger();
    {
        const unsigned herr = warp == 1 ? head_error_warp(head_err, H, lane) : 0u;
        if (tid == 32 && (herr || failed(status))) {
            if (herr) set_status(status, herr);
            *abort_flag = 1;
        }
    }
    tc_fence_before();
    cta_sync();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    constexpr uint32_t idesc_w = idesc_bf16(kTile, 80, true, true);

    int rbase = 0;   // running tile index of the CTA (barrier phases)
    int njob = 0;
    int carm = -1;   // last job whose coefficient copy was armed (thread 0)
    for (int g = aborted(abort_flag) ? gend : g0; g < gend; ++njob) {
        const int bh = g / P.ntiles, t0 = g % P.ntiles;
        const int n = min(P.ntiles - t0, gend - g);
        const int h = bh % H;
        // The previous job's reads of the coefficients and its generic writes over
        // the K ring are complete; the head's coefficients arrive on cfull.
        fence_proxy_async_smem();
        cta_sync();
        if (tid == 0) {
            mbar_arrive_expect_tx(cfull, kCoefBytes);
            bulk_load(coef, coef_img + (size_t)h * kCoefStride, kCoefBytes, cfull);
            carm = njob;
        }

        if (warp == 0) {
            if (lane == 0) {
                // K loads as far ahead as the K ring allows; V loads follow, never ahead of their K.
                int nk = 0, nv = 0;
                int karm[KS], varm[VS];  // running index of the last load armed per stage
#pragma unroll
                for (int q = 0; q < KS; ++q) karm[q] = -1;
#pragma unroll
                for (int q = 0; q < VS; ++q) varm[q] = -1;
                Stall st;
                while (nv < n) {
                    bool prog = false;
                    if (nk < n) {
                        const int r = rbase + nk, s = r % KS;
                        if (mbar_test(&kempty[s], ((r / KS) & 1) ^ 1)) {
                            if (!(stall && r == 0)) {  // test hook: the first key tile is never loaded
                                mbar_arrive_expect_tx(&kfull[s], kTileBytes);
                                tma_load_3d(kst + s * kTileBytes, &tmK, 0, (t0 + nk) * kTile, bh, &kfull[s]);
                                karm[s] = r;
                            }
                            ++nk;
                            prog = true;
                        }
                    }
                    if (nv < nk) {
                        const int r = rbase + nv, s = r % VS;
                        if (mbar_test(&vempty[s], ((r / VS) & 1) ^ 1)) {
                            mbar_arrive_expect_tx(&vfull[s], kTileBytes);
                            tma_load_3d(vst + s * kTileBytes, &tmV, 0, (t0 + nv) * kTile, bh, &vfull[s]);
                            varm[s] = r;
                            ++nv;
                            prog = true;
                        }
                    }
                    if (!st.tick(prog, abort_flag)) {
                        note_timeout(status, abort_flag);
                        break;
                    }
                }
                // Every load armed here has landed before the CTA moves on or leaves
                // (immediate unless the job was aborted).
#pragma unroll
                for (int q = 0; q < KS; ++q)
                    if (karm[q] >= 0) mbar_wait(&kfull[q], (karm[q] / KS) & 1);
#pragma unroll
                for (int q = 0; q < VS; ++q)
                    if (varm[q] >= 0) mbar_wait(&vfull[q], (varm[q] / VS) & 1);
            }
        } else if (warp == 1) {
            if (lane == 0) {
                // Base descriptors, built once; each MMA advances one by an add.
                const uint64_t dk0 = sdesc_sw128(smem_u32(kst), 16, 1024), dc0 = sdesc_sw128(smem_u32(coef), 16, 1024);
                const uint64_t dg0 = sdesc_sw128(smem_u32(xg), 1024, kGS);
                uint64_t dv[VS];  // per V stage: chunk stride (LBO) = distance to the ones chunk
#pragma unroll
                for (int s = 0; s < VS; ++s)
                    dv[s] = sdesc_sw128(smem_u32(vst + s * kTileBytes), L::kOnes - (L::kVst + s * kTileBytes), 1024);
                // Poll both queues so that neither kind of MMA waits behind the other.
                int ns = 0, nw = 0;
                Stall st;
                const bool coef_ok = wait_or_abort(cfull, njob & 1, status, abort_flag);
                while (coef_ok && nw < n) {
                    bool prog = false;
                    if (ns < n) {
                        const int r = rbase + ns, gb = r % kNG, sk = r % KS;
                        if (mbar_test(&xready[gb], (r / kNG) & 1)) {
                            tc_fence_after();
                            issue_scores_tA(tmem + gb * 2 * kKP, tmem + kA + gb * kKP, dadd(dk0, sk * kTileBytes), dc0);
                            umma_commit(&sfull[gb]);
                            umma_commit(&kempty[sk]);
                            ++ns;
                            prog = true;
                        }
                    }
                    if (nw < ns) {
                        const int r = rbase + nw, gb = r % kNG, sv = r % VS;
                        if (mbar_test(&vfull[sv], (r / VS) & 1) && mbar_test(&gready[gb], (r / kNG) & 1)) {
                            tc_fence_after();
                            const uint64_t ag = dadd(dg0, gb * 2 * kTileBytes), bv = dv[sv];
#pragma unroll
                            for (int kk = 0; kk < kTile / 16; ++kk)
                                umma_bf16(tmem + kAcc, dadd(ag, kk * 2 * kGS), dadd(bv, kk * 2048), idesc_w,
                                          (nw > 0 || kk > 0) ? 1u : 0u);
                            umma_commit(&vempty[sv]);
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
            const int grp = (warp - 2) >> 2;  // 0 .. NG-1
            const int row = epi_row(warp, lane);
            const uint32_t lane_base = (uint32_t)(32 * (warp & 3)) << 16;
            // mode 1 also stores each tile's Gamma^K buffer (bf16 hi / lo, 32 KB) for the
            // causal scan: a warp's 32 rows are four 8-row groups, one contiguous 8 KB
            // slice, which the warp stores itself (no cross-warp barrier).
            const int q4 = warp & 3;
            for (int i = (grp - rbase % kNG + kNG) % kNG; i < n; i += kNG) {
                const int r = rbase + i, sk = r % KS;
                uint8_t *gbuf = xg + grp * 2 * kTileBytes;
                if (!wait_or_abort(&kfull[sk], (r / KS) & 1, status, abort_flag)) break;
                prep_x2_row_tmem(kst + sk * kTileBytes, row, tmem + lane_base + kA + grp * kKP);
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&xready[grp]);
                if (!wait_or_abort(&sfull[grp], (r / kNG) & 1, status, abort_flag)) break;
                if (i < kNG && !wait_or_abort(cfull, njob & 1, status, abort_flag)) break;  // c_k visible
                tc_fence_after();
                float e[kKP];
                const float rs = score_row_exp128(tmem + lane_base + grp * 2 * kKP, cvec, e);
                tc_fence_before();
                const int tok = (t0 + i) * kTile + row;
                uint32_t wh[32], wl[32];
                split_row(e, tok < N ? 1.0f / rs : 0.0f, wh, wl);
                if (r >= kNG && !wait_or_abort(&wdone[grp], ((r - kNG) / kNG) & 1, status, abort_flag)) break;
                if (mode == 1) {  // the warp's previous bulk store has read its slice
                    if (lane == 0) bulk_wait_read0();
                    __syncwarp();
                }
                store_gamma_words(gbuf, row, wh, wl);
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive(&gready[grp]);
                    if (mode == 1) {
                        const size_t off = ((size_t)bh * P.ntiles + t0 + i) * (2 * kTileBytes) + 8192 * q4;
                        bulk_store(gk_out + off, gbuf + 8192 * q4, 8192);
                        bulk_commit();
                    }
                }
            }
            if (mode == 1 && lane == 0) bulk_wait_read0();
        }
        // ---- job end: the accumulated memory -> partial of this job
        cta_sync();
        float *red = reinterpret_cast<float *>(smem);  // [128][W] over the (now idle) tile buffers
        if (!aborted(abort_flag) && warp >= 2 && warp < 6) {  // group 0 covers all 128 lanes
            if (wait_or_abort(accfull, njob & 1, status, abort_flag)) {
                tc_fence_after();
                const int row = epi_row(warp, lane);
                const uint32_t lb = (uint32_t)(32 * (warp & 3)) << 16;
                uint32_t v0[32], v1[32], z[16];
                tmem_ld32(tmem + lb + kAcc, v0);
                tmem_ld32(tmem + lb + kAcc + 32, v1);
                tmem_ld16(tmem + lb + kAcc + 64, z);
                tmem_wait_ld();
                float4 *rr = reinterpret_cast<float4 *>(red + row * W);
#pragma unroll
                for (int q = 0; q < 8; ++q) {
                    rr[q] = make_float4(__uint_as_float(v0[4 * q]), __uint_as_float(v0[4 * q + 1]),
                                        __uint_as_float(v0[4 * q + 2]), __uint_as_float(v0[4 * q + 3]));
                    rr[8 + q] = make_float4(__uint_as_float(v1[4 * q]), __uint_as_float(v1[4 * q + 1]),
                                            __uint_as_float(v1[4 * q + 2]), __uint_as_float(v1[4 * q + 3]));
                }
                rr[16] = make_float4(__uint_as_float(z[0]), 0.f, 0.f, 0.f);
                tc_fence_before();
            }
        }
        cta_sync();
        if (!aborted(abort_flag)) {
            const int slot = slot_of(P, c, bh);
            float *out = part + ((size_t)c * P.slots + slot) * kKP * W;
            for (int e = tid; e < kKP * W / 4; e += kThreadsG) {
                const float4 a = reinterpret_cast<const float4 *>(red)[e], b = reinterpret_cast<const float4 *>(red + kKP * W)[e];
                reinterpret_cast<float4 *>(out)[e] = make_float4(a.x + b.x, a.y + b.y, a.z + b.z, a.w + b.w);
            }
            __threadfence();
            cta_sync();
            if (tid == 0) {
                const int njobs = last_cta_of_head(P, bh) - first_cta_of_head(P, bh) + 1;
                const unsigned old = atomicAdd(&counters[bh], 1u);
                *last_flag = (old == (unsigned)(njobs - 1));
            }
            cta_sync();
            if (*last_flag) {
                __threadfence();
                // mode 0: the bf16 hi / lo read operand, built in shared memory (over the
                // idle K ring, after the reduction buffer) and copied out with 16-byte stores
                constexpr int kImgBytes = 2 * (D_V + 16) * 128;
                uint8_t *img = smem + 128 * W * 4 + 1024;
                static_assert(128 * W * 4 + 1024 + kImgBytes <= L::kVst, "image fits over the K ring");
                combine_partials(part, P, bh, mode, img, tid, kThreadsG, io);
                if (mode == 0) {
                    cta_sync();
                    uint4 *dst = reinterpret_cast<uint4 *>(mem_img + (size_t)bh * mem_img_stride);
                    for (int e = tid; e < kImgBytes / 16; e += kThreadsG) __stcg(dst + e, reinterpret_cast<const uint4 *>(img)[e]);
                }
                if (tid == 0) counters[bh] = 0u;  // ready for the next call
            }
        }
        rbase += n;
        g += n;
        if (aborted(abort_flag)) break;
    }
    if (tid == 0 && carm >= 0) mbar_wait(cfull, carm & 1);  // the last coefficient copy has landed
    tc_fence_before();
    cta_sync();
    if (warp == 0) tmem_dealloc(tmem, kTmemCols);
}

// ------------------------------------------------------------------ read, split rows
//
// Bidirectional read with the epilogue rows split in column halves: two groups
// of 8 warps; warps w and w + 4 of a group share TMEM lanes 32 (w % 4) .. +31
// (the tile rows) and take components (or output columns) 0..31 (half 0) and
// 32..63 (half 1).  Twice the warps of a 4-warp group run the same code with
// half the per-thread work, which hides more latency per tile.
constexpr int kNGR = 2;
constexpr int kThreadsR = 64 + 256 * kNGR;

struct Read3Smem {
    static constexpr int NB = 64 + 16;
    static constexpr int kQS = 4;                                   // Q ring depth
    static constexpr int kQst = 0;
    static constexpr int kStage = kQst + kQS * kTileBytes;          // output staging [NGR][8 warps][4 KB]
    static constexpr int kCoef = kStage + kNGR * 8 * 4096;
    static constexpr int kB = kCoef + ((kCoefBytes + 1023) & ~1023);
    static constexpr int kX = kB + ((2 * NB * 128 + 1023) & ~1023);  // (max, sum) exchange [NGR][2][128][2]
    static constexpr int kBars = kX + kNGR * 2 * 128 * 2 * 8;
    static constexpr int kBytes = kBars + 256;
    static constexpr int kAlloc = kBytes + 1024;
    static_assert(kAlloc <= 232448, "shared memory budget");
};

// x^2 split of columns 32 hf .. 32 hf + 31 of this thread's row of a swizzled
// [128 x 64] bf16 tile, to the TMEM A operand at taddr (x2hi columns
// [16 hf, +16), x2lo columns [32 + 16 hf, +16)).
__device__ __forceinline__ void prep_x2_half_tmem(const uint8_t *x, int row, int hf, uint32_t taddr) {
    uint32_t h[16], l[16];
    const uint8_t *rp = x + row * 128;
#pragma unroll
    for (int c = 0; c < 4; ++c) {
        const uint4 v = *reinterpret_cast<const uint4 *>(rp + (((4 * hf + c) ^ (row & 7)) << 4));
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            h[4 * c + q] = bf2_fma(w[q], w[q], 0x80008000u);
            l[4 * c + q] = bf2_fma(w[q], w[q], h[4 * c + q] ^ 0x80008000u);
        }
    }
    tmem_st16(taddr + 16 * hf, h);
    tmem_st16(taddr + 32 + 16 * hf, l);
    tmem_wait_st();
}

// Scores of components 32 hf .. 32 hf + 31 of this thread's row (the two
// 64-column halves of the score accumulator plus c_k); returns their maximum.
__device__ __forceinline__ float score_half(uint32_t s_taddr, const float *cvec, int hf, float (&e)[32]) {
    uint32_t a[32], b[32];
    tmem_ld32(s_taddr + 32 * hf, a);
    tmem_ld32(s_taddr + 64 + 32 * hf, b);
    tmem_wait_ld();
    const float4 *c4 = reinterpret_cast<const float4 *>(cvec + 32 * hf);
    float m0 = -INFINITY, m1 = -INFINITY;
#pragma unroll
    for (int q = 0; q < 8; ++q) {
        const float4 c = c4[q];
        const float2 s0 = f2_add(f2_add(make_float2(__uint_as_float(a[4 * q]), __uint_as_float(a[4 * q + 1])),
                                        make_float2(__uint_as_float(b[4 * q]), __uint_as_float(b[4 * q + 1]))),
                                 make_float2(c.x, c.y));
        const float2 s1 = f2_add(f2_add(make_float2(__uint_as_float(a[4 * q + 2]), __uint_as_float(a[4 * q + 3])),
                                        make_float2(__uint_as_float(b[4 * q + 2]), __uint_as_float(b[4 * q + 3]))),
                                 make_float2(c.z, c.w));
        e[4 * q] = s0.x; e[4 * q + 1] = s0.y; e[4 * q + 2] = s1.x; e[4 * q + 3] = s1.y;
        m0 = fmaxf(m0, fmaxf(s0.x, s0.y));
        m1 = fmaxf(m1, fmaxf(s1.x, s1.y));
    }
    return fmaxf(m0, m1);
}

// e <- 2^(e - m); returns the sum.
__device__ __forceinline__ float exp_half(float (&e)[32], float m) {
    const float2 mm = make_float2(m, m);
    float2 s0 = make_float2(0.f, 0.f), s1 = make_float2(0.f, 0.f);
#pragma unroll
    for (int k = 0; k < 32; k += 4) {
        const float2 d0 = f2_sub(make_float2(e[k], e[k + 1]), mm), d1 = f2_sub(make_float2(e[k + 2], e[k + 3]), mm);
        e[k] = ex2(d0.x); e[k + 1] = ex2(d0.y); e[k + 2] = ex2(d1.x); e[k + 3] = ex2(d1.y);
        s0 = f2_add(s0, make_float2(e[k], e[k + 1]));
        s1 = f2_add(s1, make_float2(e[k + 2], e[k + 3]));
    }
    return (s0.x + s0.y) + (s1.x + s1.y);
}

// bf16 hi / lo words of 32 values scaled by `scale`.
__device__ __forceinline__ void split_half(const float (&e)[32], float scale, uint32_t (&wh)[16], uint32_t (&wl)[16]) {
    const float2 sc = make_float2(scale, scale);
#pragma unroll
    for (int q = 0; q < 16; ++q) {
        const float2 g = f2_mul(make_float2(e[2 * q], e[2 * q + 1]), sc);
        wh[q] = pack_bf2(g.x, g.y);
        const float2 r = f2_sub(g, make_float2(bf_lo(wh[q]), bf_hi(wh[q])));
        wl[q] = pack_bf2(r.x, r.y);
    }
}

// Output staging of one warp's 32 rows x 32 columns (4 KB): fp32 as one
// [32 x 128 B] box with 128-byte swizzle, bf16 as one [32 x 64 B] box with
// 64-byte swizzle.  The box is stored at column 32 hf.
__device__ __forceinline__ void stage_and_store_half(uint8_t *stage, const float (&o)[32], int r32, int lane,
                                                     const CUtensorMap *tmO, int o_bf16, int hf, int row0, int bh) {
    if (lane == 0) bulk_wait_read0();
    __syncwarp();
    if (o_bf16) {
        uint8_t *rp = stage + r32 * 64;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            const uint4 w = make_uint4(pack_bf2(o[8 * c], o[8 * c + 1]), pack_bf2(o[8 * c + 2], o[8 * c + 3]),
                                       pack_bf2(o[8 * c + 4], o[8 * c + 5]), pack_bf2(o[8 * c + 6], o[8 * c + 7]));
            *reinterpret_cast<uint4 *>(rp + ((c ^ ((r32 >> 1) & 3)) << 4)) = w;
        }
    } else {
        uint8_t *rp = stage + r32 * 128;
#pragma unroll
        for (int c = 0; c < 8; ++c)
            *reinterpret_cast<float4 *>(rp + ((c ^ (r32 & 7)) << 4)) =
                make_float4(o[4 * c], o[4 * c + 1], o[4 * c + 2], o[4 * c + 3]);
    }
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) {
        tma_store_3d(tmO, stage, 32 * hf, row0, bh);
        bulk_commit();
    }
}

__global__ void __launch_bounds__(kThreadsR, 1) tc_read3_kernel(
    const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmO,
    const uint8_t *__restrict__ coef_img, int H, int N, const __grid_constant__ Part P,
    const uint8_t *__restrict__ mem_img, size_t mem_img_stride, float eps, int o_bf16, unsigned *status) {
    using L = Read3Smem;
    constexpr int NB = L::NB, QS = L::kQS;
    constexpr int kTmemCols = 512;
    constexpr int kGC = kKP + 2 * NB;  // TMEM columns per group
    static_assert(kNGR * kGC <= kTmemCols, "TMEM budget");
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t *qst = smem + L::kQst, *stg = smem + L::kStage, *coef = smem + L::kCoef, *bop = smem + L::kB;
    float2 *xch = reinterpret_cast<float2 *>(smem + L::kX);
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + L::kBars);
    uint64_t *qfull = bars, *qempty = bars + QS, *xready = bars + 2 * QS, *sfull = xready + kNGR,
             *gready = sfull + kNGR, *ofull = gready + kNGR, *cfull = ofull + kNGR, *bfull = cfull + 1;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bfull + 1);
    int *abort_flag = reinterpret_cast<int *>(bfull + 2);
    static_assert((2 * QS + 4 * kNGR + 4) * 8 <= 256, "barrier area");
    const float *cvec = reinterpret_cast<const float *>(coef + 4 * kCoefMatBytes);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int c = blockIdx.x;
    const int g0 = P.start[c], gend = P.start[c + 1];
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
        for (int i = 0; i < kNGR; ++i) {
            mbar_init(&xready[i], 8);
            mbar_init(&sfull[i], 1);
            mbar_init(&gready[i], 8);
            mbar_init(&ofull[i], 1);
        }
        mbar_init(cfull, 1);
        mbar_init(bfull, 1);
        *abort_flag = 0;
        fence_mbar_init();
        tma_prefetch_desc(&tmQ);
        tma_prefetch_desc(&tmO);
    }
    tc_fence_before();
    cta_sync();
    tc_fence_after();
    pdl_trigger();  // the next call's coefficient prep waits for this kernel's completion
    const uint32_t tmem = *tmem_slot;
    constexpr uint32_t i160 = idesc_bf16(kTile, 2 * NB, false, false);
    constexpr uint32_t i80 = idesc_bf16(kTile, NB, false, false);

    int rbase = 0, njob = 0;
    int barm = -1;  // last job whose coefficient and memory-operand copies were armed
    for (int g = g0; g < gend; ++njob) {
        const int bh = g / P.ntiles, t0 = g % P.ntiles;
        const int n = min(P.ntiles - t0, gend - g);
        const int h = bh % H;
        // The previous job's MMAs and epilogues are done with the coefficients
        // and the memory operand; this head's arrive on cfull / bfull.  The memory
        // operand is written by the write kernel, which may still be finishing:
        // only the thread that copies it waits for that kernel, so the Q loads,
        // x^2 and score MMAs of the first tiles go ahead meanwhile.
        cta_sync();
        if (tid == 0) {
            mbar_arrive_expect_tx(cfull, kCoefBytes);
            bulk_load(coef, coef_img + (size_t)h * kCoefStride, kCoefBytes, cfull);
        }
        if (tid == 33) {
            if (njob == 0) pdl_wait();
            mbar_arrive_expect_tx(bfull, 2 * NB * 128);
            bulk_load(bop, mem_img + (size_t)bh * mem_img_stride, 2 * NB * 128, bfull);
        }
        barm = njob;

        if (warp == 0) {
            if (lane == 0) {
                int qarm[QS];  // running index of the last load armed per stage
#pragma unroll
                for (int q = 0; q < QS; ++q) qarm[q] = -1;
                for (int i = 0; i < n; ++i) {
                    const int r = rbase + i, s = r % QS;
                    if (!wait_or_abort(&qempty[s], ((r / QS) & 1) ^ 1, status, abort_flag)) break;
                    mbar_arrive_expect_tx(&qfull[s], kTileBytes);
                    tma_load_3d(qst + s * kTileBytes, &tmQ, 0, (t0 + i) * kTile, bh, &qfull[s]);
                    qarm[s] = r;
                }
                // every load armed here has landed before the CTA moves on or leaves
#pragma unroll
                for (int q = 0; q < QS; ++q)
                    if (qarm[q] >= 0) mbar_wait(&qfull[q], (qarm[q] / QS) & 1);
            }
        } else if (warp == 1) {
            if (lane == 0) {
                const uint64_t dq0 = sdesc_sw128(smem_u32(qst), 16, 1024), dc0 = sdesc_sw128(smem_u32(coef), 16, 1024);
                const uint64_t db0 = sdesc_sw128(smem_u32(bop), 16, 1024);
                // Read MMAs (the shorter kind, which ends a tile) go first whenever a
                // group is ready for them.
                int ns = 0, nr = 0;
                Stall st;
                const bool coef_ok = wait_or_abort(cfull, njob & 1, status, abort_flag);
                while (coef_ok && nr < n) {
                    bool prog = false;
                    if (nr < ns) {
                        const int r = rbase + nr, gb = r % kNGR;
                        if (mbar_test(&gready[gb], (r / kNGR) & 1) && (nr > 0 || mbar_test(bfull, njob & 1))) {
                            tc_fence_after();
                            const uint32_t d = tmem + gb * kGC + kKP, a = tmem + gb * kGC;
#pragma unroll
                            for (int kk = 0; kk < kKP / 16; ++kk) {
                                umma_bf16_tA(d, a + kk * 8, dadd(db0, kk * 32), i160, kk > 0 ? 1u : 0u);
                                umma_bf16_tA(d, a + 32 + kk * 8, dadd(db0, kk * 32), i80, 1u);
                            }
                            umma_commit(&ofull[gb]);
                            ++nr;
                            prog = true;
                        }
                    }
                    if (ns < n) {
                        const int r = rbase + ns, gb = r % kNGR, s = r % QS;
                        if (mbar_test(&xready[gb], (r / kNGR) & 1)) {
                            tc_fence_after();
                            issue_scores_tA(tmem + gb * kGC + kKP, tmem + gb * kGC, dadd(dq0, s * kTileBytes), dc0);
                            umma_commit(&sfull[gb]);
                            umma_commit(&qempty[s]);
                            ++ns;
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
            const int grp = (warp - 2) >> 3;          // 0 .. NGR-1
            const int hf = ((warp - 2) >> 2) & 1;     // column half
            const int quad = warp & 3;                // TMEM lane quadrant
            const int row = 32 * quad + lane;
            const uint32_t lane_base = (uint32_t)(32 * quad) << 16;
            const uint32_t gbase = tmem + lane_base + grp * kGC;
            uint8_t *stage = stg + (grp * 8 + ((warp - 2) & 7)) * 4096;
            const int pair_bar = 1 + grp * 4 + quad;  // named barrier of the two warps of these rows
            const int i0 = (grp - rbase % kNGR + kNGR) % kNGR;  // this group's first tile of the job
            for (int i = i0; i < n; i += kNGR) {
                const int r = rbase + i;
                float2 *xr = xch + ((grp * 2 + ((r / kNGR) & 1)) * 128 + row) * 2;  // [hf] (max, sum)
                if (i == i0) {  // x^2 of the group's first tile (later ones are prepared a tile ahead)
                    if (!wait_or_abort(&qfull[r % QS], (r / QS) & 1, status, abort_flag)) break;
                    prep_x2_half_tmem(qst + (r % QS) * kTileBytes, row, hf, gbase);
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&xready[grp]);
                }
                if (!wait_or_abort(&sfull[grp], (r / kNGR) & 1, status, abort_flag)) break;
                if (i == i0 && !wait_or_abort(cfull, njob & 1, status, abort_flag)) break;  // c_k visible
                tc_fence_after();
                float rs;
                {
                    float e[32];
                    const float mh = score_half(gbase + kKP, cvec, hf, e);
                    xr[hf].x = mh;
                    named_sync(pair_bar, 64);
                    const float m = fmaxf(mh, xr[hf ^ 1].x);
                    const float sh = exp_half(e, m);
                    uint32_t wh[16], wl[16];
                    split_half(e, 1.0f, wh, wl);
                    tmem_st16(gbase + 16 * hf, wh);
                    tmem_st16(gbase + 32 + 16 * hf, wl);
                    xr[hf].y = sh;
                    tmem_wait_st();
                    named_sync(pair_bar, 64);
                    rs = hf == 0 ? sh + xr[1].y : xr[0].y + sh;  // same order in both halves
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&gready[grp]);
                if (!wait_or_abort(&ofull[grp], (r / kNGR) & 1, status, abort_flag)) break;
                tc_fence_after();
                const uint32_t ob = gbase + kKP;
                float o[32];
                {
                    uint32_t a0[32], a1[32];
                    tmem_ld32(ob + 32 * hf, a0);
                    tmem_ld32(ob + NB + 32 * hf, a1);
                    const uint32_t d0 = tmem_ld1(ob + 64), d1 = tmem_ld1(ob + NB + 64);
                    tmem_wait_ld();
                    const float inv = 1.0f / (__uint_as_float(d0) + __uint_as_float(d1) + eps * rs);
                    const float2 iv = make_float2(inv, inv);
#pragma unroll
                    for (int q = 0; q < 16; ++q) {
                        const float2 t = f2_mul(f2_add(make_float2(__uint_as_float(a0[2 * q]), __uint_as_float(a0[2 * q + 1])),
                                                       make_float2(__uint_as_float(a1[2 * q]), __uint_as_float(a1[2 * q + 1]))), iv);
                        o[2 * q] = t.x;
                        o[2 * q + 1] = t.y;
                    }
                }
                tc_fence_before();
                // x^2 of the group's next tile: the read MMAs have consumed the A columns and the
                // accumulator is in registers, so its score MMAs can start while these outputs
                // are stored.
                if (i + kNGR < n) {
                    const int r2 = r + kNGR;
                    if (!wait_or_abort(&qfull[r2 % QS], (r2 / QS) & 1, status, abort_flag)) break;
                    prep_x2_half_tmem(qst + (r2 % QS) * kTileBytes, row, hf, gbase);
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&xready[grp]);
                }
                stage_and_store_half(stage, o, lane, lane, &tmO, o_bf16, hf, (t0 + i) * kTile + 32 * quad, bh);
            }
            if (lane == 0) bulk_wait_read0();  // staging reusable; kernel completion publishes the stores
        }
        rbase += n;
        g += n;
        cta_sync();
        if (aborted(abort_flag)) break;
    }
    // the last bulk copies have landed before the CTA leaves
    if (tid == 0 && barm >= 0) mbar_wait(cfull, barm & 1);
    if (tid == 33 && barm >= 0) mbar_wait(bfull, barm & 1);
    tc_fence_before();
    cta_sync();
    if (warp == 0) tmem_dealloc(tmem, kTmemCols);
}

// ------------------------------------------------------------------ causal, persistent
//
// Causal GMA ([GMA, Eq. (8b)]) over each job's tiles (chunks of C = 128
// tokens), d_r = d_v = 64, K <= 64.  With (S, Z) the prefix memory before the
// chunk, r_i the un-normalised query row sum and P = mask_{j<=i}(Gamma^Q_c Gamma^K_c^T):
//   O_i = (gQ_i [S | Z] + sum_j P_ij [V_j | 1]) split as [num | den],  O_i = num / (den + eps r_i),
// then (S, Z) += Gamma^K_c^T [V_c | 1].  The job's starting prefix is the
// exclusive prefix left in the partials by tc_write2_kernel (mode 1).
//
// Gamma^K of each chunk is not recomputed: the aggregation pass (tc_write2_kernel,
// mode 1) stores every key tile's normalised bf16 hi / lo Gamma^K, the same values
// by the same arithmetic, and this kernel loads it by bulk copy.
//
// Warps: 0 lane 0 Q / V loads, 0 lane 1 Gamma^K loads, 1 MMA issuer, 2..5 query
// group (x^2, softmax, half of the P split, outputs), 6..9 key group (the other
// half of the P split, carry of the state).  The carry runs beside the P split
// and the P [V | 1] MMAs; the next chunk's x^2 is prepared beside the P MMAs, and
// its score MMAs are issued right after them.
//
// TMEM (512 columns):
//   [0, 64)    x^2 of Q hi | lo (A operand of the score MMAs; free once they end)
//   [64, 192)  scores Q (N = 128); the softmax overwrites columns 64..127 with
//              Gamma^Q hi | lo (A operand of P + state read), so the next chunk's
//              score MMAs follow the P MMAs in issue order
//   [192, 320) P, then P hi | lo in place per 32-key block
//   [320, 400) [num | den]: one N = 208 accumulator with P for the P + state-read MMAs
//   [400, 480) state increment U = [gK_hi ; gK_lo]^T [V | 1] (N = 80)
// The B operand of the P + state-read MMAs is [Gamma^K ; S^T] (128 + 80 K-major
// rows), so P and the read of the carried state share each instruction.
// MMAs per chunk: Q scores 12, P + state read 12 (N = 208), U 8, P [V|1] 16.
struct Causal2Smem {
    static constexpr int W = kW;                           // fp32 state rows (float4 access)
    static constexpr int WX = 66;                          // carry exchange rows (float2 access)
    // B operand of the P + state-read MMAs, K-major SW128 rows of 64 components in
    // 8-row groups of 2 KB (hi rows | lo rows): 16 groups of Gamma^K (token rows, the
    // aggregation pass's stored buffer as is) then 10 groups of S^T (value rows).
    static constexpr int kGroups = (kTile + 80) / 8;
    static constexpr int kQS = 1;                          // Q ring depth
    static constexpr int kVS = 2;                          // V ring depth
    static constexpr int kQ = 0;
    static constexpr int kV = kQ + kQS * kTileBytes;       // V tiles
    // ones columns of [V | 1]: every element is 1, so one K step (16 rows, 2 KB) serves
    // all of them; each K step's descriptor points its second N chunk here (LBO)
    static constexpr int kOnes = kV + kVS * kTileBytes;
    static constexpr int kGB = kOnes + 2048;               // [Gamma^K ; S^T]
    static constexpr int kStage = kGB + kGroups * 2048;    // output staging 4 x 8 KB
    static constexpr int kCoef = kStage + 4 * 8192;
    static constexpr int kS = kCoef + kCoefBytes;          // fp32 state [64][W]
    static constexpr int kX = kS + kKP * W * 4;            // carry exchange [64][WX]
    static constexpr int kBars = kX + kKP * WX * 4;
    static constexpr int kBytes = kBars + 256;
    static constexpr int kAlloc = kBytes + 1024;
    static_assert(kOnes % 1024 == 0 && kGB % 1024 == 0 && kStage % 1024 == 0, "SW128 alignment");
    static_assert(kS % 16 == 0 && kX % 16 == 0 && kBars % 8 == 0, "alignment");
    static_assert(kAlloc <= 232448, "shared memory budget");
};

// Epilogue pieces shared by the query and the key groups of the causal
// kernel.  They are kept out of line so that both groups run one copy of the
// code: the kernel's speed is bound by instruction fetch when each role has
// its own inlined copy.
__device__ __noinline__ void x2_row(const uint8_t *x, int row, uint32_t taddr) { prep_x2_row_tmem(x, row, taddr); }

// Softmax of one score row and the bf16 hi / lo split of the responsibilities:
// to_smem == 0: un-normalised (scale 1), hi words to taddr + 0..31, lo words to
//               taddr + 32..63 (the A operand of the following MMAs);
// to_smem != 0: normalised (scale 0 for rows past N), written as row `row` of
//               the swizzled [128 x 64] hi block at gk and the lo block at gk + lo_off.
// Returns the row sum of the exponentials.
__device__ __noinline__ float gamma_row(uint32_t s_taddr, const float *cvec, int to_smem, uint32_t taddr,
                                        uint8_t *gk, int lo_off, int row, int valid) {
    float e[kKP];
    const float rs = score_row_exp128(s_taddr, cvec, e);
    tc_fence_before();
    uint32_t wh[32], wl[32];
    split_row(e, to_smem ? (valid ? 1.0f / rs : 0.0f) : 1.0f, wh, wl);
    if (!to_smem) {
        tmem_st32(taddr, wh);
        tmem_st32(taddr + 32, wl);
        tmem_wait_st();
    } else {
        uint8_t *hi = gk + row * 128, *lo = gk + lo_off + row * 128;
#pragma unroll
        for (int cc = 0; cc < 8; ++cc) {
            const uint32_t sw = (uint32_t)((cc ^ (row & 7)) << 4);
            *reinterpret_cast<uint4 *>(hi + sw) = make_uint4(wh[4 * cc], wh[4 * cc + 1], wh[4 * cc + 2], wh[4 * cc + 3]);
            *reinterpret_cast<uint4 *>(lo + sw) = make_uint4(wl[4 * cc], wl[4 * cc + 1], wl[4 * cc + 2], wl[4 * cc + 3]);
        }
    }
    return rs;
}

// One key block (32 keys) of the masked bf16 hi / lo split of P for this
// thread's query row, written in place over the block's 32 fp32 columns:
// hi words to columns [32 cb, +16), lo words to [32 cb + 16, +16).
__device__ __forceinline__ void split_p_block(const uint32_t (&pp)[32], int cb, int row, uint32_t p_taddr) {
    uint32_t wh[16], wl[16];
#pragma unroll
    for (int q = 0; q < 16; ++q) {
        const int j = cb * 32 + 2 * q;
        const float a = j <= row ? __uint_as_float(pp[2 * q]) : 0.f;
        const float b = j + 1 <= row ? __uint_as_float(pp[2 * q + 1]) : 0.f;
        wh[q] = pack_bf2(a, b);
        wl[q] = pack_bf2(a - bf_lo(wh[q]), b - bf_hi(wh[q]));
    }
    tmem_st16(p_taddr + 32 * cb, wh);
    tmem_st16(p_taddr + 32 * cb + 16, wl);
}
__device__ __forceinline__ void zero_p_block(int cb, uint32_t p_taddr) {
    uint32_t z[16];
#pragma unroll
    for (int q = 0; q < 16; ++q) z[q] = 0u;
    tmem_st16(p_taddr + 32 * cb, z);
    tmem_st16(p_taddr + 32 * cb + 16, z);
}

// Masked split of P for key blocks cb0 and cb0 + 1 of this thread's query row,
// in place.  Blocks entirely above the diagonal are written as zeros without
// reading P (the block index of the row is uniform across a warp).
__device__ __noinline__ void split_p_blocks(uint32_t p_taddr, int cb0, int row) {
    const int rb = row >> 5;
    if (cb0 + 1 <= rb) {
        uint32_t p0[32], p1[32];
        tmem_ld32(p_taddr + cb0 * 32, p0);
        tmem_ld32(p_taddr + (cb0 + 1) * 32, p1);
        tmem_wait_ld();
        split_p_block(p0, cb0, row, p_taddr);
        split_p_block(p1, cb0 + 1, row, p_taddr);
    } else if (cb0 <= rb) {
        uint32_t p0[32];
        tmem_ld32(p_taddr + cb0 * 32, p0);
        tmem_wait_ld();
        split_p_block(p0, cb0, row, p_taddr);
        zero_p_block(cb0 + 1, p_taddr);
    } else {
        zero_p_block(cb0, p_taddr);
        zero_p_block(cb0 + 1, p_taddr);
    }
    tmem_wait_st();
}

// Outputs of one query row of the causal kernel, O = num / (den + eps r) from the
// [num | den] accumulator, written into this warp's 8 KB staging area as TMA store
// boxes of [32 rows x 128 B], 128-byte swizzled: fp32, two boxes (columns 0-31 |
// 32-63); bf16, one box.  The caller issues the stores afterwards.  Once the
// accumulator is in registers, lane 0 arrives on `freed` (if given): the columns
// may be overwritten while the row is staged.
__device__ __noinline__ void stage_output_row(uint32_t o_taddr, float rq, float eps, uint8_t *stage, int lane,
                                              int o_bf16, uint64_t *freed) {
    uint32_t a0[32], a1[32];
    tmem_ld32(o_taddr, a0);
    tmem_ld32(o_taddr + 32, a1);
    const uint32_t dz = tmem_ld1(o_taddr + 64);
    tmem_wait_ld();
    tc_fence_before();
    __syncwarp();
    if (lane == 0) {
        if (freed) mbar_arrive(freed);
        bulk_wait_read0();  // this warp's previous stores have read the staging area
    }
    __syncwarp();
    const float inv = 1.0f / (__uint_as_float(dz) + eps * rq);
    auto v = [&](int k) { return __uint_as_float(k < 32 ? a0[k] : a1[k - 32]) * inv; };
    if (o_bf16) {
        uint8_t *rp = stage + lane * 128;
#pragma unroll
        for (int c = 0; c < 8; ++c) {
            const uint4 w = make_uint4(pack_bf2(v(8 * c), v(8 * c + 1)), pack_bf2(v(8 * c + 2), v(8 * c + 3)),
                                       pack_bf2(v(8 * c + 4), v(8 * c + 5)), pack_bf2(v(8 * c + 6), v(8 * c + 7)));
            *reinterpret_cast<uint4 *>(rp + ((c ^ (lane & 7)) << 4)) = w;
        }
    } else {
#pragma unroll
        for (int b = 0; b < 2; ++b) {
            uint8_t *rp = stage + b * 4096 + lane * 128;
#pragma unroll
            for (int c = 0; c < 8; ++c) {
                const int k = 32 * b + 4 * c;
                *reinterpret_cast<float4 *>(rp + ((c ^ (lane & 7)) << 4)) = make_float4(v(k), v(k + 1), v(k + 2), v(k + 3));
            }
        }
    }
    fence_proxy_async_smem();
}

// State operand: S^T inside the B operand of the P + state-read MMAs, value
// row n (n = 64 is Z; rows 65..79 stay zero) in 8-row group 16 + n / 8 (hi rows,
// lo rows 1 KB further), 64 components per 128-byte row.  Written by all 128
// threads of the key group from the fp32 state S ([64 components][kW]): item
// i < 65 * 8 is row n = i % 65, 8-component chunk c = i / 65 (consecutive threads
// take consecutive n: conflict-free reads of S).
__device__ __forceinline__ void state_operand_from_S(uint8_t *gb, const float *S, int t) {
    for (int i = t; i < 65 * 8; i += 128) {
        const int n = i % 65, c = i / 65;
        uint32_t wh[4], wl[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const float v0 = S[(8 * c + 2 * q) * kW + n], v1 = S[(8 * c + 2 * q + 1) * kW + n];
            wh[q] = pack_bf2(v0, v1);
            wl[q] = pack_bf2(v0 - bf_lo(wh[q]), v1 - bf_hi(wh[q]));
        }
        const uint32_t off = (uint32_t)((kTile / 8 + (n >> 3)) * 2048 + (n & 7) * 128 + ((c ^ (n & 7)) << 4));
        *reinterpret_cast<uint4 *>(gb + off) = make_uint4(wh[0], wh[1], wh[2], wh[3]);
        *reinterpret_cast<uint4 *>(gb + off + 1024) = make_uint4(wl[0], wl[1], wl[2], wl[3]);
    }
}

// Carry of the causal state, S += U_hi + U_lo, in two halves.  U row `row`
// holds the hi-part sums of component k = row (row < 64) or the lo-part sums
// of k = row - 64.  Thread k owns columns 0..31 of S row k and thread 64 + k
// owns columns 32..64.  S rows are kW floats apart, X rows 66.
__device__ __forceinline__ void carry_take_cols(float4 *s4, float2 *x2, const uint32_t (&own)[32],
                                                const uint32_t (&other)[32]) {
#pragma unroll
    for (int q = 0; q < 8; ++q) {
        float4 v = s4[q];
        v.x += __uint_as_float(own[4 * q]);
        v.y += __uint_as_float(own[4 * q + 1]);
        v.z += __uint_as_float(own[4 * q + 2]);
        v.w += __uint_as_float(own[4 * q + 3]);
        s4[q] = v;
    }
#pragma unroll
    for (int q = 0; q < 16; ++q) x2[q] = make_float2(__uint_as_float(other[2 * q]), __uint_as_float(other[2 * q + 1]));
}
// carry_take: adds the thread's own part of its columns to S and hands the
// partner's columns over through X (the U columns become free).
__device__ __noinline__ void carry_take(uint32_t u_taddr, float *S, float *X, int row) {
    const int kc = row & (kKP - 1), half = row >> 6;
    uint32_t a0[32], a1[32], z[16];
    tmem_ld32(u_taddr, a0);
    tmem_ld32(u_taddr + 32, a1);
    tmem_ld16(u_taddr + 64, z);
    tmem_wait_ld();
    tc_fence_before();
    float4 *s4 = reinterpret_cast<float4 *>(S + kc * kW + 32 * half);
    float2 *x2 = reinterpret_cast<float2 *>(X + kc * 66 + 32 * (1 - half));
    if (half == 0) {
        carry_take_cols(s4, x2, a0, a1);
        X[kc * 66 + 64] = __uint_as_float(z[0]);
    } else {
        carry_take_cols(s4, x2, a1, a0);
        S[kc * kW + 64] += __uint_as_float(z[0]);
    }
}
// carry_finish (after a barrier of the key group): adds the partner's part to
// the thread's columns of S.
__device__ __noinline__ void carry_finish(float *S, const float *X, int row) {
    const int kc = row & (kKP - 1), half = row >> 6;
    float *sr = S + kc * kW;
    float4 *s4 = reinterpret_cast<float4 *>(sr + 32 * half);
    const float2 *x2 = reinterpret_cast<const float2 *>(X + kc * 66 + 32 * half);
#pragma unroll
    for (int q = 0; q < 8; ++q) {
        float4 v = s4[q];
        const float2 a = x2[2 * q], b = x2[2 * q + 1];
        v.x += a.x;
        v.y += a.y;
        v.z += b.x;
        v.w += b.y;
        s4[q] = v;
    }
    if (half) sr[64] += X[kc * 66 + 64];
}
// The state operand of the next chunk from S, by the whole key group (out of
// line: one copy for the job start and the carry).
__device__ __noinline__ void state_operand(uint8_t *gb, const float *S, int t) { state_operand_from_S(gb, S, t); }

__global__ void __launch_bounds__(kThreadsG, 1) tc_causal2_kernel(
    const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmV,
    const __grid_constant__ CUtensorMap tmO, const uint8_t *__restrict__ coef_img, const uint8_t *__restrict__ gk_in,
    const float *__restrict__ prefix, int H, int N, const __grid_constant__ Part P, float eps, int o_bf16, unsigned *status) {
    using L = Causal2Smem;
    constexpr int W = L::W, QS = L::kQS, VS = L::kVS;
    constexpr int kTmemCols = 512;
    constexpr int kXQ = 0, kSQ = 64, kGQ = kSQ, kPD = 192, kO = 320, kU = 400;
    static_assert(kO == kPD + 128, "[P | num den] is one N = 208 accumulator");
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t *qst = smem + L::kQ, *vt = smem + L::kV, *gb = smem + L::kGB, *coef = smem + L::kCoef;
    float *S = reinterpret_cast<float *>(smem + L::kS), *X = reinterpret_cast<float *>(smem + L::kX);
    uint8_t *stg = smem + L::kStage;
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + L::kBars);
    uint64_t *qfull = bars + 0, *qempty = bars + QS, *vfull = bars + 2 * QS, *vempty = vfull + VS,
             *gfull = vfull + 2 * VS, *gempty = gfull + 1, *xq = gfull + 2, *sq = gfull + 3, *gq = gfull + 4,
             *sready = gfull + 5, *pfull = gfull + 6, *pready = gfull + 7, *ofull = gfull + 8, *ufull = gfull + 9,
             *cfull = gfull + 10, *xfull = gfull + 11;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(xfull + 1);
    int *abort_flag = reinterpret_cast<int *>(xfull + 2);
    static_assert((2 * QS + 2 * VS + 15) * 8 <= 256, "barrier area");
    const float *cvec = reinterpret_cast<const float *>(coef + 4 * kCoefMatBytes);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int c = blockIdx.x;
    const int g0 = P.start[c], gend = P.start[c + 1];
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
        for (int i = 0; i < VS; ++i) {
            mbar_init(&vfull[i], 1);
            mbar_init(&vempty[i], 1);
        }
        mbar_init(gfull, 1); mbar_init(gempty, 1);
        mbar_init(xq, 4); mbar_init(sq, 1); mbar_init(gq, 4); mbar_init(sready, 4);
        mbar_init(pfull, 1); mbar_init(pready, 8); mbar_init(ofull, 1); mbar_init(ufull, 1);
        mbar_init(cfull, 1); mbar_init(xfull, 1);
        *abort_flag = 0;
        fence_mbar_init();
        tma_prefetch_desc(&tmQ); tma_prefetch_desc(&tmV); tma_prefetch_desc(&tmO);
    }
    {   // constant ones columns of [V | 1]; zero B operand (the S^T padding rows must be 0)
        const uint4 one4 = make_uint4(0x3F803F80u, 0x3F803F80u, 0x3F803F80u, 0x3F803F80u);
        for (int i = tid; i < 2048 / 16; i += kThreadsG) reinterpret_cast<uint4 *>(smem + L::kOnes)[i] = one4;
        for (int i = tid; i < L::kGroups * 2048 / 16; i += kThreadsG) reinterpret_cast<uint4 *>(gb)[i] = make_uint4(0, 0, 0, 0);
    }
    tc_fence_before();
    cta_sync();
    tc_fence_after();
    pdl_trigger();  // the next call's coefficient prep waits for this kernel's completion
    const uint32_t tmem = *tmem_slot;

    int rbase = 0, njob = 0;
    int barm = -1;  // last job whose coefficient and prefix copies were armed
    for (int g = g0; g < gend; ++njob) {
        const int bh = g / P.ntiles, t0 = g % P.ntiles;
        const int n = min(P.ntiles - t0, gend - g);
        const int h = bh % H;
        // The previous job is done with the coefficients, the state and the carry area.
        // The carried-in prefix and the stored Gamma^K come from the aggregation kernel,
        // which may still be finishing: only the threads that copy them wait for it, so
        // the Q loads, x^2, score MMAs and query softmax of the first chunk go ahead.
        fence_proxy_async_smem();
        cta_sync();
        if (tid == 0) {
            mbar_arrive_expect_tx(cfull, kCoefBytes);
            bulk_load(coef, coef_img + (size_t)h * kCoefStride, kCoefBytes, cfull);
        }
        if (tid == 33) {
            if (njob == 0) pdl_wait();
            mbar_arrive_expect_tx(xfull, kKP * W * 4);
            bulk_load(S, prefix + ((size_t)c * P.slots + slot_of(P, c, bh)) * kKP * W, kKP * W * 4, xfull);
        }
        barm = njob;

        if (warp == 0) {
            if (lane == 0) {
                // Q (ring of QS) and V (ring of VS) loads, each as soon as its stage is free.
                int nq = 0, nv = 0;
                int qarm[QS], varm[VS];
#pragma unroll
                for (int q = 0; q < QS; ++q) qarm[q] = -1;
#pragma unroll
                for (int q = 0; q < VS; ++q) varm[q] = -1;
                Stall st;
                while (nv < n) {
                    bool prog = false;
                    if (nq < n) {
                        const int r = rbase + nq, s = r % QS;
                        if (mbar_test(&qempty[s], ((r / QS) & 1) ^ 1)) {
                            mbar_arrive_expect_tx(&qfull[s], kTileBytes);
                            tma_load_3d(qst + s * kTileBytes, &tmQ, 0, (t0 + nq) * kTile, bh, &qfull[s]);
                            qarm[s] = r;
                            ++nq;
                            prog = true;
                        }
                    }
                    if (nv < nq) {
                        const int r = rbase + nv, s = r % VS;
                        if (mbar_test(&vempty[s], ((r / VS) & 1) ^ 1)) {
                            mbar_arrive_expect_tx(&vfull[s], kTileBytes);
                            tma_load_3d(vt + s * kTileBytes, &tmV, 0, (t0 + nv) * kTile, bh, &vfull[s]);
                            varm[s] = r;
                            ++nv;
                            prog = true;
                        }
                    }
                    if (!st.tick(prog, abort_flag)) {
                        note_timeout(status, abort_flag);
                        break;
                    }
                }
                // every load armed here has landed before the CTA moves on or leaves
#pragma unroll
                for (int q = 0; q < QS; ++q)
                    if (qarm[q] >= 0) mbar_wait(&qfull[q], (qarm[q] / QS) & 1);
#pragma unroll
                for (int q = 0; q < VS; ++q)
                    if (varm[q] >= 0) mbar_wait(&vfull[q], (varm[q] / VS) & 1);
            } else if (lane == 1) {
                // Gamma^K of each chunk, stored by the aggregation kernel (one 32 KB buffer).
                if (njob == 0) pdl_wait();
                int ng = 0, garm = -1;
                Stall st;
                while (ng < n) {
                    const int r = rbase + ng;
                    bool prog = false;
                    if (mbar_test(gempty, (r & 1) ^ 1)) {
                        mbar_arrive_expect_tx(gfull, 2 * kTileBytes);
                        bulk_load(gb, gk_in + ((size_t)bh * P.ntiles + t0 + ng) * (2 * kTileBytes), 2 * kTileBytes, gfull);
                        garm = r;
                        ++ng;
                        prog = true;
                    }
                    if (!st.tick(prog, abort_flag)) {
                        note_timeout(status, abort_flag);
                        break;
                    }
                }
                if (garm >= 0) mbar_wait(gfull, garm & 1);
            }
        } else if (warp == 1) {
            if (lane == 0) {
                const uint64_t dq0 = sdesc_sw128(smem_u32(qst), 16, 1024);
                const uint64_t dc = sdesc_sw128(smem_u32(coef), 16, 1024);
                const uint64_t dbh = sdesc_sw128(smem_u32(gb), 16, 2048);          // K-major [Gamma^K ; S^T] hi (N = 208)
                const uint64_t dbl = dadd(dbh, 1024);                              // ... lo
                const uint64_t dgt = sdesc_sw128(smem_u32(gb), 1024, 2048);        // MN-major [Gamma^K_hi ; Gamma^K_lo]^T (M = 128)
                // MN-major [V | 1] of V stage s at K step kk: V rows 16 kk.. of the stage, the
                // ones columns at the 2 KB ones block (the LBO shrinks as the start grows)
                auto dvk = [&](int s, int kk) {
                    const uint32_t a = smem_u32(vt + s * kTileBytes) + kk * 2048;
                    return sdesc_sw128(a, smem_u32(smem + L::kOnes) - a, 1024);
                };
                constexpr uint32_t i208 = idesc_bf16(kTile, kTile + 80, false, false);
                constexpr uint32_t i80s = idesc_bf16(kTile, 80, false, true), i80u = idesc_bf16(kTile, 80, true, true);
                // Per chunk: Q scores (once the chunk's x^2 is ready and the previous P +
                // state read, which reads Gamma^Q from the score columns, is issued);
                // P + state read (after the previous chunk's P [V|1], whose P columns it
                // overwrites); P [V|1]; U whenever its inputs are loaded and the previous
                // chunk's carry has read its columns (the previous P [V|1] issued).
                // Single-thread issue order is the tensor pipe's execution order.
                int qd = 0, ud = 0, pd = 0, vd = 0;
                Stall st;
                const bool coef_ok = wait_or_abort(cfull, njob & 1, status, abort_flag);
                while (coef_ok && vd < n) {
                    bool prog = false;
                    if (ud < n && ud <= vd) {
                        const int r = rbase + ud;
                        if (mbar_test(gfull, r & 1) && mbar_test(&vfull[r % VS], (r / VS) & 1)) {
                            tc_fence_after();
                            if (ud + 1 < n) {
#pragma unroll 1
                                for (int kk = 0; kk < kTile / 16; ++kk)
                                    umma_bf16(tmem + kU, dadd(dgt, kk * 4096), dvk(r % VS, kk), i80u, kk > 0 ? 1u : 0u);
                            }
                            umma_commit(ufull);
                            ++ud;
                            if (pd >= ud) umma_commit(gempty);
                            if (vd >= ud) umma_commit(&vempty[r % VS]);
                            prog = true;
                        }
                    }
                    if (qd < n && qd <= pd) {
                        const int r = rbase + qd;
                        if (mbar_test(xq, r & 1)) {
                            tc_fence_after();
                            issue_scores_ool(tmem + kSQ, tmem + kXQ, dadd(dq0, (r % QS) * kTileBytes), dc);
                            umma_commit(sq);
                            umma_commit(&qempty[r % QS]);
                            ++qd;
                            prog = true;
                        }
                    }
                    if (pd < qd && pd == vd) {
                        const int r = rbase + pd;
                        if (mbar_test(gq, r & 1) && mbar_test(gfull, r & 1) && mbar_test(sready, r & 1)) {
                            tc_fence_after();
                            // [P | num den] = gQhi [gK ; S^T]hi^T + gQhi [gK ; S^T]lo^T + gQlo [gK ; S^T]hi^T
#pragma unroll 1
                            for (int kk = 0; kk < kKP / 16; ++kk) {
                                const uint32_t aq = tmem + kGQ + kk * 8;
                                umma_bf16_tA(tmem + kPD, aq, dadd(dbh, kk * 32), i208, kk > 0 ? 1u : 0u);
                                umma_bf16_tA(tmem + kPD, aq, dadd(dbl, kk * 32), i208, 1u);
                                umma_bf16_tA(tmem + kPD, aq + 32, dadd(dbh, kk * 32), i208, 1u);
                            }
                            umma_commit(pfull);
                            ++pd;
                            if (ud >= pd) umma_commit(gempty);
                            prog = true;
                        }
                    } else if (vd < pd) {
                        const int r = rbase + vd;
                        if (mbar_test(pready, r & 1) && mbar_test(&vfull[r % VS], (r / VS) & 1)) {
                            tc_fence_after();
                            // [num | den] += P [V | 1]; P hi / lo sit in place in the P columns:
                            // key block cb = kk / 2 holds hi words at 32 cb, lo words at 32 cb + 16.
#pragma unroll 1
                            for (int kk = 0; kk < kTile / 16; ++kk) {
                                const uint64_t bv = dvk(r % VS, kk);
                                const uint32_t ap = tmem + kPD + 32 * (kk >> 1) + 8 * (kk & 1);
                                umma_bf16_tA(tmem + kO, ap, bv, i80s, 1u);
                                umma_bf16_tA(tmem + kO, ap + 16, bv, i80s, 1u);
                            }
                            umma_commit(ofull);
                            ++vd;
                            if (ud >= vd) umma_commit(&vempty[r % VS]);
                            prog = true;
                        }
                    }
                    if (!st.tick(prog, abort_flag)) {
                        note_timeout(status, abort_flag);
                        break;
                    }
                }
            }
        } else if (warp < 6) {
            // ---------------- query group
            // Iteration i: scores and softmax of chunk i, then the outputs of chunk i - 1
            // (gq lets P + state read of chunk i overwrite its accumulator once that is in
            // registers; staging and store go beside those MMAs), the x^2 of chunk i + 1,
            // then the P split of chunk i.
            const int row = epi_row(warp, lane);
            const uint32_t lb = (uint32_t)(32 * (warp & 3)) << 16;
            uint8_t *stage = stg + (warp & 3) * 8192;
            float rq_prev = 0.f, rq = 0.f;
            for (int i = 0; i <= n; ++i) {
                const int r = rbase + i, ph = r & 1;
                if (i < n) {
                    if (i == 0) {  // x^2 of the job's first chunk (later ones are prepared a chunk ahead)
                        if (!wait_or_abort(&qfull[r % QS], (r / QS) & 1, status, abort_flag)) break;
                        x2_row(qst + (r % QS) * kTileBytes, row, tmem + lb + kXQ);
                        tc_fence_before();
                        __syncwarp();
                        if (lane == 0) mbar_arrive(xq);
                    }
                    if (!wait_or_abort(sq, ph, status, abort_flag)) break;
                    if (i == 0 && !wait_or_abort(cfull, njob & 1, status, abort_flag)) break;  // c_k visible
                    tc_fence_after();
                    rq = gamma_row(tmem + lb + kSQ, cvec, 0, tmem + lb + kGQ, nullptr, 0, row, 1);
                }
                if (i > 0) {
                    if (!wait_or_abort(ofull, ph ^ 1, status, abort_flag)) break;
                    tc_fence_after();
                    stage_output_row(tmem + lb + kO, rq_prev, eps, stage, lane, o_bf16, i < n ? gq : nullptr);
                } else {
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(gq);
                }
                __syncwarp();
                if (i > 0 && lane == 0) {
                    const int row0 = (t0 + i - 1) * kTile + 32 * (warp & 3);
                    tma_store_3d(&tmO, stage, 0, row0, bh);
                    if (!o_bf16) tma_store_3d(&tmO, stage + 4096, 32, row0, bh);
                    bulk_commit();
                }
                if (i == n) break;
                rq_prev = rq;
                // x^2 of the next chunk beside this chunk's P MMAs (the score MMAs of this
                // chunk, the only readers of the x^2 columns, have completed: sq)
                if (i + 1 < n) {
                    const int r1 = r + 1;
                    if (!wait_or_abort(&qfull[r1 % QS], (r1 / QS) & 1, status, abort_flag)) break;
                    x2_row(qst + (r1 % QS) * kTileBytes, row, tmem + lb + kXQ);
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(xq);
                }
                if (!wait_or_abort(pfull, ph, status, abort_flag)) break;
                tc_fence_after();
                // masked intra-chunk affinity, key blocks 0 and 1 -> P hi | lo (in place)
                split_p_blocks(tmem + lb + kPD, 0, row);
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(pready);
            }
            if (lane == 0) bulk_wait_read0();  // staging reusable; kernel completion publishes the stores
        } else {
            // ---------------- key group: carry of the state and half of the P split
            const int row = epi_row(warp, lane);
            const uint32_t lb = (uint32_t)(32 * (warp & 3)) << 16;
            for (int i = 0; i < n; ++i) {
                const int r = rbase + i, ph = r & 1;
                if (i == 0) {  // state operand of the job's first chunk, from the carried-in prefix
                    if (wait_or_abort(xfull, njob & 1, status, abort_flag)) state_operand(gb, S, tid - 192);
                    fence_proxy_async_smem();
                    named_sync(1, 128);  // every key thread has read S before the carry adds to it
                    if (lane == 0) mbar_arrive(sready);
                }
                const bool carry = i + 1 < n;
                if (carry) {
                    // first half of the carry, beside the P MMAs: U out of tensor memory,
                    // the partner's columns through X
                    if (!wait_or_abort(ufull, ph, status, abort_flag)) break;
                    tc_fence_after();
                    carry_take(tmem + lb + kU, S, X, row);
                }
                // masked intra-chunk affinity, key blocks 2 and 3 -> P hi | lo (in place)
                if (!wait_or_abort(pfull, ph, status, abort_flag)) break;
                tc_fence_after();
                split_p_blocks(tmem + lb + kPD, 2, row);
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(pready);
                // second half of the carry, beside the P [V | 1] MMAs: the state operand of
                // the next chunk (the state read of this chunk is done: pfull)
                if (carry) {
                    named_sync(1, 128);
                    carry_finish(S, X, row);
                    named_sync(1, 128);
                    state_operand(gb, S, tid - 192);
                    fence_proxy_async_smem();
                    named_sync(1, 128);  // every key thread has read S before the next carry
                    if (lane == 0) mbar_arrive(sready);
                }
            }
        }
        rbase += n;
        g += n;
        cta_sync();
        if (aborted(abort_flag)) break;
    }
    // the last bulk copies have landed before the CTA leaves
    if (tid == 0 && barm >= 0) mbar_wait(cfull, barm & 1);
    if (tid == 33 && barm >= 0) mbar_wait(xfull, barm & 1);
    tc_fence_before();
    cta_sync();
    if (warp == 0) tmem_dealloc(tmem, kTmemCols);
}

// ------------------------------------------------------------------ causal, single pass
//
// Causal GMA ([GMA, Eq. (8b)]) in one pass over Q_X, K_X and V_X: each CTA
// takes 128-token chunks and computes, for each, the key side (Gamma^K, kept
// in shared memory, and the chunk's memory increment U = Gamma^K^T [V | 1])
// and the query side (Gamma^Q, the masked intra-chunk P = Gamma^Q Gamma^K^T,
// P [V | 1] and the read of the prefix memory S before the chunk):
//   O_i = (sum_{j <= i in chunk} P_ij [V_j | 1] + gQ_i [S | Z]) split as [num | den],
//   O_i = num / (den + eps r_i),  r_i the un-normalised query row sum.
//
// The prefix memory before chunk t of a head is the sum of the increments of
// chunks 0 .. t-1 ("cumulative sums along the sequence dimension").  Chunks
// are handed out in (chunk index, head) order, CTA c taking every G-th one, so
// the CTAs working at one time hold consecutive chunks of each head.  Every
// chunk publishes its increment in global memory as soon as its key side is
// done; chunk t then sums, in a fixed order, the inclusive prefix published
// by the last chunk of the previous block of kBlock chunks and the increments
// of the chunks of its own block before it.  The last chunk of each block
// publishes its inclusive prefix.  The summation order depends only on t, so
// results are bitwise reproducible; the waits are bounded.  The published
// memories have one slot per chunk, written once per call; the flags carry the
// chunk index, and a reader checks them again after reading.
//
// Warps: 0 lane 0 TMA loads, 1 lane 0 MMA issue (a fixed order per chunk),
// 2..5 key group (key softmax -> Gamma^K, half of the P split, increment),
// 6..9 query group (query softmax -> Gamma^Q, half of the P split, x^2 of the
// next key and query tiles, outputs), 10..13 scan group (look-back, prefix
// operand).
//
// TMEM (512 columns):
//   [0, 64)    x^2 of K (hi | lo);  [64, 128) x^2 of Q;  both free once the
//              chunk's score MMAs are done: then [0, 80) holds U (M = 128:
//              hi-part rows 0..63, lo-part rows 64..127; N = 80 = [V | 1])
//   [128, 256) key scores (N = 64, first half), then P, then P hi | lo in place
//              per 32-key block
//   [256, 320) / [320, 384)  query scores (N = 64), then Gamma^Q hi | lo over
//              them; chunks alternate between the two, so a chunk's Gamma^Q
//              stays for its state read while the next chunk's is formed
//   [384, 464) [num | den] (N = 80)
// MMA issue order, chunk i:  U(i), P(i), state read(i - 1), P [V | 1](i),
// key scores(i + 1), query scores(i + 1).  The state read of a chunk comes one
// stage late, after the next chunk's P, so the look-back has about a chunk's
// time to finish before anything waits for it.
// MMAs per chunk: key scores 20, query scores 20 (five N = 64 products per
// K step, one accumulator), U 8, P 12 (N = 128), P [V | 1] 16, state read 12.
// Every MMA batch is unrolled with its operands a base plus constants.
namespace scan {
constexpr int kBlock = 4;              // chunks per look-back block
constexpr int kState4 = kKP * kW / 4;  // float4 of one [64][68] memory (1088)
constexpr int kQ4 = (kState4 + 127) / 128;  // float4 per key-group thread (9)
constexpr uint32_t kAggBit = 1u, kInclBit = 2u;
}  // namespace scan

struct ScanSmem {
    static constexpr int kQ = 0;                               // Q tile
    static constexpr int kK = kQ + kTileBytes;                 // K tile
    static constexpr int kV = kK + kTileBytes;                 // V tiles, 2 stages
    static constexpr int kOnes = kV + 2 * kTileBytes;          // ones columns of [V | 1] (2 KB)
    static constexpr int kGB = kOnes + 2048;                   // [Gamma^K ; S^T], 26 groups of 2 KB
    static constexpr int kGroups = (kTile + 80) / 8;
    static constexpr int kCoef = kGB + kGroups * 2048;
    static constexpr int kAgg = (kCoef + kCoefBytes + 1023) & ~1023;  // this chunk's increment [64][68] fp32
    static constexpr int kS = kAgg + kKP * kW * 4;             // exchange / prefix memory [64][68] fp32
    static constexpr int kStage = (kS + kKP * kW * 4 + 1023) & ~1023;  // output staging 4 x 8 KB
    static constexpr int kBars = kStage + 4 * 8192;
    static constexpr int kBytes = kBars + 256;
    static constexpr int kAlloc = kBytes + 1024;
    static_assert(kOnes % 1024 == 0 && kGB % 1024 == 0 && kCoef % 1024 == 0 && kStage % 1024 == 0, "SW128");
    static_assert(kAlloc <= 232448, "shared memory budget");
};

// Softmax of one N = 64 score row (s_k + c_k, max-subtracted exponentials) and
// the bf16 hi / lo split: key side (to_smem != 0): normalised (scale 0 for rows
// past N), written as row `row` of the [Gamma^K ; S^T] buffer; query side:
// un-normalised, hi words to t_out + 0..31 and lo words to t_out + 32..63.
// Returns the row sum of the exponentials.
__device__ __noinline__ float scan_softmax_row(uint32_t s_taddr, const float *cvec, int to_smem, uint32_t t_out,
                                               uint8_t *gb, int row, int valid) {
    uint32_t r0[32], r1[32];
    tmem_ld32(s_taddr, r0);
    tmem_ld32(s_taddr + 32, r1);
    tmem_wait_ld();
    tc_fence_before();
    float e[kKP];
    const float4 *c4 = reinterpret_cast<const float4 *>(cvec);
    float m0 = -INFINITY, m1 = -INFINITY;
#pragma unroll
    for (int q = 0; q < 8; ++q) {
        const float4 ca = c4[q], cb = c4[q + 8];
        const float2 a0 = f2_add(make_float2(__uint_as_float(r0[4 * q]), __uint_as_float(r0[4 * q + 1])),
                                 make_float2(ca.x, ca.y));
        const float2 a1 = f2_add(make_float2(__uint_as_float(r0[4 * q + 2]), __uint_as_float(r0[4 * q + 3])),
                                 make_float2(ca.z, ca.w));
        const float2 b0 = f2_add(make_float2(__uint_as_float(r1[4 * q]), __uint_as_float(r1[4 * q + 1])),
                                 make_float2(cb.x, cb.y));
        const float2 b1 = f2_add(make_float2(__uint_as_float(r1[4 * q + 2]), __uint_as_float(r1[4 * q + 3])),
                                 make_float2(cb.z, cb.w));
        e[4 * q] = a0.x; e[4 * q + 1] = a0.y; e[4 * q + 2] = a1.x; e[4 * q + 3] = a1.y;
        e[32 + 4 * q] = b0.x; e[32 + 4 * q + 1] = b0.y; e[32 + 4 * q + 2] = b1.x; e[32 + 4 * q + 3] = b1.y;
        m0 = fmaxf(m0, fmaxf(fmaxf(a0.x, a0.y), fmaxf(a1.x, a1.y)));
        m1 = fmaxf(m1, fmaxf(fmaxf(b0.x, b0.y), fmaxf(b1.x, b1.y)));
    }
    const float m = fmaxf(m0, m1);
    const float2 mm = make_float2(m, m);
    float2 s0 = make_float2(0.f, 0.f), s1 = make_float2(0.f, 0.f);
#pragma unroll
    for (int k = 0; k < kKP; k += 4) {
        const float2 d0 = f2_sub(make_float2(e[k], e[k + 1]), mm), d1 = f2_sub(make_float2(e[k + 2], e[k + 3]), mm);
        e[k] = ex2(d0.x); e[k + 1] = ex2(d0.y); e[k + 2] = ex2(d1.x); e[k + 3] = ex2(d1.y);
        s0 = f2_add(s0, make_float2(e[k], e[k + 1]));
        s1 = f2_add(s1, make_float2(e[k + 2], e[k + 3]));
    }
    const float rs = (s0.x + s0.y) + (s1.x + s1.y);
    uint32_t wh[32], wl[32];
    split_row(e, to_smem ? (valid ? 1.0f / rs : 0.0f) : 1.0f, wh, wl);
    if (to_smem) {
        store_gamma_words(gb, row, wh, wl);
    } else {
        tmem_st32(t_out, wh);
        tmem_st32(t_out + 32, wl);
        tmem_wait_st();
    }
    return rs;
}

// The chunk's memory increment out of the U accumulator: row `row` < 64 holds
// the hi-part sums of component row, row 64 + k the lo-part sums of component
// k (80 columns: 64 values, Z, zero padding).  Thread k keeps columns 0..31 of
// component k, thread 64 + k columns 32..64; the other half goes to the
// partner through Agg itself (each thread then reads back and overwrites only
// the half it owns).  After the key group's barrier each thread writes its
// columns of agg = hi + lo to Agg ([64][kW], shared) and to `gagg` (the
// chunk's published slot, same layout); the padding columns 65..67 are written
// as zeros.  `uread` is arrived on (lane 0) once U is in registers.
__device__ __noinline__ void scan_take_increment(uint32_t u_taddr, float *Agg, float *gagg, int row,
                                                 uint64_t *uread, int lane) {
    float *X = Agg;
    const int kc = row & (kKP - 1), half = row >> 6;
    uint32_t a0[32], a1[32], z[16];
    tmem_ld32(u_taddr, a0);
    tmem_ld32(u_taddr + 32, a1);
    tmem_ld16(u_taddr + 64, z);
    tmem_wait_ld();
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(uread);
    float *xr = X + kc * kW;
    if (half == 0) {
#pragma unroll
        for (int q = 0; q < 8; ++q)
            *reinterpret_cast<float4 *>(xr + 32 + 4 * q) =
                make_float4(__uint_as_float(a1[4 * q]), __uint_as_float(a1[4 * q + 1]),
                            __uint_as_float(a1[4 * q + 2]), __uint_as_float(a1[4 * q + 3]));
        xr[64] = __uint_as_float(z[0]);
    } else {
#pragma unroll
        for (int q = 0; q < 8; ++q)
            *reinterpret_cast<float4 *>(xr + 4 * q) =
                make_float4(__uint_as_float(a0[4 * q]), __uint_as_float(a0[4 * q + 1]),
                            __uint_as_float(a0[4 * q + 2]), __uint_as_float(a0[4 * q + 3]));
    }
    named_sync(1, 128);
    const uint32_t *own = half == 0 ? a0 : a1;
    float *ar = Agg + kc * kW + 32 * half;
    float *gr = gagg + kc * kW + 32 * half;
    const float *pr = xr + 32 * half;
#pragma unroll
    for (int q = 0; q < 8; ++q) {
        const float4 p = *reinterpret_cast<const float4 *>(pr + 4 * q);
        const float4 v = make_float4(__uint_as_float(own[4 * q]) + p.x, __uint_as_float(own[4 * q + 1]) + p.y,
                                     __uint_as_float(own[4 * q + 2]) + p.z, __uint_as_float(own[4 * q + 3]) + p.w);
        *reinterpret_cast<float4 *>(ar + 4 * q) = v;
        __stcg(reinterpret_cast<float4 *>(gr + 4 * q), v);
    }
    if (half) {
        const float4 v = make_float4(__uint_as_float(z[0]) + xr[64], 0.f, 0.f, 0.f);
        *reinterpret_cast<float4 *>(Agg + kc * kW + 64) = v;
        __stcg(reinterpret_cast<float4 *>(gagg + kc * kW + 64), v);
    }
}

__device__ __forceinline__ uint32_t ld_acquire_u32(const unsigned *p) {
    uint32_t v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ void st_release_u32(unsigned *p, uint32_t v) {
    asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// Bounded wait until the flag of chunk `t` carries `bit` (flag = (t + 1) << 2 |
// published bits).  Returns 0, or GMA_ERR_TIMEOUT when the wait runs out or
// the slot has been taken by a later chunk.
__device__ __noinline__ unsigned scan_wait_flag(const unsigned *flag, int t, uint32_t bit, const int *abort_flag) {
    const uint32_t want = (uint32_t)(t + 1);
    uint64_t t0 = 0;
    for (int spin = 0;; ++spin) {
        const uint32_t f = ld_acquire_u32(flag);
        if ((f >> 2) == want && (f & bit)) return 0u;
        if ((f >> 2) > want) return (unsigned)GMA_ERR_TIMEOUT;
        if ((spin & 255) == 255) {
            if (*reinterpret_cast<const volatile int *>(abort_flag)) return (unsigned)GMA_ERR_TIMEOUT;
            const uint64_t now = globaltimer();
            if (t0 == 0) t0 = now;
            else if (now - t0 > kWaitLimitNs) return (unsigned)GMA_ERR_TIMEOUT;
        }
    }
}

// Global state of the scan: flags [BH][R] and the published memories
// [BH][R][2][64][kW] fp32 (0: increment, 1: inclusive prefix), R = chunks per head.
struct ScanGlobal {
    unsigned *flags;
    float *ring;
    int R;
    __device__ __forceinline__ unsigned *flag(int bh, int t) const { return flags + (size_t)bh * R + (t % R); }
    __device__ __forceinline__ float *slot(int bh, int t, int kind) const {
        return ring + (((size_t)bh * R + (t % R)) * 2 + kind) * (size_t)(kKP * kW);
    }
};

// Prefix memory before chunk t of head bh, by the key group (128 threads):
// S = incl(base) + agg(base + 1) + ... + agg(t - 1), base the last chunk of the
// previous block (an empty prefix before the first block), in that order.
// The last chunk of a block then publishes incl(t) = S + agg(t).  S goes to
// the shared [64][kW] buffer.  Returns 0 or an error code (the same in every
// thread).
__device__ __noinline__ unsigned scan_lookback(const ScanGlobal &G, int bh, int t, int ntiles, const float *Agg,
                                               float *S, int tid, const int *abort_flag, unsigned *err_word,
                                               const CombineIO &io, int bar_id) {
    using namespace scan;
    const int base = (t / kBlock) * kBlock - 1;
    // thread j waits for one published memory: j = 0 the block base's prefix, j >= 1 increment base + j
    if (tid == 0) *err_word = 0u;
    named_sync(bar_id, 128);
    if (tid < t - base) {
        const int j = base + tid;
        unsigned e = 0u;
        if (tid == 0) {
            if (base >= 0) e = scan_wait_flag(G.flag(bh, base), base, kInclBit, abort_flag);
        } else {
            e = scan_wait_flag(G.flag(bh, j), j, kAggBit, abort_flag);
        }
        if (e) atomicOr(err_word, e);
    }
    named_sync(bar_id, 128);
    unsigned err = *reinterpret_cast<volatile unsigned *>(err_word);
    float4 acc[kQ4];
    if (!err) {
        const float4 *src0 = base >= 0 ? reinterpret_cast<const float4 *>(G.slot(bh, base, 1)) : nullptr;
#pragma unroll
        for (int q = 0; q < kQ4; ++q) {
            const int e4 = tid + 128 * q;
            // the first block starts from the caller's carried-in memory, if any
            acc[q] = e4 >= kState4 ? make_float4(0.f, 0.f, 0.f, 0.f)
                     : src0        ? __ldcg(src0 + e4)
                     : io.carry_vt ? io_load(io, bh, e4 / (kW / 4), 4 * (e4 % (kW / 4)))
                                   : make_float4(0.f, 0.f, 0.f, 0.f);
        }
        // increments base + 1 .. t - 1, two at a time (loads in flight together, sums in order)
        for (int j = base + 1; j < t; j += 2) {
            const bool two = j + 1 < t;
            const float4 *src0 = reinterpret_cast<const float4 *>(G.slot(bh, j, 0));
            const float4 *src1 = reinterpret_cast<const float4 *>(G.slot(bh, two ? j + 1 : j, 0));
            float4 v0[kQ4], v1[kQ4];
#pragma unroll
            for (int q = 0; q < kQ4; ++q) {
                const int e4 = tid + 128 * q;
                const bool in = e4 < kState4;
                v0[q] = in ? __ldcg(src0 + e4) : make_float4(0.f, 0.f, 0.f, 0.f);
                v1[q] = (in && two) ? __ldcg(src1 + e4) : make_float4(0.f, 0.f, 0.f, 0.f);
            }
#pragma unroll
            for (int q = 0; q < kQ4; ++q) {
                acc[q].x += v0[q].x; acc[q].y += v0[q].y; acc[q].z += v0[q].z; acc[q].w += v0[q].w;
                if (two) {
                    acc[q].x += v1[q].x; acc[q].y += v1[q].y; acc[q].z += v1[q].z; acc[q].w += v1[q].w;
                }
            }
        }
        // the slots read must still belong to the chunks they were read for
        if (tid < t - base && !(tid == 0 && base < 0)) {
            const int j = base + tid;
            const uint32_t f = ld_acquire_u32(G.flag(bh, j));
            if ((f >> 2) != (uint32_t)(j + 1)) atomicOr(err_word, (unsigned)GMA_ERR_TIMEOUT);
        }
    }
    const bool publish = (t % kBlock == kBlock - 1) && t + 1 < ntiles;
    const bool last_out = t + 1 == ntiles && io.out_vt;  // the memory after the last position, to the caller
    if (!err) {
        float4 *dst = publish ? reinterpret_cast<float4 *>(G.slot(bh, t, 1)) : nullptr;
#pragma unroll
        for (int q = 0; q < kQ4; ++q) {
            const int e4 = tid + 128 * q;
            if (e4 >= kState4) continue;
            reinterpret_cast<float4 *>(S)[e4] = acc[q];
            if (dst || last_out) {
                const float4 a = reinterpret_cast<const float4 *>(Agg)[e4];
                const float4 v = make_float4(acc[q].x + a.x, acc[q].y + a.y, acc[q].z + a.z, acc[q].w + a.w);
                if (dst) __stcg(dst + e4, v);
                if (last_out) io_store(io, bh, e4 / (kW / 4), 4 * (e4 % (kW / 4)), v);
            }
        }
    }
    // every thread's stores precede the barrier; thread 0's fence after it makes
    // them visible device-wide (cumulatively) before the flag
    named_sync(bar_id, 128);
    err = *reinterpret_cast<volatile unsigned *>(err_word);
    if (!err && publish && tid == 0) {
        __threadfence();
        st_release_u32(G.flag(bh, t), ((uint32_t)(t + 1) << 2) | kAggBit | kInclBit);
    }
    return err;
}

constexpr int kThreadsScan = 64 + 384;

__global__ void __launch_bounds__(kThreadsScan, 1) tc_scan_kernel(
    const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
    const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmO,
    const uint8_t *__restrict__ coef_img, const unsigned *__restrict__ head_err, ScanGlobal G, int H, int BH,
    int N, float eps, int o_bf16, int stall, CombineIO io, unsigned *status) {
    using L = ScanSmem;
    using namespace scan;
    constexpr int kTmemCols = 512;
    constexpr uint32_t kX = 0, kU = 0, kP = 128, kSK = kP, kSQ = 256, kO = 384;
    // query scores / Gamma^Q of chunk i: columns kSQ + 64 (i & 1)
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t *qst = smem + L::kQ, *kst = smem + L::kK, *vst = smem + L::kV, *gb = smem + L::kGB, *coef = smem + L::kCoef;
    float *Agg = reinterpret_cast<float *>(smem + L::kAgg), *S = reinterpret_cast<float *>(smem + L::kS);
    uint8_t *stg = smem + L::kStage;
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + L::kBars);
    uint64_t *qfull = bars, *qempty = bars + 1, *kfull = bars + 2, *kempty = bars + 3, *vfull = bars + 4,
             *vempty = bars + 6, *cfull = bars + 8, *cfree = bars + 9, *xk = bars + 10, *xq = bars + 11,
             *sk = bars + 12, *sq = bars + 13, *gk = bars + 14, *gq = bars + 15, *uf = bars + 16, *uread = bars + 17,
             *pf = bars + 18, *psplit = bars + 19, *of = bars + 20, *oread = bars + 21, *sready = bars + 22;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + 23);
    int *abort_flag = reinterpret_cast<int *>(bars + 24);
    unsigned *err_word = reinterpret_cast<unsigned *>(bars + 25);
    uint64_t *fin = bars + 26, *aggready = bars + 27, *aggfree = bars + 28;
    static_assert(29 * 8 <= 256, "barrier area");
    const float *cvec = reinterpret_cast<const float *>(coef + 4 * kCoefMatBytes);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int c = blockIdx.x, Gn = gridDim.x;
    const int ntiles = (N + kTile - 1) / kTile;
    const int total = BH * ntiles;
    const int n = c < total ? (total - c + Gn - 1) / Gn : 0;  // chunks of this CTA
    if (n == 0) return;

    if (warp == 0) {
        tmem_alloc(tmem_slot, kTmemCols);
        tmem_relinquish();
    }
    if (tid == 32) {
        mbar_init(qfull, 1); mbar_init(qempty, 1); mbar_init(kfull, 1); mbar_init(kempty, 1);
        mbar_init(&vfull[0], 1); mbar_init(&vfull[1], 1); mbar_init(&vempty[0], 1); mbar_init(&vempty[1], 1);
        mbar_init(cfull, 1); mbar_init(cfree, 8);
        mbar_init(xk, 4); mbar_init(xq, 4); mbar_init(sk, 1); mbar_init(sq, 1); mbar_init(gk, 4); mbar_init(gq, 4);
        mbar_init(uf, 1); mbar_init(uread, 4); mbar_init(pf, 1); mbar_init(psplit, 8); mbar_init(of, 1);
        mbar_init(oread, 4); mbar_init(sready, 4); mbar_init(fin, 1); mbar_init(aggready, 4); mbar_init(aggfree, 4);
        *abort_flag = 0;
        fence_mbar_init();
        tma_prefetch_desc(&tmQ); tma_prefetch_desc(&tmK); tma_prefetch_desc(&tmV); tma_prefetch_desc(&tmO);
    }
    {   // ones columns of [V | 1]; zero [Gamma^K ; S^T] (the S^T padding rows must be 0)
        const uint4 one4 = make_uint4(0x3F803F80u, 0x3F803F80u, 0x3F803F80u, 0x3F803F80u);
        for (int i = tid; i < 2048 / 16; i += kThreadsScan) reinterpret_cast<uint4 *>(smem + L::kOnes)[i] = one4;
        for (int i = tid; i < L::kGroups * 2048 / 16; i += kThreadsScan)
            reinterpret_cast<uint4 *>(gb)[i] = make_uint4(0, 0, 0, 0);
    }
    // Everything below reads the coefficient prep's output (images, error words,
    // cleared status and flags): wait for it, then let the next kernel launch.
    pdl_wait();
    pdl_trigger();
    {
        const unsigned herr = warp == 1 ? head_error_warp(head_err, H, lane) : 0u;
        if (tid == 32 && (herr || failed(status))) {
            if (herr) set_status(status, herr);
            *abort_flag = 1;
        }
    }
    tc_fence_before();
    cta_sync();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (!aborted(abort_flag)) {
        if (warp == 0) {
            if (lane == 0) {
                // ---------------- TMA: per chunk K, Q, V (2 stages), then the head's coefficients
                int karm = -1, qarm = -1, varm[2] = {-1, -1}, carm = -1;
                for (int i = 0; i < n; ++i) {
                    const int g = c + i * Gn, t = g / BH, bh = g % BH, h = bh % H;
                    if (!wait_or_abort(kempty, (i & 1) ^ 1, status, abort_flag)) break;
                    if (!(stall && i == 0)) {  // test hook: the first key tile is never loaded
                        mbar_arrive_expect_tx(kfull, kTileBytes);
                        tma_load_3d(kst, &tmK, 0, t * kTile, bh, kfull);
                        karm = i;
                    }
                    if (!wait_or_abort(qempty, (i & 1) ^ 1, status, abort_flag)) break;
                    mbar_arrive_expect_tx(qfull, kTileBytes);
                    tma_load_3d(qst, &tmQ, 0, t * kTile, bh, qfull);
                    qarm = i;
                    const int vs = i & 1;
                    if (!wait_or_abort(&vempty[vs], ((i >> 1) & 1) ^ 1, status, abort_flag)) break;
                    mbar_arrive_expect_tx(&vfull[vs], kTileBytes);
                    tma_load_3d(vst + vs * kTileBytes, &tmV, 0, t * kTile, bh, &vfull[vs]);
                    varm[vs] = i;
                    if (i > 0 && !wait_or_abort(cfree, (i - 1) & 1, status, abort_flag)) break;
                    mbar_arrive_expect_tx(cfull, kCoefBytes);
                    bulk_load(coef, coef_img + (size_t)h * kCoefStride, kCoefBytes, cfull);
                    carm = i;
                }
                // every load armed here has landed before the CTA leaves
                if (karm >= 0) mbar_wait(kfull, karm & 1);
                if (qarm >= 0) mbar_wait(qfull, qarm & 1);
                for (int s = 0; s < 2; ++s)
                    if (varm[s] >= 0) mbar_wait(&vfull[s], (varm[s] >> 1) & 1);
                if (carm >= 0) mbar_wait(cfull, carm & 1);
            }
        } else if (warp == 1) {
            if (lane == 0) {
                // ---------------- MMA issue, a fixed order per chunk i:
                //   U(i), P(i), P [V|1](i), key scores(i+1), state read(i), query scores(i+1)
                // (chunk 0's scores first).  Each batch waits for its inputs.
                const uint64_t dq = sdesc_sw128(smem_u32(qst), 16, 1024), dk = sdesc_sw128(smem_u32(kst), 16, 1024);
                const uint64_t dc = sdesc_sw128(smem_u32(coef), 16, 1024);
                const uint64_t dbh = sdesc_sw128(smem_u32(gb), 16, 2048), dbl = dadd(dbh, 1024);
                const uint64_t dsh = dadd(dbh, (kTile / 8) * 2048), dsl = dadd(dsh, 1024);
                const uint64_t dgt = sdesc_sw128(smem_u32(gb), 1024, 2048);
                // MN-major [V | 1] of V stage s: step kk is step 0 plus a constant (start + 2048 kk
                // bytes, LBO - 2048 kk bytes; the stages lie below the ones block)
                auto dv0 = [&](int s) {
                    const uint32_t a = smem_u32(vst + s * kTileBytes);
                    return sdesc_sw128(a, smem_u32(smem + L::kOnes) - a, 1024);
                };
                constexpr uint64_t kDvStep = 128ull - (128ull << 16);
                constexpr uint32_t i64 = idesc_bf16(kTile, 64, false, false), i128 = idesc_bf16(kTile, 128, false, false);
                constexpr uint32_t i80 = idesc_bf16(kTile, 80, false, false), i80s = idesc_bf16(kTile, 80, false, true),
                                   i80u = idesc_bf16(kTile, 80, true, true);
                // five N = 64 products per K step: x2hi a_hi, x2hi a_lo, x2lo a_hi, x b_hi, x b_lo
                auto scores = [&](uint32_t d, uint32_t x2, uint64_t dx) {
#pragma unroll
                    for (int kk = 0; kk < kDR / 16; ++kk) {
                        const uint32_t o = kk * 32;
                        umma_bf16_tA(d, x2 + kk * 8, dadd(dc, o), i64, kk > 0 ? 1u : 0u);
                        umma_bf16_tA(d, x2 + kk * 8, dadd(dc, kCoefMatBytes + o), i64, 1u);
                        umma_bf16_tA(d, x2 + 32 + kk * 8, dadd(dc, o), i64, 1u);
                        umma_bf16(d, dadd(dx, o), dadd(dc, 2 * kCoefMatBytes + o), i64, 1u);
                        umma_bf16(d, dadd(dx, o), dadd(dc, 3 * kCoefMatBytes + o), i64, 1u);
                    }
                };
                auto key_scores = [&](int i) {
                    if (!wait_or_abort(cfull, i & 1, status, abort_flag)) return false;
                    if (!wait_or_abort(xk, i & 1, status, abort_flag)) return false;
                    tc_fence_after();
                    scores(tmem + kSK, tmem + kX, dk);
                    umma_commit(sk);
                    umma_commit(kempty);
                    return true;
                };
                auto query_scores = [&](int i) {
                    if (!wait_or_abort(xq, i & 1, status, abort_flag)) return false;
                    tc_fence_after();
                    scores(tmem + kSQ + 64 * (i & 1), tmem + kX + 64, dq);
                    umma_commit(sq);
                    umma_commit(qempty);
                    return true;
                };
                // [num | den] += gQhi S^T_hi + gQhi S^T_lo + gQlo S^T_hi (the prefix memory of chunk j)
                auto state_read = [&](int j) {
                    if (!wait_or_abort(sready, j & 1, status, abort_flag)) return false;
                    tc_fence_after();
#pragma unroll
                    for (int kk = 0; kk < kKP / 16; ++kk) {
                        const uint32_t aq = tmem + kSQ + 64 * (j & 1) + kk * 8;
                        umma_bf16_tA(tmem + kO, aq, dadd(dsh, kk * 32), i80, 1u);
                        umma_bf16_tA(tmem + kO, aq, dadd(dsl, kk * 32), i80, 1u);
                        umma_bf16_tA(tmem + kO, aq + 32, dadd(dsh, kk * 32), i80, 1u);
                    }
                    umma_commit(of);
                    return true;
                };
                bool ok = key_scores(0) && query_scores(0);
                for (int i = 0; ok && i < n; ++i) {
                    const int vs = i & 1;
                    // U = [gK_hi ; gK_lo]^T [V | 1] into the x^2 columns (the scores have read them)
                    if (!(ok = wait_or_abort(gk, i & 1, status, abort_flag))) break;
                    if (!(ok = wait_or_abort(&vfull[vs], (i >> 1) & 1, status, abort_flag))) break;
                    tc_fence_after();
                    {
                        const uint64_t b0 = dv0(vs);
#pragma unroll
                        for (int kk = 0; kk < kTile / 16; ++kk)
                            umma_bf16(tmem + kU, dadd(dgt, kk * 4096), b0 + kk * kDvStep, i80u, kk > 0 ? 1u : 0u);
                    }
                    umma_commit(uf);
                    // P = gQhi gKhi^T + gQhi gKlo^T + gQlo gKhi^T
                    if (!(ok = wait_or_abort(gq, i & 1, status, abort_flag))) break;
                    tc_fence_after();
#pragma unroll
                    for (int kk = 0; kk < kKP / 16; ++kk) {
                        const uint32_t aq = tmem + kSQ + 64 * (i & 1) + kk * 8;
                        umma_bf16_tA(tmem + kP, aq, dadd(dbh, kk * 32), i128, kk > 0 ? 1u : 0u);
                        umma_bf16_tA(tmem + kP, aq, dadd(dbl, kk * 32), i128, 1u);
                        umma_bf16_tA(tmem + kP, aq + 32, dadd(dbh, kk * 32), i128, 1u);
                    }
                    umma_commit(pf);
                    // the previous chunk's prefix read (its look-back has had this chunk's key and
                    // query sides to finish)
                    if (i > 0 && !(ok = state_read(i - 1))) break;
                    // [num | den] = P [V | 1] (P hi / lo in place: key block cb = kk / 2 holds hi
                    // words at 32 cb, lo words at 32 cb + 16); the previous outputs are read
                    if (!(ok = wait_or_abort(psplit, i & 1, status, abort_flag))) break;
                    if (i > 0 && !(ok = wait_or_abort(oread, (i - 1) & 1, status, abort_flag))) break;
                    tc_fence_after();
                    {
                        const uint64_t b0 = dv0(vs);
#pragma unroll
                        for (int kk = 0; kk < kTile / 16; ++kk) {
                            const uint32_t ap = tmem + kP + 32 * (kk >> 1) + 8 * (kk & 1);
                            umma_bf16_tA(tmem + kO, ap, b0 + kk * kDvStep, i80s, kk > 0 ? 1u : 0u);
                            umma_bf16_tA(tmem + kO, ap + 16, b0 + kk * kDvStep, i80s, 1u);
                        }
                    }
                    umma_commit(&vempty[vs]);
                    if (i + 1 < n && !(ok = key_scores(i + 1))) break;
                    if (i + 1 < n && !(ok = query_scores(i + 1))) break;
                }
                if (ok) ok = state_read(n - 1);
                // every MMA issued has completed before the CTA frees its tensor memory
                umma_commit(fin);
                mbar_wait(fin, 0);
            }
        } else if (warp < 6) {
            // ---------------- key group
            const int row = epi_row(warp, lane), kt = tid - 64;
            const uint32_t lb = (uint32_t)(32 * (warp & 3)) << 16;
            if (wait_or_abort(kfull, 0, status, abort_flag)) {
                x2_row(kst, row, tmem + lb + kX);
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(xk);
            }
            for (int i = 0; i < n && !aborted(abort_flag); ++i) {
                const int g = c + i * Gn, t = g / BH, bh = g % BH;
                // key softmax -> Gamma^K (normalised, zero past N) into the [Gamma^K ; S^T] buffer
                if (!wait_or_abort(sk, i & 1, status, abort_flag)) break;
                if (!wait_or_abort(cfull, i & 1, status, abort_flag)) break;
                tc_fence_after();
                scan_softmax_row(tmem + lb + kSK, cvec, 1, 0u, gb, row, t * kTile + row < N);
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive(gk);
                    mbar_arrive(cfree);
                }
                // masked intra-chunk affinity, key blocks 2 and 3 -> P hi | lo (in place); U was
                // issued before P, so its result is ready by now too
                if (!wait_or_abort(pf, i & 1, status, abort_flag)) break;
                tc_fence_after();
                split_p_blocks(tmem + lb + kP, 2, row);
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(psplit);
                // the increment U: into Agg (once the scan group has read the previous one) and the
                // chunk's published slot
                if (!wait_or_abort(uf, i & 1, status, abort_flag)) break;
                if (i > 0 && !wait_or_abort(aggfree, (i - 1) & 1, status, abort_flag)) break;
                tc_fence_after();
                scan_take_increment(tmem + lb + kU, Agg, G.slot(bh, t, 0), row, uread, lane);
                // every thread's stores precede the barrier; thread 0's fence after it makes them
                // visible device-wide (cumulatively) before the flag
                named_sync(1, 128);
                if (kt == 0) {
                    __threadfence();
                    st_release_u32(G.flag(bh, t), ((uint32_t)(t + 1) << 2) | kAggBit);
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(aggready);
            }
        } else if (warp >= 10) {
            // ---------------- scan group: prefix memory before each chunk -> S, then its
            // bf16 hi / lo operand (S^T rows)
            const int st = tid - 320;
            for (int i = 0; i < n && !aborted(abort_flag); ++i) {
                const int g = c + i * Gn, t = g / BH, bh = g % BH;
                if (!wait_or_abort(aggready, i & 1, status, abort_flag)) break;
                const unsigned e = scan_lookback(G, bh, t, ntiles, Agg, S, st, abort_flag, err_word, io, 3);
                __syncwarp();
                if (lane == 0) mbar_arrive(aggfree);  // Agg has been read
                if (e) {
                    note_timeout(status, abort_flag);
                    break;
                }
                // the previous chunk's state read has read its operand rows
                if (i > 0 && !wait_or_abort(of, (i - 1) & 1, status, abort_flag)) break;
                named_sync(3, 128);
                state_operand(gb, S, st);
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(sready);
            }
        } else {
            // ---------------- query group
            const int row = epi_row(warp, lane);
            const uint32_t lb = (uint32_t)(32 * (warp & 3)) << 16;
            uint8_t *stage = stg + (warp & 3) * 8192;
            float rq_prev = 0.f;
            int t_prev = 0, bh_prev = 0, n_out = 0;
            // outputs of chunk j: O = num / (den + eps r), staged and stored by TMA
            auto scan_output = [&](uint32_t o_taddr, float r, int tj, int bhj) {
                if (!wait_or_abort(of, n_out & 1, status, abort_flag)) return false;
                ++n_out;
                tc_fence_after();
                stage_output_row(o_taddr, r, eps, stage, lane, o_bf16, oread);
                __syncwarp();
                if (lane == 0) {
                    const int row0 = tj * kTile + 32 * (warp & 3);
                    tma_store_3d(&tmO, stage, 0, row0, bhj);
                    if (!o_bf16) tma_store_3d(&tmO, stage + 4096, 32, row0, bhj);
                    bulk_commit();
                }
                return true;
            };
            if (wait_or_abort(qfull, 0, status, abort_flag)) {
                x2_row(qst, row, tmem + lb + kX + 64);
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(xq);
            }
            for (int i = 0; i < n && !aborted(abort_flag); ++i) {
                const int g = c + i * Gn, t = g / BH, bh = g % BH;
                // query softmax -> Gamma^Q hi | lo (un-normalised) over the score columns
                if (!wait_or_abort(sq, i & 1, status, abort_flag)) break;
                if (!wait_or_abort(cfull, i & 1, status, abort_flag)) break;
                tc_fence_after();
                const uint32_t sqc = tmem + lb + kSQ + 64 * (i & 1);
                const float rq = scan_softmax_row(sqc, cvec, 0, sqc, nullptr, row, 1);
                tc_fence_before();
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive(gq);
                    mbar_arrive(cfree);
                }
                // masked intra-chunk affinity, key blocks 0 and 1 -> P hi | lo (in place)
                if (!wait_or_abort(pf, i & 1, status, abort_flag)) break;
                tc_fence_after();
                split_p_blocks(tmem + lb + kP, 0, row);
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(psplit);
                // x^2 of the next key and query tiles (their columns are free once the increment
                // is read out)
                if (i + 1 < n) {
                    if (!wait_or_abort(uread, i & 1, status, abort_flag)) break;
                    if (!wait_or_abort(kfull, (i + 1) & 1, status, abort_flag)) break;
                    tc_fence_after();
                    x2_row(kst, row, tmem + lb + kX);
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(xk);
                    if (!wait_or_abort(qfull, (i + 1) & 1, status, abort_flag)) break;
                    x2_row(qst, row, tmem + lb + kX + 64);
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(xq);
                }
                // outputs of the previous chunk (its state read follows this chunk's P)
                if (i > 0 && !scan_output(tmem + lb + kO, rq_prev, t_prev, bh_prev)) break;
                rq_prev = rq;
                t_prev = t;
                bh_prev = bh;
            }
            if (!aborted(abort_flag)) scan_output(tmem + lb + kO, rq_prev, t_prev, bh_prev);
            if (lane == 0) bulk_wait_read0();  // staging reusable; kernel completion publishes the stores
        }
    }
    tc_fence_before();
    cta_sync();
    if (warp == 0) tmem_dealloc(tmem, kTmemCols);
}

// ------------------------------------------------------------------ host side


// [BH][N][d] bf16 tensor (d = 32 or 64), boxes of 64 columns x 128 rows x 1
// head, 128-byte swizzle; rows past N and columns past d read as zero (so a
// d = 32 tile arrives zero-padded to the 64-column layout the kernels use).
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

// O [BH][N][64] (fp32 or bf16) for TMA stores of 32-row boxes, 128-byte swizzle.
bool make_out_map(CUtensorMap *map, void *base, int BH, int N, bool bf16) {
    auto fn = encode_fn();
    if (!fn) return false;
    const int es = bf16 ? 2 : 4;
    cuuint64_t dims[3] = {64, (cuuint64_t)N, (cuuint64_t)BH};
    cuuint64_t strides[2] = {(cuuint64_t)64 * es, (cuuint64_t)N * 64 * es};
    cuuint32_t box[3] = {(cuuint32_t)(128 / es), 32, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = fn(map, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, base, dims,
                    strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// O [BH][N][64] (fp32 or bf16) for TMA stores of [32 rows x 32 columns]
// boxes: 128-byte swizzle for fp32, 64-byte swizzle for bf16.
bool make_out_map_half(CUtensorMap *map, void *base, int BH, int N, bool bf16) {
    auto fn = encode_fn();
    if (!fn) return false;
    const int es = bf16 ? 2 : 4;
    cuuint64_t dims[3] = {64, (cuuint64_t)N, (cuuint64_t)BH};
    cuuint64_t strides[2] = {(cuuint64_t)64 * es, (cuuint64_t)N * 64 * es};
    cuuint32_t box[3] = {32, 32, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = fn(map, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, base, dims,
                    strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                    bf16 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_NONE,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}


// Workspace of the persistent kernels: status | per-head job counters |
// per-block parameter-error words of the coefficient prep | per-head coefficient images | job partials
// [ctas][slots][KP][kW] | per-head read operand images | (causal) Gamma^K of every key tile.  Nothing needs
// clearing by the caller: coef_prep_tc_kernel resets the status word and the
// counters, and writes every error word.
struct TcLayout2 {
    Part P;
    int nctas = 0;
    size_t counters = 0, head_err = 0, coef = 0, part = 0, mem = 0, mem_stride = 0, gk = 0, total = 0;
};

// End of the range that starts at tile a when a range may cost m (tiles, plus
// kSwitchTiles per head boundary crossed); at least one tile.  The rest of a's
// head first, then as many whole heads as the budget pays for (each its tiles
// plus the switch), then part of one more head if the budget left exceeds the
// switch: constant time, so the cuts of a call cost O(CTAs) per search step
// whatever the number of heads.
int range_end(int a, int ntiles, int total, long long m) {
    const int head_end = (a / ntiles + 1) * ntiles;
    const long long first = std::min<long long>(m, head_end - a);
    long long b = a + first, left = m - first;
    if (left <= 0 || b >= total) return b > a ? (int)b : a + 1;
    const long long whole = left / (kSwitchTiles + ntiles), heads_left = (total - b) / ntiles;
    if (whole >= heads_left) return total;
    b += whole * ntiles;
    left -= whole * (kSwitchTiles + ntiles);
    if (left > kSwitchTiles) b += left - kSwitchTiles;  // < ntiles: part of the next head
    return (int)b;
}

// Cuts with the smallest largest range cost that needs at most nct ranges
// (binary search on the cost, greedy ranges); the slot count is the largest
// number of heads a range touches.
void part_cuts(Part *P, int ntiles, int total, int nct) {
    P->ntiles = ntiles;
    P->total = total;
    const long long heads = (total + ntiles - 1) / ntiles;
    long long lo = (total + nct - 1) / nct, hi = total + kSwitchTiles * heads;
    auto count = [&](long long m) {
        int n = 0;
        for (int a = 0; a < total; a = range_end(a, ntiles, total, m)) ++n;
        return n;
    };
    while (lo < hi) {
        const long long mid = (lo + hi) / 2;
        if (count(mid) <= nct) hi = mid; else lo = mid + 1;
    }
    int n = 0, slots = 1;
    for (int a = 0; a < total;) {
        const int b = range_end(a, ntiles, total, lo);
        P->start[n++] = a;
        slots = std::max(slots, (b - 1) / ntiles - a / ntiles + 1);
        a = b;
    }
    P->start[n] = total;
    P->nctas = n;
    P->slots = slots;
}

TcLayout2 tc_layout2(const Problem &p, int splits, int causal) {
    TcLayout2 L;
    const int ntiles = (p.N + kTile - 1) / kTile;
    const int total = p.BH() * ntiles;
    int nct = splits > 0 ? splits : num_sms();
    nct = nct < 1 ? 1 : (nct > total ? total : nct);
    nct = nct > kMaxPartCtas ? kMaxPartCtas : nct;
    part_cuts(&L.P, ntiles, total, nct);
    L.nctas = L.P.nctas;
    size_t off = kStatusBytes;
    L.counters = off;
    off = align256(off + sizeof(unsigned) * (size_t)p.BH());
    L.head_err = off;
    off = align256(off + sizeof(unsigned) * (size_t)p.H * kPrepBlocks);
    L.coef = off;
    off = align256(off + kCoefStride * p.H);
    L.part = off;
    off = align256(off + sizeof(float) * (size_t)L.nctas * L.P.slots * kKP * kW);
    L.mem_stride = ((size_t)2 * (p.d_v + 16) * 128 + 1023) & ~size_t(1023);
    L.mem = off;
    off = align256(off + L.mem_stride * p.BH());
    if (causal == 1) {  // Gamma^K of every key tile (bf16 hi / lo), from the aggregation to the scan
        L.gk = off;
        off = align256(off + (size_t)2 * kTileBytes * p.BH() * ntiles);
    }
    L.total = off;
    return L;
}

// Workspace of the single-pass causal scan: status | per-block parameter-error
// words | per-head coefficient images | look-back flags [BH][R] | published
// memories [BH][R][2][64][kW] fp32 (R = chunks per head).  coef_prep_tc_kernel clears the
// status word and the flags; every other region is written before it is read.
struct ScanLayout {
    int R = 0, grid = 0;
    size_t head_err = 0, coef = 0, flags = 0, ring = 0, total = 0;
};

ScanLayout scan_layout(const Problem &p, int splits) {
    ScanLayout L;
    const int ntiles = (p.N + kTile - 1) / kTile;
    // one slot per chunk: a slot is written once per call, so no reader can see
    // it change under it (a ring of fewer slots is only safe while no chunk lags
    // the chunks that reuse its slot, which nothing guarantees)
    L.R = ntiles;
    const long long total = (long long)p.BH() * ntiles;
    long long g = splits > 0 ? splits : num_sms();
    L.grid = (int)(g < total ? g : total);
    size_t off = kStatusBytes;
    L.head_err = off;
    off = align256(off + sizeof(unsigned) * (size_t)p.H * kPrepBlocks);
    L.coef = off;
    off = align256(off + kCoefStride * p.H);
    L.flags = off;
    off = align256(off + sizeof(unsigned) * (size_t)p.BH() * L.R);
    L.ring = off;
    off = align256(off + sizeof(float) * (size_t)p.BH() * L.R * 2 * kKP * kW);
    L.total = off;
    return L;
}

// The causal call on the single-pass kernel: coefficient prep (which also
// clears the look-back flags), then the scan.
// io.carry_vt: the prefix starts from the caller's memory; io.out_vt: the
// prefix after the last position is written there.
cudaError_t run_scan(const Problem &p, const ScanLayout &L, uint8_t *ws, cudaStream_t s, StageClock &clk,
                     CombineIO io = CombineIO{nullptr, nullptr, nullptr, nullptr, 0}) {
    unsigned *status = reinterpret_cast<unsigned *>(ws);
    unsigned *head_err = reinterpret_cast<unsigned *>(ws + L.head_err);
    unsigned *flags = reinterpret_cast<unsigned *>(ws + L.flags);
    uint8_t *coef = ws + L.coef;
    CUtensorMap tq, tk, tv, to;
    if (!make_map(&tq, p.Q, p.BH(), p.N, p.d_r) || !make_map(&tk, p.Kx, p.BH(), p.N, p.d_r) ||
        !make_map(&tv, p.V, p.BH(), p.N, 64) || !make_out_map(&to, p.O, p.BH(), p.N, p.o_bf16))
        return cudaErrorInvalidValue;
    clk.mark();
    GMA_TRY(launch_pdl(coef_prep_tc_kernel, dim3(kPrepBlocks, p.H), dim3(128), 0, s, p.mu, p.sigma2, p.log_pi, p.K,
                       p.d_r, coef, status, head_err, flags, p.BH() * L.R));
    clk.mark();
    GMA_TRY(set_smem(tc_scan_kernel, ScanSmem::kAlloc));
    const ScanGlobal G{flags, reinterpret_cast<float *>(ws + L.ring), L.R};
    GMA_TRY(launch_pdl(tc_scan_kernel, dim3(L.grid), dim3(kThreadsScan), ScanSmem::kAlloc, s, tq, tk, tv, to,
                       static_cast<const uint8_t *>(coef), static_cast<const unsigned *>(head_err), G, p.H, p.BH(),
                       p.N, p.eps, p.o_bf16 ? 1 : 0, p.test_stall ? 1 : 0, io, status));
    clk.mark();
    return cudaSuccess;
}

// Read operand image of a caller's memory [Vt | Z] (fp32) for each head, the
// same bf16 hi | lo layout the combine builds: row n < 64 holds Vt[:, n], row 64
// Z, rows 65 .. 79 zero; column k of every row is component k (zero past K).
// It is the first kernel of its call after the coefficient prep, so its first
// warp also turns the prep's parameter checks into the call's status (the read
// kernel then returns at once).
__global__ void __launch_bounds__(256) pack_memory_tc_kernel(const float *__restrict__ Vt, const float *__restrict__ Z,
                                                             int K, uint8_t *__restrict__ mem, size_t stride,
                                                             const unsigned *__restrict__ head_err, int H,
                                                             unsigned *status) {
    constexpr int NBR = 64 + 16;
    const int bh = blockIdx.x;
    if (bh == 0 && threadIdx.x < 32) {
        const unsigned herr = head_error_warp(head_err, H, threadIdx.x);
        if (herr && threadIdx.x == 0) set_status(status, herr);
    }
    __nv_bfloat16 *bhi = reinterpret_cast<__nv_bfloat16 *>(mem + (size_t)bh * stride);
    __nv_bfloat16 *blo = reinterpret_cast<__nv_bfloat16 *>(mem + (size_t)bh * stride + NBR * 128);
    for (int e = threadIdx.x; e < NBR * kKP; e += blockDim.x) {
        const int n = e / kKP, k = e % kKP;
        const float v = k >= K  ? 0.f
                        : n < 64 ? Vt[((size_t)bh * K + k) * 64 + n]
                        : n == 64 ? Z[(size_t)bh * K + k]
                                  : 0.f;
        const __nv_bfloat16 vh = __float2bfloat16_rn(v);
        const uint32_t off = sw128_offset(n, k, 1024) / 2;
        bhi[off] = vh;
        blo[off] = __float2bfloat16_rn(v - __bfloat162float(vh));
    }
}

// The bidirectional call: coefficient prep, the key side (write) and the query
// side (read).  io.out_vt: also the fp32 memory; read = false: stop after the
// write (the latent memory alone); pack_from: read the caller's memory
// (io.carry_vt / carry_z) instead of writing one.
cudaError_t run_bidir2(const Problem &p, const TcLayout2 &L, uint8_t *ws, cudaStream_t s, StageClock &clk,
                       CombineIO io = CombineIO{nullptr, nullptr, nullptr, nullptr, 0}, bool read = true,
                       bool pack_from = false) {
    unsigned *status = reinterpret_cast<unsigned *>(ws);
    unsigned *counters = reinterpret_cast<unsigned *>(ws + L.counters);
    float *part = reinterpret_cast<float *>(ws + L.part);
    uint8_t *mem = ws + L.mem;
    uint8_t *coef = ws + L.coef;
    CUtensorMap tq, tk, tv, to;
    if (!make_map(&tq, p.Q, p.BH(), p.N, p.d_r) || !make_map(&tk, p.Kx, p.BH(), p.N, p.d_r) ||
        !make_map(&tv, p.V, p.BH(), p.N, 64) || !make_out_map_half(&to, p.O, p.BH(), p.N, p.o_bf16))
        return cudaErrorInvalidValue;
    unsigned *head_err = reinterpret_cast<unsigned *>(ws + L.head_err);
    clk.mark();
    GMA_TRY(launch_pdl(coef_prep_tc_kernel, dim3(kPrepBlocks, p.H), dim3(128), 0, s, p.mu, p.sigma2, p.log_pi, p.K,
                       p.d_r, coef, status, head_err, counters, p.BH()));
    clk.mark();
    if (pack_from) {
        // after the prep (a plain launch: the read's dependent-launch wait then
        // covers both), so the read sees the coefficients and the operand images
        pack_memory_tc_kernel<<<p.BH(), 256, 0, s>>>(io.carry_vt, io.carry_z, p.K, mem, L.mem_stride, head_err, p.H,
                                                     status);
        GMA_TRY(cudaGetLastError());
    } else {
        GMA_TRY(set_smem(tc_write2_kernel, Write2Smem::kAlloc));
        GMA_TRY(launch_pdl(tc_write2_kernel, dim3(L.nctas), dim3(kThreadsG), Write2Smem::kAlloc, s, tk, tv, coef,
                           head_err, p.H, p.N, L.P, part, counters, mem, L.mem_stride, static_cast<uint8_t *>(nullptr),
                           0, p.test_stall ? 1 : 0, io, status));
    }
    clk.mark();
    if (!read) return cudaSuccess;
    GMA_TRY(set_smem(tc_read3_kernel, Read3Smem::kAlloc));
    GMA_TRY(launch_pdl(tc_read3_kernel, dim3(L.nctas), dim3(kThreadsR), Read3Smem::kAlloc, s, tq, to, coef, p.H, p.N,
                       L.P, mem, L.mem_stride, p.eps, p.o_bf16 ? 1 : 0, status));
    clk.mark();
    return cudaSuccess;
}

// The causal call: coefficient prep, aggregation (job prefixes, stored Gamma^K)
// and the chunk scan.  io.carry_vt: the prefix starts from the caller's memory;
// io.out_vt: the prefix after the last position is written there.
cudaError_t run_causal2(const Problem &p, const TcLayout2 &L, uint8_t *ws, cudaStream_t s, StageClock &clk,
                        CombineIO io = CombineIO{nullptr, nullptr, nullptr, nullptr, 0}) {
    unsigned *status = reinterpret_cast<unsigned *>(ws);
    unsigned *counters = reinterpret_cast<unsigned *>(ws + L.counters);
    float *part = reinterpret_cast<float *>(ws + L.part);
    uint8_t *coef = ws + L.coef;
    CUtensorMap tq, tk, tv, to;
    if (!make_map(&tq, p.Q, p.BH(), p.N, p.d_r) || !make_map(&tk, p.Kx, p.BH(), p.N, p.d_r) ||
        !make_map(&tv, p.V, p.BH(), p.N, 64) || !make_out_map(&to, p.O, p.BH(), p.N, p.o_bf16))
        return cudaErrorInvalidValue;
    unsigned *head_err = reinterpret_cast<unsigned *>(ws + L.head_err);
    clk.mark();
    GMA_TRY(launch_pdl(coef_prep_tc_kernel, dim3(kPrepBlocks, p.H), dim3(128), 0, s, p.mu, p.sigma2, p.log_pi, p.K,
                       p.d_r, coef, status, head_err, counters, p.BH()));
    clk.mark();
    GMA_TRY(set_smem(tc_write2_kernel, Write2Smem::kAlloc));
    GMA_TRY(launch_pdl(tc_write2_kernel, dim3(L.nctas), dim3(kThreadsG), Write2Smem::kAlloc, s, tk, tv, coef, head_err,
                       p.H, p.N, L.P, part, counters, static_cast<uint8_t *>(nullptr), size_t(0), ws + L.gk, 1,
                       p.test_stall ? 1 : 0, io, status));
    clk.mark();
    GMA_TRY(set_smem(tc_causal2_kernel, Causal2Smem::kAlloc));
    GMA_TRY(launch_pdl(tc_causal2_kernel, dim3(L.nctas), dim3(kThreadsG), Causal2Smem::kAlloc, s, tq, tv, to, coef,
                       static_cast<const uint8_t *>(ws + L.gk), part, p.H, p.N, L.P, p.eps, p.o_bf16 ? 1 : 0, status));
    clk.mark();
    return cudaSuccess;
}

}  // namespace

const char *const kTcStages[3][8] = {
    {nullptr},
    {"prep", "tc_write", "tc_read", nullptr},
    {"prep", "tc_aggregate", "tc_causal", nullptr},
};

const char *const kTcScanStages[8] = {"prep", "tc_scan", nullptr};

const char *const kAuxTcStages[5][8] = {
    {"prep", "tc_write", nullptr},
    {nullptr},
    {nullptr},
    {"prep", "pack", "tc_read", nullptr},
    {"prep", "tc_aggregate", "tc_causal", nullptr},
};

bool tc_supported(const Problem &p, int causal) {
    if (p.dtype != GMA_BF16 || (p.d_r != kDR && p.d_r != kDR / 2) || p.K > kKP) return false;
    if (causal == 0) return p.d_v == 64;
    return causal == 1 && p.d_v == 64;
}

int tc_partition(int ntiles, int total, int max_ctas, int *starts, int starts_len, int *switch_tiles) {
    if (ntiles < 1 || total < 1 || total % ntiles != 0 || max_ctas < 1 || !starts) return -1;
    if (switch_tiles) *switch_tiles = kSwitchTiles;
    int nct = max_ctas > total ? total : max_ctas;
    nct = nct > kMaxPartCtas ? kMaxPartCtas : nct;
    Part P;
    part_cuts(&P, ntiles, total, nct);
    if (starts_len < P.nctas + 1) return -1;
    for (int i = 0; i <= P.nctas; ++i) starts[i] = P.start[i];
    return P.nctas;
}

size_t tc_workspace(const Problem &p, int causal, int splits) { return tc_layout2(p, splits, causal).total; }

size_t tc_carry_workspace(const Problem &p) { return tc_layout2(p, 0, 1).total; }

size_t tc_scan_workspace(const Problem &p, int splits) { return scan_layout(p, splits).total; }

cudaError_t tc_bidir(const Problem &p, int splits, void *ws, cudaStream_t s, StageClock &clk) {
    TcLayout2 L = tc_layout2(p, splits, 0);
    uint8_t *w = static_cast<uint8_t *>(ws);
    return run_bidir2(p, L, w, s, clk);
}

cudaError_t tc_causal(const Problem &p, int splits, void *ws, cudaStream_t s, StageClock &clk) {
    TcLayout2 L = tc_layout2(p, splits, 1);
    return run_causal2(p, L, static_cast<uint8_t *>(ws), s, clk);
}

cudaError_t tc_causal_1pass(const Problem &p, int splits, void *ws, cudaStream_t s, StageClock &clk) {
    return run_scan(p, scan_layout(p, splits), static_cast<uint8_t *>(ws), s, clk);
}

cudaError_t tc_latent_memory(const Problem &p, int splits, float *Vt, float *Z, void *ws, cudaStream_t s,
                             StageClock &clk) {
    TcLayout2 L = tc_layout2(p, splits, 0);
    return run_bidir2(p, L, static_cast<uint8_t *>(ws), s, clk, CombineIO{nullptr, nullptr, Vt, Z, p.K}, false);
}

cudaError_t tc_read_memory(const Problem &p, const float *Vt, const float *Z, void *ws, cudaStream_t s,
                           StageClock &clk) {
    TcLayout2 L = tc_layout2(p, 0, 0);
    return run_bidir2(p, L, static_cast<uint8_t *>(ws), s, clk, CombineIO{Vt, Z, nullptr, nullptr, p.K}, true,
                      true);
}

cudaError_t tc_causal_carry(const Problem &p, int splits, const float *Vt_in, const float *Z_in, float *Vt_out,
                            float *Z_out, void *ws, cudaStream_t s, StageClock &clk) {
    TcLayout2 L = tc_layout2(p, splits, 1);
    return run_causal2(p, L, static_cast<uint8_t *>(ws), s, clk, CombineIO{Vt_in, Z_in, Vt_out, Z_out, p.K});
}

cudaError_t tc_causal_carry_1pass(const Problem &p, int splits, const float *Vt_in, const float *Z_in,
                                  float *Vt_out, float *Z_out, void *ws, cudaStream_t s, StageClock &clk) {
    return run_scan(p, scan_layout(p, splits), static_cast<uint8_t *>(ws), s, clk,
                    CombineIO{Vt_in, Z_in, Vt_out, Z_out, p.K});
}

}  // namespace gma
