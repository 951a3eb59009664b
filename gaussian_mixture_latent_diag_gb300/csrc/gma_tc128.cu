// gma_tc128.cu -- tcgen05 tensor-core kernels for the causal GMA forward with
// d_r = d_v = 128 and K <= 128 components (bf16 inputs, fp32 accumulation).
//
// The numerics are those of the 64-wide kernels (gma_tc.cu): the log-density
// as a GEMM on the expanded quadratic ([GMA, Eqs. (2)-(3)]),
//   s_ik log2(e) = sum_j x_ij^2 a_kj + x_ij b_kj + c_k,
// with a, b split into bf16 hi + lo and x^2 = x2hi + x2lo exactly, so that the
// five products x2hi ahi + x2hi alo + x2lo ahi + x bhi + x blo carry ~16
// significant bits; the softmax over k in fp32 on the tensor-memory rows; and
// Gamma and the causal state split into bf16 hi + lo for the value
// contractions (hi.hi, hi.lo and lo.hi kept).
//
// At 128 components and 128 value columns every per-chunk operand is four
// times that of the 64-wide kernels, which sets the layout:
//   tc128_prep_kernel       per-head coefficient image: eight 16 KB slabs
//                           (a_hi, a_lo, b_hi, b_lo for routing columns 0-63,
//                           then for 64-127) streamed through a shared-memory
//                           ring by the score MMAs, and c_k.
//   tc128_aggregate_kernel  key side of every tile: Gamma^K, the memory
//                           increment Gamma^K^T V_X summed over each job (a
//                           contiguous tile range of one head), and the key
//                           mass (column sums of Gamma^K) of every tile; the
//                           last job of each head to finish turns the jobs'
//                           memories into exclusive prefixes, in job order.
//   tc128_causal_kernel     the chunked scan ([GMA, Eq. (8b)]), one 128-token
//                           chunk at a time: Gamma^Q, Gamma^K (recomputed, never
//                           stored), U = Gamma^Q Gamma^K^T masked to j <= i
//                           (P), num = P V_X + Gamma^Q S, S += Gamma^K^T V_X.
// The key mass enters only through the denominator:
//   Gamma^Q_i Z^(i) = e_i . Zp + sum_{j <= i in chunk} P_ij,
// with e_i the un-normalised query responsibilities and Zp the key mass before
// the chunk (fp32 sums from the aggregation), so the state needs no column of
// ones and fits in 128 tensor-memory columns.
//
// Paper: "Gaussian Mixture Attention: Linear-Time Sequence Mixing via
// Probabilistic Latent Routing" (arXiv 2606.18283), cited [GMA, ...].
#include <cuda.h>
#include <cuda_bf16.h>
#include <cudaTypedefs.h>

#include <cmath>

#include "gma_internal.h"
#include "tc_common.cuh"
#include "tc_ptx.cuh"

namespace gma {
namespace {

using namespace ptx;

constexpr int kT = 128;                  // tokens per tile / chunk (UMMA M)
constexpr int kD = 128;                  // d_r = d_v
constexpr int kKC = 128;                 // padded number of components
constexpr int kHalf = kT * 128;          // one [128 rows x 64 bf16] SW128 block (16 KB)
constexpr int kTileB = 2 * kHalf;        // a [128 x 128] bf16 tile as two column halves
constexpr int kSlab = kKC * 128;         // one coefficient slab [128 components x 64 columns] bf16
constexpr int kSlabs = 8;                // a_hi, a_lo, b_hi, b_lo of each column half
constexpr int kCoefC = kSlabs * kSlab;   // offset of c[128] (fp32) in a head's image
constexpr size_t kImgStride = kCoefC + 1024;
constexpr int kPrepBlocks128 = kKC / 8;
constexpr int kPartFloats = kKC * kD + kKC;  // a job's memory: S [128][128], then Z [128]
constexpr int kGroupB = 4096;            // Gamma buffer: bytes per 8-token group (hi|lo x 2 halves)
constexpr float kLog2e128 = 1.4426950408889634f;

// ------------------------------------------------------------------ coefficient prep
// Grid (KC / 8, H) x 128: block (b, h) writes components 8b .. 8b + 7 of head h's
// image.  Thread t takes component 8b + t / 16 and routing columns 8 (t % 16) ..
// + 7, writes them into the four slabs of their column half (K-major SW128 rows
// of 64 columns, one row per component) and, with the other 15 threads of its
// component, sums the log-determinant terms for c_k (-inf for padded
// components).  Parameter checks go to err[h * 16 + b].  Being the first kernel
// of a call, it also clears the status word and the per-head job counters.
__global__ void __launch_bounds__(128) tc128_prep_kernel(const float *__restrict__ mu,
                                                         const float *__restrict__ sigma2,
                                                         const float *__restrict__ log_pi, int K,
                                                         uint8_t *__restrict__ img, unsigned *status,
                                                         unsigned *head_err, unsigned *counters, int BH) {
    const int tid = threadIdx.x, h = blockIdx.y;
    const int gt = (blockIdx.y * gridDim.x + blockIdx.x) * blockDim.x + tid;
    uint8_t *coef = img + (size_t)h * kImgStride;
    const int k = blockIdx.x * 8 + (tid >> 4), j0 = (tid & 15) * 8;
    const bool realk = k < K;
    // The previous call's kernels may still read the status, counters and images,
    // and the kernel before this one may have written the parameters: they are read
    // only after the dependency wait, their lines brought into L2 meanwhile.
    if (realk) {
        prefetch_l2(sigma2 + ((size_t)h * K + k) * kD + j0);
        prefetch_l2(mu + ((size_t)h * K + k) * kD + j0);
        if ((tid & 15) == 0) prefetch_l2(log_pi + (size_t)h * K + k);
    }
    pdl_wait();
    pdl_trigger();
    if (gt == 0) *status = 0u;
    for (int i = gt; i < BH; i += gridDim.x * gridDim.y * blockDim.x) counters[i] = 0u;
    float sv[8], mv[8];
    if (realk) {
        const float4 *s4 = reinterpret_cast<const float4 *>(sigma2 + ((size_t)h * K + k) * kD + j0);
        const float4 *m4 = reinterpret_cast<const float4 *>(mu + ((size_t)h * K + k) * kD + j0);
        const float4 s0 = s4[0], s1 = s4[1], m0 = m4[0], m1 = m4[1];
        sv[0] = s0.x; sv[1] = s0.y; sv[2] = s0.z; sv[3] = s0.w; sv[4] = s1.x; sv[5] = s1.y; sv[6] = s1.z; sv[7] = s1.w;
        mv[0] = m0.x; mv[1] = m0.y; mv[2] = m0.z; mv[3] = m0.w; mv[4] = m1.x; mv[5] = m1.y; mv[6] = m1.z; mv[7] = m1.w;
    } else {
#pragma unroll
        for (int q = 0; q < 8; ++q) { sv[q] = 1.f; mv[q] = 0.f; }
    }
    bool bad = false;
    float det = 0.f;
    uint32_t ah[4], al[4], bh[4], bl[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
        float a[2], b[2];
#pragma unroll
        for (int v = 0; v < 2; ++v) {
            const float s2 = sv[2 * u + v], m = mv[2 * u + v];
            if (realk && (!(s2 > 0.f) || !isfinite(s2) || !isfinite(m))) bad = true;
            const float inv = realk ? __frcp_rn(s2) : 0.f;
            a[v] = (-0.5f * kLog2e128) * inv;
            b[v] = (kLog2e128 * m) * inv;
            det += realk ? m * m * inv + __logf(s2) : 0.f;
        }
        ah[u] = pack_bf2(a[0], a[1]);
        al[u] = pack_bf2(a[0] - bf_lo(ah[u]), a[1] - bf_hi(ah[u]));
        bh[u] = pack_bf2(b[0], b[1]);
        bl[u] = pack_bf2(b[0] - bf_lo(bh[u]), b[1] - bf_hi(bh[u]));
    }
#pragma unroll
    for (int o = 8; o > 0; o >>= 1) det += __shfl_xor_sync(0xffffffffu, det, o);
    const float lp = realk ? log_pi[(size_t)h * K + k] : 0.f;
    if ((tid & 15) == 0 && realk && !isfinite(lp)) bad = true;
    const int any = __syncthreads_or(bad ? 1 : 0);
    uint8_t *slabs = coef + (j0 >> 6) * 4 * kSlab;
    const uint32_t off = sw128_offset(k, j0 & 63, 1024);  // 16-byte aligned (j0 % 8 == 0)
    *reinterpret_cast<uint4 *>(slabs + off) = make_uint4(ah[0], ah[1], ah[2], ah[3]);
    *reinterpret_cast<uint4 *>(slabs + kSlab + off) = make_uint4(al[0], al[1], al[2], al[3]);
    *reinterpret_cast<uint4 *>(slabs + 2 * kSlab + off) = make_uint4(bh[0], bh[1], bh[2], bh[3]);
    *reinterpret_cast<uint4 *>(slabs + 3 * kSlab + off) = make_uint4(bl[0], bl[1], bl[2], bl[3]);
    if ((tid & 15) == 0) reinterpret_cast<float *>(coef + kCoefC)[k] = realk ? kLog2e128 * (lp - 0.5f * det) : -INFINITY;
    if (tid == 0) head_err[h * kPrepBlocks128 + blockIdx.x] = any ? (unsigned)GMA_ERR_NONFINITE_PARAM : 0u;
}

// Parameter-error check by one whole warp: any prep block that failed fails the call.
__device__ __forceinline__ unsigned head_error_warp128(const unsigned *head_err, int H, int lane) {
    unsigned e = 0u;
    for (int i = lane; i < H * kPrepBlocks128; i += 32) e |= __ldcg(head_err + i);
    return __reduce_or_sync(0xffffffffu, e);
}

// ------------------------------------------------------------------ shared device pieces

struct Part128 {
    int ntiles;  // tiles per head
    int total;   // B*H*ntiles
    int tpc;     // tiles per CTA
    int slots;   // job memories per CTA (upper bound on its jobs)
};
__host__ __device__ inline int first_cta128(const Part128 &P, int bh) { return (bh * P.ntiles) / P.tpc; }
__host__ __device__ inline int last_cta128(const Part128 &P, int bh) { return ((bh + 1) * P.ntiles - 1) / P.tpc; }
__host__ __device__ inline int slot128(const Part128 &P, int c, int bh) { return bh - (c * P.tpc) / P.ntiles; }

// x^2 of this thread's row of a [128 x 128] bf16 tile (two SW128 column halves)
// as the tensor-memory A operand of the score MMAs: x2hi of routing column j at
// 32-bit column j / 2 of `taddr` (pairs, low half first), x2lo 64 columns further.
__device__ __noinline__ void x2_row128(const uint8_t *x, int row, uint32_t taddr) {
#pragma unroll
    for (int hf = 0; hf < 2; ++hf) {
        uint32_t h[32], l[32];
        const uint8_t *rp = x + hf * kHalf + row * 128;
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
        tmem_st32(taddr + 32 * hf, h);
        tmem_st32(taddr + 64 + 32 * hf, l);
    }
    tmem_wait_st();
}

// Score MMAs of one side of a chunk, 40 instructions (N = 128, all components),
// slab by slab through the coefficient ring: for column half hf and K step kk
// of it (routing columns 64 hf + 16 kk ..):
//   a_hi: x2hi a_hi + x2lo a_hi;  a_lo: x2hi a_lo;  b_hi: x b_hi;  b_lo: x b_lo.
// d: accumulator; ax: x^2 operand in tensor memory (x2hi +0, x2lo +64); dx0:
// descriptor of the x tile's first column half; dring0: descriptor of ring slot
// 0 (NS slots of 16 KB, slab s always in slot s % NS).  Unrolled, every operand
// a base plus a constant: a rolled loop that builds descriptors costs several
// times the MMA itself.
//
// Slab schedule (SlabOrder): the sides of a job take the eight slabs in
// alternating order, forward then backward, so a side begins with the NS slabs
// the previous side ended with, still in the ring, and loads only the other
// 8 - NS (the first side of a job loads all 8).  full[slot] completes once per
// load (bit `slot` of *fpar is the parity of the next one), empty[slot] is
// committed after a load's last use: at once for slabs that the next side does
// not reuse, after the next side for the last NS slabs of a side.  Returns
// false (after recording the timeout) if a slab never arrived.
struct SlabOrder {
    int first, last;  // the side is the first / last of its job
};
template <int NS, bool FWD>
__device__ __noinline__ bool issue_scores128(uint32_t d, uint32_t ax, uint64_t dx0, uint64_t dring0, uint32_t *fpar,
                                             SlabOrder so, uint64_t *full, uint64_t *empty, unsigned *status,
                                             int *abort_flag) {
    constexpr uint32_t i128 = idesc_bf16(kT, 128, false, false);
    static_assert(NS <= 4, "the first and last NS positions of a side must not overlap");
    uint32_t fp = *fpar;
#pragma unroll
    for (int k = 0; k < kSlabs; ++k) {
        const int sl = FWD ? k : kSlabs - 1 - k, slot = sl % NS, hf = sl >> 2, m = sl & 3;
        if (so.first || k >= NS) {  // a fresh load
            if (!mbar_wait(&full[slot], (fp >> slot) & 1u)) {
                note_timeout(status, abort_flag);
                return false;
            }
            fp ^= 1u << slot;
        }
        tc_fence_after();
        const uint64_t db = dadd(dring0, slot * kSlab);
#pragma unroll
        for (int k4 = 0; k4 < 4; ++k4) {
            const int kk = 4 * hf + k4;
            const uint64_t bb = dadd(db, k4 * 32);
            const uint32_t acc = (k > 0 || k4 > 0) ? 1u : 0u;
            if (m == 0) {
                umma_bf16_tA(d, ax + kk * 8, bb, i128, acc);
                umma_bf16_tA(d, ax + 64 + kk * 8, bb, i128, 1u);
            } else if (m == 1) {
                umma_bf16_tA(d, ax + kk * 8, bb, i128, acc);
            } else {
                umma_bf16(d, dadd(dx0, hf * kHalf + k4 * 32), bb, i128, acc);
            }
        }
        if (k < kSlabs - NS || so.last) umma_commit(&empty[slot]);  // this load's last use
    }
    *fpar = fp;
    return true;
}

// Position p of a forward side takes unit unit_at<PAIRS>(p) of the image.  Slabs
// go in image order.  The four 32 KB pairs go as [b ; a] of column half 0, then
// [a ; b] of half 1 ([b_hi ; b_lo] = 4 MMAs, [a_hi ; a_lo] = 8): with two slots,
// each fresh load of a side then follows an 8-MMA pair (in image order one of
// them would follow a 4-MMA pair, half the time to hide its load).
template <bool PAIRS>
__device__ __forceinline__ int unit_at(int p) { return PAIRS ? (p < 2 ? 1 - p : p) : p; }

// Producer side of the slab schedule: the loads of one side (all NU units for
// the first side of a job, else the NU - NS the previous side did not leave in
// the ring), each once the slot's previous load has had its last use.  A unit
// is UB bytes of the coefficient image (a slab, or a pair of adjacent slabs);
// the unit at position p (unit_at) always goes to slot p % NS.  Bit `slot` of
// *lpar is the parity of the slot's load count; bit `slot` of *lmask is set once
// the slot has been loaded.  Returns false on a timeout.
template <int NS, int NU, int UB>
__device__ __forceinline__ bool load_units128(uint8_t *ring, const uint8_t *himg, int fwd, int first, uint32_t *lpar,
                                              uint32_t *lmask, uint64_t *full, uint64_t *empty, unsigned *status,
                                              int *abort_flag) {
    uint32_t lp = *lpar;
    for (int k = first ? 0 : NS; k < NU; ++k) {
        const int pos = fwd ? k : NU - 1 - k, u = unit_at<(UB > kSlab)>(pos), slot = pos % NS;
        if (!wait_or_abort(&empty[slot], ((lp >> slot) & 1u) ^ 1u, status, abort_flag)) return false;
        lp ^= 1u << slot;
        *lmask |= 1u << slot;
        mbar_arrive_expect_tx(&full[slot], UB);
        bulk_load(ring + slot * UB, himg + u * UB, UB, &full[slot]);
        *lpar = lp;
    }
    return true;
}
template <int NS>
__device__ __forceinline__ bool load_slabs128(uint8_t *ring, const uint8_t *himg, int fwd, int first, uint32_t *lpar,
                                              uint32_t *lmask, uint64_t *full, uint64_t *empty, unsigned *status,
                                              int *abort_flag) {
    return load_units128<NS, kSlabs, kSlab>(ring, himg, fwd, first, lpar, lmask, full, empty, status, abort_flag);
}

// Waits (bounded) until the last load into every slot that has been loaded has
// landed, so that no slab copy is in flight when the CTA moves on or leaves.
template <int NS>
__device__ __forceinline__ void drain_slabs128(uint32_t lpar, uint32_t lmask, uint64_t *full) {
#pragma unroll
    for (int q = 0; q < NS; ++q)
        if ((lmask >> q) & 1u) mbar_wait(&full[q], ((lpar >> q) & 1u) ^ 1u);
}

// Score MMAs of one key tile of the aggregation, 24 instructions: the slabs
// stream as four 32 KB pairs -- [a_hi ; a_lo] and [b_hi ; b_lo] of each column
// half, adjacent in the image, so each pair is one N = 256 B operand (rows: the
// 128 components' hi parts, then their lo parts) -- and per K step
//   D[:, 0:256] += x2hi [a_hi | a_lo],  D[:, 0:128] += x2lo a_hi,  D[:, 0:256] += x [b_hi | b_lo];
// the score of component k is D[:, k] + D[:, 128 + k] (+ c_k).  Pairs in the
// snake order of issue_scores128, in the order of unit_at<true> (the pair at
// position p in slot p % NS).
template <int NS, bool FWD>
__device__ __noinline__ bool issue_score_pairs128(uint32_t d, uint32_t ax, uint64_t dx0, uint64_t dring0,
                                                  uint32_t *fpar, SlabOrder so, uint64_t *full, uint64_t *empty,
                                                  unsigned *status, int *abort_flag) {
    constexpr uint32_t i256 = idesc_bf16(kT, 256, false, false), i128 = idesc_bf16(kT, 128, false, false);
    constexpr int NU = kSlabs / 2;
    static_assert(2 * NS <= NU, "the first and last NS positions of a side must not overlap");
    uint32_t fp = *fpar;
#pragma unroll
    for (int k = 0; k < NU; ++k) {
        const int pos = FWD ? k : NU - 1 - k, u = unit_at<true>(pos), slot = pos % NS, hf = u >> 1;
        const bool a_pair = (u & 1) == 0;
        if (so.first || k >= NS) {  // a fresh load
            if (!mbar_wait(&full[slot], (fp >> slot) & 1u)) {
                note_timeout(status, abort_flag);
                return false;
            }
            fp ^= 1u << slot;
        }
        tc_fence_after();
        const uint64_t db = dadd(dring0, slot * 2 * kSlab);
#pragma unroll
        for (int k4 = 0; k4 < 4; ++k4) {
            const int kk = 4 * hf + k4;
            const uint64_t bb = dadd(db, k4 * 32);
            const uint32_t acc = (k > 0 || k4 > 0) ? 1u : 0u;
            if (a_pair) {
                umma_bf16_tA(d, ax + kk * 8, bb, i256, acc);
                umma_bf16_tA(d, ax + 64 + kk * 8, bb, i128, 1u);
            } else {
                umma_bf16(d, dadd(dx0, hf * kHalf + k4 * 32), bb, i256, acc);
            }
        }
        if (k < NU - NS || so.last) umma_commit(&empty[slot]);  // this load's last use
    }
    *fpar = fp;
    return true;
}

// Score row of the N = 256 accumulator: e_k = s_k + c_k into registers (s_k the
// sum of columns k and 128 + k, c from the head's image in global memory);
// returns the row maximum.  exp_row128 then turns e into 2^(e - max) and
// returns the row sum: the accumulator is free between the two.
__device__ __forceinline__ float score_sum256(uint32_t taddr, const float *cg, float (&e)[kKC]) {
    float m = -INFINITY;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        uint32_t a[32], b[32];
        tmem_ld32(taddr + 32 * q, a);
        tmem_ld32(taddr + 128 + 32 * q, b);
        tmem_wait_ld();
        const float4 *c4 = reinterpret_cast<const float4 *>(cg + 32 * q);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const float4 c = __ldg(c4 + i);
            const float2 x0 = f2_add(f2_add(make_float2(__uint_as_float(a[4 * i]), __uint_as_float(a[4 * i + 1])),
                                            make_float2(__uint_as_float(b[4 * i]), __uint_as_float(b[4 * i + 1]))),
                                     make_float2(c.x, c.y));
            const float2 x1 = f2_add(f2_add(make_float2(__uint_as_float(a[4 * i + 2]), __uint_as_float(a[4 * i + 3])),
                                            make_float2(__uint_as_float(b[4 * i + 2]), __uint_as_float(b[4 * i + 3]))),
                                     make_float2(c.z, c.w));
            e[32 * q + 4 * i] = x0.x;
            e[32 * q + 4 * i + 1] = x0.y;
            e[32 * q + 4 * i + 2] = x1.x;
            e[32 * q + 4 * i + 3] = x1.y;
            m = fmaxf(m, fmaxf(fmaxf(x0.x, x0.y), fmaxf(x1.x, x1.y)));
        }
    }
    return m;
}
__device__ __forceinline__ float exp_row128(float (&e)[kKC], float m) {
    const float2 mm = make_float2(m, m);
    float2 s0 = make_float2(0.f, 0.f), s1 = make_float2(0.f, 0.f);
#pragma unroll
    for (int k = 0; k < kKC; k += 4) {
        const float2 d0 = f2_sub(make_float2(e[k], e[k + 1]), mm), d1 = f2_sub(make_float2(e[k + 2], e[k + 3]), mm);
        e[k] = ex2(d0.x);
        e[k + 1] = ex2(d0.y);
        e[k + 2] = ex2(d1.x);
        e[k + 3] = ex2(d1.y);
        s0 = f2_add(s0, make_float2(e[k], e[k + 1]));
        s1 = f2_add(s1, make_float2(e[k + 2], e[k + 3]));
    }
    return (s0.x + s0.y) + (s1.x + s1.y);
}

// The other MMA batches of a chunk, out of line so that the compiler keeps
// their 16-24 descriptors as a base plus constants instead of hoisting them all
// out of the chunk loop (and spilling them).  All have M = N = 128.
// num = Gamma^Q S: A = Gamma^Q hi | lo in tensor memory (aq0: hi, +64: lo), B =
// the state operand (dS: hi, MN-major; lo 32 KB further); hi.hi, hi.lo, lo.hi.
__device__ __noinline__ void issue_num128(uint32_t d, uint32_t aq0, uint64_t dS) {
    constexpr uint32_t ikm = idesc_bf16(kT, 128, false, true);
#pragma unroll
    for (int kk = 0; kk < kKC / 16; ++kk) {
        const uint64_t bs = dadd(dS, kk * 2048);
        umma_bf16_tA(d, aq0 + kk * 8, bs, ikm, kk > 0 ? 1u : 0u);
        umma_bf16_tA(d, aq0 + kk * 8, dadd(bs, 2 * kHalf), ikm, 1u);
        umma_bf16_tA(d, aq0 + 64 + kk * 8, bs, ikm, 1u);
    }
}
// U = Gamma^Q Gamma^K^T: B = Gamma^K (dG: hi, K-major rows = keys; lo 1 KB further).
__device__ __noinline__ void issue_u128(uint32_t d, uint32_t aq0, uint64_t dG) {
    constexpr uint32_t ikk = idesc_bf16(kT, 128, false, false);
#pragma unroll
    for (int kk = 0; kk < kKC / 16; ++kk) {
        const uint64_t bg = dadd(dG, (kk >> 2) * 2048 + (kk & 3) * 32);
        umma_bf16_tA(d, aq0 + kk * 8, bg, ikk, kk > 0 ? 1u : 0u);
        umma_bf16_tA(d, aq0 + kk * 8, dadd(bg, 1024), ikk, 1u);
        umma_bf16_tA(d, aq0 + 64 + kk * 8, bg, ikk, 1u);
    }
}
// S (+)= Gamma^K^T V: A = Gamma^K^T (dGT: hi, MN-major; lo 1 KB further), B = V
// (dV, MN-major); `acc` = 0 starts the sum.
__device__ __noinline__ void issue_supd128(uint32_t d, uint64_t dGT, uint64_t dV, uint32_t acc) {
    constexpr uint32_t imm = idesc_bf16(kT, 128, true, true);
#pragma unroll
    for (int kk = 0; kk < kT / 16; ++kk) {
        const uint64_t b = dadd(dV, kk * 2048), a = dadd(dGT, kk * 2 * kGroupB);
        umma_bf16(d, a, b, imm, (acc || kk > 0) ? 1u : 0u);
        umma_bf16(d, dadd(a, 1024), b, imm, 1u);
    }
}
// num += P V: A = P hi / lo in place in the U columns (key block cb = kk / 2: hi
// words at 32 cb, lo words at 32 cb + 16), B = V (dV, MN-major).
__device__ __noinline__ void issue_pv128(uint32_t d, uint32_t ap0, uint64_t dV) {
    constexpr uint32_t ikm = idesc_bf16(kT, 128, false, true);
#pragma unroll
    for (int kk = 0; kk < kT / 16; ++kk) {
        const uint64_t b = dadd(dV, kk * 2048);
        const uint32_t ap = ap0 + 32 * (kk >> 1) + 8 * (kk & 1);
        umma_bf16_tA(d, ap, b, ikm, 1u);
        umma_bf16_tA(d, ap + 16, b, ikm, 1u);
    }
}

// Score row -> e_k = 2^(s_k + c_k - max) in registers; returns the row sum.
__device__ __forceinline__ float score_exp128(uint32_t taddr, const float *cvec, float (&e)[kKC]) {
    float m = -INFINITY;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        uint32_t r[32];
        tmem_ld32(taddr + 32 * q, r);
        tmem_wait_ld();
        const float4 *c4 = reinterpret_cast<const float4 *>(cvec + 32 * q);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const float4 c = c4[i];
            const float2 a = f2_add(make_float2(__uint_as_float(r[4 * i]), __uint_as_float(r[4 * i + 1])),
                                    make_float2(c.x, c.y));
            const float2 b = f2_add(make_float2(__uint_as_float(r[4 * i + 2]), __uint_as_float(r[4 * i + 3])),
                                    make_float2(c.z, c.w));
            e[32 * q + 4 * i] = a.x;
            e[32 * q + 4 * i + 1] = a.y;
            e[32 * q + 4 * i + 2] = b.x;
            e[32 * q + 4 * i + 3] = b.y;
            m = fmaxf(m, fmaxf(fmaxf(a.x, a.y), fmaxf(b.x, b.y)));
        }
    }
    const float2 mm = make_float2(m, m);
    float2 s0 = make_float2(0.f, 0.f), s1 = make_float2(0.f, 0.f);
#pragma unroll
    for (int k = 0; k < kKC; k += 4) {
        const float2 d0 = f2_sub(make_float2(e[k], e[k + 1]), mm), d1 = f2_sub(make_float2(e[k + 2], e[k + 3]), mm);
        e[k] = ex2(d0.x);
        e[k + 1] = ex2(d0.y);
        e[k + 2] = ex2(d1.x);
        e[k + 3] = ex2(d1.y);
        s0 = f2_add(s0, make_float2(e[k], e[k + 1]));
        s1 = f2_add(s1, make_float2(e[k + 2], e[k + 3]));
    }
    return (s0.x + s0.y) + (s1.x + s1.y);
}

// bf16 hi / lo words of e[8 w .. 8 w + 7] scaled by `sc` (4 words each).
__device__ __forceinline__ void split8(const float (&e)[kKC], int w, float sc, uint32_t (&h)[4], uint32_t (&l)[4]) {
    const float2 s2 = make_float2(sc, sc);
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        const float2 g = f2_mul(make_float2(e[8 * w + 2 * q], e[8 * w + 2 * q + 1]), s2);
        h[q] = pack_bf2(g.x, g.y);
        const float2 r = f2_sub(g, make_float2(bf_lo(h[q]), bf_hi(h[q])));
        l[q] = pack_bf2(r.x, r.y);
    }
}

// Normalised Gamma^K row `row` (e scaled by sc) into the Gamma buffer: 8-token
// groups of 4 KB = [hi, components 0-63 | lo, 0-63 | hi, 64-127 | lo, 64-127],
// each 1 KB block an SW128 atom (8 rows of 128 bytes).  The same bytes are the
// K-major B operand of U (rows = tokens) and the MN-major A operand of the
// state update (rows = tokens, 64 components per row).
__device__ __forceinline__ void store_gamma128(uint8_t *gbuf, int row, const float (&e)[kKC], float sc) {
    uint8_t *rb = gbuf + (row >> 3) * kGroupB + (row & 7) * 128;
#pragma unroll
    for (int w = 0; w < 16; ++w) {  // 8 components per 16-byte chunk
        uint32_t h[4], l[4];
        split8(e, w, sc, h, l);
        const int atom = w >> 3, c = w & 7;
        uint8_t *p = rb + atom * 2048 + ((c ^ (row & 7)) << 4);
        *reinterpret_cast<uint4 *>(p) = make_uint4(h[0], h[1], h[2], h[3]);
        *reinterpret_cast<uint4 *>(p + 1024) = make_uint4(l[0], l[1], l[2], l[3]);
    }
}

// ------------------------------------------------------------------ aggregation
//
// Warps: 0 lane 0 K / V tile loads, lane 1 coefficient slab pairs; 1 lane 0 MMA
// issue; 2..5 epilogue (one thread per tile row / component).
// TMEM: x^2 [0, 128); scores [128, 384) (N = 256: hi-part and lo-part
// products); the job's memory increment S (M = 128 components, N = 128 value
// columns) [384, 512).  Per tile: 24 score MMAs, then 16 state MMAs
// (Gamma^K_hi, Gamma^K_lo times V, both operands MN-major).  The epilogue loads
// a tile's scores into registers, frees the accumulator, prepares the next
// tile's x^2, and only then runs the softmax and stores Gamma^K, so the next
// score MMAs overlap it.  The key mass of a tile (column sums of Gamma^K) is
// left as four per-warp partial rows (a fixed-order butterfly over each warp's
// 32 rows): the scan adds them in warp order, and the job's total is summed in
// registers and combined across the warps once, at the job's end.
struct Agg128Smem {
    static constexpr int kKS = 2, kCS = 2;              // K stages; slab-pair slots
    static constexpr int kK = 0;                        // K stages
    static constexpr int kV = kK + kKS * kTileB;        // V stage
    static constexpr int kG = kV + kTileB;              // Gamma^K buffer (16 groups x 4 KB)
    static constexpr int kCf = kG + 16 * kGroupB;       // slab-pair ring (32 KB slots)
    static constexpr int kBars = kCf + kCS * 2 * kSlab;
    static constexpr int kBytes = kBars + 256;
    static constexpr int kAlloc = kBytes + 1024;
    static_assert(kV % 1024 == 0 && kG % 1024 == 0 && kCf % 1024 == 0, "SW128 alignment");
    static_assert(kAlloc <= 232448, "shared memory budget");
};
constexpr int kThreadsAgg = 64 + 128;

// Column sums over the warp's 32 rows of v[128] (butterfly reduce-scatter, a
// fixed order): on return lane l holds the sums of columns base .. base + 3 in
// v[0..3], base = 64 b4 + 32 b3 + 16 b2 + 8 b1 + 4 b0 (b4..b0 the bits of l).
__device__ __forceinline__ int column_sums_warp(float (&v)[kKC], int lane) {
    int base = 0;
#pragma unroll
    for (int o = 16, n = 64; o > 0; o >>= 1, n >>= 1) {
        const bool up = (lane & o) != 0;
#pragma unroll
        for (int i = 0; i < n; ++i) {
            const float mine = up ? v[n + i] : v[i];
            const float other = up ? v[i] : v[n + i];
            v[i] = mine + __shfl_xor_sync(0xffffffffu, other, o);
        }
        base += up ? n : 0;
    }
    return base;
}

// The combine of head bh's job memories (fp32, kPartFloats each), in job order,
// by the whole CTA: mode 1 replaces each by the exclusive prefix before it,
// mode 0 writes their sum to the head's memory.  Each thread takes NQ float4
// slots per round and keeps the loads of NB jobs for all of them in flight at
// once (the sums stay in job order).
__device__ __noinline__ void combine_jobs128(float *__restrict__ part, float *__restrict__ mem, const Part128 &P,
                                             int bh, int mode, int tid) {
    constexpr int kP4 = kPartFloats / 4, NQ = 4, NB = 4;
    const int cf = first_cta128(P, bh), cl = last_cta128(P, bh);
    for (int e0 = tid; e0 < kP4; e0 += NQ * kThreadsAgg) {
        float4 acc[NQ];
#pragma unroll
        for (int q = 0; q < NQ; ++q) acc[q] = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int cb = cf; cb <= cl; cb += NB) {
            float4 v[NB][NQ];
#pragma unroll
            for (int u = 0; u < NB; ++u) {
                const int cc = cb + u;
                const float4 *src = reinterpret_cast<const float4 *>(
                    part + ((size_t)cc * P.slots + (cc <= cl ? slot128(P, cc, bh) : 0)) * kPartFloats);
#pragma unroll
                for (int q = 0; q < NQ; ++q) {
                    const int e4 = e0 + q * kThreadsAgg;
                    v[u][q] = (cc <= cl && e4 < kP4) ? __ldcg(src + e4) : make_float4(0.f, 0.f, 0.f, 0.f);
                }
            }
#pragma unroll
            for (int u = 0; u < NB; ++u) {
                const int cc = cb + u;
                if (cc > cl) break;
                float4 *dst = reinterpret_cast<float4 *>(part + ((size_t)cc * P.slots + slot128(P, cc, bh)) *
                                                                     kPartFloats);
#pragma unroll
                for (int q = 0; q < NQ; ++q) {
                    const int e4 = e0 + q * kThreadsAgg;
                    if (e4 >= kP4) continue;
                    if (mode == 1) __stcg(dst + e4, acc[q]);
                    acc[q].x += v[u][q].x;
                    acc[q].y += v[u][q].y;
                    acc[q].z += v[u][q].z;
                    acc[q].w += v[u][q].w;
                }
            }
        }
        if (mode == 0) {
#pragma unroll
            for (int q = 0; q < NQ; ++q) {
                const int e4 = e0 + q * kThreadsAgg;
                if (e4 < kP4) __stcg(reinterpret_cast<float4 *>(mem + (size_t)bh * kPartFloats) + e4, acc[q]);
            }
        }
    }
}

__global__ void __launch_bounds__(kThreadsAgg, 1) tc128_aggregate_kernel(
    const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
    const uint8_t *__restrict__ coef_img, const unsigned *__restrict__ head_err, int H, int N, Part128 P,
    float *__restrict__ part, float *__restrict__ ztile, float *__restrict__ mem, unsigned *__restrict__ counters,
    int mode, int stall, unsigned *status) {
    using L = Agg128Smem;
    constexpr int KS = L::kKS, CS = L::kCS;
    constexpr int kX = 0, kSC = 128, kSA = 384, kTmemCols = 512;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t *kst = smem + L::kK, *vst = smem + L::kV, *gbuf = smem + L::kG, *ring = smem + L::kCf;
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + L::kBars);
    uint64_t *kfull = bars, *kempty = kfull + KS, *vfull = kempty + KS, *vempty = vfull + 1, *cffull = vempty + 1,
             *cfempty = cffull + CS, *xready = cfempty + CS, *sfull = xready + 1, *sfree = sfull + 1,
             *gready = sfree + 1, *wdone = gready + 1, *accfull = wdone + 1, *zjob = accfull + 1;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(zjob + 1);
    int *abort_flag = reinterpret_cast<int *>(zjob + 2);
    int *last_flag = abort_flag + 1;
    static_assert((2 * KS + 2 + 2 * CS + 7) * 8 + 16 <= 256, "barrier area");

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int c = blockIdx.x;
    const int g0 = c * P.tpc, gend = min(P.total, g0 + P.tpc);
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
        mbar_init(vfull, 1);
        mbar_init(vempty, 1);
        for (int i = 0; i < CS; ++i) {
            mbar_init(&cffull[i], 1);
            mbar_init(&cfempty[i], 1);
        }
        mbar_init(xready, 4);
        mbar_init(sfull, 1);
        mbar_init(sfree, 4);
        mbar_init(gready, 4);
        mbar_init(wdone, 1);
        mbar_init(accfull, 1);
        mbar_init(zjob, 4);
        *abort_flag = 0;
        fence_mbar_init();
        tma_prefetch_desc(&tmK);
        tma_prefetch_desc(&tmV);
    }
    // Everything below reads the coefficient prep's output: wait for it, then let
    // the next kernel launch.
    pdl_wait();
    pdl_trigger();
    {
        const unsigned herr = warp == 1 ? head_error_warp128(head_err, H, lane) : 0u;
        if (tid == 32 && (herr || failed(status))) {
            if (herr) set_status(status, herr);
            *abort_flag = 1;
        }
    }
    tc_fence_before();
    cta_sync();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    int rbase = 0, njob = 0;
    // slab ring state of the producer (load parities) and of the MMA thread (full
    // parities), per slot; slab_lmask: the slots loaded at least once
    uint32_t slab_lpar = 0u, slab_fpar = 0u, slab_lmask = 0u;
    for (int g = aborted(abort_flag) ? gend : g0; g < gend; ++njob) {
        const int bh = g / P.ntiles, t0 = g % P.ntiles;
        const int n = min(P.ntiles - t0, gend - g);
        const int h = bh % H;
        const uint8_t *himg = coef_img + (size_t)h * kImgStride;
        cta_sync();  // the previous job is done with the Gamma buffer and the job memory
        if (warp == 0) {
            if (lane == 0) {
                // K two stages ahead, V one stage
                int karm[KS], varm = -1;
#pragma unroll
                for (int q = 0; q < KS; ++q) karm[q] = -1;
                for (int i = 0; i < n; ++i) {
                    const int r = rbase + i, s = r % KS;
                    if (!wait_or_abort(&kempty[s], ((r / KS) & 1) ^ 1, status, abort_flag)) break;
                    if (!(stall && r == 0)) {  // test hook: the first key tile is never loaded
                        mbar_arrive_expect_tx(&kfull[s], kTileB);
                        tma_load_3d(kst + s * kTileB, &tmK, 0, (t0 + i) * kT, bh, &kfull[s]);
                        tma_load_3d(kst + s * kTileB + kHalf, &tmK, 64, (t0 + i) * kT, bh, &kfull[s]);
                        karm[s] = r;
                    }
                    if (i >= 1) {
                        const int rv = r - 1;
                        if (!wait_or_abort(vempty, (rv & 1) ^ 1, status, abort_flag)) break;
                        mbar_arrive_expect_tx(vfull, kTileB);
                        tma_load_3d(vst, &tmV, 0, (t0 + i - 1) * kT, bh, vfull);
                        tma_load_3d(vst + kHalf, &tmV, 64, (t0 + i - 1) * kT, bh, vfull);
                        varm = rv;
                    }
                }
                if (!aborted(abort_flag)) {
                    const int rv = rbase + n - 1;
                    if (wait_or_abort(vempty, (rv & 1) ^ 1, status, abort_flag)) {
                        mbar_arrive_expect_tx(vfull, kTileB);
                        tma_load_3d(vst, &tmV, 0, (t0 + n - 1) * kT, bh, vfull);
                        tma_load_3d(vst + kHalf, &tmV, 64, (t0 + n - 1) * kT, bh, vfull);
                        varm = rv;
                    }
                }
                // every load armed here has landed before the CTA moves on or leaves
#pragma unroll
                for (int q = 0; q < KS; ++q)
                    if (karm[q] >= 0) mbar_wait(&kfull[q], (karm[q] / KS) & 1);
                if (varm >= 0) mbar_wait(vfull, varm & 1);
            } else if (lane == 1) {
                // slab pairs: one side per key tile, alternating direction
                for (int i = 0; i < n; ++i)
                    if (!load_units128<CS, kSlabs / 2, 2 * kSlab>(ring, himg, (i & 1) == 0, i == 0, &slab_lpar,
                                                                  &slab_lmask, cffull, cfempty, status, abort_flag))
                        break;
                // every slab load armed here has landed before the CTA moves on or leaves
                drain_slabs128<CS>(slab_lpar, slab_lmask, cffull);
            }
        } else if (warp == 1) {
            if (lane == 0) {
                bool ok = true;
                const uint64_t dk0 = sdesc_sw128(smem_u32(kst), 16, 1024), dring0 = sdesc_sw128(smem_u32(ring), 16, 1024);
                const uint64_t dgt = sdesc_sw128(smem_u32(gbuf), 2048, kGroupB);  // Gamma^K^T hi, MN-major A
                const uint64_t dv = sdesc_sw128(smem_u32(vst), kHalf, 1024);       // V, MN-major B
                // scores(i + 1) go before the state MMAs of tile i: the epilogue frees the
                // score accumulator and prepares the next x^2 before tile i's softmax
                auto scores = [&](int i) {
                    const int r = rbase + i;
                    if (!wait_or_abort(xready, r & 1, status, abort_flag)) return false;
                    if (!wait_or_abort(&kfull[r % KS], (r / KS) & 1, status, abort_flag)) return false;
                    if (r > 0 && !wait_or_abort(sfree, (r - 1) & 1, status, abort_flag)) return false;
                    tc_fence_after();
                    const SlabOrder so{i == 0, i == n - 1};
                    const uint64_t dx = dadd(dk0, (r % KS) * kTileB);
                    if (!((i & 1) == 0 ? issue_score_pairs128<CS, true>(tmem + kSC, tmem + kX, dx, dring0, &slab_fpar,
                                                                        so, cffull, cfempty, status, abort_flag)
                                       : issue_score_pairs128<CS, false>(tmem + kSC, tmem + kX, dx, dring0, &slab_fpar,
                                                                         so, cffull, cfempty, status, abort_flag)))
                        return false;
                    umma_commit(sfull);
                    umma_commit(&kempty[r % KS]);
                    return true;
                };
                ok = scores(0);
                for (int i = 0; ok && i < n; ++i) {
                    const int r = rbase + i;
                    if (i + 1 < n && !(ok = scores(i + 1))) break;
                    if (!(ok = wait_or_abort(gready, r & 1, status, abort_flag))) break;
                    if (!(ok = wait_or_abort(vfull, r & 1, status, abort_flag))) break;
                    tc_fence_after();
                    issue_supd128(tmem + kSA, dgt, dv, i > 0 ? 1u : 0u);
                    umma_commit(wdone);
                    umma_commit(vempty);
                }
                umma_commit(accfull);
            }
        } else {
            // ---------------- epilogue: one thread per tile row (and per component)
            const int row = epi_row(warp, lane), ew = warp - 2;
            const uint32_t lb = (uint32_t)(32 * (warp & 3)) << 16;
            const float *cg = reinterpret_cast<const float *>(himg + kCoefC);
            float zacc[4] = {0.f, 0.f, 0.f, 0.f};
            int zbase = 0;
            auto x2 = [&](int i) {  // x^2 of tile i, once the previous score MMAs are done (sfull)
                const int r = rbase + i;
                if (!wait_or_abort(&kfull[r % KS], (r / KS) & 1, status, abort_flag)) return false;
                x2_row128(kst + (r % KS) * kTileB, row, tmem + lb + kX);
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(xready);
                return true;
            };
            bool ok = x2(0);
            for (int i = 0; ok && i < n; ++i) {
                const int r = rbase + i;
                if (!(ok = wait_or_abort(sfull, r & 1, status, abort_flag))) break;
                tc_fence_after();
                float e[kKC];
                const float mx = score_sum256(tmem + lb + kSC, cg, e);
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(sfree);
                if (i + 1 < n && !(ok = x2(i + 1))) break;
                const float rs = exp_row128(e, mx);
                const int tok = (t0 + i) * kT + row;
                const float sc = tok < N ? 1.0f / rs : 0.0f;
                if (r > 0 && !(ok = wait_or_abort(wdone, (r - 1) & 1, status, abort_flag))) break;
                store_gamma128(gbuf, row, e, sc);
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(gready);
                // key mass of the tile: this warp's column sums of the normalised Gamma^K
#pragma unroll
                for (int k = 0; k < kKC; ++k) e[k] *= sc;
                zbase = column_sums_warp(e, lane);
                if (mode == 1)
                    __stcg(reinterpret_cast<float4 *>(ztile + (((size_t)bh * P.ntiles + t0 + i) * 4 + ew) * kKC + zbase),
                           make_float4(e[0], e[1], e[2], e[3]));
#pragma unroll
                for (int q = 0; q < 4; ++q) zacc[q] += e[q];
            }
            // job end: the memory increment and key mass -> this job's memory slot; the
            // warps' key-mass partials meet in the (now idle) Gamma buffer
            if (ok && wait_or_abort(accfull, njob & 1, status, abort_flag)) {
                tc_fence_after();
                float *out = part + ((size_t)c * P.slots + slot128(P, c, bh)) * kPartFloats;
#pragma unroll 1
                for (int q = 0; q < 4; ++q) {
                    uint32_t v[32];
                    tmem_ld32(tmem + lb + kSA + 32 * q, v);
                    tmem_wait_ld();
                    float4 *o4 = reinterpret_cast<float4 *>(out + (size_t)row * kD + 32 * q);
#pragma unroll
                    for (int u = 0; u < 8; ++u)
                        __stcg(o4 + u, make_float4(__uint_as_float(v[4 * u]), __uint_as_float(v[4 * u + 1]),
                                                   __uint_as_float(v[4 * u + 2]), __uint_as_float(v[4 * u + 3])));
                }
                tc_fence_before();
                float *zw = reinterpret_cast<float *>(gbuf);  // [4 warps][128]
                *reinterpret_cast<float4 *>(zw + ew * kKC + zbase) = make_float4(zacc[0], zacc[1], zacc[2], zacc[3]);
                __syncwarp();
                if (lane == 0) mbar_arrive(zjob);
                if (wait_or_abort(zjob, njob & 1, status, abort_flag))
                    __stcg(out + kKC * kD + row, ((zw[row] + zw[kKC + row]) + zw[2 * kKC + row]) + zw[3 * kKC + row]);
            }
        }
        // ---- the head's last job to finish combines the job memories in job order:
        // mode 1, each replaced by the exclusive prefix before it; mode 0, the sum of all
        // of them into the head's memory
        __threadfence();
        cta_sync();
        if (!aborted(abort_flag)) {
            if (tid == 0) {
                const int njobs = last_cta128(P, bh) - first_cta128(P, bh) + 1;
                const unsigned old = atomicAdd(&counters[bh], 1u);
                *last_flag = (old == (unsigned)(njobs - 1));
            }
            cta_sync();
            if (*last_flag) {
                __threadfence();
                combine_jobs128(part, mem, P, bh, mode, tid);
                if (tid == 0) counters[bh] = 0u;  // ready for the next call
            }
        }
        rbase += n;
        g += n;
        if (aborted(abort_flag)) break;
    }
    tc_fence_before();
    cta_sync();
    if (warp == 0) tmem_dealloc(tmem, kTmemCols);
}

// ------------------------------------------------------------------ causal chunk scan
//
// One 128-token chunk at a time per CTA (its tile range, as in the
// aggregation; the job's carried-in prefix comes from there).  Warps: 0 lane 0
// Q / K / V tile loads, lane 1 coefficient slabs; 1 lane 0 MMA issue, lane 1
// the job's prefix; 2..5 query group (components 64-127 of the query and of
// the key softmax, P split of key blocks 0 and 1, outputs, then the next
// chunk's x^2 of K); 6..9 key group (components 0-63 of both softmaxes, P split
// of key blocks 2 and 3, state operand, then the next chunk's x^2 of Q).
//
// The Q and K tile buffers also hold the query and key softmaxes' exchanges once
// their score MMAs are done (the next tiles load after that), and the V tile buffer the
// output staging once the state update and P V are done (the next value tile
// loads once the stores have read it).
//
// TMEM (512 columns):
//   [0, 128)    A: x^2 of Q (hi | lo), then the key scores, then U, then P hi /
//               lo in place per 32-key block
//   [128, 256)  query scores, then Gamma^Q hi [128, 192) | lo [192, 256) in place
//   [256, 384)  B: x^2 of K, then num (N = 128)
//   [384, 512)  S, the fp32 state (M = 128 components, N = 128 value columns)
// The x^2 of both sides of the next chunk are prepared while this chunk ends,
// so the key score MMAs follow the query ones at once (each MMA's accumulator
// may be a column range an earlier MMA reads as its A operand: a single thread
// issues them, and issue order is execution order).
// MMA issue order per chunk: Q scores (40), K scores (40), num = Gamma^Q S (24:
// hi.hi, hi.lo, lo.hi), U (24), S += Gamma^K^T V (16), num += P V (16).
//
// Shared memory R (64 KB) holds either the state operand S (bf16 hi and lo, 32
// KB each, MN-major: rows = components, two 64-column halves) or Gamma^K (the
// 4 KB groups of store_gamma128): the key softmax writes Gamma^K once num has
// read S, and the state operand of the next chunk is written once U and the
// state update have read Gamma^K.  At a job start it receives the fp32 prefix.
struct Causal128Smem {
    static constexpr int kCS = 4;
    static constexpr int kQ = 0, kK = kQ + kTileB, kV = kK + kTileB;
    static constexpr int kR = kV + kTileB;              // state operand | Gamma^K | fp32 prefix (64 KB)
    static constexpr int kCf = kR + 65536;              // coefficient slab ring
    static constexpr int kC = kCf + kCS * kSlab;        // c [128] fp32
    static constexpr int kZp = kC + 512;                // key mass before the chunk [128] fp32
    static constexpr int kRs = kZp + 512;               // key group's P row sums [128] fp32
    static constexpr int kBars = kRs + 512;
    static constexpr int kBytes = kBars + 512;
    static constexpr int kAlloc = kBytes + 1024;
    static_assert(kR % 1024 == 0 && kCf % 1024 == 0, "SW128 alignment");
    static_assert(kAlloc <= 232448, "shared memory budget");
};
constexpr int kThreadsC128 = 64 + 256;

// One 32-key block of the masked bf16 hi / lo split of P for query row `row`,
// in place (hi words at 32 cb, lo words at 32 cb + 16); returns the block's
// sum of the masked fp32 values.
__device__ __forceinline__ float split_p_block128(uint32_t p_taddr, int cb, int row) {
    uint32_t wh[16], wl[16];
    float sum = 0.f;
    if (32 * cb > row) {
#pragma unroll
        for (int q = 0; q < 16; ++q) wh[q] = wl[q] = 0u;
    } else {
        uint32_t pp[32];
        tmem_ld32(p_taddr + 32 * cb, pp);
        tmem_wait_ld();
#pragma unroll
        for (int q = 0; q < 16; ++q) {
            const int j = cb * 32 + 2 * q;
            const float a = j <= row ? __uint_as_float(pp[2 * q]) : 0.f;
            const float b = j + 1 <= row ? __uint_as_float(pp[2 * q + 1]) : 0.f;
            sum += a + b;
            wh[q] = pack_bf2(a, b);
            wl[q] = pack_bf2(a - bf_lo(wh[q]), b - bf_hi(wh[q]));
        }
    }
    tmem_st16(p_taddr + 32 * cb, wh);
    tmem_st16(p_taddr + 32 * cb + 16, wl);
    return sum;
}

__device__ __noinline__ float split_p_blocks128(uint32_t p_taddr, int cb0, int row) {
    const float s0 = split_p_block128(p_taddr, cb0, row);
    const float s1 = split_p_block128(p_taddr, cb0 + 1, row);
    tmem_wait_st();
    return s0 + s1;
}

// Query softmax of one row: Gamma^Q = e (un-normalised) as bf16 hi | lo in place
// of the scores; returns r = sum_k e_k and writes e . Zp to *den0.
__device__ __noinline__ float query_row128(uint32_t s_taddr, const float *cvec, const float *zp, float *den0) {
    float e[kKC];
    const float r = score_exp128(s_taddr, cvec, e);
    float d0 = 0.f, d1 = 0.f;
#pragma unroll
    for (int k = 0; k < kKC; k += 2) {
        d0 = fmaf(e[k], zp[k], d0);
        d1 = fmaf(e[k + 1], zp[k + 1], d1);
    }
    *den0 = d0 + d1;
#pragma unroll
    for (int w4 = 0; w4 < 4; ++w4) {  // components 32 w4 .. 32 w4 + 31
        uint32_t h[16], l[16];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            uint32_t hh[4], ll[4];
            split8(e, 4 * w4 + u, 1.0f, hh, ll);
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                h[4 * u + q] = hh[q];
                l[4 * u + q] = ll[q];
            }
        }
        tmem_st16(s_taddr + 16 * w4, h);
        tmem_st16(s_taddr + 64 + 16 * w4, l);
    }
    tmem_wait_st();
    return r;
}

// Query softmax of half `hf` of one row (components 64 hf .. 64 hf + 63), run by
// the threads of both warp groups that own the row: Gamma^Q = e (un-normalised)
// as bf16 hi | lo in place of the scores -- hi words of the half's components at
// s_taddr + 32 hf, lo words at s_taddr + 64 + 32 hf, written only once both
// halves have read their scores.  The halves' maxima, then their row sums and
// e . Zp sums, meet in xb ([max | sum | e.Zp][half][128] fp32) through the
// mbarriers mx and ms (8 warps each, phase ph).  Returns false on a timeout;
// *r and *den0 get the whole row's sums (half 0 + half 1).
__device__ __noinline__ bool query_half128(uint32_t s_taddr, const float *cvec, const float *zp, int hf, int row,
                                           float *xb, uint64_t *mx, uint64_t *ms, uint32_t ph, float *r,
                                           float *den0, unsigned *status, int *abort_flag) {
    float e[64];
    float m = -INFINITY;
#pragma unroll
    for (int q = 0; q < 2; ++q) {
        uint32_t v[32];
        tmem_ld32(s_taddr + 64 * hf + 32 * q, v);
        tmem_wait_ld();
        const float4 *c4 = reinterpret_cast<const float4 *>(cvec + 64 * hf + 32 * q);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const float4 c = c4[i];
            const float2 a = f2_add(make_float2(__uint_as_float(v[4 * i]), __uint_as_float(v[4 * i + 1])),
                                    make_float2(c.x, c.y));
            const float2 b = f2_add(make_float2(__uint_as_float(v[4 * i + 2]), __uint_as_float(v[4 * i + 3])),
                                    make_float2(c.z, c.w));
            e[32 * q + 4 * i] = a.x;
            e[32 * q + 4 * i + 1] = a.y;
            e[32 * q + 4 * i + 2] = b.x;
            e[32 * q + 4 * i + 3] = b.y;
            m = fmaxf(m, fmaxf(fmaxf(a.x, a.y), fmaxf(b.x, b.y)));
        }
    }
    tc_fence_before();
    const int lane = threadIdx.x & 31;
    xb[hf * kT + row] = m;
    __syncwarp();
    if (lane == 0) mbar_arrive(mx);
    if (!wait_or_abort(mx, ph, status, abort_flag)) return false;  // both halves' scores are read
    tc_fence_after();
    const float2 mm = make_float2(fmaxf(xb[row], xb[kT + row]), fmaxf(xb[row], xb[kT + row]));
    float2 s0 = make_float2(0.f, 0.f), s1 = make_float2(0.f, 0.f);
    float d0 = 0.f, d1 = 0.f;
    const float *zh = zp + 64 * hf;
#pragma unroll
    for (int k = 0; k < 64; k += 4) {
        const float2 x0 = f2_sub(make_float2(e[k], e[k + 1]), mm), x1 = f2_sub(make_float2(e[k + 2], e[k + 3]), mm);
        e[k] = ex2(x0.x);
        e[k + 1] = ex2(x0.y);
        e[k + 2] = ex2(x1.x);
        e[k + 3] = ex2(x1.y);
        s0 = f2_add(s0, make_float2(e[k], e[k + 1]));
        s1 = f2_add(s1, make_float2(e[k + 2], e[k + 3]));
        d0 = fmaf(e[k], zh[k], d0);
        d1 = fmaf(e[k + 1], zh[k + 1], d1);
        d0 = fmaf(e[k + 2], zh[k + 2], d0);
        d1 = fmaf(e[k + 3], zh[k + 3], d1);
    }
#pragma unroll
    for (int w4 = 0; w4 < 2; ++w4) {  // components 64 hf + 32 w4 .. + 31
        uint32_t h[16], l[16];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            uint32_t hh[4], ll[4];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const float a = e[32 * w4 + 8 * u + 2 * q], b = e[32 * w4 + 8 * u + 2 * q + 1];
                hh[q] = pack_bf2(a, b);
                ll[q] = pack_bf2(a - bf_lo(hh[q]), b - bf_hi(hh[q]));
            }
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                h[4 * u + q] = hh[q];
                l[4 * u + q] = ll[q];
            }
        }
        tmem_st16(s_taddr + 32 * hf + 16 * w4, h);
        tmem_st16(s_taddr + 64 + 32 * hf + 16 * w4, l);
    }
    tmem_wait_st();
    xb[2 * kT + hf * kT + row] = (s0.x + s0.y) + (s1.x + s1.y);
    xb[4 * kT + hf * kT + row] = d0 + d1;
    __syncwarp();
    if (lane == 0) mbar_arrive(ms);
    if (!wait_or_abort(ms, ph, status, abort_flag)) return false;
    *r = xb[2 * kT + row] + xb[3 * kT + row];
    *den0 = xb[4 * kT + row] + xb[5 * kT + row];
    return true;
}

// Key softmax of half `hf` of one row (components 64 hf .. 64 hf + 63), run by
// the threads of both warp groups that own the row: the halves' maxima and sums
// meet in xb ([max | sum][half][128] fp32) through the mbarriers mx and ms (8
// warps each, phase ph); the row sum is the half-0 sum plus the half-1 sum.
// The half's normalised Gamma^K goes into R (its 64-component atom of the 4 KB
// groups) once `freed` says num has read S from there.  Returns false on a
// timeout.
__device__ __noinline__ bool key_half128(uint32_t s_taddr, const float *cvec, int hf, int valid, uint8_t *R,
                                         int row, float *xb, uint64_t *mx, uint64_t *ms, uint64_t *freed,
                                         uint32_t ph, unsigned *status, int *abort_flag) {
    float e[64];
    float m = -INFINITY;
#pragma unroll
    for (int q = 0; q < 2; ++q) {
        uint32_t v[32];
        tmem_ld32(s_taddr + 64 * hf + 32 * q, v);
        tmem_wait_ld();
        const float4 *c4 = reinterpret_cast<const float4 *>(cvec + 64 * hf + 32 * q);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const float4 c = c4[i];
            const float2 a = f2_add(make_float2(__uint_as_float(v[4 * i]), __uint_as_float(v[4 * i + 1])),
                                    make_float2(c.x, c.y));
            const float2 b = f2_add(make_float2(__uint_as_float(v[4 * i + 2]), __uint_as_float(v[4 * i + 3])),
                                    make_float2(c.z, c.w));
            e[32 * q + 4 * i] = a.x;
            e[32 * q + 4 * i + 1] = a.y;
            e[32 * q + 4 * i + 2] = b.x;
            e[32 * q + 4 * i + 3] = b.y;
            m = fmaxf(m, fmaxf(fmaxf(a.x, a.y), fmaxf(b.x, b.y)));
        }
    }
    tc_fence_before();
    const int lane = threadIdx.x & 31;
    xb[hf * kT + row] = m;
    __syncwarp();
    if (lane == 0) mbar_arrive(mx);
    if (!wait_or_abort(mx, ph, status, abort_flag)) return false;
    const float M = fmaxf(xb[row], xb[kT + row]);
    const float2 mm = make_float2(M, M);
    float2 s0 = make_float2(0.f, 0.f), s1 = make_float2(0.f, 0.f);
#pragma unroll
    for (int k = 0; k < 64; k += 4) {
        const float2 d0 = f2_sub(make_float2(e[k], e[k + 1]), mm), d1 = f2_sub(make_float2(e[k + 2], e[k + 3]), mm);
        e[k] = ex2(d0.x);
        e[k + 1] = ex2(d0.y);
        e[k + 2] = ex2(d1.x);
        e[k + 3] = ex2(d1.y);
        s0 = f2_add(s0, make_float2(e[k], e[k + 1]));
        s1 = f2_add(s1, make_float2(e[k + 2], e[k + 3]));
    }
    xb[2 * kT + hf * kT + row] = (s0.x + s0.y) + (s1.x + s1.y);
    __syncwarp();
    if (lane == 0) mbar_arrive(ms);
    if (!wait_or_abort(ms, ph, status, abort_flag)) return false;
    const float sc = valid ? 1.0f / (xb[2 * kT + row] + xb[3 * kT + row]) : 0.0f;
    if (!wait_or_abort(freed, ph, status, abort_flag)) return false;
    const float2 s2 = make_float2(sc, sc);
    uint8_t *rb = R + (row >> 3) * kGroupB + (row & 7) * 128 + hf * 2048;
#pragma unroll
    for (int w = 0; w < 8; ++w) {  // 8 components per 16-byte chunk
        uint32_t h[4], l[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const float2 g = f2_mul(make_float2(e[8 * w + 2 * q], e[8 * w + 2 * q + 1]), s2);
            h[q] = pack_bf2(g.x, g.y);
            const float2 r = f2_sub(g, make_float2(bf_lo(h[q]), bf_hi(h[q])));
            l[q] = pack_bf2(r.x, r.y);
        }
        uint8_t *p = rb + ((w ^ (row & 7)) << 4);
        *reinterpret_cast<uint4 *>(p) = make_uint4(h[0], h[1], h[2], h[3]);
        *reinterpret_cast<uint4 *>(p + 1024) = make_uint4(l[0], l[1], l[2], l[3]);
    }
    return true;
}

// State operand row k (component k) from 128 fp32 values: bf16 hi at R, lo at R +
// 32 KB, MN-major SW128: value column n of half n / 64 at row k of that half's
// [128 x 64] block.
__device__ __forceinline__ void state_row128(uint8_t *R, int k, const uint32_t (&v)[32], int q) {
    // v: value columns 32 q .. 32 q + 31
    const int hf = q >> 1;
    uint8_t *rb = R + hf * kHalf + (k >> 3) * 1024 + (k & 7) * 128;
#pragma unroll
    for (int c4 = 0; c4 < 4; ++c4) {  // 8 columns per 16-byte chunk
        const int cc = 4 * (q & 1) + c4;
        uint32_t h[4], l[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const float a = __uint_as_float(v[8 * c4 + 2 * u]), b = __uint_as_float(v[8 * c4 + 2 * u + 1]);
            h[u] = pack_bf2(a, b);
            l[u] = pack_bf2(a - bf_lo(h[u]), b - bf_hi(h[u]));
        }
        uint8_t *p = rb + ((cc ^ (k & 7)) << 4);
        *reinterpret_cast<uint4 *>(p) = make_uint4(h[0], h[1], h[2], h[3]);
        *reinterpret_cast<uint4 *>(p + 2 * kHalf) = make_uint4(l[0], l[1], l[2], l[3]);
    }
}

// The state operand from the fp32 state in tensor memory (this thread's row k).
__device__ __noinline__ void state_operand128(uint32_t s_taddr, uint8_t *R, int k) {
#pragma unroll 1
    for (int q = 0; q < 4; ++q) {
        uint32_t v[32];
        tmem_ld32(s_taddr + 32 * q, v);
        tmem_wait_ld();
        state_row128(R, k, v, q);
    }
}

// Job start, by the key group: this thread's row k of the carried-in fp32 prefix
// (row-major [128][128] in R) into the state columns of tensor memory and into
// the state operand, which overwrites R once every key thread has read its row
// (each warp arrives on `read`, phase `ph`, and waits for the other three).
// Returns false on a timeout.
__device__ __noinline__ bool init_state128(uint8_t *R, int k, uint32_t s_taddr, uint64_t *read, uint32_t ph,
                                           unsigned *status, int *abort_flag) {
    uint32_t v0[32], v1[32], v2[32], v3[32];
    const uint4 *src = reinterpret_cast<const uint4 *>(R + k * 512);
#pragma unroll
    for (int u = 0; u < 8; ++u) {
        const uint4 a = src[u], b = src[8 + u], c = src[16 + u], d = src[24 + u];
        v0[4 * u] = a.x; v0[4 * u + 1] = a.y; v0[4 * u + 2] = a.z; v0[4 * u + 3] = a.w;
        v1[4 * u] = b.x; v1[4 * u + 1] = b.y; v1[4 * u + 2] = b.z; v1[4 * u + 3] = b.w;
        v2[4 * u] = c.x; v2[4 * u + 1] = c.y; v2[4 * u + 2] = c.z; v2[4 * u + 3] = c.w;
        v3[4 * u] = d.x; v3[4 * u + 1] = d.y; v3[4 * u + 2] = d.z; v3[4 * u + 3] = d.w;
    }
    __syncwarp();
    if ((threadIdx.x & 31) == 0) mbar_arrive(read);
    if (!wait_or_abort(read, ph, status, abort_flag)) return false;
    tmem_st32(s_taddr, v0);
    tmem_st32(s_taddr + 32, v1);
    tmem_st32(s_taddr + 64, v2);
    tmem_st32(s_taddr + 96, v3);
    state_row128(R, k, v0, 0);
    state_row128(R, k, v1, 1);
    state_row128(R, k, v2, 2);
    state_row128(R, k, v3, 3);
    tmem_wait_st();
    return true;
}

// Outputs of one chunk's query rows, O = num / den, by each query warp for its
// 32 rows: staged in the warp's 8 KB slice of `stage` and written by TMA stores
// (which clip rows past N): fp32 O in two rounds of 64 columns (two boxes of 32
// rows x 32 columns each, 128-byte swizzle), bf16 O in one round (two boxes of
// 32 rows x 64 columns).  The whole accumulator row is read first (the second
// fp32 half into registers), and lane 0 arrives on `xfree` (if given), so the
// columns can take the next tile's operands while the stores go out; lane 0
// issues the stores and waits until they have read the staging slice.
__device__ __noinline__ void output_rows128(uint32_t o_taddr, float inv, uint8_t *stage, int lane, int o_bf16,
                                            const CUtensorMap *tmO, int row0, int bh, uint64_t *xfree) {
    const int sw = lane & 7;
    if (o_bf16) {
#pragma unroll 1
        for (int q = 0; q < 4; ++q) {
            uint32_t v[32];
            tmem_ld32(o_taddr + 32 * q, v);
            tmem_wait_ld();
            uint8_t *rp = stage + (q >> 1) * 4096 + lane * 128;
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                uint32_t w[4];
#pragma unroll
                for (int z = 0; z < 4; ++z)
                    w[z] = pack_bf2(__uint_as_float(v[8 * u + 2 * z]) * inv, __uint_as_float(v[8 * u + 2 * z + 1]) * inv);
                *reinterpret_cast<uint4 *>(rp + (((4 * (q & 1) + u) ^ sw) << 4)) = make_uint4(w[0], w[1], w[2], w[3]);
            }
        }
        tc_fence_before();
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
            if (xfree) mbar_arrive(xfree);
            tma_store_3d(tmO, stage, 0, row0, bh);
            tma_store_3d(tmO, stage + 4096, 64, row0, bh);
            bulk_commit();
            bulk_wait_read0();
        }
        __syncwarp();
        return;
    }
    // columns 0 .. 63 staged, 64 .. 127 held in registers
#pragma unroll 1
    for (int b = 0; b < 2; ++b) {
        uint32_t v[32];
        tmem_ld32(o_taddr + 32 * b, v);
        tmem_wait_ld();
        uint8_t *rp = stage + b * 4096 + lane * 128;
#pragma unroll
        for (int c = 0; c < 8; ++c)
            *reinterpret_cast<float4 *>(rp + ((c ^ sw) << 4)) =
                make_float4(__uint_as_float(v[4 * c]) * inv, __uint_as_float(v[4 * c + 1]) * inv,
                            __uint_as_float(v[4 * c + 2]) * inv, __uint_as_float(v[4 * c + 3]) * inv);
    }
    uint32_t h0[32], h1[32];
    tmem_ld32(o_taddr + 64, h0);
    tmem_ld32(o_taddr + 96, h1);
    tmem_wait_ld();
    tc_fence_before();
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) {
        if (xfree) mbar_arrive(xfree);
        tma_store_3d(tmO, stage, 0, row0, bh);
        tma_store_3d(tmO, stage + 4096, 32, row0, bh);
        bulk_commit();
        bulk_wait_read0();  // the slice is read before the second round overwrites it
    }
    __syncwarp();
#pragma unroll
    for (int b = 0; b < 2; ++b) {
        const uint32_t *v = b ? h1 : h0;
        uint8_t *rp = stage + b * 4096 + lane * 128;
#pragma unroll
        for (int c = 0; c < 8; ++c)
            *reinterpret_cast<float4 *>(rp + ((c ^ sw) << 4)) =
                make_float4(__uint_as_float(v[4 * c]) * inv, __uint_as_float(v[4 * c + 1]) * inv,
                            __uint_as_float(v[4 * c + 2]) * inv, __uint_as_float(v[4 * c + 3]) * inv);
    }
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) {
        tma_store_3d(tmO, stage, 64, row0, bh);
        tma_store_3d(tmO, stage + 4096, 96, row0, bh);
        bulk_commit();
        bulk_wait_read0();
    }
    __syncwarp();
}

__global__ void __launch_bounds__(kThreadsC128, 1) tc128_causal_kernel(
    const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
    const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmO,
    const uint8_t *__restrict__ coef_img, const float *__restrict__ part, const float *__restrict__ ztile, int H,
    int N, Part128 P, float eps, int o_bf16, unsigned *status) {
    using L = Causal128Smem;
    constexpr int CS = L::kCS;
    // kA: x^2 of Q, then the key scores, U and P; kB: x^2 of K, then num and O
    constexpr int kA = 0, kGQ = 128, kB = 256, kSA = 384, kTmemCols = 512;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t *qst = smem + L::kQ, *kst = smem + L::kK, *vst = smem + L::kV, *R = smem + L::kR, *ring = smem + L::kCf;
    float *cvec = reinterpret_cast<float *>(smem + L::kC), *zp = reinterpret_cast<float *>(smem + L::kZp);
    float *rsk = reinterpret_cast<float *>(smem + L::kRs);
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + L::kBars);
    uint64_t *qfull = bars, *qempty = bars + 1, *kfull = bars + 2, *kempty = bars + 3, *vfull = bars + 4,
             *vempty = bars + 5, *cffull = bars + 6, *cfempty = cffull + CS, *xq = cfempty + CS, *xk = xq + 1,
             *sq = xq + 2, *sk = xq + 3, *gq = xq + 4, *gk = xq + 5, *sready = xq + 6, *ndone = xq + 7,
             *ufull = xq + 8, *wdone = xq + 9, *pready = xq + 10, *ofull = xq + 11, *cfull = xq + 12,
             *xfull = xq + 13, *pread = xq + 14, *kmx = xq + 15, *ksm = xq + 16, *qmx = xq + 17,
             *qsm = xq + 18;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(qsm + 1);
    int *abort_flag = reinterpret_cast<int *>(qsm + 2);
    static_assert((6 + 2 * CS + 19) * 8 + 16 <= 512, "barrier area");

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int c = blockIdx.x;
    const int g0 = c * P.tpc, gend = min(P.total, g0 + P.tpc);
    if (failed(status) || g0 >= gend) return;

    if (warp == 0) {
        tmem_alloc(tmem_slot, kTmemCols);
        tmem_relinquish();
    }
    if (tid == 32) {
        for (int i = 0; i < 6; ++i) mbar_init(&bars[i], 1);
        mbar_init(qempty, 8);  // both groups, once the query softmax exchange in the Q buffer is done
        mbar_init(kempty, 8);  // both groups, once the key softmax exchange in the K buffer is done
        mbar_init(vempty, 4);  // the query warps, once their outputs staged in the V buffer are out
        for (int i = 0; i < CS; ++i) {
            mbar_init(&cffull[i], 1);
            mbar_init(&cfempty[i], 1);
        }
        mbar_init(xq, 4); mbar_init(xk, 4); mbar_init(sq, 1); mbar_init(sk, 1);
        mbar_init(gq, 8); mbar_init(gk, 8); mbar_init(sready, 4); mbar_init(ndone, 1);
        mbar_init(ufull, 1); mbar_init(wdone, 1); mbar_init(pready, 8); mbar_init(ofull, 1);
        mbar_init(cfull, 1); mbar_init(xfull, 1); mbar_init(pread, 4);
        mbar_init(kmx, 8); mbar_init(ksm, 8); mbar_init(qmx, 8); mbar_init(qsm, 8);
        *abort_flag = 0;
        fence_mbar_init();
        tma_prefetch_desc(&tmQ); tma_prefetch_desc(&tmK); tma_prefetch_desc(&tmV); tma_prefetch_desc(&tmO);
    }
    tc_fence_before();
    cta_sync();
    tc_fence_after();
    pdl_trigger();  // the next call's coefficient prep waits for this kernel's completion
    // The key group reads the aggregation's per-tile key mass directly.
    if (warp >= 6) pdl_wait();
    const uint32_t tmem = *tmem_slot;

    int rbase = 0, njob = 0;
    int barm = -1;  // last job whose c vector and prefix copies were armed
    uint32_t slab_lpar = 0u, slab_fpar = 0u, slab_lmask = 0u;  // slab ring state (see issue_scores128)
    for (int g = g0; g < gend; ++njob) {
        const int bh = g / P.ntiles, t0 = g % P.ntiles;
        const int n = min(P.ntiles - t0, gend - g);
        const int h = bh % H;
        const uint8_t *himg = coef_img + (size_t)h * kImgStride;
        // The previous job is done with c, R and the key mass.
        fence_proxy_async_smem();
        cta_sync();
        if (tid == 0) {
            mbar_arrive_expect_tx(cfull, 512);
            bulk_load(cvec, himg + kCoefC, 512, cfull);
        }
        if (tid == 33) {
            if (njob == 0) pdl_wait();  // the prefixes come from the aggregation kernel
            const float *pre = part + ((size_t)c * P.slots + slot128(P, c, bh)) * kPartFloats;
            mbar_arrive_expect_tx(xfull, 65536 + 512);
            bulk_load(R, pre, 65536, xfull);
            bulk_load(zp, pre + kKC * kD, 512, xfull);
        }
        barm = njob;

        if (warp == 0) {
            if (lane == 0) {
                int qa = -1, ka = -1, va = -1;
                for (int i = 0; i < n; ++i) {
                    const int r = rbase + i, y = (t0 + i) * kT;
                    if (!wait_or_abort(qempty, (r & 1) ^ 1, status, abort_flag)) break;
                    mbar_arrive_expect_tx(qfull, kTileB);
                    tma_load_3d(qst, &tmQ, 0, y, bh, qfull);
                    tma_load_3d(qst + kHalf, &tmQ, 64, y, bh, qfull);
                    qa = r;
                    if (!wait_or_abort(kempty, (r & 1) ^ 1, status, abort_flag)) break;
                    mbar_arrive_expect_tx(kfull, kTileB);
                    tma_load_3d(kst, &tmK, 0, y, bh, kfull);
                    tma_load_3d(kst + kHalf, &tmK, 64, y, bh, kfull);
                    ka = r;
                    if (!wait_or_abort(vempty, (r & 1) ^ 1, status, abort_flag)) break;
                    mbar_arrive_expect_tx(vfull, kTileB);
                    tma_load_3d(vst, &tmV, 0, y, bh, vfull);
                    tma_load_3d(vst + kHalf, &tmV, 64, y, bh, vfull);
                    va = r;
                }
                if (qa >= 0) mbar_wait(qfull, qa & 1);
                if (ka >= 0) mbar_wait(kfull, ka & 1);
                if (va >= 0) mbar_wait(vfull, va & 1);
            } else if (lane == 1) {
                // slabs: two sides per chunk (query forward, key backward)
                for (int i = 0; i < 2 * n; ++i)
                    if (!load_slabs128<CS>(ring, himg, (i & 1) == 0, i == 0, &slab_lpar, &slab_lmask, cffull, cfempty,
                                           status, abort_flag))
                        break;
                drain_slabs128<CS>(slab_lpar, slab_lmask, cffull);
            }
        } else if (warp == 1) {
            if (lane == 0) {
                // base descriptors; every MMA below adds a constant to one of them
                const uint64_t dq0 = sdesc_sw128(smem_u32(qst), 16, 1024), dk0 = sdesc_sw128(smem_u32(kst), 16, 1024);
                const uint64_t dring0 = sdesc_sw128(smem_u32(ring), 16, 1024);
                const uint64_t dS = sdesc_sw128(smem_u32(R), kHalf, 1024);     // state operand hi, MN-major B
                const uint64_t dG = sdesc_sw128(smem_u32(R), 16, kGroupB);      // Gamma^K hi, K-major B
                const uint64_t dGT = sdesc_sw128(smem_u32(R), 2048, kGroupB);   // Gamma^K^T hi, MN-major A
                const uint64_t dV = sdesc_sw128(smem_u32(vst), kHalf, 1024);    // V, MN-major B
                for (int i = 0; i < n; ++i) {
                    const int r = rbase + i, ph = r & 1;
                    // query scores
                    if (!wait_or_abort(xq, ph, status, abort_flag) || !wait_or_abort(qfull, ph, status, abort_flag)) break;
                    tc_fence_after();
                    if (!issue_scores128<CS, true>(tmem + kGQ, tmem + kA, dq0, dring0, &slab_fpar, SlabOrder{i == 0, 0},
                                                   cffull, cfempty, status, abort_flag))
                        break;
                    umma_commit(sq);
                    // key scores, into the x^2 columns of Q that the query scores read (issue order
                    // is execution order), from the x^2 of K prepared during the previous chunk
                    if (!wait_or_abort(xk, ph, status, abort_flag) || !wait_or_abort(kfull, ph, status, abort_flag)) break;
                    tc_fence_after();
                    if (!issue_scores128<CS, false>(tmem + kA, tmem + kB, dk0, dring0, &slab_fpar,
                                                    SlabOrder{0, i == n - 1}, cffull, cfempty, status, abort_flag))
                        break;
                    umma_commit(sk);
                    // num = Gamma^Q S (hi.hi, hi.lo, lo.hi)
                    if (!wait_or_abort(gq, ph, status, abort_flag) || !wait_or_abort(sready, ph, status, abort_flag)) break;
                    tc_fence_after();
                    issue_num128(tmem + kB, tmem + kGQ, dS);
                    umma_commit(ndone);
                    // U = Gamma^Q Gamma^K^T
                    if (!wait_or_abort(gk, ph, status, abort_flag)) break;
                    tc_fence_after();
                    issue_u128(tmem + kA, tmem + kGQ, dG);
                    umma_commit(ufull);
                    // S += Gamma^K^T V (hi, lo)
                    if (!wait_or_abort(vfull, ph, status, abort_flag)) break;
                    tc_fence_after();
                    issue_supd128(tmem + kSA, dGT, dV, 1u);
                    umma_commit(wdone);
                    // num += P V (P hi / lo in place in the U columns)
                    if (!wait_or_abort(pready, ph, status, abort_flag)) break;
                    tc_fence_after();
                    issue_pv128(tmem + kB, tmem + kA, dV);
                    umma_commit(ofull);
                }
            }
        } else if (warp < 6) {
            // ---------------- query group: query softmax, half of the key softmax, half of
            // the P split, the outputs, and the next chunk's x^2 of K
            const int row = epi_row(warp, lane);
            const uint32_t lb = (uint32_t)(32 * (warp & 3)) << 16;
            float *xb = reinterpret_cast<float *>(kst);  // key softmax exchange (the K tile is consumed)
            float *xq_b = reinterpret_cast<float *>(qst);  // query softmax exchange (the Q tile is consumed)
            auto x2k = [&](int r) {  // x^2 of the key tile of chunk r, into the kB columns
                if (!wait_or_abort(kfull, r & 1, status, abort_flag)) return false;
                x2_row128(kst, row, tmem + lb + kB);
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(xk);
                return true;
            };
            bool ok = x2k(rbase);
            for (int i = 0; ok && i < n; ++i) {
                const int r = rbase + i, ph = r & 1;
                if (!(ok = wait_or_abort(sq, ph, status, abort_flag))) break;
                if (i == 0 && !(ok = wait_or_abort(cfull, njob & 1, status, abort_flag))) break;  // c_k visible
                if (!(ok = wait_or_abort(sready, ph, status, abort_flag))) break;                 // key mass Zp visible
                tc_fence_after();
                // components 64 .. 127 of the query softmax (exchange in the consumed Q tile)
                float rq, den0;
                if (!(ok = query_half128(tmem + lb + kGQ, cvec, zp, 1, row, xq_b, qmx, qsm, ph, &rq, &den0, status,
                                         abort_flag)))
                    break;
                fence_proxy_async_smem();  // the exchange's writes, before the next Q tile lands there
                tc_fence_before();
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive(gq);
                    mbar_arrive(qempty);
                }
                // components 64 .. 127 of the key softmax
                if (!(ok = wait_or_abort(sk, ph, status, abort_flag))) break;
                tc_fence_after();
                if (!(ok = key_half128(tmem + lb + kA, cvec, 1, (t0 + i) * kT + row < N, R, row, xb, kmx, ksm, ndone,
                                       ph, status, abort_flag)))
                    break;
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive(gk);
                    mbar_arrive(kempty);  // this warp is done with the exchange in the K buffer
                }
                if (!(ok = wait_or_abort(ufull, ph, status, abort_flag))) break;
                tc_fence_after();
                const float rs0 = split_p_blocks128(tmem + lb + kA, 0, row);
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(pready);
                if (!(ok = wait_or_abort(ofull, ph, status, abort_flag))) break;
                if (!(ok = wait_or_abort(pready, ph, status, abort_flag))) break;  // the key group's row sums
                tc_fence_after();
                // outputs staged in the V tile buffer (the state update and P V, its last
                // readers, are complete: ofull), which the next value tile may then reuse
                output_rows128(tmem + lb + kB, 1.0f / (den0 + (rs0 + rsk[row]) + eps * rq), vst + (warp & 3) * 8192,
                               lane, o_bf16, &tmO, (t0 + i) * kT + 32 * (warp & 3), bh, nullptr);
                tc_fence_before();
                if (lane == 0) mbar_arrive(vempty);
                // the next chunk's x^2 of K, now that this chunk's outputs are out of kB
                if (i + 1 < n && !(ok = x2k(r + 1))) break;
            }
        } else {
            // ---------------- key group: the next chunk's x^2 of Q, half of the key softmax,
            // half of the P split, the state operand
            const int row = epi_row(warp, lane);
            const uint32_t lb = (uint32_t)(32 * (warp & 3)) << 16;
            float *xb = reinterpret_cast<float *>(kst);
            float *xq_b = reinterpret_cast<float *>(qst);
            auto x2q = [&](int r) {  // x^2 of the query tile of chunk r, into the kA columns
                if (!wait_or_abort(qfull, r & 1, status, abort_flag)) return false;
                x2_row128(qst, row, tmem + lb + kA);
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(xq);
                return true;
            };
            // job start: the carried-in state (fp32 rows in R) -> tensor memory and the
            // state operand
            if (wait_or_abort(xfull, njob & 1, status, abort_flag))
                init_state128(R, row, tmem + lb + kSA, pread, njob & 1, status, abort_flag);
            fence_proxy_async_smem();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(sready);
            bool ok = x2q(rbase);
            for (int i = 0; ok && i < n; ++i) {
                const int r = rbase + i, ph = r & 1;
                const float *zr = ztile + ((size_t)bh * P.ntiles + t0 + i) * 4 * kKC + row;
                const float zt = ((__ldcg(zr) + __ldcg(zr + kKC)) + __ldcg(zr + 2 * kKC)) + __ldcg(zr + 3 * kKC);
                // components 0 .. 63 of the query softmax
                if (!(ok = wait_or_abort(sq, ph, status, abort_flag))) break;
                if (i == 0 && !(ok = wait_or_abort(cfull, njob & 1, status, abort_flag))) break;  // c_k visible
                if (!(ok = wait_or_abort(sready, ph, status, abort_flag))) break;                 // every Zp row
                tc_fence_after();
                {
                    float rq_, den0_;
                    if (!(ok = query_half128(tmem + lb + kGQ, cvec, zp, 0, row, xq_b, qmx, qsm, ph, &rq_, &den0_,
                                             status, abort_flag)))
                        break;
                }
                fence_proxy_async_smem();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive(gq);
                    mbar_arrive(qempty);
                }
                if (!(ok = wait_or_abort(sk, ph, status, abort_flag))) break;
                tc_fence_after();
                // components 0 .. 63 of the key softmax; Gamma^K into R once num has read S
                if (!(ok = key_half128(tmem + lb + kA, cvec, 0, (t0 + i) * kT + row < N, R, row, xb, kmx, ksm, ndone,
                                       ph, status, abort_flag)))
                    break;
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive(gk);
                    mbar_arrive(kempty);
                }
                if (!(ok = wait_or_abort(ufull, ph, status, abort_flag))) break;
                tc_fence_after();
                rsk[row] = split_p_blocks128(tmem + lb + kA, 2, row);
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(pready);
                // the next chunk's state operand and key mass, once U and the state
                // update have read Gamma^K; then its x^2 of Q, once P V has read P (kA)
                if (!(ok = wait_or_abort(wdone, ph, status, abort_flag))) break;
                tc_fence_after();
                if (i + 1 < n) {
                    state_operand128(tmem + lb + kSA, R, row);
                    zp[row] += zt;
                    fence_proxy_async_smem();
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(sready);
                    if (!(ok = wait_or_abort(ofull, ph, status, abort_flag))) break;
                    tc_fence_after();
                    if (!(ok = x2q(r + 1))) break;
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

// ------------------------------------------------------------------ bidirectional read
//
// Eq. (7) at d_r = d_v = 128: O = Gamma^Q [Vt | Z] / (. + eps) from the head's
// memory (the aggregation's mode-0 total).  Per query tile: x^2, 40 score MMAs
// (slabs in the snake order, one side per tile), the query softmax (Gamma^Q =
// e un-normalised, in place; e . Z and the row sum r in fp32), num = Gamma^Q Vt
// (24 MMAs against the memory's bf16 hi | lo operand, built in shared memory at
// each job start), O = num / (e . Z + eps r) staged and stored by TMA.
// Warps: 0 lane 0 Q loads (two stages), lane 1 slabs; 1 lane 0 MMA issue; 2..5
// epilogue.  TMEM: x^2 of tile t at [128 (t % 2), +128); scores -> Gamma^Q
// [256, 384); num [384, 512).  The next tile's score MMAs run beside this
// tile's outputs.
struct Read128Smem {
    static constexpr int kQS = 2, kCS = 4;
    static constexpr int kQ = 0;                        // Q stages
    static constexpr int kR = kQ + kQS * kTileB;        // memory operand (hi 32 KB | lo 32 KB)
    static constexpr int kCf = kR + 65536;              // coefficient slab ring
    static constexpr int kStage = kCf + kCS * kSlab;    // output staging, 4 warps x 8 KB
    static constexpr int kC = kStage + 4 * 8192;        // c [128] fp32
    static constexpr int kZ = kC + 512;                 // Z [128] fp32
    static constexpr int kBars = kZ + 512;
    static constexpr int kBytes = kBars + 256;
    static constexpr int kAlloc = kBytes + 1024;
    static_assert(kR % 1024 == 0 && kCf % 1024 == 0 && kStage % 1024 == 0, "SW128 alignment");
    static_assert(kAlloc <= 232448, "shared memory budget");
};
constexpr int kThreadsRead128 = 64 + 128;

__global__ void __launch_bounds__(kThreadsRead128, 1) tc128_read_kernel(
    const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmO,
    const uint8_t *__restrict__ coef_img, const float *__restrict__ mem, int H, Part128 P, float eps, int o_bf16,
    unsigned *status) {
    using L = Read128Smem;
    constexpr int QS = L::kQS, CS = L::kCS;
    constexpr int kX0 = 0, kGQ = 256, kO = 384, kTmemCols = 512;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t *qst = smem + L::kQ, *R = smem + L::kR, *ring = smem + L::kCf, *stg = smem + L::kStage;
    float *cvec = reinterpret_cast<float *>(smem + L::kC), *zs = reinterpret_cast<float *>(smem + L::kZ);
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + L::kBars);
    uint64_t *qfull = bars, *qempty = qfull + QS, *cffull = qempty + QS, *cfempty = cffull + CS,
             *xq = cfempty + CS, *sq = xq + 2, *gq = sq + 1, *nfull = gq + 1, *ofree = nfull + 1, *sready = ofree + 1,
             *cfull = sready + 1;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(cfull + 1);
    int *abort_flag = reinterpret_cast<int *>(cfull + 2);
    static_assert((2 * QS + 2 * CS + 9) * 8 + 16 <= 256, "barrier area");

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
        for (int i = 0; i < CS; ++i) {
            mbar_init(&cffull[i], 1);
            mbar_init(&cfempty[i], 1);
        }
        mbar_init(&xq[0], 4); mbar_init(&xq[1], 4); mbar_init(sq, 1); mbar_init(gq, 4); mbar_init(nfull, 1);
        mbar_init(ofree, 4); mbar_init(sready, 4); mbar_init(cfull, 1);
        *abort_flag = 0;
        fence_mbar_init();
        tma_prefetch_desc(&tmQ);
        tma_prefetch_desc(&tmO);
    }
    tc_fence_before();
    cta_sync();
    tc_fence_after();
    pdl_trigger();  // the next call's coefficient prep waits for this kernel's completion
    // the epilogue reads the aggregation's memories directly
    if (warp >= 2) pdl_wait();
    const uint32_t tmem = *tmem_slot;

    int rbase = 0, njob = 0;
    uint32_t slab_lpar = 0u, slab_fpar = 0u, slab_lmask = 0u;  // slab ring state (see issue_scores128)
    for (int g = g0; g < gend; ++njob) {
        const int bh = g / P.ntiles, t0 = g % P.ntiles;
        const int n = min(P.ntiles - t0, gend - g);
        const int h = bh % H;
        const uint8_t *himg = coef_img + (size_t)h * kImgStride;
        fence_proxy_async_smem();
        cta_sync();  // the previous job is done with c, the memory operand and Z
        if (tid == 0) {
            mbar_arrive_expect_tx(cfull, 512);
            bulk_load(cvec, himg + kCoefC, 512, cfull);
        }
        if (warp == 0) {
            if (lane == 0) {
                int qarm[QS];
#pragma unroll
                for (int q = 0; q < QS; ++q) qarm[q] = -1;
                for (int i = 0; i < n; ++i) {
                    const int r = rbase + i, s = r % QS;
                    if (!wait_or_abort(&qempty[s], ((r / QS) & 1) ^ 1, status, abort_flag)) break;
                    mbar_arrive_expect_tx(&qfull[s], kTileB);
                    tma_load_3d(qst + s * kTileB, &tmQ, 0, (t0 + i) * kT, bh, &qfull[s]);
                    tma_load_3d(qst + s * kTileB + kHalf, &tmQ, 64, (t0 + i) * kT, bh, &qfull[s]);
                    qarm[s] = r;
                }
#pragma unroll
                for (int q = 0; q < QS; ++q)
                    if (qarm[q] >= 0) mbar_wait(&qfull[q], (qarm[q] / QS) & 1);
            } else if (lane == 1) {
                for (int i = 0; i < n; ++i)
                    if (!load_slabs128<CS>(ring, himg, (i & 1) == 0, i == 0, &slab_lpar, &slab_lmask, cffull, cfempty,
                                           status, abort_flag))
                        break;
                drain_slabs128<CS>(slab_lpar, slab_lmask, cffull);
            }
        } else if (warp == 1) {
            if (lane == 0) {
                const uint64_t dq0 = sdesc_sw128(smem_u32(qst), 16, 1024), dring0 = sdesc_sw128(smem_u32(ring), 16, 1024);
                const uint64_t dS = sdesc_sw128(smem_u32(R), kHalf, 1024);
                for (int i = 0; i < n; ++i) {
                    const int r = rbase + i, ph = r & 1;
                    if (!wait_or_abort(&xq[r & 1], (r >> 1) & 1, status, abort_flag) ||
                        !wait_or_abort(&qfull[r % QS], (r / QS) & 1, status, abort_flag))
                        break;
                    tc_fence_after();
                    const SlabOrder so{i == 0, i == n - 1};
                    const uint32_t ax = tmem + kX0 + 128 * (r & 1);
                    const uint64_t dx = dadd(dq0, (r % QS) * kTileB);
                    if (!((i & 1) == 0 ? issue_scores128<CS, true>(tmem + kGQ, ax, dx, dring0, &slab_fpar, so, cffull,
                                                                   cfempty, status, abort_flag)
                                       : issue_scores128<CS, false>(tmem + kGQ, ax, dx, dring0, &slab_fpar, so, cffull,
                                                                    cfempty, status, abort_flag)))
                        break;
                    umma_commit(sq);
                    umma_commit(&qempty[r % QS]);
                    // num = Gamma^Q [Vt], once the previous tile's outputs are out of its columns
                    if (!wait_or_abort(gq, ph, status, abort_flag)) break;
                    if (i == 0 && !wait_or_abort(sready, njob & 1, status, abort_flag)) break;
                    if (r > 0 && !wait_or_abort(ofree, (r - 1) & 1, status, abort_flag)) break;
                    tc_fence_after();
                    issue_num128(tmem + kO, tmem + kGQ, dS);
                    umma_commit(nfull);
                }
            }
        } else {
            // ---------------- epilogue: one thread per tile row (and per memory row)
            const int row = epi_row(warp, lane);
            const uint32_t lb = (uint32_t)(32 * (warp & 3)) << 16;
            uint8_t *stage = stg + (warp & 3) * 8192;
            // job start: the head's memory (fp32 [Vt | Z] rows) -> the bf16 hi | lo operand and Z
            {
                const float *mr = mem + (size_t)bh * kPartFloats + (size_t)row * kD;
#pragma unroll 1
                for (int q = 0; q < 4; ++q) {
                    uint32_t v[32];
#pragma unroll
                    for (int u = 0; u < 8; ++u) {
                        const float4 a = __ldcg(reinterpret_cast<const float4 *>(mr + 32 * q) + u);
                        v[4 * u] = __float_as_uint(a.x);
                        v[4 * u + 1] = __float_as_uint(a.y);
                        v[4 * u + 2] = __float_as_uint(a.z);
                        v[4 * u + 3] = __float_as_uint(a.w);
                    }
                    state_row128(R, row, v, q);
                }
                zs[row] = __ldcg(mem + (size_t)bh * kPartFloats + kKC * kD + row);
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(sready);
            }
            auto x2 = [&](int r) {
                if (!wait_or_abort(&qfull[r % QS], (r / QS) & 1, status, abort_flag)) return false;
                x2_row128(qst + (r % QS) * kTileB, row, tmem + lb + kX0 + 128 * (r & 1));
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&xq[r & 1]);
                return true;
            };
            bool ok = x2(rbase) && wait_or_abort(cfull, njob & 1, status, abort_flag) &&
                      wait_or_abort(sready, njob & 1, status, abort_flag);  // c and every Z row visible
            for (int i = 0; ok && i < n; ++i) {
                const int r = rbase + i, ph = r & 1;
                if (!(ok = wait_or_abort(sq, ph, status, abort_flag))) break;
                tc_fence_after();
                float den0;
                const float rq = query_row128(tmem + lb + kGQ, cvec, zs, &den0);
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(gq);
                // the next tile's x^2 (its buffer was read by tile i - 1's score MMAs)
                if (i + 1 < n && !(ok = x2(r + 1))) break;
                if (!(ok = wait_or_abort(nfull, ph, status, abort_flag))) break;
                tc_fence_after();
                output_rows128(tmem + lb + kO, 1.0f / (den0 + eps * rq), stage, lane, o_bf16, &tmO,
                               (t0 + i) * kT + 32 * (warp & 3), bh, ofree);
                tc_fence_before();
            }
        }
        rbase += n;
        g += n;
        cta_sync();
        if (aborted(abort_flag)) break;
    }
    if (tid == 0 && njob > 0) mbar_wait(cfull, (njob - 1) & 1);
    tc_fence_before();
    cta_sync();
    if (warp == 0) tmem_dealloc(tmem, kTmemCols);
}

// ------------------------------------------------------------------ host side

// [BH][N][128] bf16 tensor, boxes of 64 columns x 128 rows x 1 head, 128-byte
// swizzle (two boxes per tile); rows past N read as zero.
bool make_map128(CUtensorMap *map, const void *base, int BH, int N) {
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[3] = {(cuuint64_t)kD, (cuuint64_t)N, (cuuint64_t)BH};
    cuuint64_t strides[2] = {(cuuint64_t)kD * 2, (cuuint64_t)N * kD * 2};
    cuuint32_t box[3] = {64, (cuuint32_t)kT, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// O [BH][N][128] (fp32 or bf16) for TMA stores of [32 rows x 128 bytes] boxes,
// 128-byte swizzle.
bool make_out_map128(CUtensorMap *map, void *base, int BH, int N, bool bf16) {
    auto fn = encode_fn();
    if (!fn) return false;
    const int es = bf16 ? 2 : 4;
    cuuint64_t dims[3] = {(cuuint64_t)kD, (cuuint64_t)N, (cuuint64_t)BH};
    cuuint64_t strides[2] = {(cuuint64_t)kD * es, (cuuint64_t)N * kD * es};
    cuuint32_t box[3] = {(cuuint32_t)(128 / es), 32, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = fn(map, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, base, dims,
                    strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// Workspace: status | per-head job counters | prep error words | per-head
// coefficient images | job memories [ctas][slots][kPartFloats] | key mass of
// every tile [BH][ntiles][4][128] (per-warp partials) | per-head memories
// [BH][kPartFloats] (bidirectional).  The prep clears the status and the counters;
// everything else is written before it is read.
struct Tc128Layout {
    Part128 P;
    int nctas = 0;
    size_t counters = 0, head_err = 0, coef = 0, part = 0, ztile = 0, mem = 0, total = 0;
};

Tc128Layout tc128_layout(const Problem &p, int splits) {
    Tc128Layout L;
    const int ntiles = (p.N + kT - 1) / kT;
    const int total = p.BH() * ntiles;
    int nct = splits > 0 ? splits : num_sms();
    nct = nct < 1 ? 1 : (nct > total ? total : nct);
    const int tpc = (total + nct - 1) / nct;
    L.nctas = (total + tpc - 1) / tpc;
    L.P = Part128{ntiles, total, tpc, tpc / ntiles + 2};
    size_t off = kStatusBytes;
    L.counters = off;
    off = align256(off + sizeof(unsigned) * (size_t)p.BH());
    L.head_err = off;
    off = align256(off + sizeof(unsigned) * (size_t)p.H * kPrepBlocks128);
    L.coef = off;
    off = align256(off + kImgStride * p.H);
    L.part = off;
    off = align256(off + sizeof(float) * (size_t)L.nctas * L.P.slots * kPartFloats);
    L.ztile = off;  // key mass of every tile as four per-warp partial rows
    off = align256(off + sizeof(float) * (size_t)p.BH() * ntiles * 4 * kKC);
    L.mem = off;  // the bidirectional call's per-head memories
    off = align256(off + sizeof(float) * (size_t)p.BH() * kPartFloats);
    L.total = off;
    return L;
}

}  // namespace

bool tc128_supported(const Problem &p, int causal) {
    return (causal == 0 || causal == 1) && p.dtype == GMA_BF16 && p.d_r == kD && p.d_v == kD && p.K <= kKC;
}

size_t tc128_workspace(const Problem &p, int splits) { return tc128_layout(p, splits).total; }

cudaError_t tc128_causal(const Problem &p, int splits, void *workspace, cudaStream_t s, StageClock &clk) {
    const Tc128Layout L = tc128_layout(p, splits);
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    unsigned *status = reinterpret_cast<unsigned *>(ws);
    unsigned *counters = reinterpret_cast<unsigned *>(ws + L.counters);
    unsigned *head_err = reinterpret_cast<unsigned *>(ws + L.head_err);
    uint8_t *coef = ws + L.coef;
    float *part = reinterpret_cast<float *>(ws + L.part);
    float *ztile = reinterpret_cast<float *>(ws + L.ztile);
    CUtensorMap tq, tk, tv, to;
    if (!make_map128(&tq, p.Q, p.BH(), p.N) || !make_map128(&tk, p.Kx, p.BH(), p.N) ||
        !make_map128(&tv, p.V, p.BH(), p.N) || !make_out_map128(&to, p.O, p.BH(), p.N, p.o_bf16))
        return cudaErrorInvalidValue;
    clk.mark();
    GMA_TRY(launch_pdl(tc128_prep_kernel, dim3(kPrepBlocks128, p.H), dim3(128), 0, s, p.mu, p.sigma2, p.log_pi, p.K,
                       coef, status, head_err, counters, p.BH()));
    clk.mark();
    GMA_TRY(set_smem(tc128_aggregate_kernel, Agg128Smem::kAlloc));
    GMA_TRY(launch_pdl(tc128_aggregate_kernel, dim3(L.nctas), dim3(kThreadsAgg), Agg128Smem::kAlloc, s, tk, tv,
                       static_cast<const uint8_t *>(coef), static_cast<const unsigned *>(head_err), p.H, p.N, L.P,
                       part, ztile, static_cast<float *>(nullptr), counters, 1, p.test_stall ? 1 : 0, status));
    clk.mark();
    GMA_TRY(set_smem(tc128_causal_kernel, Causal128Smem::kAlloc));
    GMA_TRY(launch_pdl(tc128_causal_kernel, dim3(L.nctas), dim3(kThreadsC128), Causal128Smem::kAlloc, s, tq, tk, tv,
                       to, static_cast<const uint8_t *>(coef), static_cast<const float *>(part),
                       static_cast<const float *>(ztile), p.H, p.N, L.P, p.eps, p.o_bf16 ? 1 : 0, status));
    clk.mark();
    return cudaSuccess;
}

cudaError_t tc128_bidir(const Problem &p, int splits, void *workspace, cudaStream_t s, StageClock &clk) {
    const Tc128Layout L = tc128_layout(p, splits);
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    unsigned *status = reinterpret_cast<unsigned *>(ws);
    unsigned *counters = reinterpret_cast<unsigned *>(ws + L.counters);
    unsigned *head_err = reinterpret_cast<unsigned *>(ws + L.head_err);
    uint8_t *coef = ws + L.coef;
    float *part = reinterpret_cast<float *>(ws + L.part);
    float *mem = reinterpret_cast<float *>(ws + L.mem);
    CUtensorMap tq, tk, tv, to;
    if (!make_map128(&tq, p.Q, p.BH(), p.N) || !make_map128(&tk, p.Kx, p.BH(), p.N) ||
        !make_map128(&tv, p.V, p.BH(), p.N) || !make_out_map128(&to, p.O, p.BH(), p.N, p.o_bf16))
        return cudaErrorInvalidValue;
    clk.mark();
    GMA_TRY(launch_pdl(tc128_prep_kernel, dim3(kPrepBlocks128, p.H), dim3(128), 0, s, p.mu, p.sigma2, p.log_pi, p.K,
                       coef, status, head_err, counters, p.BH()));
    clk.mark();
    GMA_TRY(set_smem(tc128_aggregate_kernel, Agg128Smem::kAlloc));
    GMA_TRY(launch_pdl(tc128_aggregate_kernel, dim3(L.nctas), dim3(kThreadsAgg), Agg128Smem::kAlloc, s, tk, tv,
                       static_cast<const uint8_t *>(coef), static_cast<const unsigned *>(head_err), p.H, p.N, L.P,
                       part, static_cast<float *>(nullptr), mem, counters, 0, p.test_stall ? 1 : 0, status));
    clk.mark();
    GMA_TRY(set_smem(tc128_read_kernel, Read128Smem::kAlloc));
    GMA_TRY(launch_pdl(tc128_read_kernel, dim3(L.nctas), dim3(kThreadsRead128), Read128Smem::kAlloc, s, tq, to,
                       static_cast<const uint8_t *>(coef), static_cast<const float *>(mem), p.H, L.P, p.eps,
                       p.o_bf16 ? 1 : 0, status));
    clk.mark();
    return cudaSuccess;
}

}  // namespace gma
