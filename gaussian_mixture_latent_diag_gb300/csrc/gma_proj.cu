// gma_proj.cu -- the Q/K/V projections in front of the hot path, as a tcgen05
// tensor-core GEMM that writes the head-major layouts the GMA kernels read.
//
// Paper: "Gaussian Mixture Attention: Linear-Time Sequence Mixing via
// Probabilistic Latent Routing" (arXiv 2606.18283), Eq. (4): the layer input
// X is projected to the routing rows Q_X, K_X and the values V_X (the display
// equation was lost in extraction; the plainest reading is Q_X = X W_Q etc.).
// With X [B, N, D] and each weight stored one output feature per row
// (W_Q [H d_r, D]):
//   Q_X[b, h, n, c] = sum_i X[b, n, i] W_Q[h d_r + c, i]     (likewise K_X, V_X)
//
// One CTA computes a 128-token x 256-feature tile of one projection (the
// widest MMA, N = 256, is the one that reaches the dense tensor rate, and the
// wide tile halves the re-reads of X from L2):
//   thread 0      TMA producer: X and W tiles of 64 input features (one 128-byte
//                 swizzle atom per row) into a ring of kProjStages stages
//   thread 32     MMA issuer: 4 x tcgen05.mma (M = 128, N = 256, K = 16) per
//                 stage, fp32 accumulator in tensor memory; each stage is
//                 released by tcgen05.commit when its MMAs complete
//   warps 0-3     epilogue: row m = 32 w + lane of the accumulator, rounded to
//                 bf16 (or kept fp32) and stored into the head-major output
// Every wait is bounded; a wait that runs out records GMA_ERR_TIMEOUT, and the
// CTA still waits (bounded) for the loads it armed and frees its tensor memory.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "gma_internal.h"
#include "tc_ptx.cuh"

namespace gma {
namespace {

using namespace ptx;

constexpr int kProjM = 128;     // tokens per tile
constexpr int kProjN = 256;     // output features per tile
constexpr int kProjK = 64;      // input features per stage (128 bytes of bf16)
constexpr int kProjStages = 2;  // 96 KB of stages: two CTAs per SM (2 x 256 TMEM columns)
constexpr int kProjXBytes = kProjM * kProjK * 2;  // 16 KB X tile
constexpr int kProjWBytes = kProjN * kProjK * 2;  // 32 KB W tile
constexpr int kProjSmem = kProjStages * (kProjXBytes + kProjWBytes) + 1024;

__device__ __forceinline__ uint64_t dadd(uint64_t desc, uint32_t bytes) { return desc + (uint64_t)(bytes >> 4); }

struct ProjOut {
    void *y[3];    // Q_X, K_X, V_X: [B][H][N][d_p]
    int d[3];      // d_r, d_r, d_v
    int tiles[3];  // feature tiles of each projection
};

// grid (tiles of Q + K + V features, ceil(B N / 128)), 128 threads.
template <bool OUT_BF16>
__global__ void __launch_bounds__(128) proj_kernel(const __grid_constant__ CUtensorMap tmX,
                                                   const __grid_constant__ CUtensorMap tmWq,
                                                   const __grid_constant__ CUtensorMap tmWk,
                                                   const __grid_constant__ CUtensorMap tmWv, ProjOut out, int Bn,
                                                   int N, int H, int D, unsigned *status) {
    extern __shared__ __align__(1024) uint8_t proj_smem[];
    // SW128 tiles want 1024-byte aligned stages
    uint8_t *base = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(proj_smem) + 1023) & ~uintptr_t(1023));
    uint8_t *sx = base;                                    // [stage][128 x 64] bf16
    uint8_t *sw = base + kProjStages * kProjXBytes;        // [stage][256 x 64] bf16
    __shared__ uint64_t full[kProjStages], empty[kProjStages], done;
    __shared__ uint32_t tmem_slot;
    __shared__ int abort_flag;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    int p = 0, t = blockIdx.x;
    while (p < 2 && t >= out.tiles[p]) t -= out.tiles[p++];
    const CUtensorMap *tmW = p == 0 ? &tmWq : (p == 1 ? &tmWk : &tmWv);
    const int o0 = t * kProjN, m0 = blockIdx.y * kProjM;
    const int nk = (D + kProjK - 1) / kProjK;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kProjStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        mbar_init(&done, 1);
        abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 0) {
        tmem_alloc(&tmem_slot, kProjN);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_slot;

    if (threadIdx.x == 0) {
        // producer: stage kb % S is refilled once the MMAs of kb - S released it
        tma_prefetch_desc(&tmX);
        tma_prefetch_desc(tmW);
        int armed = 0;
        for (int kb = 0; kb < nk; ++kb) {
            const int s = kb % kProjStages;
            if (kb >= kProjStages && !mbar_wait(&empty[s], ((kb / kProjStages) - 1) & 1)) {
                atomicCAS(status, 0u, (unsigned)GMA_ERR_TIMEOUT);
                atomicExch(&abort_flag, 1);
                break;
            }
            if (*reinterpret_cast<volatile int *>(&abort_flag)) break;
            mbar_arrive_expect_tx(&full[s], kProjXBytes + kProjWBytes);
            tma_load_3d(sx + s * kProjXBytes, &tmX, kb * kProjK, m0, 0, &full[s]);
            tma_load_3d(sw + s * kProjWBytes, tmW, kb * kProjK, o0, 0, &full[s]);
            armed = kb + 1;
        }
        // every load armed here has landed before the CTA leaves
        for (int kb = armed - kProjStages < 0 ? 0 : armed - kProjStages; kb < armed; ++kb)
            mbar_wait(&full[kb % kProjStages], (kb / kProjStages) & 1);
    } else if (threadIdx.x == 32) {
        // MMA issuer
        constexpr uint32_t idesc = idesc_bf16(kProjM, kProjN, false, false);
        for (int kb = 0; kb < nk; ++kb) {
            const int s = kb % kProjStages;
            if (!mbar_wait(&full[s], (kb / kProjStages) & 1)) {
                atomicCAS(status, 0u, (unsigned)GMA_ERR_TIMEOUT);
                atomicExch(&abort_flag, 1);
                break;
            }
            if (*reinterpret_cast<volatile int *>(&abort_flag)) break;
            tc_fence_after();
            const uint64_t da = sdesc_sw128(smem_u32(sx + s * kProjXBytes), 16, 1024);
            const uint64_t db = sdesc_sw128(smem_u32(sw + s * kProjWBytes), 16, 1024);
#pragma unroll
            for (int kk = 0; kk < kProjK / 16; ++kk)
                umma_bf16(tmem, dadd(da, kk * 32), dadd(db, kk * 32), idesc, (kb > 0 || kk > 0) ? 1u : 0u);
            umma_commit(&empty[s]);
        }
        umma_commit(&done);
    }
    __syncwarp();

    // epilogue: warp w holds rows 32 w .. 32 w + 31 of the tile in its TMEM lanes
    const bool ok = mbar_wait(&done, 0);
    if (!ok) atomicCAS(status, 0u, (unsigned)GMA_ERR_TIMEOUT);
    tc_fence_after();
    const int m = m0 + warp * 32 + lane;
    const bool write = ok && !*reinterpret_cast<volatile int *>(&abort_flag) && m < Bn * N;
    const int dp = out.d[p];
    const int O = H * dp;
    const int b = m / N, n = m % N;
#pragma unroll 1
    for (int c0 = 0; c0 < kProjN; c0 += 32) {
        uint32_t r[32];
        tmem_ld32(tmem + ((uint32_t)(warp * 32) << 16) + c0, r);
        tmem_wait_ld();
        if (!write) continue;
        // 32 consecutive features o0 + c0 .. + 31: one head when d_p >= 32,
        // else 32 / d_p heads of d_p features each
        const int seg = dp < 32 ? dp : 32;
#pragma unroll 1
        for (int s0 = 0; s0 < 32; s0 += seg) {
            const int o = o0 + c0 + s0;
            if (o >= O) break;
            const int h = o / dp, c = o % dp;
            const size_t off = (((size_t)b * H + h) * N + n) * dp + c;
            if (OUT_BF16) {
                uint4 *dst = reinterpret_cast<uint4 *>(static_cast<__nv_bfloat16 *>(out.y[p]) + off);
                for (int q = 0; q < seg / 8; ++q) {
                    const int i = s0 + 8 * q;
                    dst[q] = make_uint4(pack_bf2(__uint_as_float(r[i]), __uint_as_float(r[i + 1])),
                                        pack_bf2(__uint_as_float(r[i + 2]), __uint_as_float(r[i + 3])),
                                        pack_bf2(__uint_as_float(r[i + 4]), __uint_as_float(r[i + 5])),
                                        pack_bf2(__uint_as_float(r[i + 6]), __uint_as_float(r[i + 7])));
                }
            } else {
                float4 *dst = reinterpret_cast<float4 *>(static_cast<float *>(out.y[p]) + off);
                for (int q = 0; q < seg / 4; ++q) {
                    const int i = s0 + 4 * q;
                    dst[q] = make_float4(__uint_as_float(r[i]), __uint_as_float(r[i + 1]), __uint_as_float(r[i + 2]),
                                         __uint_as_float(r[i + 3]));
                }
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, kProjN);
}

PFN_cuTensorMapEncodeTiled_v12000 proj_encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
    });
    return fn;
}

// [rows][D] bf16 matrix, boxes of 64 features x box_rows rows, 128-byte
// swizzle; rows past `rows` and features past D read as zero.
bool proj_map(CUtensorMap *map, const void *ptr, int rows, int D, int box_rows) {
    auto fn = proj_encode_fn();
    if (!fn) return false;
    cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)rows, 1};
    cuuint64_t strides[2] = {(cuuint64_t)D * 2, (cuuint64_t)D * 2 * rows};
    cuuint32_t box[3] = {kProjK, (cuuint32_t)box_rows, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(ptr), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

size_t proj_workspace() { return kStatusBytes; }

cudaError_t tc_project_qkv(const void *X, const void *Wq, const void *Wk, const void *Wv, void *Q, void *Kx, void *V,
                           bool out_bf16, int B, int N, int D, int H, int d_r, int d_v, void *ws, cudaStream_t s) {
    CUtensorMap tx, tq, tk, tv;
    const int M = B * N;
    if (!proj_map(&tx, X, M, D, kProjM) || !proj_map(&tq, Wq, H * d_r, D, kProjN) ||
        !proj_map(&tk, Wk, H * d_r, D, kProjN) || !proj_map(&tv, Wv, H * d_v, D, kProjN))
        return cudaErrorInvalidValue;
    ProjOut out;
    out.y[0] = Q; out.y[1] = Kx; out.y[2] = V;
    out.d[0] = d_r; out.d[1] = d_r; out.d[2] = d_v;
    for (int p = 0; p < 3; ++p) out.tiles[p] = (H * out.d[p] + kProjN - 1) / kProjN;
    unsigned *status = static_cast<unsigned *>(ws);
    cudaError_t e = cudaMemsetAsync(status, 0, sizeof(unsigned), s);
    if (e != cudaSuccess) return e;
    const dim3 grid(out.tiles[0] + out.tiles[1] + out.tiles[2], (M + kProjM - 1) / kProjM);
    if (out_bf16) {
        e = cudaFuncSetAttribute(proj_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, kProjSmem);
        if (e != cudaSuccess) return e;
        proj_kernel<true><<<grid, 128, kProjSmem, s>>>(tx, tq, tk, tv, out, B, N, H, D, status);
    } else {
        e = cudaFuncSetAttribute(proj_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, kProjSmem);
        if (e != cudaSuccess) return e;
        proj_kernel<false><<<grid, 128, kProjSmem, s>>>(tx, tq, tk, tv, out, B, N, H, D, status);
    }
    return cudaGetLastError();
}

}  // namespace gma
