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
// Persistent kernel, one CTA per SM, each CTA taking every gridDim.x-th tile
// (128 tokens x 256 features of one projection; feature tiles vary fastest, so
// the CTAs running side by side share the same tokens' X tile in L2):
//   warp 0, lane 0   TMA producer: X and W tiles of 64 input features (one
//                    128-byte swizzle atom per row) into a ring of kProjStages stages
//   warp 1, lane 0   MMA issuer: 4 x tcgen05.mma (M = 128, N = 256, K = 16) per
//                    stage into one of two fp32 accumulators in tensor memory
//                    (2 x 256 columns); each stage is released by tcgen05.commit
//                    when its MMAs complete, each accumulator when its tile's do
//   warps 2-5        epilogue: accumulator row 32 (w % 4) + lane, rounded to bf16
//                    (or kept fp32) and stored into the head-major output, while
//                    the MMAs of the next tile fill the other accumulator
// Every wait is bounded; a wait that runs out records GMA_ERR_TIMEOUT and the
// CTA winds down: it still waits (bounded) for the loads and MMAs it issued and
// frees its tensor memory.
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
constexpr int kProjStages = 4;  // 192 KB of stages: one CTA per SM
constexpr int kProjXBytes = kProjM * kProjK * 2;  // 16 KB X tile
constexpr int kProjWBytes = kProjN * kProjK * 2;  // 32 KB W tile
constexpr int kProjSmem = kProjStages * (kProjXBytes + kProjWBytes) + 1024;
constexpr int kProjThreads = 192;                 // producer warp, MMA warp, 4 epilogue warps

__device__ __forceinline__ uint64_t dadd(uint64_t desc, uint32_t bytes) { return desc + (uint64_t)(bytes >> 4); }

struct ProjOut {
    void *y[3];    // Q_X, K_X, V_X: [B][H][N][d_p]
    int d[3];      // d_r, d_r, d_v
    int tiles[3];  // feature tiles of each projection
};

__device__ __forceinline__ bool aborted(const int *flag) { return *reinterpret_cast<const volatile int *>(flag) != 0; }
__device__ __forceinline__ void give_up(unsigned *status, int *flag) {
    atomicCAS(status, 0u, (unsigned)GMA_ERR_TIMEOUT);
    atomicExch(flag, 1);
}

template <bool OUT_BF16>
__device__ __forceinline__ void store_row_chunk(const ProjOut &out, int p, int dp, int H, int N, int b, int n, int o0,
                                                const uint32_t (&r)[32]) {
    // 32 consecutive features o0 .. o0 + 31: one head when d_p >= 32, else
    // 32 / d_p heads of d_p features each
    const int O = H * dp;
    const int seg = dp < 32 ? dp : 32;
#pragma unroll 1
    for (int s0 = 0; s0 < 32; s0 += seg) {
        const int o = o0 + s0;
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

// grid min(tiles, SMs), kProjThreads threads.  Tile t: row tile t / FT,
// feature tile t % FT over the Q, K, V feature tiles in that order.
template <bool OUT_BF16>
__global__ void __launch_bounds__(kProjThreads, 1) proj_kernel(const __grid_constant__ CUtensorMap tmX,
                                                               const __grid_constant__ CUtensorMap tmWq,
                                                               const __grid_constant__ CUtensorMap tmWk,
                                                               const __grid_constant__ CUtensorMap tmWv,
                                                               ProjOut out, int Bn, int N, int H, int D,
                                                               int stall, unsigned *status) {
    extern __shared__ __align__(1024) uint8_t proj_smem[];
    // SW128 tiles want 1024-byte aligned stages
    uint8_t *base = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(proj_smem) + 1023) & ~uintptr_t(1023));
    uint8_t *sx = base;                                    // [stage][128 x 64] bf16
    uint8_t *sw = base + kProjStages * kProjXBytes;        // [stage][256 x 64] bf16
    __shared__ uint64_t full[kProjStages], empty[kProjStages], acc_full[2], acc_empty[2], drain;
    __shared__ uint32_t tmem_slot;
    __shared__ int abort_flag;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int FT = out.tiles[0] + out.tiles[1] + out.tiles[2];
    const int M = Bn * N;
    const int ntiles = FT * ((M + kProjM - 1) / kProjM);
    const int nk = (D + kProjK - 1) / kProjK;
    // tile -> projection, first feature, first token
    auto decode_tile = [&](int t, int &p, int &o0, int &m0) {
        int f = t % FT;
        m0 = (t / FT) * kProjM;
        p = 0;
        while (p < 2 && f >= out.tiles[p]) f -= out.tiles[p++];
        o0 = f * kProjN;
    };

    if (threadIdx.x == 0) {
        for (int s = 0; s < kProjStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(&acc_full[a], 1);
            mbar_init(&acc_empty[a], 4);
        }
        mbar_init(&drain, 1);
        abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 0) {
        tmem_alloc(&tmem_slot, 2 * kProjN);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_slot;

    if (warp == 0) {
        if (lane == 0) {
            // producer: stage g % S is refilled once the MMAs of g - S released it
            tma_prefetch_desc(&tmX);
            tma_prefetch_desc(&tmWq);
            tma_prefetch_desc(&tmWk);
            tma_prefetch_desc(&tmWv);
            long g = 0;
            for (int t = blockIdx.x; t < ntiles && !aborted(&abort_flag); t += gridDim.x) {
                int p, o0, m0;
                decode_tile(t, p, o0, m0);
                const CUtensorMap *tmW = p == 0 ? &tmWq : (p == 1 ? &tmWk : &tmWv);
                for (int kb = 0; kb < nk; ++kb, ++g) {
                    const int s = (int)(g % kProjStages);
                    if (g >= kProjStages && !mbar_wait(&empty[s], (uint32_t)((g / kProjStages) - 1) & 1)) {
                        give_up(status, &abort_flag);
                        break;
                    }
                    if (stall && g == 0) continue;  // test hook: the first stage is never loaded
                    mbar_arrive_expect_tx(&full[s], kProjXBytes + kProjWBytes);
                    tma_load_3d(sx + s * kProjXBytes, &tmX, kb * kProjK, m0, 0, &full[s]);
                    tma_load_3d(sw + s * kProjWBytes, tmW, kb * kProjK, o0, 0, &full[s]);
                }
            }
            // every load armed here has landed before the CTA leaves
            for (long j = g - kProjStages < 0 ? 0 : g - kProjStages; j < g; ++j)
                if (!(stall && j == 0)) mbar_wait(&full[j % kProjStages], (uint32_t)(j / kProjStages) & 1);
        }
        __syncwarp();
    } else if (warp == 1) {
        if (lane == 0) {
            constexpr uint32_t idesc = idesc_bf16(kProjM, kProjN, false, false);
            long g = 0;
            int i = 0;  // this CTA's tile count
            for (int t = blockIdx.x; t < ntiles && !aborted(&abort_flag); t += gridDim.x, ++i) {
                const int a = i & 1;
                if (i >= 2 && !mbar_wait(&acc_empty[a], (uint32_t)((i >> 1) - 1) & 1)) {
                    give_up(status, &abort_flag);
                    break;
                }
                tc_fence_after();
                const uint32_t acc = tmem + a * kProjN;
                bool ok = true;
                for (int kb = 0; kb < nk; ++kb, ++g) {
                    const int s = (int)(g % kProjStages);
                    if (!mbar_wait(&full[s], (uint32_t)(g / kProjStages) & 1)) {
                        give_up(status, &abort_flag);
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint64_t da = sdesc_sw128(smem_u32(sx + s * kProjXBytes), 16, 1024);
                    const uint64_t db = sdesc_sw128(smem_u32(sw + s * kProjWBytes), 16, 1024);
#pragma unroll
                    for (int kk = 0; kk < kProjK / 16; ++kk)
                        umma_bf16(acc, dadd(da, kk * 32), dadd(db, kk * 32), idesc, (kb > 0 || kk > 0) ? 1u : 0u);
                    umma_commit(&empty[s]);
                }
                if (!ok) break;
                umma_commit(&acc_full[a]);
            }
            // everything issued has completed before tensor memory is freed
            umma_commit(&drain);
            mbar_wait(&drain, 0);
        }
        __syncwarp();
    } else {
        // epilogue warps 2-5: tensor-memory lane quarter w % 4
        const int quarter = warp & 3;
        int i = 0;
        for (int t = blockIdx.x; t < ntiles; t += gridDim.x, ++i) {
            const int a = i & 1;
            if (!mbar_wait(&acc_full[a], (uint32_t)(i >> 1) & 1)) {
                give_up(status, &abort_flag);
                break;
            }
            if (aborted(&abort_flag)) break;
            tc_fence_after();
            int p, o0, m0;
            decode_tile(t, p, o0, m0);
            const int m = m0 + quarter * 32 + lane;
            const bool write = m < M;
            const int b = m / N, n = m % N;
            const int dp = out.d[p];
#pragma unroll 1
            for (int c0 = 0; c0 < kProjN; c0 += 32) {
                uint32_t r[32];
                tmem_ld32(tmem + a * kProjN + ((uint32_t)(quarter * 32) << 16) + c0, r);
                tmem_wait_ld();
                if (write) store_row_chunk<OUT_BF16>(out, p, dp, H, N, b, n, o0 + c0, r);
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&acc_empty[a]);
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, 2 * kProjN);
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
                           bool out_bf16, int B, int N, int D, int H, int d_r, int d_v, bool stall, void *ws,
                           cudaStream_t s) {
    CUtensorMap tx, tq, tk, tv;
    const int M = B * N;
    if (!proj_map(&tx, X, M, D, kProjM) || !proj_map(&tq, Wq, H * d_r, D, kProjN) ||
        !proj_map(&tk, Wk, H * d_r, D, kProjN) || !proj_map(&tv, Wv, H * d_v, D, kProjN))
        return cudaErrorInvalidValue;
    ProjOut out;
    out.y[0] = Q; out.y[1] = Kx; out.y[2] = V;
    out.d[0] = d_r; out.d[1] = d_r; out.d[2] = d_v;
    for (int p = 0; p < 3; ++p) out.tiles[p] = (H * out.d[p] + kProjN - 1) / kProjN;
    const long ntiles = (long)(out.tiles[0] + out.tiles[1] + out.tiles[2]) * ((M + kProjM - 1) / kProjM);
    int dev = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    unsigned *status = static_cast<unsigned *>(ws);
    e = cudaMemsetAsync(status, 0, sizeof(unsigned), s);
    if (e != cudaSuccess) return e;
    const int grid = (int)(ntiles < sms ? ntiles : sms);
    if (out_bf16) {
        e = cudaFuncSetAttribute(proj_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, kProjSmem);
        if (e != cudaSuccess) return e;
        proj_kernel<true><<<grid, kProjThreads, kProjSmem, s>>>(tx, tq, tk, tv, out, B, N, H, D, stall ? 1 : 0,
                                                                status);
    } else {
        e = cudaFuncSetAttribute(proj_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, kProjSmem);
        if (e != cudaSuccess) return e;
        proj_kernel<false><<<grid, kProjThreads, kProjSmem, s>>>(tx, tq, tk, tv, out, B, N, H, D, stall ? 1 : 0,
                                                                 status);
    }
    return cudaGetLastError();
}

}  // namespace gma
