// tc_common.cuh -- device and host helpers shared by the tensor-core kernel
// translation units (gma_tc.cu: d_r <= 64, d_v = 64, K <= 64; gma_tc128.cu:
// d_r = d_v = 128, K <= 128): status words, bounded waits, barriers, the
// 128-byte-swizzle offset and descriptor arithmetic, and the host-side tensor
// map encoder and dependent launch.  Internal linkage: each translation unit
// has its own copy.
#pragma once

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "gma_internal.h"
#include "tc_ptx.cuh"

namespace gma {
namespace {

using namespace ptx;

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

// A shared-memory descriptor advanced by `bytes` (the start-address field is
// the address >> 4 in the low bits; addresses stay below 256 KB, so a plain
// add never carries out of the field).  Lets the single MMA-issuing thread
// build each descriptor once and advance it with one add per MMA.
__device__ __forceinline__ uint64_t dadd(uint64_t desc, uint32_t bytes) { return desc + (uint64_t)(bytes >> 4); }

// Aborts the CTA's work on a timed-out wait: records the status once.
__device__ __forceinline__ void note_timeout(unsigned *status, int *abort_flag) {
    set_status(status, GMA_ERR_TIMEOUT);
    *reinterpret_cast<volatile int *>(abort_flag) = 1;
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
// CTA and named barriers of the warp-specialised kernels.  Roles run long
// single-lane loops (the TMA and MMA threads, the last store wait of an
// epilogue warp), and the barrier instructions expect whole warps: each warp
// reconverges first.
__device__ __forceinline__ void cta_sync() {
    __syncwarp();
    __syncthreads();
}
__device__ __forceinline__ void named_sync(int id, int nthreads) {
    __syncwarp();
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}
// Row of the tile / TMEM lane handled by an epilogue thread (warp w may only
// read TMEM lanes 32*(w%4) .. 32*(w%4)+31).
__device__ __forceinline__ int epi_row(int warp, int lane) { return 32 * (warp & 3) + lane; }

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

// Launch with programmatic stream serialisation: the kernel may start while
// the previous kernel of the stream finishes; it waits (pdl_wait) before
// touching what that kernel writes.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s, Args... args) {
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
    return cudaLaunchKernelEx(&cfg, kern, static_cast<KArgs>(args)...);
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

}  // namespace
}  // namespace gma
