// gma_noalloc.cu -- gma_forward_bidir_noalloc: the bidirectional forward
// with its scratch memory in a fixed, file-scope device array, for callers
// that cannot allocate device memory themselves.
//
// The array is part of this library's device image: every GPU that loads
// the library holds GMA_NOALLOC_SCRATCH_BYTES of it until the process exits.
// Its device address is looked up once per device (cudaGetSymbolAddress,
// with that device current) on the first call made on that device; later
// calls reuse the cached address.  In host code the array's name is only a
// host-side stand-in for the symbol, never a device address, which is why
// the address is looked up rather than taken.
#include <mutex>

#include "gma_internal.h"

namespace {

constexpr size_t kNoallocScratchBytes = GMA_NOALLOC_SCRATCH_BYTES;
constexpr int kMaxDevices = 64;

__device__ __align__(256) unsigned char g_noalloc_scratch[kNoallocScratchBytes];

std::mutex g_setup_mutex;
void *g_scratch_addr[kMaxDevices] = {};

// Device address of g_noalloc_scratch on the current device (looked up once
// per device), or nullptr on failure.
void *scratch_on_current_device() {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        (void)cudaGetLastError();
        return nullptr;
    }
    std::lock_guard<std::mutex> lock(g_setup_mutex);
    if (!g_scratch_addr[dev]) {
        void *ptr = nullptr;
        cudaError_t err = cudaGetSymbolAddress(&ptr, g_noalloc_scratch);
        if (err != cudaSuccess || !ptr) {
            (void)cudaGetLastError();
            return nullptr;
        }
        g_scratch_addr[dev] = ptr;
    }
    return g_scratch_addr[dev];
}

}  // namespace

extern "C" gma_status gma_forward_bidir_noalloc(
    const void *Q_X, const void *K_X, const void *V_X, gma_dtype dtype, const float *mu,
    const float *sigma2, const float *log_pi, float eps, void *O, int B, int H, int N, int d_r,
    int d_v, int K, const gma_options *options, void *stream) {
    // Size check first: a request that cannot fit never touches the device.
    const size_t need = gma_workspace_size(B, H, N, d_r, d_v, K, dtype, 0, options);
    if (need == 0) return GMA_ERR_UNSUPPORTED_SHAPE;
    if (need > kNoallocScratchBytes) return GMA_ERR_WORKSPACE_TOO_SMALL;
    void *scratch = scratch_on_current_device();
    if (!scratch) return GMA_ERR_CUDA;
    // Everything the kernels need at zero (the status word) is cleared by the
    // call itself; every other scratch region is fully written before it is read.
    return gma_forward_bidir(Q_X, K_X, V_X, dtype, mu, sigma2, log_pi, eps, O, B, H, N, d_r, d_v,
                             K, options, scratch, kNoallocScratchBytes, stream);
}
