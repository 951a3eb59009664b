// gma_noalloc.cu -- gma_forward_bidir_noalloc: the bidirectional forward
// with its scratch memory in a fixed, file-scope device array, for callers
// that cannot allocate device memory themselves.
//
// The array is part of this library's device image: every GPU that loads
// the library holds GMA_NOALLOC_SCRATCH_BYTES of it until the process exits.
// In host code the array's name is only a host-side stand-in for the symbol,
// never a device address, so every call looks the address up
// (cudaGetSymbolAddress) in the CUDA context current on the calling thread.
// The lookup allocates nothing and launches nothing; an address cached from an
// earlier call could belong to a context that has since been destroyed
// (cudaDeviceReset) or to another context on the same device.
#include "gma_internal.h"

namespace {

constexpr size_t kNoallocScratchBytes = GMA_NOALLOC_SCRATCH_BYTES;

__device__ __align__(256) unsigned char g_noalloc_scratch[kNoallocScratchBytes];

// Device address of g_noalloc_scratch in the current context, or nullptr.
void *scratch_in_current_context() {
    void *ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || !ptr) {
        (void)cudaGetLastError();
        return nullptr;
    }
    return ptr;
}

}  // namespace

extern "C" gma_status gma_forward_bidir_noalloc(
    const void *Q_X, const void *K_X, const void *V_X, gma_dtype dtype, const float *mu,
    const float *sigma2, const float *log_pi, float eps, void *O, int B, int H, int N, int d_r,
    int d_v, int K, const gma_options *options, void *stream) {
    // Argument errors first, as gma_forward_bidir reports them; then the size
    // check, so a request that cannot fit never touches the device.
    if (!Q_X || !K_X || !V_X || !mu || !sigma2 || !log_pi || !O) return GMA_ERR_INVALID_ARG;
    if (dtype != GMA_F32 && dtype != GMA_BF16) return GMA_ERR_INVALID_ARG;
    if (options && (options->chunk < 0 || options->splits < 0)) return GMA_ERR_INVALID_ARG;
    const size_t need = gma_workspace_size(B, H, N, d_r, d_v, K, dtype, 0, options);
    if (need == 0) return GMA_ERR_UNSUPPORTED_SHAPE;
    if (need > kNoallocScratchBytes) return GMA_ERR_WORKSPACE_TOO_SMALL;
    void *scratch = scratch_in_current_context();
    if (!scratch) return GMA_ERR_CUDA;
    // Everything the kernels need at zero (the status word, the job counters)
    // is cleared by the call itself; every other scratch region is fully
    // written before it is read.
    return gma_forward_bidir(Q_X, K_X, V_X, dtype, mu, sigma2, log_pi, eps, O, B, H, N, d_r, d_v,
                             K, options, scratch, kNoallocScratchBytes, stream);
}
