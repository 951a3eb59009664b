// gma_combine.cu -- gma_combine_memories: the rank-order sum of latent
// memories that stitches a sequence sharded over N back together.
//
// The latent memory of [GMA, Eqs. (5)-(6)] is a sum over positions, so the
// memories of consecutive key/value blocks add up to the memory of their
// union, and the prefix memory of the causal variant ([GMA, Eq. (8b)]) at a
// block boundary is the sum of the memories of every earlier block.  The
// rows are summed one after another in row order (row 0 first), in fp32, so
// every caller that holds the same rows gets bitwise the same result.
#include "gma_internal.h"

namespace {

__global__ void __launch_bounds__(256) combine_rows_kernel(const float *__restrict__ parts, long long n, int count,
                                                           float *__restrict__ out) {
    const long long stride = (long long)gridDim.x * blockDim.x;
    for (long long e = (long long)blockIdx.x * blockDim.x + threadIdx.x; e < n; e += stride) {
        float acc = parts[e];
        for (int r = 1; r < count; ++r) acc += parts[(long long)r * n + e];
        out[e] = acc;
    }
}

bool overlaps(const void *a, size_t na, const void *b, size_t nb) {
    auto pa = reinterpret_cast<uintptr_t>(a), pb = reinterpret_cast<uintptr_t>(b);
    return pa < pb + nb && pb < pa + na;
}

}  // namespace

extern "C" gma_status gma_combine_memories(const float *parts, int P, long long n, int count, float *out,
                                           void *stream) {
    if (!parts || !out) return GMA_ERR_INVALID_ARG;
    if (reinterpret_cast<uintptr_t>(parts) % 4 != 0 || reinterpret_cast<uintptr_t>(out) % 4 != 0)
        return GMA_ERR_INVALID_ARG;
    if (P < 1 || n < 1 || count < 1 || count > P || n > (1LL << 40) / P) return GMA_ERR_UNSUPPORTED_SHAPE;
    if (overlaps(out, sizeof(float) * (size_t)n, parts, sizeof(float) * (size_t)n * P)) return GMA_ERR_INVALID_ARG;
    const long long blocks = (n + 255) / 256;
    combine_rows_kernel<<<(unsigned)(blocks < 4096 ? blocks : 4096), 256, 0, static_cast<cudaStream_t>(stream)>>>(
        parts, n, count, out);
    if (cudaGetLastError() != cudaSuccess) return GMA_ERR_CUDA;
    return GMA_OK;
}
