// gma_tc.cu -- tcgen05 tensor-core kernels (placeholder: not eligible yet).
#include "gma_internal.h"

namespace gma {
bool tc_supported(const Problem &, int) { return false; }
size_t tc_workspace(const Problem &, int, int) { return 0; }
const char *const kTcStages[3][8] = {{nullptr}, {nullptr}, {nullptr}};
cudaError_t tc_bidir(const Problem &, int, void *, cudaStream_t, StageClock &) { return cudaErrorNotSupported; }
cudaError_t tc_causal(const Problem &, int, void *, cudaStream_t, StageClock &) { return cudaErrorNotSupported; }
}  // namespace gma
