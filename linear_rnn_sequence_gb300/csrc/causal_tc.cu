// causal_tc.cu -- tensor-core (tcgen05 / TMA / TMEM) chunkwise causal kernel.
// Not built yet: every shape is served by the CUDA-core kernel for now.
#include "la_internal.h"

namespace la {
bool causal_tc_supported(const FwdArgs &) { return false; }
size_t causal_tc_workspace(int, int, int, int) { return 0; }
cudaError_t launch_causal_tc(const FwdArgs &) { return cudaErrorNotSupported; }
}  // namespace la
