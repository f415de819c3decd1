// tcgen05 fused chunk kernel (placeholder until the kernel lands).
#include "gdn_internal.cuh"

namespace gdn {

bool fused_tc_supported(int, int, int) { return false; }

cudaError_t launch_fused_tc(const Problem &, const Workspace &, int, int, cudaStream_t) {
    return cudaErrorNotSupported;
}

}  // namespace gdn
