// verify_tc.cu -- tensor-core (tcgen05) tree verification.  Placeholder until
// the kernel lands: reports every shape as unsupported.
#include "tv_internal.cuh"

namespace tv {

bool verify_tc_supported(const VerifyArgs &) { return false; }

cudaError_t launch_verify_tc(const VerifyArgs &, cudaStream_t) { return cudaErrorNotSupported; }

}  // namespace tv
