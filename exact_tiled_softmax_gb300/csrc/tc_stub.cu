// Placeholder until the tensor-core kernels land: report them unsupported.
#include "internal.h"
namespace exattn {
bool tc_fwd_supported(const Problem&) { return false; }
cudaError_t launch_tc_fwd(const FwdArgs&, cudaStream_t) { return cudaErrorNotSupported; }
bool tc_bwd_supported(const Problem&) { return false; }
cudaError_t launch_tc_bwd(const BwdArgs&, cudaStream_t) { return cudaErrorNotSupported; }
}  // namespace exattn
