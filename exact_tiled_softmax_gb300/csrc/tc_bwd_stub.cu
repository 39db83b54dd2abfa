// The tensor-core reverse kernel is not built yet: the reverse pass runs on
// the SIMT kernels for every shape.
#include "internal.h"
namespace exattn {
bool tc_bwd_supported(const Problem&) { return false; }
cudaError_t launch_tc_bwd(const BwdArgs&, cudaStream_t) { return cudaErrorNotSupported; }
}  // namespace exattn
