// Placeholder until the tensor-core kernels land.
#include "cpattn_internal.h"
namespace cpattn {
bool tc_fwd_available() { return false; }
bool tc_bwd_available() { return false; }
cudaError_t launch_tc_fwd(const FwdArgs&, cudaStream_t) { return cudaErrorNotSupported; }
cudaError_t launch_tc_bwd(const BwdArgs&, cudaStream_t) { return cudaErrorNotSupported; }
}  // namespace cpattn
