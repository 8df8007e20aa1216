// Tensor-core ring backward (not in this build yet: the CUDA-core kernel runs).
#include "cpattn_internal.h"
namespace cpattn {
bool tc_bwd_available() { return false; }
cudaError_t launch_tc_bwd(const BwdArgs&, cudaStream_t) { return cudaErrorNotSupported; }
}  // namespace cpattn
