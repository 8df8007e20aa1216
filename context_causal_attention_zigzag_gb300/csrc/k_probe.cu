// A probe of the bounded-wait path: one CTA waits, with the same helper the
// tensor-core kernels use, on an mbarrier phase that nothing completes.  The
// wait gives up after its limit, raises the device error word and returns;
// no fault, no hang, and the context stays usable.
#include <cuda_runtime.h>
#include <stdint.h>

#include "cpattn_internal.h"
#include "tc_ptx.cuh"

namespace cpattn {
namespace {

__global__ void wait_probe_kernel(int* err, uint64_t limit_ns) {
  __shared__ __align__(8) uint64_t bar_storage;
  __shared__ int abort_flag;
  const uint32_t bar = tc::smem_u32(&bar_storage);
  if (threadIdx.x == 0) {
    tc::mbar_init(bar, 1);
    abort_flag = 0;
    tc::fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    tc::WaitCtl wc{&abort_flag, err, limit_ns};
    (void)tc::mbar_wait(bar, 0, wc);  // no arrival ever comes: gives up after limit_ns
  }
}

}  // namespace

cudaError_t launch_wait_probe(int* err, uint64_t limit_ns, cudaStream_t stream) {
  wait_probe_kernel<<<1, 32, 0, stream>>>(err, limit_ns);
  return cudaGetLastError();
}

}  // namespace cpattn
