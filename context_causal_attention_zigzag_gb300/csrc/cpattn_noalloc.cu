// Allocation-free ring backward.
//
// cpattn_ring_bwd needs a caller-provided device workspace: the float32
// per-query-head dK / dV partials of the tensor-core kernels (the CUDA-core
// kernels keep their float32 dQ, dK and dV there instead) and the Delta rows.
// Some callers cannot provide one: code that runs under a memory manager
// owning all of the device memory (a framework's caching allocator, a
// serving runtime that reserves HBM at start-up) and forbids allocations
// behind its back, or code on a latency-critical loop where a cudaMalloc /
// cudaFree would synchronise the device.
// For them the scratch lives in a fixed-size array in this library's own
// device image: every GPU that loads the library holds it until the process
// exits, and no call allocates anything.
#include <cuda_runtime.h>
#include <stddef.h>

#include "cpattn.h"

namespace {

// 64 MiB: the workspace of, e.g., B=1, S=1024, H=32, Hkv=8, D=128 (40 MiB).
constexpr size_t kScratchBytes = (size_t)64 << 20;

// Shared by every call on a device; keeps the last call's contents.
static __device__ __align__(256) unsigned char g_bwd_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
void* g_scratch_addr[kMaxDevices] = {nullptr};

// Device address of the scratch array on the current device.  The first call
// on a device looks it up (cudaGetSymbolAddress, with that device current);
// later calls reuse the cached address.
void* scratch_on_current_device() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  if (g_scratch_addr[dev] == nullptr) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_bwd_scratch) != cudaSuccess || ptr == nullptr)
      return nullptr;
    g_scratch_addr[dev] = ptr;
  }
  return g_scratch_addr[dev];
}

}  // namespace

extern "C" int cpattn_ring_bwd_noalloc(const void* q, const void* k, const void* v,
                                       const void* out, const void* dout, const float* lse,
                                       void* dq, void* dk, void* dv, int B, int H, int Hkv, int S,
                                       int D, int cp_size, int layout, int causal, int dtype,
                                       float softmax_scale, cpattn_stream_t stream) {
  if (B < 0 || H < 1 || Hkv < 1 || S < 0 || D < 1) return CPATTN_ERR_INVALID_ARG;
  const size_t need = cpattn_ring_bwd_workspace_bytes(B, H, Hkv, S, D, dtype);
  if (need > kScratchBytes) return CPATTN_ERR_WORKSPACE;
  void* scratch = scratch_on_current_device();
  if (scratch == nullptr) return CPATTN_ERR_CUDA;
  // The backward writes every workspace element before it reads it (Delta
  // by its pre-pass, each partial or accumulator slot once by the kernel that
  // owns it), so whatever an earlier call left in the array does not leak
  // into this one.
  return cpattn_ring_bwd(q, k, v, out, dout, lse, dq, dk, dv, B, H, Hkv, S, D, cp_size, layout,
                         causal, dtype, softmax_scale, scratch, kScratchBytes, stream);
}
