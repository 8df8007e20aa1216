// Microbenchmark: aggregate rate at which bulk asynchronous copies
// (cp.async.bulk global -> shared, completing on an mbarrier) bring a
// region that sits in L2 into shared memory when every SM streams it, the
// way the attention kernels stream one kv head's K and V tiles.  One CTA per
// SM, one thread issues 32 KB copies into a ring of six shared-memory stages
// (at most six copies in flight), consuming nothing.  Access patterns:
//   lockstep  every CTA walks the region's chunks in order from one of eight
//             neighbouring starts (the CTAs in flight read the same chunks at
//             about the same time, as the natural-order tile walks do);
//   skewed    CTA c starts 3c chunks in (a window of about 450 chunks);
//   spread    CTA c starts c * nchunks / grid chunks in (every chunk of the
//             region is being read by some CTA at any time).
// Every wait is bounded (2 s of the global timer), after which the kernel
// records an error, waits (again bounded) for its copies in flight and
// stops.  Not part of the library.
//
//   python -m context_causal_attention_zigzag_gb300.microbench --load
#include <cuda_runtime.h>
#include <stdint.h>
#include <stdio.h>

namespace {

constexpr int kStages = 6;
constexpr int kChunk = 32768;
constexpr uint64_t kLimitNs = 2000000000ull;

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ uint64_t gtimer() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
__device__ __forceinline__ void mbar_init(uint32_t b, uint32_t n) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(b), "r"(n) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint32_t b, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(b), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ bool mbar_try(uint32_t b, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}"
      : "=r"(ok)
      : "r"(b), "r"(parity)
      : "memory");
  return ok != 0;
}
__device__ __forceinline__ bool mbar_wait(uint32_t b, uint32_t parity) {
  const uint64_t t0 = gtimer();
  while (!mbar_try(b, parity))
    if (gtimer() - t0 > kLimitNs) return false;
  return true;
}
__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes,
                                          uint32_t b) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
          "r"(dst),
      "l"(src), "r"(bytes), "r"(b)
      : "memory");
}

// CTA c copies chunks (start(c) + i) % nchunks for i < reps.
__global__ void __launch_bounds__(32, 1)
    load_kernel(const uint8_t* buf, int64_t nchunks, int reps, int pattern,
                unsigned long long* ns, int* err) {
  extern __shared__ __align__(1024) uint8_t sm[];
  if (threadIdx.x != 0) return;
  const uint32_t ring = smem_u32(sm);
  const uint32_t bars = ring + kStages * kChunk;
  for (int s = 0; s < kStages; ++s) mbar_init(bars + 8 * s, 1);
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  const int64_t c = blockIdx.x;
  const int64_t start = pattern == 0 ? (c & 7) : pattern == 1 ? 3 * c : (c * nchunks) / gridDim.x;
  const uint64_t t0 = gtimer();
  int issued = 0, waited = 0;
  bool ok = true;
  for (int i = 0; i < reps + kStages; ++i) {
    if (i >= kStages) {
      const int j = i - kStages;
      if (!mbar_wait(bars + 8 * (j % kStages), (j / kStages) & 1)) {
        ok = false;
        break;
      }
      ++waited;
    }
    if (i < reps) {
      const int s = i % kStages;
      mbar_expect_tx(bars + 8 * s, kChunk);
      bulk_load(ring + s * kChunk, buf + ((start + i) % nchunks) * kChunk, kChunk, bars + 8 * s);
      ++issued;
    }
  }
  if (!ok) {
    atomicExch(err, 1);
    for (int j = waited; j < issued; ++j)
      if (!mbar_wait(bars + 8 * (j % kStages), (j / kStages) & 1)) break;
  }
  ns[blockIdx.x] = gtimer() - t0;
}

}  // namespace

int main() {
  int sms = 0;
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, 0);
  const int64_t max_bytes = (int64_t)1 << 30;
  uint8_t* buf = nullptr;
  unsigned long long* ns = nullptr;
  int* err = nullptr;
  if (cudaMalloc(&buf, max_bytes) != cudaSuccess) return 1;
  cudaMalloc(&ns, sizeof(unsigned long long) * sms);
  cudaMalloc(&err, sizeof(int));
  cudaMemset(buf, 0, max_bytes);
  cudaMemset(err, 0, sizeof(int));
  const int smem = kStages * kChunk + 8 * kStages;
  cudaFuncSetAttribute(load_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  const char* names[] = {"lockstep", "skewed", "spread"};
  struct Case {
    int64_t region;
    int pattern;
  } cases[] = {{32 << 20, 0}, {64 << 20, 0}, {64 << 20, 1}, {64 << 20, 2},
               {96 << 20, 2}, {512 << 20, 0}, {512 << 20, 2}};
  const int reps = 3000;
  for (const Case& cs : cases) {
    const int64_t nchunks = cs.region / kChunk;
    load_kernel<<<sms, 32, smem>>>(buf, nchunks, 200, cs.pattern, ns, err);  // warm-up
    cudaEvent_t a, b;
    cudaEventCreate(&a);
    cudaEventCreate(&b);
    cudaEventRecord(a);
    load_kernel<<<sms, 32, smem>>>(buf, nchunks, reps, cs.pattern, ns, err);
    cudaEventRecord(b);
    cudaError_t e = cudaEventSynchronize(b);
    int herr = 0;
    cudaMemcpy(&herr, err, sizeof(int), cudaMemcpyDeviceToHost);
    if (e != cudaSuccess || herr) {
      printf("error %s, wait limit %d\n", cudaGetErrorString(e), herr);
      return 1;
    }
    float ms = 0.f;
    cudaEventElapsedTime(&ms, a, b);
    const double bytes = (double)sms * reps * kChunk;
    printf("%3d SMs, region %5.0f MB, %-8s: %.3f ms, %.2f TB/s into shared memory "
           "(%.1f GB/s per SM)\n",
           sms, cs.region / 1048576.0, names[cs.pattern], ms, bytes / (ms * 1e-3) / 1e12,
           bytes / sms / (ms * 1e-3) / 1e9);
  }
  return 0;
}
