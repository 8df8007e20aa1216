// Microbenchmark: aggregate throughput of bulk asynchronous reductions
// (cp.reduce.async.bulk .add.f32, shared -> global) from every SM into a
// float32 buffer, the primitive a K/V-major attention backward would use to
// add each tile's dQ partial (128 query rows x 128 features, 64 KB) into a
// float32 accumulator.  One CTA per SM issues `chunk`-byte reductions of a
// shared-memory tile to tile-sized slots of the buffer, walking the slots so
// that the CTAs in flight touch `live` distinct tiles (the accumulator's
// working set), with up to four tiles in flight per SM.  Reported: bytes
// reduced per second over all SMs, for a working set inside L2 and one
// larger than L2.  The kernel has no spin-waits (only the bulk-group waits,
// which end when the copies do); not part of the library.
//
//   python -m context_causal_attention_zigzag_gb300.microbench --reduce
#include <cuda_runtime.h>
#include <stdint.h>
#include <stdio.h>

namespace {

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ uint64_t gtimer() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
__device__ __forceinline__ void bulk_reduce_add_f32(float* dst, uint32_t src, uint32_t bytes) {
  asm volatile("cp.reduce.async.bulk.global.shared::cta.bulk_group.add.f32 [%0], [%1], %2;" ::"l"(
                   dst),
               "r"(src), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void bulk_commit() {
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
template <int N>
__device__ __forceinline__ void bulk_wait_read() {
  asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}
template <int N>
__device__ __forceinline__ void bulk_wait() {
  asm volatile("cp.async.bulk.wait_group %0;" ::"n"(N) : "memory");
}

constexpr int kTileBytes = 65536;

// Each CTA reduces its shared tile `reps` times; rep i of CTA c goes to tile
// slot (i * grid + c) % live of the buffer (live tiles of 64 KB).
__global__ void __launch_bounds__(128, 1)
    reduce_kernel(float* buf, int live, int reps, int chunk, unsigned long long* ns) {
  extern __shared__ __align__(1024) uint8_t sm[];
  for (int i = threadIdx.x; i < kTileBytes / 4; i += blockDim.x)
    reinterpret_cast<float*>(sm)[i] = 1.0f;
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  __syncthreads();
  if (threadIdx.x == 0) {
    const uint32_t src = smem_u32(sm);
    const uint64_t t0 = gtimer();
    for (int i = 0; i < reps; ++i) {
      const int64_t slot = ((int64_t)i * gridDim.x + blockIdx.x) % live;
      char* dst = reinterpret_cast<char*>(buf) + slot * kTileBytes;
      for (int off = 0; off < kTileBytes; off += chunk)
        bulk_reduce_add_f32(reinterpret_cast<float*>(dst + off), src + off, (uint32_t)chunk);
      bulk_commit();
      bulk_wait_read<3>();  // at most four tiles' reductions still reading shared memory
    }
    bulk_wait<0>();
    ns[blockIdx.x] = gtimer() - t0;
  }
}

// The same tile-sized reductions from registers: every thread adds float4
// values with red.global.add.v4.f32 (the load/store path instead of the bulk
// copy engine).
__global__ void __launch_bounds__(512, 1)
    red_v4_kernel(float* buf, int live, int reps, unsigned long long* ns) {
  const float4 one = make_float4(1.f, 1.f, 1.f, 1.f);
  const uint64_t t0 = gtimer();
  for (int i = 0; i < reps; ++i) {
    const int64_t slot = ((int64_t)i * gridDim.x + blockIdx.x) % live;
    float4* dst = reinterpret_cast<float4*>(reinterpret_cast<char*>(buf) + slot * kTileBytes);
    for (int e = threadIdx.x; e < kTileBytes / 16; e += blockDim.x)
      asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(dst + e), "f"(one.x),
                   "f"(one.y), "f"(one.z), "f"(one.w)
                   : "memory");
  }
  __syncthreads();
  if (threadIdx.x == 0) ns[blockIdx.x] = gtimer() - t0;
}

}  // namespace

int main() {
  int sms = 0;
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, 0);
  const int64_t big_tiles = (int64_t)8192;  // 512 MB of float32 accumulator
  float* buf = nullptr;
  unsigned long long* ns = nullptr;
  if (cudaMalloc(&buf, big_tiles * kTileBytes) != cudaSuccess) return 1;
  cudaMalloc(&ns, sizeof(unsigned long long) * sms);
  cudaMemset(buf, 0, big_tiles * kTileBytes);
  cudaFuncSetAttribute(reduce_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kTileBytes);
  const int reps = 400;
  struct Case {
    int live;
    int chunk;
    int grid;  // 0: every SM
  } cases[] = {{16, 65536, 0}, {1024, 65536, 0}, {1024, 16384, 0}, {1024, 4096, 0},
               {8192, 65536, 0}, {8192, 16384, 0},
               // fewer SMs issuing: a per-SM limit keeps the per-SM rate, an
               // aggregate (L2) limit lets it rise
               {1024, 65536, 8}, {1024, 65536, 38}, {1024, 65536, 76}};
  for (const Case& c : cases) {
    const int grid = c.grid ? c.grid : sms;
    reduce_kernel<<<grid, 128, kTileBytes>>>(buf, c.live, 20, c.chunk, ns);  // warm-up
    cudaEvent_t a, b;
    cudaEventCreate(&a);
    cudaEventCreate(&b);
    cudaEventRecord(a);
    reduce_kernel<<<grid, 128, kTileBytes>>>(buf, c.live, reps, c.chunk, ns);
    cudaEventRecord(b);
    cudaError_t e = cudaEventSynchronize(b);
    if (e != cudaSuccess) {
      printf("error %s\n", cudaGetErrorString(e));
      return 1;
    }
    float ms = 0.f;
    cudaEventElapsedTime(&ms, a, b);
    const double bytes = (double)grid * reps * kTileBytes;
    printf("%3d SMs, live %5d tiles (%6.1f MB) chunk %6d B: %.3f ms, %.2f TB/s reduced "
           "(%.1f GB/s per SM)\n",
           grid, c.live, c.live * (double)kTileBytes / 1e6, c.chunk, ms,
           bytes / (ms * 1e-3) / 1e12, bytes / grid / (ms * 1e-3) / 1e9);
  }
  for (int grid : {sms, 8}) {
    for (int live : {1024, 8192}) {
      red_v4_kernel<<<grid, 512>>>(buf, live, 20, ns);  // warm-up
      cudaEvent_t a, b;
      cudaEventCreate(&a);
      cudaEventCreate(&b);
      cudaEventRecord(a);
      red_v4_kernel<<<grid, 512>>>(buf, live, reps, ns);
      cudaEventRecord(b);
      cudaError_t e = cudaEventSynchronize(b);
      if (e != cudaSuccess) {
        printf("error %s\n", cudaGetErrorString(e));
        return 1;
      }
      float ms = 0.f;
      cudaEventElapsedTime(&ms, a, b);
      const double bytes = (double)grid * reps * kTileBytes;
      printf("red.v4 %3d SMs, live %5d tiles (%6.1f MB): %.3f ms, %.2f TB/s reduced "
             "(%.1f GB/s per SM)\n",
             grid, live, live * (double)kTileBytes / 1e6, ms, bytes / (ms * 1e-3) / 1e12,
             bytes / grid / (ms * 1e-3) / 1e9);
    }
  }
  return 0;
}
