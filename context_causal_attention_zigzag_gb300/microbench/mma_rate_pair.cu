// Microbenchmark: cycles per tcgen05.mma (kind::f16, bf16, fp32 accumulate)
// issued by a CTA pair with cta_group::2, M = 256 (128 rows per SM), K = 16,
// N in {128, 256}, SS and TS forms, back to back from the even CTA of each
// 2-CTA cluster: either one thread building the operand descriptors per
// instruction, or a whole warp with the descriptors built once and one
// elected lane issuing (the attention kernels' style).  Each SM's tensor core does the same per-SM work
// as a cta_group::1 M=128 instruction of the same N, so the per-SM cycles are
// directly comparable with mma_rate.cu.  One CTA per SM (the shared-memory
// request keeps two CTAs off one SM); every mbarrier wait is bounded.  It
// measures the ceiling a CTA-pair attention kernel would run against; it is
// not part of the library.
//
// Pair protocol (PTX ISA, tcgen05): both CTAs allocate TMEM with
// tcgen05.alloc.cta_group::2 from the same warp; a cluster barrier makes the
// peer's TMEM and shared memory ready before the even CTA issues; the commit
// multicasts to the barrier of both CTAs; both CTAs wait for it and pass a
// second cluster barrier before deallocating.
//
//   python -m context_causal_attention_zigzag_gb300.microbench
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdio.h>
#include <stdint.h>
#include "tc_ptx.cuh"
using namespace cpattn::tc;

namespace {

constexpr uint32_t kCols = 256;          // TMEM columns per SM
constexpr int kSmemReq = 160 * 1024;     // one CTA per SM

__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;"
               ::: "memory");
}
__device__ __forceinline__ void alloc2(uint32_t dst, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void relinquish2() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void dealloc2(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void mma2_ss(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, 1, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d),
      "l"(a), "l"(b), "r"(idesc)
      : "memory");
}
__device__ __forceinline__ void mma2_ts(uint32_t d, uint32_t a, uint64_t b, uint32_t idesc) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, 1, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d),
      "r"(a), "l"(b), "r"(idesc)
      : "memory");
}
// Arrive once on the barrier at offset `bar` of both CTAs of the pair when
// every tcgen05 operation this thread issued has completed.
__device__ __forceinline__ void commit2_both(uint32_t bar) {
  asm volatile(
      "{\n\t.reg .b16 m;\n\tmov.b16 m, 3;\n\t"
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 "
      "[%0], m;\n\t}" ::"r"(bar)
      : "memory");
}

}  // namespace

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(128, 1)
    pair_rate_kernel(int mode, int reps, unsigned long long* out, int* err, int wide) {
  extern __shared__ uint8_t raw_[];
  uint32_t raw = smem_u32(raw_);
  uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* sm = raw_ + (base - raw);
  const uint32_t sA = base, sB = base + 32768;
  const uint32_t bar0 = base + 98304;
  uint32_t* slot = (uint32_t*)(sm + 98304 + 64);
  volatile int* ab = (volatile int*)(sm + 98304 + 68);
  const int warp = threadIdx.x >> 5;
  const uint32_t crank = cluster_rank();
  for (int i = threadIdx.x; i < 98304 / 16; i += blockDim.x)
    reinterpret_cast<uint4*>(sm)[i] = make_uint4(0x3f803f80u, 0, 0x3f803f80u, 0);
  if (threadIdx.x == 0) {
    mbar_init(bar0, 1);
    *ab = 0;
    fence_mbar_init();
  }
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  if (warp == 0) {
    alloc2(smem_u32(slot), kCols);
    relinquish2();
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();
  tc_fence_after();
  const uint32_t tmem = *slot;
  WaitCtl wc{ab, err};
  // mode 0: SS N=128, 1: SS N=256, 2: TS N=128 (A at columns 128..191)
  const int N = mode == 1 ? 256 : 128;
  const bool ts = mode == 2;
  unsigned long long t0 = 0, t1 = 0;
  if (wide && crank == 0 && warp == 1) {
    const bool leader = elect_one();
    const uint32_t idesc = idesc_bf16(256, N, false, ts);
    const uint64_t dA = sdesc_sw128(sA, 16, 1024), dB = sdesc_sw128(sB, 16, 1024);
    const uint64_t dBmn = sdesc_sw128(sB, 16384, 1024);
    t0 = clock64();
    for (int r = 0; r < reps; ++r) {
      if (leader) {
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          const uint32_t off = (kk >> 2) * 16384 + (kk & 3) * 32;
          if (!ts)
            mma2_ss(tmem, sdesc_advance(dA, off), sdesc_advance(dB, off), idesc);
          else
            mma2_ts(tmem, tmem + 128 + kk * 8, sdesc_advance(dBmn, kk * 2048), idesc);
        }
      }
    }
    if (leader) commit2_both(bar0);
    const bool ok = __all_sync(0xffffffffu, mbar_wait(bar0, 0, wc));
    t1 = clock64();
    if (leader) out[blockIdx.x / 2] = ok ? (t1 - t0) : 0ull;
  }
  if (!wide && crank == 0 && threadIdx.x == 0) {
    const uint32_t idesc = idesc_bf16(256, N, false, ts);
    t0 = clock64();
    for (int r = 0; r < reps; ++r) {
      for (int kk = 0; kk < 8; ++kk) {
        const uint32_t off = (kk >> 2) * 16384 + (kk & 3) * 32;
        if (!ts)
          mma2_ss(tmem, sdesc_sw128(sA + off, 16, 1024), sdesc_sw128(sB + off, 16, 1024), idesc);
        else
          mma2_ts(tmem, tmem + 128 + kk * 8, sdesc_sw128(sB + kk * 2048, 16384, 1024), idesc);
      }
    }
    commit2_both(bar0);
  }
  if (threadIdx.x == 0) {
    const bool ok = mbar_wait(bar0, 0, wc);
    t1 = clock64();
    if (crank == 0 && !wide) out[blockIdx.x / 2] = ok ? (t1 - t0) : 0ull;
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();
  if (warp == 0) {
    tc_fence_after();
    dealloc2(tmem, kCols);
  }
}

int main() {
  int sms = 0;
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, 0);
  const int grid = sms & ~1;
  unsigned long long* d;
  int* err;
  cudaMalloc(&d, sizeof(unsigned long long) * grid);
  cudaMalloc(&err, 4);
  cudaMemset(err, 0, 4);
  cudaFuncSetAttribute(pair_rate_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemReq);
  const char* names[] = {"pair SS M=256 N=128", "pair SS M=256 N=256", "pair TS M=256 N=128"};
  for (int wide : {0, 1})
  for (int mode = 0; mode < 3; ++mode) {
    const int reps = 200;
    cudaMemset(d, 0, sizeof(unsigned long long) * grid);
    pair_rate_kernel<<<grid, 128, kSmemReq>>>(mode, reps, d, err, wide);
    cudaError_t e = cudaDeviceSynchronize();
    if (e != cudaSuccess) {
      printf("error %s\n", cudaGetErrorString(e));
      return 1;
    }
    unsigned long long h[1024];
    cudaMemcpy(h, d, sizeof(unsigned long long) * (grid / 2), cudaMemcpyDeviceToHost);
    double sum = 0;
    int n = 0;
    for (int i = 0; i < grid / 2; ++i)
      if (h[i]) {
        sum += h[i];
        ++n;
      }
    const int N = mode == 1 ? 256 : 128;
    const double per = n ? sum / n / (reps * 8.0) : 0.0;
    // Per SM: 128 rows x N x 16 x 2 flops per instruction.
    const double ideal = 128.0 * N * 16 * 2 / 8192.0;
    printf("%s %s: %.1f cycles per MMA (per-SM ideal at 8192 flop/clk/SM: %.1f) -> %.0f%% (%d pairs)\n",
           wide ? "warp-issued" : "one-thread", names[mode], per, ideal,
           per > 0 ? 100 * ideal / per : 0.0, n);
  }
  int herr = 0;
  cudaMemcpy(&herr, err, 4, cudaMemcpyDeviceToHost);
  printf("err word %d\n", herr);
  return 0;
}
