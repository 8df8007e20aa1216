// Microbenchmark: cycles per tcgen05.mma (kind::f16, bf16, cta_group::1) for
// the SS and TS forms at M=128, N in {64, 128, 256}, K=16, issued back to back by
// one thread, optionally while eight other warps load / store TMEM the way the
// attention kernels' softmax warps do.  Two issue styles: one thread
// (`if (threadIdx.x == 0)`) building each operand descriptor per
// instruction, or a whole warp running the loop with the descriptors built
// once and one elected lane issuing (the style of the attention kernels).  Modes 4 and 5 issue N=128 MMAs that
// alternate between two independent accumulators (two chains interleaved
// instruction by instruction) instead of one accumulation chain.  One CTA of 384 threads per SM on every
// SM; every wait is bounded.  It measures the per-instruction ceiling the
// attention kernels run against; it is not part of the library.
//
//   python -m context_causal_attention_zigzag_gb300.microbench
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdio.h>
#include <stdint.h>
#include "tc_ptx.cuh"
using namespace cpattn::tc;

__global__ void __launch_bounds__(384, 1) rate_kernel(int mode, int reps, unsigned long long* out, int* err, int noise, int wide) {
  extern __shared__ uint8_t raw_[];
  uint32_t raw = smem_u32(raw_);
  uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* sm = raw_ + (base - raw);
  // A: 32 KB at base, B: 64 KB at base + 32 KB; barriers after.
  uint32_t sA = base, sB = base + 32768;
  uint32_t bar0 = base + 98304;
  uint32_t* slot = (uint32_t*)(sm + 98304 + 64);
  volatile int* ab = (volatile int*)(sm + 98304 + 68);
  int warp = threadIdx.x >> 5;
  for (int i = threadIdx.x; i < 98304 / 16; i += blockDim.x)
    reinterpret_cast<uint4*>(sm)[i] = make_uint4(0x3f803f80u, 0, 0x3f803f80u, 0);
  if (threadIdx.x == 0) {
    mbar_init(bar0, 1);
    *ab = 0;
    fence_mbar_init();
  }
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  if (warp == 0) {
    tmem_alloc(smem_u32(slot), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  uint32_t tmem = *slot;
  WaitCtl wc{ab, err};
  if (noise && warp >= 4) {
    // Softmax-like TMEM traffic: every warp of warpgroups 1-2 loads and
    // stores 32 columns of its sub-partition in a loop (columns 384..511).
    const uint32_t tl = tmem + ((uint32_t)((warp & 3) * 32) << 16) + 384 + 32 * ((warp >> 2) - 1) * 2;
    uint32_t r[32];
    for (int it = 0; it < reps * 6 && !*ab; ++it) {
      tmem_ld32(tl, r);
      tmem_wait_ld_regs(r);
      for (int j = 0; j < 32; ++j) r[j] += 1u;
      tmem_st32(tl + 32, r);
      tmem_wait_st();
    }
  }
  if (!wide && threadIdx.x == 0) {
    const int N = (mode == 1 || mode == 3) ? 256 : (mode >= 6 ? 64 : 128);
    const bool ts = mode == 2 || mode == 3 || mode == 5 || mode == 7;
    const bool two = mode == 4 || mode == 5;
    const uint32_t idesc = idesc_bf16(128, N, false, ts);
    unsigned long long t0 = clock64();
    for (int r = 0; r < reps; ++r) {
      for (int kk = 0; kk < 8; ++kk) {
        const uint32_t off = (kk >> 2) * 16384 + (kk & 3) * 32;
        // two chains: D at columns 128 and 256 (the noise warps use 384-511)
        const uint32_t d = two ? 128u + 128u * (uint32_t)(kk & 1) : (ts ? 256u : 0u);
        if (!ts)
          mma_ss(tmem + d, sdesc_sw128(sA + off, 16, 1024), sdesc_sw128(sB + off, 16, 1024), idesc,
                 1);
        else
          mma_ts(tmem + d, tmem + 0 + kk * 8, sdesc_sw128(sB + kk * 2048, 16384, 1024), idesc, 1);
      }
    }
    mma_commit(bar0);
    bool ok = mbar_wait(bar0, 0, wc);
    unsigned long long t1 = clock64();
    out[blockIdx.x] = ok ? (t1 - t0) : 0ull;
  }
  if (wide && warp == 1) {
    const bool leader = elect_one();
    const int N = (mode == 1 || mode == 3) ? 256 : (mode >= 6 ? 64 : 128);
    const bool ts = mode == 2 || mode == 3 || mode == 5 || mode == 7;
    const bool two = mode == 4 || mode == 5;
    const uint32_t idesc = idesc_bf16(128, N, false, ts);
    const uint64_t dA = sdesc_sw128(sA, 16, 1024), dB = sdesc_sw128(sB, 16, 1024);
    const uint64_t dBmn = sdesc_sw128(sB, 16384, 1024);
    unsigned long long t0 = clock64();
    for (int r = 0; r < reps; ++r) {
      if (leader) {
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          const uint32_t off = (kk >> 2) * 16384 + (kk & 3) * 32;
          const uint32_t d = two ? 128u + 128u * (uint32_t)(kk & 1) : (ts ? 256u : 0u);
          if (!ts)
            mma_ss(tmem + d, sdesc_advance(dA, off), sdesc_advance(dB, off), idesc, 1);
          else
            mma_ts(tmem + d, tmem + 0 + kk * 8, sdesc_advance(dBmn, kk * 2048), idesc, 1);
        }
      }
    }
    if (leader) mma_commit(bar0);
    const bool ok = __all_sync(0xffffffffu, mbar_wait(bar0, 0, wc));
    unsigned long long t1 = clock64();
    if (leader) out[blockIdx.x] = ok ? (t1 - t0) : 0ull;
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

int main() {
  int sms = 0;
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, 0);
  unsigned long long* d;
  int* err;
  cudaMalloc(&d, sizeof(unsigned long long) * sms);
  cudaMalloc(&err, 4);
  cudaMemset(err, 0, 4);
  int smem = 98304 + 1024 + 128;
  cudaFuncSetAttribute(rate_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  const char* names[] = {"SS N=128", "SS N=256", "TS N=128", "TS N=256",
                         "SS N=128 two chains", "TS N=128 two chains", "SS N=64", "TS N=64"};
  for (int wide : {0, 1})
  for (int mode = 0; mode < 8; ++mode) {
    for (int noise : {0, 1}) {
      const int grid = sms;
      const int reps = 200;
      rate_kernel<<<grid, 384, smem>>>(mode, reps, d, err, noise, wide);
      cudaError_t e = cudaDeviceSynchronize();
      if (e != cudaSuccess) { printf("error %s\n", cudaGetErrorString(e)); return 1; }
      unsigned long long h[1024];
      cudaMemcpy(h, d, sizeof(unsigned long long) * grid, cudaMemcpyDeviceToHost);
      double mx = 0, sum = 0;
      for (int i = 0; i < grid; ++i) { sum += h[i]; if (h[i] > mx) mx = h[i]; }
      const int N = (mode == 1 || mode == 3) ? 256 : (mode >= 6 ? 64 : 128);
      double per = sum / grid / (reps * 8.0);
      double ideal = 128.0 * N * 16 * 2 / 8192.0;
      printf("%s %s tmem-noise=%d: %.1f cycles per MMA (ideal at 8192 flop/clk/SM: %.1f) -> %.0f%%\n",
             wide ? "warp-issued" : "one-thread", names[mode], noise, per, ideal, 100 * ideal / per);
    }
  }
  int herr = 0;
  cudaMemcpy(&herr, err, 4, cudaMemcpyDeviceToHost);
  printf("err word %d\n", herr);
  return 0;
}
