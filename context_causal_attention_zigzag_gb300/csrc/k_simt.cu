// fp32 CUDA-core ring kernels: the exact-fp32 path (dtype float32, e.g. the
// S=256 / D=64 case) and the fallback for shapes the tensor-core kernels do
// not take (chunks that are not a multiple of 256 tokens, D = 64 in bf16).
//
// Forward: one CTA per (64 query rows of one rank, batch*head).  The CTA walks
// the ring -- step t brings the K/V shard of rank (r - t) mod cp -- in 64-key
// tiles, skips tiles that no query of the block sees (wholly in the causal
// future, or outside the packed documents of its rows), masks the rest
// element-wise against each row's key window (natural positions), and keeps the
// online-softmax state (running max m, running sum l, unnormalised O) in
// registers ("Sequence Parallelism IV", sections 4-5).  A 64 x 64 score tile
// is spread over 256 threads as 4 x 4 blocks; row max and row sum are reduced
// across the 16 threads of a row with warp shuffles.
//
// Backward, two kernels, no atomics (every gradient element is written once,
// so the result does not depend on scheduling):
//   dK/dV: one CTA per (64 key rows of one source rank, batch*kv head).  It
//   follows its K/V tile around the ring (step t: receiving rank (s + t) mod
//   cp), over every query head of the group, recomputes P from the saved LSE
//   and accumulates dK, dV in registers, written to the float32 accumulators
//   at the end.
//   dQ: one CTA per (64 query rows of one rank, batch*head), the forward's
//   tile walk over the K/V of every ring step; P, dP and dS recomputed per
//   tile, dQ in registers, written at the end.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <limits.h>
#include <stdint.h>

#include "cpattn_internal.h"

namespace cpattn {
namespace {

constexpr int BM = kSimtTile;  // query rows per tile
constexpr int BN = kSimtTile;  // key rows per tile
constexpr int NT = 256;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kLog2e = 1.4426950408889634f;

__device__ __forceinline__ float to_f(float x) { return x; }
__device__ __forceinline__ float to_f(__nv_bfloat16 x) { return __bfloat162float(x); }
__device__ __forceinline__ void from_f(float* p, float x) { *p = x; }
__device__ __forceinline__ void from_f(__nv_bfloat16* p, float x) { *p = __float2bfloat16_rn(x); }

// Copies rows [pos0, pos0 + n) of head x of a [B, S, X, D] tensor into a
// row-padded float tile (stride D + 1); rows n..63 are zero.
template <typename T, int D>
__device__ __forceinline__ void load_tile(float* dst, const T* src, int b, int pos0, int n, int x,
                                          int X, int S) {
  constexpr int DP = D + 1;
  for (int e = threadIdx.x; e < BM * D; e += NT) {
    int row = e / D, d = e - row * D;
    float val = 0.f;
    if (row < n) val = to_f(src[(((int64_t)b * S + pos0 + row) * X + x) * D + d]);
    dst[row * DP + d] = val;
  }
}

__device__ __forceinline__ float max16(float v) {
#pragma unroll
  for (int off = 8; off > 0; off >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, off, 16));
  return v;
}
__device__ __forceinline__ float sum16(float v) {
#pragma unroll
  for (int off = 8; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off, 16);
  return v;
}

template <int D>
constexpr int fwd_smem_bytes() {
  return (BM * (D + 1) + 2 * BN * (D + 1) + BM * (BN + 1)) * (int)sizeof(float);
}
template <int D>
constexpr int bwd_smem_bytes() {
  return (2 * BN * (D + 1) + 2 * BM * (D + 1) + BM * (BN + 1)) * (int)sizeof(float);
}

template <typename T, int D, bool STEP>
__global__ void __launch_bounds__(NT) simt_fwd_kernel(const FwdArgs a) {
  constexpr int DP = D + 1, PP = BN + 1, DV = D / 16;
  extern __shared__ float smem[];
  float* Qs = smem;
  float* Ks = Qs + BM * DP;
  float* Vs = Ks + BN * DP;
  float* Ps = Vs + BN * DP;
  __shared__ int q_lo[BM], q_hi[BM];  // key window of each query row
  __shared__ int k_nat[BN];
  __shared__ int s_lo, s_hi;

  const RingShape& sh = a.sh;
  const int tid = threadIdx.x, ty = tid >> 4, tx = tid & 15;
  const int nblk = (sh.L + BM - 1) / BM;
  const int r = blockIdx.x / nblk, qb = blockIdx.x - r * nblk;
  const int b = blockIdx.y / sh.H, h = blockIdx.y - b * sh.H;
  const int g = h / (sh.H / sh.Hkv);
  const int q0 = r * sh.L + qb * BM;
  const int qn = min(BM, sh.L - qb * BM);
  const T* qp = static_cast<const T*>(a.q);
  const T* kp = static_cast<const T*>(a.k);
  const T* vp = static_cast<const T*>(a.v);

  load_tile<T, D>(Qs, qp, b, q0, qn, h, sh.H, sh.S);
  if (tid < BM) {
    int lo = INT_MAX, hi = -1;  // padding rows see nothing
    if (tid < qn) query_window(sh, natural_pos(sh, q0 + tid), lo, hi);
    q_lo[tid] = lo;
    q_hi[tid] = hi;
  }
  __syncthreads();
  if (tid < 32) {
    int lo = min(q_lo[tid], q_lo[tid + 32]), hi = max(q_hi[tid], q_hi[tid + 32]);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      lo = min(lo, __shfl_xor_sync(0xffffffffu, lo, off));
      hi = max(hi, __shfl_xor_sync(0xffffffffu, hi, off));
    }
    if (tid == 0) {
      s_lo = lo;
      s_hi = hi;
    }
  }
  __syncthreads();
  const int blk_lo = s_lo, blk_hi = s_hi;  // keys some row of the block sees

  float m[4], l[4], o[4][DV];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    m[i] = -INFINITY;
    l[i] = 0.f;
#pragma unroll
    for (int dd = 0; dd < DV; ++dd) o[i][dd] = 0.f;
  }

  // Ring: steps t_begin..t_end-1, the shard of rank (r - t) mod cp each.
  // All-gather (kv_natural): one pass over the whole K/V in natural order.
  const bool nat_kv = sh.kv_natural != 0;
  const int n_pass = nat_kv ? 1 : a.t_end - a.t_begin;
  for (int pass = 0; pass < n_pass; ++pass) {
    const int t = a.t_begin + pass;
    const int s = ring_source(r, t, sh.cp);
    const int kbase = nat_kv ? 0 : s * sh.L, klen = nat_kv ? sh.S : sh.L;
    unsigned long long tiles = 0;
    for (int kb = 0; kb < klen; kb += BN) {
      const int k0 = kbase + kb, kn = min(BN, klen - kb);
      __syncthreads();  // the previous tile is fully consumed
      int live = 0;
      if (tid < BN) {
        int kpos = tid < kn ? (nat_kv ? k0 + tid : natural_pos(sh, k0 + tid)) : INT_MAX;
        k_nat[tid] = kpos;
        live = tid < kn && kpos >= blk_lo && kpos <= blk_hi;
      }
      if (!__syncthreads_or(live)) continue;  // no row of the block sees the tile
      if (nat_kv) {
        // Census: the ring step at which the tile's first key would arrive.
        if (a.tiles_rt != nullptr && tid == 0)
          atomicAdd(&a.tiles_rt[r * sh.cp +
                                ring_step_of(r, chunk_owner(sh, k_nat[0] / sh.c), sh.cp)],
                    1ull);
      } else {
        ++tiles;
      }
      load_tile<T, D>(Ks, kp, b, k0, kn, g, sh.Hkv, sh.S);
      load_tile<T, D>(Vs, vp, b, k0, kn, g, sh.Hkv, sh.S);
      __syncthreads();

      float sc[4][4];
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) sc[i][j] = 0.f;
#pragma unroll 8
      for (int d = 0; d < D; ++d) {
        float qv[4], kv[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) qv[i] = Qs[(ty * 4 + i) * DP + d];
#pragma unroll
        for (int j = 0; j < 4; ++j) kv[j] = Ks[(tx + 16 * j) * DP + d];
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
          for (int j = 0; j < 4; ++j) sc[i][j] = fmaf(qv[i], kv[j], sc[i][j]);
      }

#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int row = ty * 4 + i;
        const int lo = q_lo[row], hi = q_hi[row];
        float mx = -INFINITY;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int col = tx + 16 * j;
          const bool ok = col < kn && k_nat[col] >= lo && k_nat[col] <= hi;
          sc[i][j] = ok ? sc[i][j] * sh.scale_log2 : -INFINITY;
          mx = fmaxf(mx, sc[i][j]);
        }
        mx = max16(mx);
        const float mnew = fmaxf(m[i], mx);
        float alpha = 1.f, rs = 0.f, p[4];
        if (mnew == -INFINITY) {
#pragma unroll
          for (int j = 0; j < 4; ++j) p[j] = 0.f;
        } else {
          alpha = exp2f(m[i] - mnew);
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            p[j] = exp2f(sc[i][j] - mnew);
            rs += p[j];
          }
        }
        rs = sum16(rs);
        l[i] = l[i] * alpha + rs;
        m[i] = mnew;
#pragma unroll
        for (int dd = 0; dd < DV; ++dd) o[i][dd] *= alpha;
#pragma unroll
        for (int j = 0; j < 4; ++j) Ps[row * PP + tx + 16 * j] = p[j];
      }
      __syncthreads();

#pragma unroll 4
      for (int c = 0; c < BN; ++c) {
        float pv[4], vv[DV];
#pragma unroll
        for (int i = 0; i < 4; ++i) pv[i] = Ps[(ty * 4 + i) * PP + c];
#pragma unroll
        for (int dd = 0; dd < DV; ++dd) vv[dd] = Vs[c * DP + tx + 16 * dd];
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
          for (int dd = 0; dd < DV; ++dd) o[i][dd] = fmaf(pv[i], vv[dd], o[i][dd]);
      }
    }
    if (a.tiles_rt != nullptr && tid == 0 && tiles != 0)
      atomicAdd(&a.tiles_rt[r * sh.cp + t], tiles);
  }

#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int row = ty * 4 + i;
    if (row >= qn) continue;
    const bool empty = !(l[i] > 0.f);
    const float inv = empty ? 0.f : 1.f / l[i];
    const int64_t base = (((int64_t)b * sh.S + q0 + row) * sh.H + h) * D;
    if constexpr (STEP) {
      float* op = static_cast<float*>(a.out);
#pragma unroll
      for (int dd = 0; dd < DV; ++dd) op[base + tx + 16 * dd] = o[i][dd] * inv;
    } else {
      T* op = static_cast<T*>(a.out);
#pragma unroll
      for (int dd = 0; dd < DV; ++dd) from_f(op + base + tx + 16 * dd, o[i][dd] * inv);
    }
    if (tx == 0)
      a.lse[((int64_t)b * sh.H + h) * sh.S + q0 + row] =
          empty ? -INFINITY : (m[i] + log2f(l[i])) * kLn2;
  }
}

template <typename T, int D>
__global__ void __launch_bounds__(NT) simt_bwd_kernel(const BwdArgs a) {
  constexpr int DP = D + 1, PP = BN + 1, DV = D / 16;
  extern __shared__ float smem[];
  float* Ks = smem;
  float* Vs = Ks + BN * DP;
  float* Qs = Vs + BN * DP;
  float* Os = Qs + BM * DP;  // dO tile
  float* Ps = Os + BM * DP;  // P, then dS
  __shared__ int q_lo[BM], q_hi[BM];  // key window of each query row
  __shared__ int k_nat[BN];
  __shared__ float lse2[BM];  // LSE in base 2
  __shared__ float dlt[BM];
  __shared__ int s_kmin, s_kmax;

  const RingShape& sh = a.sh;
  const int tid = threadIdx.x, ty = tid >> 4, tx = tid & 15;
  // Ring: the CTA's 64 key rows lie in source rank s's shard.  All-gather
  // (kv_natural): 64 rows of the natural-order K/V.
  const bool nat_kv = sh.kv_natural != 0;
  const int nblk = (sh.L + BN - 1) / BN;
  const int s = nat_kv ? 0 : blockIdx.x / nblk, kb = blockIdx.x - s * nblk;
  const int b = blockIdx.y / sh.Hkv, g = blockIdx.y - b * sh.Hkv;
  const int grp = sh.H / sh.Hkv;
  const int k0 = nat_kv ? blockIdx.x * BN : s * sh.L + kb * BN;
  const int kn = nat_kv ? min(BN, sh.S - k0) : min(BN, sh.L - kb * BN);
  const T* qp = static_cast<const T*>(a.q);
  const T* kp = static_cast<const T*>(a.k);
  const T* vp = static_cast<const T*>(a.v);
  const T* dop = static_cast<const T*>(a.dout);

  load_tile<T, D>(Ks, kp, b, k0, kn, g, sh.Hkv, sh.S);
  load_tile<T, D>(Vs, vp, b, k0, kn, g, sh.Hkv, sh.S);
  if (tid < BN)
    k_nat[tid] = tid < kn ? (nat_kv ? k0 + tid : natural_pos(sh, k0 + tid)) : INT_MAX;
  __syncthreads();
  if (tid < 32) {
    int mn = min(k_nat[tid], k_nat[tid + 32]);
    int mx = max(tid < kn ? k_nat[tid] : -1, tid + 32 < kn ? k_nat[tid + 32] : -1);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      mn = min(mn, __shfl_xor_sync(0xffffffffu, mn, off));
      mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, off));
    }
    if (tid == 0) {
      s_kmin = mn;
      s_kmax = mx;
    }
  }
  __syncthreads();
  const int kmin = s_kmin, kmax = s_kmax;

  float dk[4][DV], dv[4][DV];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int dd = 0; dd < DV; ++dd) dk[i][dd] = dv[i][dd] = 0.f;

  for (int hh = 0; hh < grp; ++hh) {
    const int h = g * grp + hh;
    for (int t = 0; t < sh.cp; ++t) {
      // the rank holding this K/V at step t (all-gather: every rank, in order)
      const int r = nat_kv ? t : (s + t) % sh.cp;
      for (int qb = 0; qb < sh.L; qb += BM) {
        const int q0 = r * sh.L + qb, qn = min(BM, sh.L - qb);
        __syncthreads();
        int live = 0;
        if (tid < BM) {
          int lo = INT_MAX, hi = -1;  // padding rows see nothing
          if (tid < qn) query_window(sh, natural_pos(sh, q0 + tid), lo, hi);
          q_lo[tid] = lo;
          q_hi[tid] = hi;
          live = lo <= kmax && hi >= kmin;
          if (tid < qn) {
            int64_t li = ((int64_t)b * sh.H + h) * sh.S + q0 + tid;
            lse2[tid] = a.lse[li] * kLog2e;
            dlt[tid] = a.delta[li];
          } else {
            lse2[tid] = 0.f;
            dlt[tid] = 0.f;
          }
        }
        if (!__syncthreads_or(live)) continue;
        if (a.tiles_kv_rt != nullptr && !nat_kv && tid == 0)
          atomicAdd(&a.tiles_kv_rt[r * sh.cp + t], 1ull);
        load_tile<T, D>(Qs, qp, b, q0, qn, h, sh.H, sh.S);
        load_tile<T, D>(Os, dop, b, q0, qn, h, sh.H, sh.S);
        __syncthreads();

        float sc[4][4], dp[4][4];
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
          for (int j = 0; j < 4; ++j) sc[i][j] = dp[i][j] = 0.f;
#pragma unroll 4
        for (int d = 0; d < D; ++d) {
          float qv[4], ov[4], kv[4], vv[4];
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            qv[i] = Qs[(ty * 4 + i) * DP + d];
            ov[i] = Os[(ty * 4 + i) * DP + d];
          }
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            kv[j] = Ks[(tx + 16 * j) * DP + d];
            vv[j] = Vs[(tx + 16 * j) * DP + d];
          }
#pragma unroll
          for (int i = 0; i < 4; ++i)
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              sc[i][j] = fmaf(qv[i], kv[j], sc[i][j]);
              dp[i][j] = fmaf(ov[i], vv[j], dp[i][j]);
            }
        }
        // P and dS for this thread's 4 x 4 block (query rows ty*4+i, keys tx+16j).
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int row = ty * 4 + i;
          const int lo = q_lo[row], hi = q_hi[row];
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const int col = tx + 16 * j;
            const bool ok = col < kn && k_nat[col] >= lo && k_nat[col] <= hi;
            const float p = ok ? exp2f(sc[i][j] * sh.scale_log2 - lse2[row]) : 0.f;
            sc[i][j] = p;
            dp[i][j] = p * (dp[i][j] - dlt[row]);
            Ps[row * PP + col] = p;
          }
        }
        __syncthreads();
        // dV[key][d] += sum_q P[q][key] dO[q][d]   (keys ty*4+i, d = tx+16dd)
#pragma unroll 4
        for (int qq = 0; qq < BM; ++qq) {
          float pv[4], ov[DV];
#pragma unroll
          for (int i = 0; i < 4; ++i) pv[i] = Ps[qq * PP + ty * 4 + i];
#pragma unroll
          for (int dd = 0; dd < DV; ++dd) ov[dd] = Os[qq * DP + tx + 16 * dd];
#pragma unroll
          for (int i = 0; i < 4; ++i)
#pragma unroll
            for (int dd = 0; dd < DV; ++dd) dv[i][dd] = fmaf(pv[i], ov[dd], dv[i][dd]);
        }
        __syncthreads();
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
          for (int j = 0; j < 4; ++j) Ps[(ty * 4 + i) * PP + tx + 16 * j] = dp[i][j];
        __syncthreads();
        // dK[key][d] += sum_q dS[q][key] Q[q][d]
#pragma unroll 4
        for (int qq = 0; qq < BM; ++qq) {
          float sv[4], qv[DV];
#pragma unroll
          for (int i = 0; i < 4; ++i) sv[i] = Ps[qq * PP + ty * 4 + i];
#pragma unroll
          for (int dd = 0; dd < DV; ++dd) qv[dd] = Qs[qq * DP + tx + 16 * dd];
#pragma unroll
          for (int i = 0; i < 4; ++i)
#pragma unroll
            for (int dd = 0; dd < DV; ++dd) dk[i][dd] = fmaf(sv[i], qv[dd], dk[i][dd]);
        }
      }
    }
  }

  // This CTA owns its key rows over every query: plain float32 stores into the
  // accumulators (the conversion kernel follows).
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int row = ty * 4 + i;
    if (row >= kn) continue;
    const int64_t base = (((int64_t)b * sh.S + k0 + row) * sh.Hkv + g) * D;
#pragma unroll
    for (int dd = 0; dd < DV; ++dd) {
      a.dk_acc[base + tx + 16 * dd] = sh.scale * dk[i][dd];
      a.dv_acc[base + tx + 16 * dd] = dv[i][dd];
    }
  }
}

// dQ, query-major (see the file header).
template <typename T, int D>
__global__ void __launch_bounds__(NT) simt_dq_kernel(const BwdArgs a) {
  constexpr int DP = D + 1, PP = BN + 1, DV = D / 16;
  extern __shared__ float smem[];
  float* Qs = smem;
  float* Os = Qs + BM * DP;  // dO tile
  float* Ks = Os + BM * DP;
  float* Vs = Ks + BN * DP;
  float* Ps = Vs + BN * DP;  // dS
  __shared__ int q_lo[BM], q_hi[BM];  // key window of each query row
  __shared__ int k_nat[BN];
  __shared__ float lse2[BM];  // LSE in base 2
  __shared__ float dlt[BM];
  __shared__ int s_lo, s_hi;

  const RingShape& sh = a.sh;
  const int tid = threadIdx.x, ty = tid >> 4, tx = tid & 15;
  const int nblk = (sh.L + BM - 1) / BM;
  const int r = blockIdx.x / nblk, qb = blockIdx.x - r * nblk;
  const int b = blockIdx.y / sh.H, h = blockIdx.y - b * sh.H;
  const int g = h / (sh.H / sh.Hkv);
  const int q0 = r * sh.L + qb * BM;
  const int qn = min(BM, sh.L - qb * BM);
  const T* qp = static_cast<const T*>(a.q);
  const T* kp = static_cast<const T*>(a.k);
  const T* vp = static_cast<const T*>(a.v);
  const T* dop = static_cast<const T*>(a.dout);

  load_tile<T, D>(Qs, qp, b, q0, qn, h, sh.H, sh.S);
  load_tile<T, D>(Os, dop, b, q0, qn, h, sh.H, sh.S);
  if (tid < BM) {
    int lo = INT_MAX, hi = -1;  // padding rows see nothing
    float l2 = 0.f, dl = 0.f;
    if (tid < qn) {
      query_window(sh, natural_pos(sh, q0 + tid), lo, hi);
      const int64_t li = ((int64_t)b * sh.H + h) * sh.S + q0 + tid;
      l2 = a.lse[li] * kLog2e;
      dl = a.delta[li];
    }
    q_lo[tid] = lo;
    q_hi[tid] = hi;
    lse2[tid] = l2;
    dlt[tid] = dl;
  }
  __syncthreads();
  if (tid < 32) {
    int lo = min(q_lo[tid], q_lo[tid + 32]), hi = max(q_hi[tid], q_hi[tid + 32]);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      lo = min(lo, __shfl_xor_sync(0xffffffffu, lo, off));
      hi = max(hi, __shfl_xor_sync(0xffffffffu, hi, off));
    }
    if (tid == 0) {
      s_lo = lo;
      s_hi = hi;
    }
  }
  __syncthreads();
  const int blk_lo = s_lo, blk_hi = s_hi;  // keys some row of the block sees

  float dq[4][DV];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int dd = 0; dd < DV; ++dd) dq[i][dd] = 0.f;

  // Ring: every step t, the shard of rank (r - t) mod cp.  All-gather
  // (kv_natural): one pass over the whole K/V in natural order.
  const bool nat_kv = sh.kv_natural != 0;
  const int n_pass = nat_kv ? 1 : sh.cp;
  for (int t = 0; t < n_pass; ++t) {
    const int s = ring_source(r, t, sh.cp);
    const int kbase = nat_kv ? 0 : s * sh.L, klen = nat_kv ? sh.S : sh.L;
    for (int kb = 0; kb < klen; kb += BN) {
      const int k0 = kbase + kb, kn = min(BN, klen - kb);
      __syncthreads();  // the previous tile is fully consumed
      int live = 0;
      if (tid < BN) {
        int kpos = tid < kn ? (nat_kv ? k0 + tid : natural_pos(sh, k0 + tid)) : INT_MAX;
        k_nat[tid] = kpos;
        live = tid < kn && kpos >= blk_lo && kpos <= blk_hi;
      }
      if (!__syncthreads_or(live)) continue;  // no row of the block sees the tile
      if (a.tiles_q_rt != nullptr && !nat_kv && tid == 0)
        atomicAdd(&a.tiles_q_rt[r * sh.cp + t], 1ull);
      load_tile<T, D>(Ks, kp, b, k0, kn, g, sh.Hkv, sh.S);
      load_tile<T, D>(Vs, vp, b, k0, kn, g, sh.Hkv, sh.S);
      __syncthreads();

      float sc[4][4], dp[4][4];
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) sc[i][j] = dp[i][j] = 0.f;
#pragma unroll 4
      for (int d = 0; d < D; ++d) {
        float qv[4], ov[4], kv[4], vv[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          qv[i] = Qs[(ty * 4 + i) * DP + d];
          ov[i] = Os[(ty * 4 + i) * DP + d];
        }
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          kv[j] = Ks[(tx + 16 * j) * DP + d];
          vv[j] = Vs[(tx + 16 * j) * DP + d];
        }
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            sc[i][j] = fmaf(qv[i], kv[j], sc[i][j]);
            dp[i][j] = fmaf(ov[i], vv[j], dp[i][j]);
          }
      }
      // dS = P (dP - Delta) for this thread's 4 x 4 block (query rows
      // ty*4+i, keys tx+16j), P from the saved LSE.
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int row = ty * 4 + i;
        const int lo = q_lo[row], hi = q_hi[row];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int col = tx + 16 * j;
          const bool ok = col < kn && k_nat[col] >= lo && k_nat[col] <= hi;
          const float p = ok ? exp2f(sc[i][j] * sh.scale_log2 - lse2[row]) : 0.f;
          Ps[row * PP + col] = p * (dp[i][j] - dlt[row]);
        }
      }
      __syncthreads();
      // dQ[q][d] += sum_key dS[q][key] K[key][d]   (rows ty*4+i, d = tx+16dd)
#pragma unroll 4
      for (int c = 0; c < BN; ++c) {
        float sv[4], kv[DV];
#pragma unroll
        for (int i = 0; i < 4; ++i) sv[i] = Ps[(ty * 4 + i) * PP + c];
#pragma unroll
        for (int dd = 0; dd < DV; ++dd) kv[dd] = Ks[c * DP + tx + 16 * dd];
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
          for (int dd = 0; dd < DV; ++dd) dq[i][dd] = fmaf(sv[i], kv[dd], dq[i][dd]);
      }
    }
  }

#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int row = ty * 4 + i;
    if (row >= qn) continue;
    float* dst = a.dq_acc + (((int64_t)b * sh.S + q0 + row) * sh.H + h) * D;
#pragma unroll
    for (int dd = 0; dd < DV; ++dd) dst[tx + 16 * dd] = sh.scale * dq[i][dd];
  }
}

template <typename T, int D, bool STEP>
cudaError_t fwd_as(const FwdArgs& a, cudaStream_t stream) {
  constexpr int smem = fwd_smem_bytes<D>();
  auto kern = simt_fwd_kernel<T, D, STEP>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  const int nblk = (a.sh.L + BM - 1) / BM;
  dim3 grid(nblk * a.sh.cp, a.sh.B * a.sh.H);
  kern<<<grid, NT, smem, stream>>>(a);
  return cudaGetLastError();
}

template <typename T, int D>
cudaError_t bwd_as(const BwdArgs& a, cudaStream_t stream) {
  constexpr int smem = bwd_smem_bytes<D>();
  auto kern = simt_bwd_kernel<T, D>;
  auto kern_dq = simt_dq_kernel<T, D>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(kern_dq, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  const int nblk = (a.sh.L + BN - 1) / BN;
  dim3 grid(a.sh.kv_natural ? (a.sh.S + BN - 1) / BN : nblk * a.sh.cp, a.sh.B * a.sh.Hkv);
  kern<<<grid, NT, smem, stream>>>(a);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const int qblk = (a.sh.L + BM - 1) / BM;
  dim3 grid_dq(qblk * a.sh.cp, a.sh.B * a.sh.H);
  kern_dq<<<grid_dq, NT, smem, stream>>>(a);
  return cudaGetLastError();
}

template <typename T>
cudaError_t fwd_dispatch(const FwdArgs& a, cudaStream_t stream) {
  if (a.sh.D == 128)
    return a.step_mode ? fwd_as<T, 128, true>(a, stream) : fwd_as<T, 128, false>(a, stream);
  return a.step_mode ? fwd_as<T, 64, true>(a, stream) : fwd_as<T, 64, false>(a, stream);
}

}  // namespace

cudaError_t launch_simt_fwd(const FwdArgs& a, int dtype, cudaStream_t stream) {
  if (a.sh.B == 0 || a.sh.H == 0 || a.sh.S == 0) return cudaSuccess;
  return dtype == 1 ? fwd_dispatch<__nv_bfloat16>(a, stream) : fwd_dispatch<float>(a, stream);
}

cudaError_t launch_simt_bwd(const BwdArgs& a, int dtype, cudaStream_t stream) {
  if (a.sh.B == 0 || a.sh.H == 0 || a.sh.S == 0) return cudaSuccess;
  if (dtype == 1)
    return a.sh.D == 128 ? bwd_as<__nv_bfloat16, 128>(a, stream)
                         : bwd_as<__nv_bfloat16, 64>(a, stream);
  return a.sh.D == 128 ? bwd_as<float, 128>(a, stream) : bwd_as<float, 64>(a, stream);
}

}  // namespace cpattn
