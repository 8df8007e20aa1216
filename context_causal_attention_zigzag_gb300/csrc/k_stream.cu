// Bandwidth-bound kernels of the ring: zigzag permute / unpermute, the exact
// LSE merge of two partials, the backward pre-pass (Delta = dO . O and zeroing
// of the gradient accumulators) and the float32 -> output dtype conversion of
// dQ, dK, dV; the per-position document bounds of a packed sequence; and the
// all-to-all transposes of the Ulysses variant.
//
// All of them move data in 16-byte vectors with consecutive threads on
// consecutive vectors, and size their grids as a multiple of the SM count.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <limits.h>
#include <stdint.h>

#include "cpattn_internal.h"

namespace cpattn {
namespace {

int sm_count() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 148;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 148;
  return n > 0 ? n : 148;
}

int grid_for(int64_t work_items, int threads, int per_sm) {
  int64_t want = (work_items + threads - 1) / threads;
  int64_t cap = (int64_t)sm_count() * per_sm;
  if (want > cap) want = cap;
  return (int)(want < 1 ? 1 : want);
}

// ---------------------------------------------------------------------------
// Permute.  A tensor [outer, S, inner] moves as outer * nchunk runs of
// c * inner contiguous bytes (a chunk keeps its internal order), so the copy
// is a gather of runs: run (o, sharded chunk ci) <-> (o, natural chunk nc).
// The natural side may be shorter (S_nat <= S tokens): natural positions from
// S_nat on are padding, written as zeros into the sharded tensor and dropped
// on the way back.
// ---------------------------------------------------------------------------
template <typename V>
__global__ void __launch_bounds__(256) permute_runs_kernel(const char* __restrict__ in,
                                                           char* __restrict__ out, int64_t S,
                                                           int64_t S_nat, int64_t inner_bytes,
                                                           int cp, int per_rank, int64_t c,
                                                           int64_t run_vecs, int64_t blocks_per_run,
                                                           bool inverse) {
  // Block -> (run, part of the run); the run's offsets once per block, then
  // a plain strided copy of its vectors.
  constexpr int U = 4;
  const int64_t nchunk = (int64_t)cp * per_rank;
  const int64_t run = blockIdx.x / blocks_per_run;  // (outer index, sharded chunk)
  const int64_t part = blockIdx.x - run * blocks_per_run;
  const int64_t ci = run % nchunk, o = run / nchunk;
  const int r = (int)(ci / per_rank), j = (int)(ci % per_rank);
  const int64_t nc = (per_rank == 1 || j == 0) ? r : 2 * cp - 1 - r;  // natural chunk
  // Tokens of this run that are real (not padding); a whole number of
  // vectors (the launcher picks V so that S_nat * inner_bytes and the run
  // length are multiples of it).
  int64_t real = S_nat - nc * c;
  real = real < 0 ? 0 : (real > c ? c : real);
  const int64_t real_vecs = real * inner_bytes / (int64_t)sizeof(V);
  const int64_t sh_off = (o * S + ci * c) * inner_bytes;
  const int64_t nat_off = (o * S_nat + nc * c) * inner_bytes;
  const V* src = reinterpret_cast<const V*>(in + (inverse ? sh_off : nat_off));
  V* dst = reinterpret_cast<V*>(out + (inverse ? nat_off : sh_off));
  // Sharding writes the whole run (zeros for padding); unsharding writes
  // only the real tokens.
  const int64_t nwrite = inverse ? real_vecs : run_vecs;
  const int64_t step = blocks_per_run * (int64_t)blockDim.x;
  for (int64_t e0 = part * blockDim.x + threadIdx.x; e0 < nwrite; e0 += step * U) {
    V val[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int64_t e = e0 + u * step;
      val[u] = e < real_vecs ? src[e] : V{};
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int64_t e = e0 + u * step;
      if (e < nwrite) dst[e] = val[u];
    }
  }
}

template <typename V>
cudaError_t permute_as(const void* in, void* out, int64_t outer, int64_t S, int64_t S_nat,
                       int64_t inner_bytes, const RingShape& sh, bool inverse,
                       cudaStream_t stream) {
  const int64_t run_bytes = (int64_t)sh.c * inner_bytes;
  const int64_t run_vecs = run_bytes / (int64_t)sizeof(V);
  const int64_t nruns = outer * (int64_t)sh.cp * sh.per_rank;
  if (nruns == 0 || run_vecs == 0) return cudaSuccess;
  // About eight resident blocks per SM in total, no more per run than its
  // vectors can keep busy.
  const int64_t target = (int64_t)sm_count() * 8;
  int64_t bpr = (target + nruns - 1) / nruns;
  const int64_t useful = (run_vecs + 256 * 4 - 1) / (256 * 4);
  if (bpr > useful) bpr = useful;
  if (bpr < 1) bpr = 1;
  const int64_t grid = nruns * bpr;
  if (grid > INT32_MAX) return cudaErrorInvalidConfiguration;
  permute_runs_kernel<V><<<(unsigned)grid, 256, 0, stream>>>(
      static_cast<const char*>(in), static_cast<char*>(out), S, S_nat, inner_bytes, sh.cp,
      sh.per_rank, (int64_t)sh.c, run_vecs, bpr, inverse);
  return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// LSE merge: one warp per row (b, s, h); each lane moves float4s.
// ---------------------------------------------------------------------------
template <int D>
__global__ void __launch_bounds__(256) lse_merge_kernel(const float* o_a, const float* l_a,
                                                        const float* o_b, const float* l_b,
                                                        float* o, float* l, int B, int S, int H) {
  constexpr int VPR = D / 4;  // float4 per row
  const int lane = threadIdx.x & 31;
  const int64_t rows = (int64_t)B * S * H;
  const int64_t warp0 = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
  for (int64_t row = warp0; row < rows; row += nwarps) {
    int64_t b = row / ((int64_t)S * H);
    int64_t s = (row / H) % S;
    int64_t h = row % H;
    int64_t li = (b * H + h) * S + s;
    float la = l_a[li], lb = l_b[li];
    float hi = fmaxf(la, lb), lo = fminf(la, lb);
    float L, wa, wb;
    if (hi == -INFINITY) {
      L = -INFINITY;
      wa = 0.f;
      wb = 0.f;
    } else {
      L = hi + log1pf(expf(lo - hi));
      wa = expf(la - L);
      wb = expf(lb - L);
    }
    float4 va[(VPR + 31) / 32], vb[(VPR + 31) / 32];
#pragma unroll
    for (int u = 0; u * 32 < VPR; ++u) {
      int e = lane + u * 32;
      if (e < VPR) {
        va[u] = reinterpret_cast<const float4*>(o_a + row * D)[e];
        vb[u] = reinterpret_cast<const float4*>(o_b + row * D)[e];
      }
    }
    __syncwarp();  // every lane has read before any lane writes (in-place merge)
#pragma unroll
    for (int u = 0; u * 32 < VPR; ++u) {
      int e = lane + u * 32;
      if (e < VPR) {
        float4 r;
#if CPATTN_MUTATION == 3
        r = make_float4(wa * va[u].x, wa * va[u].y, wa * va[u].z, wa * va[u].w);  // planted
        (void)wb;
#else
        r.x = wa * va[u].x + wb * vb[u].x;
        r.y = wa * va[u].y + wb * vb[u].y;
        r.z = wa * va[u].z + wb * vb[u].z;
        r.w = wa * va[u].w + wb * vb[u].w;
#endif
        reinterpret_cast<float4*>(o + row * D)[e] = r;
      }
    }
    if (lane == 0) l[li] = L;
    __syncwarp();
  }
}

// Loads N consecutive elements of T (N * sizeof(T) in {4, 8, 16} bytes, aligned)
// as one vector and widens them to float.
template <typename T, int N>
__device__ __forceinline__ void load_vec(const T* p, float* f) {
  if constexpr (sizeof(T) == 4) {
    if constexpr (N == 4) {
      float4 x = *reinterpret_cast<const float4*>(p);
      f[0] = x.x; f[1] = x.y; f[2] = x.z; f[3] = x.w;
    } else {
      float2 x = *reinterpret_cast<const float2*>(p);
      f[0] = x.x; f[1] = x.y;
    }
  } else {
    if constexpr (N == 4) {
      uint2 x = *reinterpret_cast<const uint2*>(p);
      float2 lo = __bfloat1622float2(*reinterpret_cast<__nv_bfloat162*>(&x.x));
      float2 hi = __bfloat1622float2(*reinterpret_cast<__nv_bfloat162*>(&x.y));
      f[0] = lo.x; f[1] = lo.y; f[2] = hi.x; f[3] = hi.y;
    } else {
      uint32_t x = *reinterpret_cast<const uint32_t*>(p);
      float2 lo = __bfloat1622float2(*reinterpret_cast<__nv_bfloat162*>(&x));
      f[0] = lo.x; f[1] = lo.y;
    }
  }
}

// ---------------------------------------------------------------------------
// Backward pre-pass: delta[b,h,s] = sum_d dout * out (fp32), zero the float32
// dQ accumulator row (one warp per row), and zero the dK / dV accumulators
// (grid-stride, float4).
// ---------------------------------------------------------------------------
template <typename T, int D>
__global__ void __launch_bounds__(256) bwd_prep_kernel(const T* __restrict__ out,
                                                       const T* __restrict__ dout,
                                                       float* __restrict__ delta,
                                                       float* __restrict__ dq_acc,
                                                       float4* __restrict__ dk_acc,
                                                       float4* __restrict__ dv_acc,
                                                       int64_t n4_kv, int B, int S, int H,
                                                       float delta_scale) {
  const int lane = threadIdx.x & 31;
  const int64_t warp0 = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
  constexpr int EPL = D / 32;  // elements per lane: one 4-, 8- or 16-byte vector
  // A warp takes R consecutive rows (b, s, h) of the [B, S, H, D] tensors per
  // iteration: R * D contiguous elements of each, all loads in flight at once.
  constexpr int R = (sizeof(T) == 4 && D == 128) ? 2 : 4;
  const int64_t rows = (int64_t)B * S * H;
  for (int64_t row0 = warp0 * R; row0 < rows; row0 += nwarps * R) {
    float a[R][EPL], b[R][EPL];
#pragma unroll
    for (int r = 0; r < R; ++r) {
      if (row0 + r < rows) {
        load_vec<T, EPL>(out + (row0 + r) * D + lane * EPL, a[r]);
        load_vec<T, EPL>(dout + (row0 + r) * D + lane * EPL, b[r]);
      } else {
#pragma unroll
        for (int e = 0; e < EPL; ++e) a[r][e] = b[r][e] = 0.f;
      }
    }
    float mine = 0.f;  // lane r keeps row r's sum
#pragma unroll
    for (int r = 0; r < R; ++r) {
      float acc = 0.f;
#pragma unroll
      for (int e = 0; e < EPL; ++e) acc = fmaf(a[r][e], b[r][e], acc);
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
      if (lane == r) mine = acc;
    }
    if (dq_acc != nullptr) {
#pragma unroll
      for (int r = 0; r < R; ++r) {
        if (row0 + r >= rows) continue;
        float* dq = dq_acc + (row0 + r) * D + lane * EPL;
        if constexpr (EPL == 4) {
          *reinterpret_cast<float4*>(dq) = make_float4(0.f, 0.f, 0.f, 0.f);
        } else {
          *reinterpret_cast<float2*>(dq) = make_float2(0.f, 0.f);
        }
      }
    }
    if (lane < R && row0 + lane < rows) {
      const int64_t row = row0 + lane;
      const int64_t bi = row / ((int64_t)S * H), si = (row / H) % S, hi = row % H;
      delta[(bi * H + hi) * S + si] = mine * delta_scale;
    }
  }
  const float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n4_kv;
       i += (int64_t)gridDim.x * blockDim.x) {
    dk_acc[i] = z;
    dv_acc[i] = z;
  }
}

// dst[i] = (out dtype) src[i] for the three gradient accumulators, 4
// elements per thread-iteration; element counts are multiples of 4.
template <typename O>
__device__ __forceinline__ void store4(O* dst, int64_t i, float4 x);
template <>
__device__ __forceinline__ void store4<float>(float* dst, int64_t i, float4 x) {
  reinterpret_cast<float4*>(dst)[i] = x;
}
template <>
__device__ __forceinline__ void store4<__nv_bfloat16>(__nv_bfloat16* dst, int64_t i, float4 x) {
  uint2 v;
  __nv_bfloat162 lo = __floats2bfloat162_rn(x.x, x.y), hi = __floats2bfloat162_rn(x.z, x.w);
  v.x = *reinterpret_cast<uint32_t*>(&lo);
  v.y = *reinterpret_cast<uint32_t*>(&hi);
  reinterpret_cast<uint2*>(dst)[i] = v;
}

// Sum of the per-query-head dK / dV partials over each kv head's group.
template <typename O>
__global__ void __launch_bounds__(256) grad_reduce_kernel(const float4* __restrict__ dk_part,
                                                          const float4* __restrict__ dv_part,
                                                          O* __restrict__ dk, O* __restrict__ dv,
                                                          int64_t rows_kv, int H, int Hkv,
                                                          int D4) {
  const int grp = H / Hkv;
  const int64_t total = rows_kv * D4;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t row = i / D4;  // (b*S + s)*Hkv + g
    const int d4 = (int)(i - row * D4);
    const int64_t bs = row / Hkv;
    const int g = (int)(row - bs * Hkv);
    const int64_t p0 = ((bs * H + (int64_t)g * grp) * D4) + d4;
    float4 a = dk_part[p0], b = dv_part[p0];
    for (int hh = 1; hh < grp; ++hh) {
      const float4 x = dk_part[p0 + (int64_t)hh * D4], y = dv_part[p0 + (int64_t)hh * D4];
      a.x += x.x; a.y += x.y; a.z += x.z; a.w += x.w;
      b.x += y.x; b.y += y.y; b.z += y.z; b.w += y.w;
    }
    store4<O>(dk, i, a);
    store4<O>(dv, i, b);
  }
}

template <typename O>
__global__ void __launch_bounds__(256) grad_convert_kernel(const float4* __restrict__ q4,
                                                           const float4* __restrict__ k4,
                                                           const float4* __restrict__ v4,
                                                           O* __restrict__ dq, O* __restrict__ dk,
                                                           O* __restrict__ dv, int64_t nq4,
                                                           int64_t nkv4) {
  const int64_t total = nq4 + 2 * nkv4;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total;
       i += (int64_t)gridDim.x * blockDim.x) {
    if (i < nq4) {
      store4<O>(dq, i, q4[i]);
    } else if (i < nq4 + nkv4) {
      store4<O>(dk, i - nq4, k4[i - nq4]);
    } else {
      store4<O>(dv, i - nq4 - nkv4, v4[i - nq4 - nkv4]);
    }
  }
}

// ---------------------------------------------------------------------------
// Document bounds.  Position p belongs to the document d with
// cu[d] <= p < cu[d+1] (binary search over the offsets); threads d < ndocs
// also check the offsets themselves (the caller guarantees 1 <= ndocs <= S,
// so every offset is checked).
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256) doc_bounds_kernel(const int* __restrict__ cu, int ndocs,
                                                         int S, int2* __restrict__ docs,
                                                         int* err) {
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t x = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; x < S; x += stride) {
    const int p = (int)x;
    if (x < ndocs) {
      bool bad = cu[x] >= cu[x + 1];
      if (x == 0) bad = bad || cu[0] != 0 || cu[ndocs] != S;
      if (bad) atomicExch(err, kErrBadDocs);
    }
    int lo = 0, hi = ndocs;  // invariant: cu[lo] <= p < cu[hi] for valid offsets
    while (hi - lo > 1) {
      const int mid = lo + (hi - lo) / 2;
      if (cu[mid] <= p)
        lo = mid;
      else
        hi = mid;
    }
    int first = cu[lo], end = cu[lo + 1];
    if (first < 0 || first > p) first = p;  // only for broken offsets
    if (end <= p || end > S) end = p + 1;
    docs[p] = make_int2(first, end);
  }
}

// ---------------------------------------------------------------------------
// Sequence <-> head all-to-all (Ulysses, and the first level of the
// hierarchical schedule).  Sequence -> head: each (head owner r, b, row m)
// row of the output is nx*D contiguous elements read from one sharded row of
// the input (the token at natural position natural_pos(inner, m)), so the
// copy moves 16-byte vectors of those runs.  Head -> sequence: each
// (b, sharded p, head x) row of D elements sums the head owners holding x.
// ---------------------------------------------------------------------------
__device__ __forceinline__ int a2a_x0(const A2aShape& a, int r) {
  return (int)(((long long)r * a.x_num) / a.x_den);
}

template <typename V>
__global__ void __launch_bounds__(256) a2a_to_head_kernel(const char* __restrict__ in,
                                                          char* __restrict__ out,
                                                          const A2aShape a, int elt) {
  const int64_t row_vecs = (int64_t)a.nx * a.D * elt / (int64_t)sizeof(V);
  const int64_t total = (int64_t)a.ranks * a.B * a.sh.S * row_vecs;
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total; i += stride) {
    const int64_t row = i / row_vecs, e = i - row * row_vecs;
    const int m = (int)(row % a.sh.S);
    const int64_t rb = row / a.sh.S;
    const int b = (int)(rb % a.B), r = (int)(rb / a.B);
    const int p = sharded_pos(a.sh, natural_pos(a.inner, m));
    const int64_t src = ((((int64_t)b * a.sh.S + p) * a.X + a2a_x0(a, r)) * a.D) * elt +
                        e * (int64_t)sizeof(V);
    reinterpret_cast<V*>(out)[i] = *reinterpret_cast<const V*>(in + src);
  }
}

template <typename T>
__device__ __forceinline__ float a2a_ld(const T* p);
template <>
__device__ __forceinline__ float a2a_ld<float>(const float* p) { return *p; }
template <>
__device__ __forceinline__ float a2a_ld<__nv_bfloat16>(const __nv_bfloat16* p) {
  return __bfloat162float(*p);
}
template <typename T>
__device__ __forceinline__ void a2a_st(T* p, float x);
template <>
__device__ __forceinline__ void a2a_st<float>(float* p, float x) { *p = x; }
template <>
__device__ __forceinline__ void a2a_st<__nv_bfloat16>(__nv_bfloat16* p, float x) {
  *p = __float2bfloat16_rn(x);
}

// One thread per 4 elements of an output row (D is a multiple of 4).
template <typename T>
__global__ void __launch_bounds__(256) a2a_to_seq_kernel(const T* __restrict__ in,
                                                         T* __restrict__ out, const A2aShape a) {
  const int q4 = a.D / 4;
  const int64_t total = (int64_t)a.B * a.sh.S * a.X * q4;
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total; i += stride) {
    const int d = (int)(i % q4) * 4;
    const int64_t row = i / q4;  // (b, p, x)
    const int x = (int)(row % a.X);
    const int64_t bp = row / a.X;
    const int p = (int)(bp % a.sh.S), b = (int)(bp / a.sh.S);
    const int m = sharded_pos(a.inner, natural_pos(a.sh, p));
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
    for (int r = 0; r < a.ranks; ++r) {
      const int x0 = a2a_x0(a, r);
      if (x < x0 || x >= x0 + a.nx) continue;
      const T* src = in + ((((int64_t)r * a.B + b) * a.sh.S + m) * a.nx + (x - x0)) * a.D + d;
#pragma unroll
      for (int u = 0; u < 4; ++u) acc[u] += a2a_ld<T>(src + u);
    }
    T* dst = out + row * a.D + d;
#pragma unroll
    for (int u = 0; u < 4; ++u) a2a_st<T>(dst + u, acc[u]);
  }
}

// LSE: out[r, b, h', m] = in[b, r*hc + h', p(m)] (to heads) and back, p(m)
// the sharded position of the token at row m of the head owners' order.
__global__ void __launch_bounds__(256) lse_a2a_kernel(const float* __restrict__ in,
                                                      float* __restrict__ out,
                                                      const RingShape sh, const RingShape inner,
                                                      int ranks, int B, int H, bool to_seq) {
  const int hc = H / ranks;
  const int64_t total = (int64_t)B * H * sh.S;
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total; i += stride) {
    // i indexes the sharded [B, H, S] tensor: (b, h, p)
    const int p = (int)(i % sh.S);
    const int64_t bh = i / sh.S;
    const int h = (int)(bh % H), b = (int)(bh / H);
    const int r = h / hc, hh = h - r * hc;
    const int64_t j =
        (((int64_t)r * B + b) * hc + hh) * sh.S + sharded_pos(inner, natural_pos(sh, p));
    if (to_seq)
      out[i] = in[j];
    else
      out[j] = in[i];
  }
}

}  // namespace

cudaError_t launch_a2a(const void* in, void* out, const A2aShape& a, bool to_seq, int dtype,
                       cudaStream_t stream) {
  const int elt = dtype == 1 ? 2 : 4;
  const int64_t rows = (int64_t)a.ranks * a.B * a.sh.S;
  if (rows == 0 || a.nx == 0) return cudaSuccess;
  if (!to_seq) {
    const int64_t row_bytes = (int64_t)a.nx * a.D * elt;
    const uint64_t align = (uint64_t)(reinterpret_cast<uintptr_t>(in) |
                                      reinterpret_cast<uintptr_t>(out)) |
                           (uint64_t)row_bytes | (uint64_t)((int64_t)a.X * a.D * elt);
    if ((align & 15) == 0) {
      a2a_to_head_kernel<uint4><<<grid_for(rows * row_bytes / 16, 256, 8), 256, 0, stream>>>(
          static_cast<const char*>(in), static_cast<char*>(out), a, elt);
    } else {
      a2a_to_head_kernel<uint32_t><<<grid_for(rows * row_bytes / 4, 256, 8), 256, 0, stream>>>(
          static_cast<const char*>(in), static_cast<char*>(out), a, elt);
    }
    return cudaGetLastError();
  }
  const int64_t n = (int64_t)a.B * a.sh.S * a.X * (a.D / 4);
  if (dtype == 1)
    a2a_to_seq_kernel<__nv_bfloat16><<<grid_for(n, 256, 8), 256, 0, stream>>>(
        static_cast<const __nv_bfloat16*>(in), static_cast<__nv_bfloat16*>(out), a);
  else
    a2a_to_seq_kernel<float><<<grid_for(n, 256, 8), 256, 0, stream>>>(
        static_cast<const float*>(in), static_cast<float*>(out), a);
  return cudaGetLastError();
}

cudaError_t launch_lse_a2a(const float* in, float* out, const RingShape& sh,
                           const RingShape& inner, int ranks, int B, int H, bool to_seq,
                           cudaStream_t stream) {
  const int64_t n = (int64_t)B * H * sh.S;
  if (n == 0) return cudaSuccess;
  lse_a2a_kernel<<<grid_for(n, 256, 8), 256, 0, stream>>>(in, out, sh, inner, ranks, B, H,
                                                          to_seq);
  return cudaGetLastError();
}

cudaError_t launch_doc_bounds(const int* cu, int ndocs, int S, int2* docs, int* err,
                              cudaStream_t stream) {
  if (S == 0) return cudaSuccess;
  doc_bounds_kernel<<<grid_for(S, 256, 4), 256, 0, stream>>>(cu, ndocs, S, docs, err);
  return cudaGetLastError();
}

cudaError_t launch_permute(const void* in, void* out, int64_t outer, int64_t S, int64_t S_nat,
                           int64_t inner_bytes, const RingShape& sh, bool inverse,
                           cudaStream_t stream) {
  int64_t run_bytes = (int64_t)sh.c * inner_bytes;
  uintptr_t a = reinterpret_cast<uintptr_t>(in) | reinterpret_cast<uintptr_t>(out);
  // Every run starts at a multiple of run_bytes (plus whole rows of S_nat
  // tokens on the natural side) from the base pointers.
  uint64_t align = (uint64_t)a | (uint64_t)run_bytes | (uint64_t)(S_nat * inner_bytes);
#define CPATTN_PERMUTE_AS(V) \
  permute_as<V>(in, out, outer, S, S_nat, inner_bytes, sh, inverse, stream)
  if ((align & 15) == 0) return CPATTN_PERMUTE_AS(uint4);
  if ((align & 7) == 0) return CPATTN_PERMUTE_AS(uint2);
  if ((align & 3) == 0) return CPATTN_PERMUTE_AS(uint32_t);
  if ((align & 1) == 0) return CPATTN_PERMUTE_AS(uint16_t);
  return CPATTN_PERMUTE_AS(uint8_t);
#undef CPATTN_PERMUTE_AS
}

cudaError_t launch_lse_merge(const float* o_a, const float* l_a, const float* o_b,
                             const float* l_b, float* o, float* l, int B, int S, int H, int D,
                             cudaStream_t stream) {
  int64_t rows = (int64_t)B * S * H;
  if (rows == 0) return cudaSuccess;
  int grid = grid_for(rows * 32, 256, 8);
  if (D == 128)
    lse_merge_kernel<128><<<grid, 256, 0, stream>>>(o_a, l_a, o_b, l_b, o, l, B, S, H);
  else
    lse_merge_kernel<64><<<grid, 256, 0, stream>>>(o_a, l_a, o_b, l_b, o, l, B, S, H);
  return cudaGetLastError();
}

cudaError_t launch_bwd_prep(const void* out, const void* dout, float* delta, float* dq_acc,
                            float* dk_acc, float* dv_acc, int64_t n_kv, int B, int S, int H,
                            int D, int dtype, float delta_scale, cudaStream_t stream) {
  int64_t rows = (int64_t)B * S * H;
  if (rows == 0) return cudaSuccess;
  int grid = grid_for(rows * 32, 256, 8);
  float4* dk4 = reinterpret_cast<float4*>(dk_acc);
  float4* dv4 = reinterpret_cast<float4*>(dv_acc);
  const int64_t n4 = n_kv / 4;
  if (dtype == 1) {
    auto o = static_cast<const __nv_bfloat16*>(out);
    auto d = static_cast<const __nv_bfloat16*>(dout);
    if (D == 128)
      bwd_prep_kernel<__nv_bfloat16, 128>
          <<<grid, 256, 0, stream>>>(o, d, delta, dq_acc, dk4, dv4, n4, B, S, H, delta_scale);
    else
      bwd_prep_kernel<__nv_bfloat16, 64>
          <<<grid, 256, 0, stream>>>(o, d, delta, dq_acc, dk4, dv4, n4, B, S, H, delta_scale);
  } else {
    auto o = static_cast<const float*>(out);
    auto d = static_cast<const float*>(dout);
    if (D == 128)
      bwd_prep_kernel<float, 128><<<grid, 256, 0, stream>>>(o, d, delta, dq_acc, dk4, dv4, n4, B,
                                                            S, H, delta_scale);
    else
      bwd_prep_kernel<float, 64><<<grid, 256, 0, stream>>>(o, d, delta, dq_acc, dk4, dv4, n4, B,
                                                           S, H, delta_scale);
  }
  return cudaGetLastError();
}

cudaError_t launch_grad_reduce(const float* dk_part, const float* dv_part, void* dk, void* dv,
                               int B, int S, int H, int Hkv, int D, int out_dtype,
                               cudaStream_t stream) {
  const int64_t rows_kv = (int64_t)B * S * Hkv;
  const int D4 = D / 4;
  if (rows_kv == 0) return cudaSuccess;
  int grid = grid_for(rows_kv * D4, 256, 8);
  auto k4 = reinterpret_cast<const float4*>(dk_part);
  auto v4 = reinterpret_cast<const float4*>(dv_part);
  if (out_dtype == 1)
    grad_reduce_kernel<__nv_bfloat16><<<grid, 256, 0, stream>>>(
        k4, v4, static_cast<__nv_bfloat16*>(dk), static_cast<__nv_bfloat16*>(dv), rows_kv, H, Hkv,
        D4);
  else
    grad_reduce_kernel<float><<<grid, 256, 0, stream>>>(
        k4, v4, static_cast<float*>(dk), static_cast<float*>(dv), rows_kv, H, Hkv, D4);
  return cudaGetLastError();
}

cudaError_t launch_grad_convert(const float* dq_acc, const float* dk_acc, const float* dv_acc,
                                void* dq, void* dk, void* dv, int64_t n_q, int64_t n_kv,
                                int out_dtype, cudaStream_t stream) {
  const int64_t nq4 = n_q / 4, nkv4 = n_kv / 4;  // D is a multiple of 64
  const int64_t total = nq4 + 2 * nkv4;
  if (total == 0) return cudaSuccess;
  int grid = grid_for(total, 256, 8);
  auto q4 = reinterpret_cast<const float4*>(dq_acc);
  auto k4 = reinterpret_cast<const float4*>(dk_acc);
  auto v4 = reinterpret_cast<const float4*>(dv_acc);
  if (out_dtype == 1)
    grad_convert_kernel<__nv_bfloat16><<<grid, 256, 0, stream>>>(
        q4, k4, v4, static_cast<__nv_bfloat16*>(dq), static_cast<__nv_bfloat16*>(dk),
        static_cast<__nv_bfloat16*>(dv), nq4, nkv4);
  else
    grad_convert_kernel<float><<<grid, 256, 0, stream>>>(q4, k4, v4, static_cast<float*>(dq),
                                                         static_cast<float*>(dk),
                                                         static_cast<float*>(dv), nq4, nkv4);
  return cudaGetLastError();
}

}  // namespace cpattn
