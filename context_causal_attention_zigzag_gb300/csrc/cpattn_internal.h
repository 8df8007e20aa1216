// Internal interfaces between the C-ABI layer (cpattn_api.cu) and the kernel
// translation units.  Not installed; not part of the ABI.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "cpattn.h"

// Planted mistakes for the mutation tests: a build with -DCPATTN_MUTATION=n
// (n > 0, into a build folder of its own) compiles mistake n into the
// library, so that the tests can show that the GPU parity checks catch it.
// The regular build is always 0.
#ifndef CPATTN_MUTATION
#define CPATTN_MUTATION 0
#endif

namespace cpattn {

// Shape of one ring problem.  Positions are token indices along S.
struct RingShape {
  int B, H, Hkv, S, D;
  int cp;        // context-parallel size (number of virtual ranks)
  int layout;    // CPATTN_LAYOUT_*
  int causal;    // 1: key j visible to query i iff natural(j) <= natural(i)
  int per_rank;  // chunks per rank: 2 (zigzag) or 1 (contiguous)
  int L;         // tokens per rank, S / cp
  int c;         // chunk length, L / per_rank
  float scale;       // softmax scale
  float scale_log2;  // softmax scale * log2(e): scores are kept in base 2
  // Packed documents ("Context Parallelism for Long-Context Training",
  // "Prove attention equivalence" and "Test sequence divisibility and
  // padding"): docs[p] = (first position, one past the last position) of the
  // document holding natural position p; a token sees only its own document.
  // nullptr: the whole sequence is one document.
  const int2* docs;
  // K/V schedule.  0, ring: K, V (dK, dV) are in sharded order like Q and
  // the tiles of rank (r - t) mod cp arrive at step t ("Sequence Parallelism
  // IV", section 4).  1, all-gather: every rank holds the whole K, V (dK,
  // dV) in natural order and walks it chunk by chunk in natural order
  // ("Context Parallelism in MegaDLMs", key-value communication patterns).
  int kv_natural;
  // ceil(2^32 / (c / 128)) when 128 divides c (else 0), for chunk_of_tile.
  unsigned long long tile_magic;
};

// Rank owning natural chunk kc, and the chunk's slot in that rank's shard.
__host__ __device__ inline int chunk_owner(const RingShape& s, int kc) {
  return (s.per_rank == 1 || kc < s.cp) ? kc : 2 * s.cp - 1 - kc;
}
__host__ __device__ inline int chunk_slot(const RingShape& s, int kc) {
  return (s.per_rank == 1 || kc < s.cp) ? 0 : 1;
}
// Sharded position of natural position n (inverse of natural_pos).
__host__ __device__ inline int sharded_pos(const RingShape& s, int n) {
  if (s.per_rank == 1) return n;
  const int kc = n / s.c, off = n - kc * s.c;
  return chunk_owner(s, kc) * s.L + chunk_slot(s, kc) * s.c + off;
}

// Ring step at which rank r holds the K/V of rank src (r, src in [0, cp)).
__host__ __device__ inline int ring_step_of(int r, int src, int cp) {
#if CPATTN_MUTATION == 2
  const int t = src - r;  // planted: the ring turned the other way
#else
  const int t = r - src;
#endif
  return t < 0 ? t + cp : t;
}

// Natural chunk of the tile with natural index m (tiles of 128 tokens):
// m / (c / 128) as (m * tile_magic) >> 32 with tile_magic = ceil(2^32 / (c /
// 128)) (RingShape::tile_magic), so that a step of a tile walk divides
// nothing.  Exact while m * (c / 128) < 2^32 (the tensor-core paths take
// S < 2^23, where both factors are below 2^16).
__host__ __device__ inline int chunk_of_tile(int m, unsigned long long tile_magic) {
  return (int)(((unsigned long long)(unsigned)m * tile_magic) >> 32);
}

// Order of the persistent kernels' work items.  An item is (group, rank,
// sub): `group` the head (or kv head) whose tiles the item reads, `rank` its
// place in cost order (rank 0 visits the most tiles), `sub` one of `inner`
// items of equal cost (the query heads of a kv head).  The ranks are cut into
// cost bands, the band outermost; inside a band the items go group by group,
// so that the CTAs in flight share one group's tiles through L2.  CTA c takes
// items c, 2*grid - 1 - c, 2*grid + c, ... (item_index), which over a list
// sorted by cost gives every CTA about the same work; the bands make the
// list sorted to within one band's cost spread.  The band count is the
// power of two at or above 16 * grid / (items per group), at least 2 and at
// most the number of ranks: two bands where a group holds many waves of items
// (long sequences, whose CTAs in flight then stay within one or two groups,
// so that L2 holds their tiles), more as a group's items shrink against the
// grid (short sequences).  With max_groups > 0 the count is also held to the
// largest power of two that keeps about max_groups groups in flight (a wave
// meets grid * bands / per_group groups), for kernels whose every item
// streams its group's tiles in full.
__host__ __device__ inline int cost_band_count(int per_group, int nrank, int grid,
                                               int max_groups) {
  const int want = (16 * grid + per_group - 1) / per_group;
  int nb = 2;
  while (nb < want) nb *= 2;
  if (max_groups > 0)
    while (nb > 2 && (long long)grid * nb > (long long)max_groups * per_group) nb /= 2;
  return nb < nrank ? nb : nrank;
}

__host__ __device__ inline void banded_item(int idx, int ngroups, int nrank, int inner, int grid,
                                            int max_groups, int& group, int& rank, int& sub) {
  const int nb = cost_band_count(nrank * inner, nrank, grid, max_groups);
  const int bsz = (nrank + nb - 1) / nb;  // ranks per band; the last band may hold fewer
  const int band_items = ngroups * bsz * inner;
  const int band = idx / band_items;
  int rem = idx - band * band_items;
  const int left = nrank - band * bsz;
  const int bw = bsz < left ? bsz : left;
  group = rem / (bw * inner);
  rem -= group * bw * inner;
  const int r = rem / inner;
  rank = band * bsz + r;
  sub = rem - r * inner;
}

// Keys visible to the query at natural position i: the natural range [lo, hi].
// Both ends are non-decreasing in i, so the keys that some query of a run of
// consecutive positions i0..i1 sees form the single range [lo(i0), hi(i1)].
__host__ __device__ inline void query_window(const RingShape& s, int i, int& lo, int& hi) {
  if (s.docs != nullptr) {
    const int2 d = s.docs[i];
    lo = d.x;
    hi = s.causal ? i : d.y - 1;
  } else {
    lo = 0;
    hi = s.causal ? i : s.S - 1;
  }
}

// Queries that see the key at natural position j: the natural range [lo, hi]
// (non-decreasing in j, like query_window).
__host__ __device__ inline void key_window(const RingShape& s, int j, int& lo, int& hi) {
  if (s.docs != nullptr) {
    const int2 d = s.docs[j];
    lo = s.causal ? j : d.x;
    hi = d.y - 1;
  } else {
    lo = s.causal ? j : 0;
    hi = s.S - 1;
  }
}

// Tiles of edge T, counted from the chunk start x0 (chunk length c), that
// overlap the natural range [lo, hi]: [t_lo, t_hi), empty when t_lo >= t_hi.
__host__ __device__ inline void tiles_overlapping(int x0, int c, int T, int lo, int hi,
                                                  int& t_lo, int& t_hi) {
  if (hi < x0 || lo > x0 + c - 1 || lo > hi) {
    t_lo = 0;
    t_hi = 0;
    return;
  }
  t_lo = ((lo > x0 ? lo : x0) - x0) / T;
  t_hi = ((hi < x0 + c - 1 ? hi : x0 + c - 1) - x0) / T + 1;
}

// Natural position of sharded position p.  Rank r = p / L owns, in order,
// chunk r and (zigzag only) chunk 2*cp-1-r ("Sequence Parallelism IV",
// section 3).
__host__ __device__ inline int natural_pos(const RingShape& s, int p) {
  if (s.per_rank == 1) return p;
  int r = p / s.L, w = p - r * s.L;
  int j = w / s.c, off = w - j * s.c;
  int chunk = j == 0 ? r : 2 * s.cp - 1 - r;
  return chunk * s.c + off;
}

// Natural chunk id of the j-th chunk of rank r.
__host__ __device__ inline int rank_chunk(const RingShape& s, int r, int j) {
  return (s.per_rank == 1 || j == 0) ? r : 2 * s.cp - 1 - r;
}

// Ring source: at step t rank r holds the K/V of rank (r - t) mod cp.
__host__ __device__ inline int ring_source(int r, int t, int cp) {
#if CPATTN_MUTATION == 2
  return (r + t) % cp;  // planted: the ring turned the other way
#else
  int s = (r - t) % cp;
  return s < 0 ? s + cp : s;
#endif
}

struct FwdArgs {
  RingShape sh;
  const void* q;
  const void* k;
  const void* v;
  void* out;     // dtype [B,S,H,D] (full forward) or float32 partial (step mode)
  float* lse;    // [B,H,S]
  int t_begin;   // ring steps processed: [t_begin, t_end)
  int t_end;
  int step_mode; // 1: out is a float32 partial, empty rows -> (0, -inf)
  unsigned long long* tiles_rt;  // optional [cp][cp] census (device)
  int* err;      // device error word
};

struct BwdArgs {
  RingShape sh;
  const void* q;
  const void* k;
  const void* v;
  const void* dout;
  const float* lse;    // [B,H,S]
  const float* delta;  // [B,H,S], dout . out (times the softmax scale on the tensor-core path)
  // CUDA-core path: float32 accumulators, pre-zeroed by the pre-pass.
  float* dq_acc;       // [B,S,H,D]   receives scale * dS K
  float* dk_acc;       // [B,S,Hkv,D] receives scale * dS^T Q
  float* dv_acc;       // [B,S,Hkv,D] receives P^T dO
  // Tensor-core path: per-query-head partials of dK / dV (float32, summed
  // over each kv head's group afterwards) and dQ written directly.
  float* dk_part;      // [B,S,H,D]
  float* dv_part;      // [B,S,H,D]
  void* dq;            // [B,S,H,D] float32 if dq_f32 else bf16
  int dq_f32;
  int* err;
  // Optional [cp][cp] census of the tiles each walk visits, per receiving
  // rank r and ring step t: the K/V-major walk (dK / dV) and the query-major
  // walk (dQ).  Ring schedule only (not filled when kv_natural).
  unsigned long long* tiles_kv_rt;
  unsigned long long* tiles_q_rt;
};

// Kernel launchers; each returns the launch error (cudaSuccess if queued).
// Ulysses all-to-all ("Sequence Parallelism IV", section 7).  A tensor
// [B, S, X, D] in sharded order (rank r owns sharded rows [r*L, (r+1)*L))
// <-> [cp][B, S, nx, D] in natural order, rank r holding heads
// x0(r) .. x0(r)+nx-1 with x0(r) = (r * x_num) / x_den.  Seq -> head copies;
// head -> seq sums the ranks that hold a head (kv heads shared by ranks).
// dtype: CPATTN_F32 / CPATTN_BF16 (the element type; sums in float32).
// Sequence <-> head all-to-all.  The sequence owners hold [B, S, X, D] in
// the sharded order of `sh` (cp ranks); the `ranks` head owners each hold
// [B, S, nx, D] with the sequence axis in the sharded order of `inner`:
// natural order (cp = 1) for the Ulysses variant, the second level's shard
// order for the hierarchical (a2a+p2p) schedule.  Of each shape only cp,
// per_rank, S, L and c are used.
struct A2aShape {
  RingShape sh;
  RingShape inner;
  int ranks;
  int B, X, nx, x_num, x_den, D;
};
cudaError_t launch_a2a(const void* in, void* out, const A2aShape& a, bool to_seq, int dtype,
                       cudaStream_t stream);
// LSE [B, H, S] in `sh` order <-> [ranks][B, H/ranks, S] in `inner` order
// (query heads only).
cudaError_t launch_lse_a2a(const float* in, float* out, const RingShape& sh,
                           const RingShape& inner, int ranks, int B, int H, bool to_seq,
                           cudaStream_t stream);

// docs[p] for every natural position p from document offsets cu[0..ndocs]
// (cu[0] = 0, strictly increasing, cu[ndocs] = S).  Offsets that break those
// rules set the device error word to kErrBadDocs; every entry is still
// clamped to first <= p < one-past-last, so the kernels stay in bounds.
cudaError_t launch_doc_bounds(const int* cu, int ndocs, int S, int2* docs, int* err,
                              cudaStream_t stream);
constexpr int kErrTimeout = 1;
constexpr int kErrBadDocs = 2;
constexpr int kErrLaunch = 3;  // a kernel found its launch unusable (shared-memory alignment)

// Flags callers OR into the dtype argument (include/cpattn.h).
constexpr int kDtypeFlags = CPATTN_GRAD_F32 | CPATTN_BWD_ONEPASS;

// Natural <-> sharded along S; the natural tensor holds S_nat <= S tokens
// (the rest is padding: zeros when sharding, dropped when unsharding).
cudaError_t launch_permute(const void* in, void* out, int64_t outer, int64_t S, int64_t S_nat,
                           int64_t inner_bytes, const RingShape& sh, bool inverse,
                           cudaStream_t stream);
cudaError_t launch_simt_fwd(const FwdArgs& a, int dtype, cudaStream_t stream);
cudaError_t launch_tc_fwd(const FwdArgs& a, cudaStream_t stream);
cudaError_t launch_lse_merge(const float* o_a, const float* l_a, const float* o_b,
                             const float* l_b, float* o, float* l, int B, int S, int H, int D,
                             cudaStream_t stream);
// delta[b,h,s] = delta_scale * (dout . out) of the row (the tensor-core
// backward takes it pre-multiplied by the softmax scale).
cudaError_t launch_bwd_prep(const void* out, const void* dout, float* delta, float* dq_acc,
                            float* dk_acc, float* dv_acc, int64_t n_kv, int B, int S, int H,
                            int D, int dtype, float delta_scale, cudaStream_t stream);
cudaError_t launch_simt_bwd(const BwdArgs& a, int dtype, cudaStream_t stream);
cudaError_t launch_tc_bwd(const BwdArgs& a, cudaStream_t stream);
// One-pass tensor-core backward: dK / dV partials as launch_tc_bwd, dQ added
// into a.dq_acc (float32 [B,S,H,D], zeroed by the caller).
cudaError_t launch_tc_bwd_onepass(const BwdArgs& a, cudaStream_t stream);
// dk[b,s,g,:] = sum of dk_part[b,s,h,:] over the query heads h of kv head g
// (and the same for dv), written in the output dtype.
cudaError_t launch_grad_reduce(const float* dk_part, const float* dv_part, void* dk, void* dv,
                               int B, int S, int H, int Hkv, int D, int out_dtype,
                               cudaStream_t stream);
// Converts the three float32 gradient accumulators to the output dtype
// (CPATTN_F32 or CPATTN_BF16) in one launch; n_q / n_kv elements each.
cudaError_t launch_grad_convert(const float* dq_acc, const float* dk_acc, const float* dv_acc,
                                void* dq, void* dk, void* dv, int64_t n_q, int64_t n_kv,
                                int out_dtype, cudaStream_t stream);

// One CTA whose bounded mbarrier wait gives up after limit_ns (raising *err).
cudaError_t launch_wait_probe(int* err, uint64_t limit_ns, cudaStream_t stream);

// Whether this build carries the tensor-core kernels.
bool tc_fwd_available();
bool tc_bwd_available();

// Tile edges of the kernels (tokens).
constexpr int kSimtTile = 64;
constexpr int kTcTile = 128;

}  // namespace cpattn
