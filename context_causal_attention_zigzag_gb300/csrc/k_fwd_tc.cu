// Tensor-core ring forward for sm_103a: tcgen05.mma with TMEM accumulators,
// TMA-staged bf16 tiles, warp-specialised, persistent.
//
// The ring ("Sequence Parallelism IV", sections 4-5) on one GPU: every
// virtual rank's Q/K/V shard sits in HBM; "receiving" the K/V of rank
// (r - t) mod cp at ring step t is a change of the base row the TMA reads.
// A work item is 256 query rows of one (batch, head) -- two 128-row tiles of
// one chunk.  Its CTA streams the K/V tiles of ring steps t = 0..cp-1, skips
// the tiles that no query of the item sees (wholly in the causal future, or,
// for packed documents, outside the documents of the item's rows: never
// loaded), and keeps the online softmax state; the two tiles on the causal
// diagonal (the item's own rows) are taken last.  Each softmax thread masks
// its row element-wise against the row's key window only on tiles that
// window cuts (the diagonal, document borders).  The rescale of O when the running
// maximum moves is the softmax-state correction; it is skipped while the
// maximum grows by less than 2^8, which leaves the result exact because the
// final normalisation uses the same stale maximum.
//
// CTA = 384 threads:
//   warp 0      TMA producer (the warp runs the loop, one elected lane
//               issues): Q pair once per item, K and V tiles into a
//               ring of five 32 KB slots (K(j), V(j), K(j+1), ... take
//               consecutive slots; a slot is freed as soon as the MMAs that
//               read it retire, so loads run up to two tiles ahead).
//   warp 1      TMEM owner and MMA issuer (the warp runs the control flow,
//               one elected lane issues):
//               S_i = Q_i K^T  (SS form, 128x128x128, fp32 in TMEM),
//               O_i += P_i V   (TS form: P read from TMEM, V MN-major).
//   warps 4-7   softmax of query tile 0, warps 8-11 of tile 1: one thread
//               per row (TMEM lane), row max / sum in fp32, P -> bf16
//               written back over S in TMEM, conditional O rescale,
//               epilogue O / l -> HBM and LSE.
// TMEM (512 columns): S0 [0,128) S1 [128,256) O0 [256,384) O1 [384,512);
// P_i occupies the first 64 columns of S_i (bf16 pairs).
// The MMA order per K/V tile j is PV0(j), S0(j+1), PV1(j), S1(j+1): while
// one softmax warpgroup works on its tile, the tensor core runs the other's.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "cpattn_internal.h"
#include "tc_ptx.cuh"

namespace cpattn {
namespace {

using namespace tc;

constexpr int kT = 128;                     // tile edge (rows, keys)
constexpr int kD = 128;                     // head dim
constexpr int kBoxBytes = kT * 64 * 2;      // [128 rows][64 bf16] = 16 KB
constexpr int kTileBytes = 2 * kBoxBytes;   // [128 rows][128 bf16] = 32 KB
constexpr int kSlots = 5;  // K/V ring: K(j), V(j) take consecutive slots
constexpr int kThreads = 384;

constexpr int kOffQ = 0;
constexpr int kOffRing = kOffQ + 2 * kTileBytes;
constexpr int kOffBar = kOffRing + kSlots * kTileBytes;
// barriers
constexpr int kBarQFull = 0;
constexpr int kBarQEmpty = 1;
constexpr int kBarFull = 2;                 // [kSlots]
constexpr int kBarEmpty = kBarFull + kSlots;  // [kSlots]
constexpr int kBarS = kBarEmpty + kSlots;     // [2]
constexpr int kBarP = kBarS + 2;             // [2]
constexpr int kBarO = kBarP + 2;             // [2]
constexpr int kBarDrain = kBarO + 2;
constexpr int kNumBars = kBarDrain + 1;
constexpr int kOffMisc = kOffBar + kNumBars * 8;
constexpr int kSmemBytes = kOffMisc + 16 + 1024;  // + slack for 1024-B alignment

__host__ __device__ constexpr uint32_t col_s(int i) { return 128u * (uint32_t)i; }
__host__ __device__ constexpr uint32_t col_o(int i) { return 256u + 128u * (uint32_t)i; }

constexpr uint32_t kIdescQK = idesc_bf16(128, 128, false, false);
constexpr uint32_t kIdescPV = idesc_bf16(128, 128, false, true);

constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleThreshold = 8.0f;  // log2 units

// Flags of one K/V tile for the item's two query tiles.
constexpr int kUse0 = 1, kUse1 = 2;

// Whether the 128 keys from natural position k0 meet the range [lo, hi].
__device__ __forceinline__ bool tile_meets(int k0, int lo, int hi) {
  return k0 <= hi && k0 + kT - 1 >= lo;
}

struct Item {
  int b, h, g, r, qc, a, qrow;  // qc: natural chunk, a: natural tile of query tile 0
};

// Work items: groups are the (batch, kv head) pairs, ranks the query pairs
// in order of decreasing cost (natural query position), each rank the query
// heads of the kv head, in cost bands (banded_item).  The CTAs running at the
// same time therefore share one kv head's K/V (2 * S * D * 2 bytes) through
// L2, and every round of the snake deal holds items of similar cost.
__device__ __forceinline__ Item decode_item(const RingShape& sh, int idx) {
  const int grp = sh.H / sh.Hkv;
  const int npair = sh.S / (2 * kT);
  int gi, rank, sub;
  banded_item(idx, sh.B * sh.Hkv, npair, grp, gridDim.x, 0, gi, rank, sub);
  const int pr = npair - 1 - rank;
  Item it;
  it.b = gi / sh.Hkv;
  it.g = gi - it.b * sh.Hkv;
  it.h = it.g * grp + sub;
  const int nat0 = pr * 2 * kT;
  it.qc = nat0 / sh.c;
  const int off = nat0 - it.qc * sh.c;
  int jq;
  if (sh.per_rank == 1 || it.qc < sh.cp) {
    it.r = it.qc;
    jq = 0;
  } else {
    it.r = 2 * sh.cp - 1 - it.qc;
    jq = 1;
  }
  it.qrow = it.r * sh.L + jq * sh.c + off;
  it.a = nat0 / kT;
  return it;
}

// The K/V tiles an item visits.  Query tile i sees the keys [lo[i], hi[i]]
// (natural positions); a tile is visited when either window meets it.  The
// walk takes the tiles in natural order, earliest first, whichever rank
// holds them: the CTAs in flight hold the query tiles of one kv head and so
// start on the same K/V tile and read the same K / V tiles at about the same
// time (one fetch from HBM serves them all through L2); under the causal
// rule the two diagonal tiles, the item's own rows, come last.  `step` is
// the ring step at which the tile's rank delivers it, (r - s) mod cp; a call
// for a range of ring steps [t_begin, t_end) visits only those steps' tiles.
//
// All-gather schedule (sh.kv_natural): K/V rows are natural positions, the
// same order, every step; `step` still reports the ring step at which the
// chunk's owner would have delivered it, so the census is the same.
struct KvSeq {
  int cp, per, L, c, t_begin, t_end, r, a;
  int lo[2], hi[2];
  int m, m_hi;
  bool natural;
  unsigned long long magic;  // RingShape::tile_magic, for chunk_of_tile

  __device__ __forceinline__ void init(const RingShape& sh, int t_begin_, int t_end_,
                                       const Item& it) {
    cp = sh.cp;
    per = sh.per_rank;
    L = sh.L;
    c = sh.c;
    t_begin = t_begin_;
    t_end = t_end_;
    r = it.r;
    a = it.a;
    int x;
    for (int i = 0; i < 2; ++i) {
      query_window(sh, (a + i) * kT, lo[i], x);
      query_window(sh, (a + i) * kT + kT - 1, x, hi[i]);
    }
    natural = sh.kv_natural != 0;
    m = lo[0] / kT;
    m_hi = hi[1] >= lo[0] ? hi[1] / kT : -1;
    magic = sh.tile_magic;
  }

  __device__ __forceinline__ int flags(int k0) const {
    return (tile_meets(k0, lo[0], hi[0]) ? kUse0 : 0) | (tile_meets(k0, lo[1], hi[1]) ? kUse1 : 0);
  }

  // kvrow: sharded row of the tile (natural row in the all-gather schedule);
  // fl: kUse* flags; step: ring step; knat: natural position of the tile's
  // first key.
  __device__ __forceinline__ bool next(int& kvrow, int& fl, int& step, int& knat) {
    while (m <= m_hi) {
      const int k0 = m * kT;
      const int chunk = chunk_of_tile(m, magic);
      ++m;
      fl = flags(k0);
      if (fl == 0) continue;
      const int s = (per == 1 || chunk < cp) ? chunk : 2 * cp - 1 - chunk;
      step = ring_step_of(r, s, cp);
      if (!natural && (step < t_begin || step >= t_end)) continue;
      const int slot = (per == 1 || chunk < cp) ? 0 : 1;
      kvrow = natural ? k0 : s * L + slot * c + (k0 - chunk * c);
      knat = k0;
      return true;
    }
    return false;
  }
};

__device__ __forceinline__ int item_index(int k, int cta, int grid) {
  // Snake order over the cost-sorted list balances the persistent CTAs.
  return k * grid + ((k & 1) ? (grid - 1 - cta) : cta);
}

__global__ void __launch_bounds__(kThreads, 1)
    tc_fwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                  const __grid_constant__ CUtensorMap tm_v, const FwdArgs args, int n_items) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (base - raw);
  const uint32_t sQ = base + kOffQ, sRing = base + kOffRing;
  auto slot = [&](uint32_t n) { return sRing + (n % kSlots) * kTileBytes; };
  const uint32_t bars = base + kOffBar;
  auto bar = [&](int i) { return bars + 8u * (uint32_t)i; };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kOffMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kOffMisc + 4);

  const RingShape& sh = args.sh;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const WaitCtl wc{abort_flag, args.err};

  if (threadIdx.x == 0) {
    mbar_init(bar(kBarQFull), 1);
    mbar_init(bar(kBarQEmpty), 1);
    for (int s = 0; s < kSlots; ++s) {
      mbar_init(bar(kBarFull + s), 1);
      mbar_init(bar(kBarEmpty + s), 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(bar(kBarS + i), 1);
      mbar_init(bar(kBarP + i), 128);
      mbar_init(bar(kBarO + i), 1);
    }
    mbar_init(bar(kBarDrain), 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    // ------------------------------------------------------------------ TMA
    // The whole warp runs the loop; one elected lane issues the copies.
    {
      const bool leader = elect_one();
      auto wwait = [&](uint32_t bar_addr, uint32_t parity) {
        return __all_sync(0xffffffffu, mbar_wait(bar_addr, parity, wc));
      };
      if (leader) {
        tma_prefetch_desc(&tm_q);
        tma_prefetch_desc(&tm_k);
        tma_prefetch_desc(&tm_v);
      }
      uint32_t seq = 0, q_armed = 0, armed[kSlots] = {0};
      bool ok = true;
      for (int k = 0; ok; ++k) {
        const int idx = item_index(k, blockIdx.x, gridDim.x);
        if (idx >= n_items) break;
        const Item it = decode_item(sh, idx);
        if (!wwait(bar(kBarQEmpty), (k & 1) ^ 1)) {
          ok = false;
          break;
        }
        ++q_armed;
        const int row0 = it.b * sh.S + it.qrow;
        if (leader) {
          mbar_arrive_expect_tx(bar(kBarQFull), 2 * kTileBytes);
          for (int tq = 0; tq < 2; ++tq)
            for (int half = 0; half < 2; ++half)
              tma_load_3d(sQ + tq * kTileBytes + half * kBoxBytes, &tm_q, bar(kBarQFull),
                          half * 64, it.h, row0 + tq * kT);
        }
        KvSeq kseq;
        kseq.init(sh, args.t_begin, args.t_end, it);
        int kvrow, fl, step, knat;
        while (ok && kseq.next(kvrow, fl, step, knat)) {
          const int krow = it.b * sh.S + kvrow;
          for (int which = 0; which < 2; ++which) {  // K(j), then V(j)
            const uint32_t n = seq++;
            const int sl = n % kSlots;
            if (!wwait(bar(kBarEmpty + sl), ((n / kSlots) & 1) ^ 1)) {
              ok = false;
              break;
            }
            ++armed[sl];
            if (leader) {
              mbar_arrive_expect_tx(bar(kBarFull + sl), kTileBytes);
              for (int half = 0; half < 2; ++half)
                tma_load_3d(slot(n) + half * kBoxBytes, which == 0 ? &tm_k : &tm_v,
                            bar(kBarFull + sl), half * 64, it.g, krow);
            }
          }
        }
      }
      if (!ok) {
        // Let the copies already issued land before the CTA exits.
        if (q_armed) mbar_drain(bar(kBarQFull), (q_armed - 1) & 1);
        for (int s = 0; s < kSlots; ++s)
          if (armed[s]) mbar_drain(bar(kBarFull + s), (armed[s] - 1) & 1);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------------ MMA
    // The whole warp runs the control flow (its values stay warp-uniform);
    // one elected lane issues the MMAs and commits.
    {
      const bool leader = elect_one();
      // A wait that the whole warp agrees on, so its control flow stays uniform.
      auto wwait = [&](uint32_t bar_addr, uint32_t parity) {
        return __all_sync(0xffffffffu, mbar_wait(bar_addr, parity, wc));
      };
      uint32_t kv_it = 0, p_ph[2] = {0, 0};
      bool ok = true;
      // Operand descriptors, computed once and advanced by byte offsets: Q
      // tile 0, ring slot 0 read K-major (K for S) and MN-major (V for P V).
      const uint64_t d_q = sdesc_sw128(sQ, 16, 1024);
      const uint64_t d_k = sdesc_sw128(sRing, 16, 1024);
      const uint64_t d_v = sdesc_sw128(sRing, kBoxBytes, 1024);
      auto slot_off = [](uint32_t n) { return (n % kSlots) * (uint32_t)kTileBytes; };
      for (int k = 0; ok; ++k) {
        const int idx = item_index(k, blockIdx.x, gridDim.x);
        if (idx >= n_items) break;
        const Item it = decode_item(sh, idx);
        if (!wwait(bar(kBarQFull), k & 1)) {
          ok = false;
          break;
        }
        tc_fence_after();
        KvSeq seq;
        seq.init(sh, args.t_begin, args.t_end, it);
        int kvrow, fl, step, knat;
        bool have = seq.next(kvrow, fl, step, knat);
        if (!have) {
          if (leader) mma_commit(bar(kBarQEmpty));
          continue;
        }
        unsigned long long census = 0;
        int census_step = step;
        // S for the first tile: K(j) is ring entry 2*kv_it, V(j) entry 2*kv_it + 1.
        uint32_t kn = 2 * kv_it;
        if (!wwait(bar(kBarFull + kn % kSlots), (kn / kSlots) & 1)) {
          ok = false;
          break;
        }
        tc_fence_after();
        for (int i = 0; i < 2; ++i) {
          if (!(fl & (kUse0 << i))) continue;
          const uint64_t a0 = sdesc_advance(d_q, i * kTileBytes);
          const uint64_t b0 = sdesc_advance(d_k, slot_off(kn));
          if (leader) {
#pragma unroll
            for (int kk = 0; kk < kD / 16; ++kk) {
              const uint32_t off = (kk >> 2) * kBoxBytes + (kk & 3) * 32;
              mma_ss(tmem + col_s(i), sdesc_advance(a0, off), sdesc_advance(b0, off), kIdescQK,
                     kk > 0);
            }
            mma_commit(bar(kBarS + i));
          }
        }
        if (leader) mma_commit(bar(kBarEmpty + kn % kSlots));
        // acc[i]: query tile i has had a P V product in this item.
        uint32_t acc[2] = {0, 0};
        while (true) {
          int nkvrow, nfl = 0, nstep = 0, nknat;
          const bool have_next = seq.next(nkvrow, nfl, nstep, nknat);
          const uint32_t vn = 2 * kv_it + 1, nkn = 2 * kv_it + 2;
          if (!wwait(bar(kBarFull + vn % kSlots), (vn / kSlots) & 1)) {
            ok = false;
            break;
          }
          tc_fence_after();
          bool k_ready = false;
          for (int i = 0; i < 2; ++i) {
            if (fl & (kUse0 << i)) {
              if (!wwait(bar(kBarP + i), p_ph[i])) {
                ok = false;
                break;
              }
              p_ph[i] ^= 1;
              tc_fence_after();
              const uint64_t bv = sdesc_advance(d_v, slot_off(vn));
              if (leader) {
#pragma unroll
                for (int kk = 0; kk < kT / 16; ++kk)
                  mma_ts(tmem + col_o(i), tmem + col_s(i) + kk * 8, sdesc_advance(bv, kk * 2048),
                         kIdescPV, acc[i] | (kk > 0));
              }
              acc[i] = 1;
            }
            if (have_next && (nfl & (kUse0 << i))) {
              if (!k_ready) {
                if (!wwait(bar(kBarFull + nkn % kSlots), (nkn / kSlots) & 1)) {
                  ok = false;
                  break;
                }
                tc_fence_after();
                k_ready = true;
              }
              const uint64_t a0 = sdesc_advance(d_q, i * kTileBytes);
              const uint64_t b0 = sdesc_advance(d_k, slot_off(nkn));
              if (leader) {
#pragma unroll
                for (int kk = 0; kk < kD / 16; ++kk) {
                  const uint32_t off = (kk >> 2) * kBoxBytes + (kk & 3) * 32;
                  mma_ss(tmem + col_s(i), sdesc_advance(a0, off), sdesc_advance(b0, off),
                         kIdescQK, kk > 0);
                }
                mma_commit(bar(kBarS + i));
              }
            }
          }
          if (!ok) break;
          if (leader) {
            mma_commit(bar(kBarEmpty + vn % kSlots));
            if (have_next) mma_commit(bar(kBarEmpty + nkn % kSlots));
          }
          if (args.tiles_rt != nullptr) {
            if (step != census_step) {
              if (leader) atomicAdd(&args.tiles_rt[it.r * sh.cp + census_step], census);
              census = 0;
              census_step = step;
            }
            census += (unsigned long long)(((fl & kUse0) ? 1 : 0) + ((fl & kUse1) ? 1 : 0));
          }
          ++kv_it;
          if (!have_next) break;
          kvrow = nkvrow;
          fl = nfl;
          step = nstep;
        }
        if (!ok) break;
        if (leader) {
          if (args.tiles_rt != nullptr && census)
            atomicAdd(&args.tiles_rt[it.r * sh.cp + census_step], census);
          // O(i) is released only to a softmax warpgroup that waits for it:
          // the one whose query tile saw at least one K/V tile of the item.
          if (acc[0]) mma_commit(bar(kBarO + 0));
          if (acc[1]) mma_commit(bar(kBarO + 1));
          mma_commit(bar(kBarQEmpty));
        }
      }
      if (!ok) {
        // Let every MMA already issued retire before TMEM is released.
        if (leader) mma_commit(bar(kBarDrain));
        mbar_drain(bar(kBarDrain), 0);
      }
    }
  } else if (warp >= 4) {
    // -------------------------------------------------------------- softmax
    const int ti = (warp - 4) >> 2;  // query tile of this warpgroup
    const int wq = warp & 3;         // TMEM sub-partition = rows 32*wq ..
    const int row = wq * 32 + lane;  // row within the tile
    const uint32_t tl = tmem + ((uint32_t)(wq * 32) << 16);
    const uint32_t colS = col_s(ti), colO = col_o(ti);
    const float sl2 = sh.scale_log2;
    uint32_t s_ph = 0, o_ph = 0;
    bool ok = true;
    for (int k = 0; ok; ++k) {
      const int idx = item_index(k, blockIdx.x, gridDim.x);
      if (idx >= n_items) break;
      const Item it = decode_item(sh, idx);
      KvSeq seq;
      seq.init(sh, args.t_begin, args.t_end, it);
      // This row's key window (natural positions).
      int w_lo, w_hi;
      query_window(sh, (it.a + ti) * kT + row, w_lo, w_hi);
      float m = -INFINITY, l = 0.f;
      int nt = 0;
      int kvrow, fl, step, knat;
      while (seq.next(kvrow, fl, step, knat)) {
        if (!(fl & (kUse0 << ti))) continue;
        const int j_lo = w_lo - knat, j_hi = w_hi - knat;  // visible columns
        const bool cut = j_lo > 0 || j_hi < kT - 1;
        if (!__all_sync(0xffffffffu, mbar_wait(bar(kBarS + ti), s_ph, wc))) {
          ok = false;
          break;
        }
        s_ph ^= 1;
        tc_fence_after();
        uint32_t r[128];
        tmem_ld32(tl + colS + 0, r + 0);
        tmem_ld32(tl + colS + 32, r + 32);
        tmem_ld32(tl + colS + 64, r + 64);
        tmem_ld32(tl + colS + 96, r + 96);
        tmem_wait_ld_regs(r);
        reg_fence32(r + 32);
        reg_fence32(r + 64);
        reg_fence32(r + 96);
        if (cut) {
#pragma unroll
          for (int j = 0; j < 128; ++j)
#if CPATTN_MUTATION == 1
            if (j < j_lo || j >= j_hi) r[j] = __float_as_uint(-INFINITY);  // planted: seam
#else
            if (j < j_lo || j > j_hi) r[j] = __float_as_uint(-INFINITY);
#endif
        }
        float mx0 = __uint_as_float(r[0]), mx1 = __uint_as_float(r[1]);
        float mx2 = __uint_as_float(r[2]), mx3 = __uint_as_float(r[3]);
#pragma unroll
        for (int j = 4; j < 128; j += 4) {
          mx0 = fmaxf(mx0, __uint_as_float(r[j]));
          mx1 = fmaxf(mx1, __uint_as_float(r[j + 1]));
          mx2 = fmaxf(mx2, __uint_as_float(r[j + 2]));
          mx3 = fmaxf(mx3, __uint_as_float(r[j + 3]));
        }
        const float m_tile = fmaxf(fmaxf(mx0, mx1), fmaxf(mx2, mx3)) * sl2;
        const float m_new = fmaxf(m, m_tile);
        const bool need = m_new > m + kRescaleThreshold;
        const bool rescale = __any_sync(0xffffffffu, need);
        float alpha = 1.f;
        if (rescale) {
          // A row that has seen no key yet keeps m = -inf and alpha = 1.
          alpha = m_new == -INFINITY ? 1.f : ex2(m - m_new);
          l *= alpha;
          m = m_new;
        }
        const float nm = m == -INFINITY ? 0.f : -m;
        float l0 = 0.f, l1 = 0.f;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          uint32_t p[32];
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            const float a0 = ex2(fmaf(__uint_as_float(r[64 * h + 2 * j]), sl2, nm));
            const float a1 = ex2(fmaf(__uint_as_float(r[64 * h + 2 * j + 1]), sl2, nm));
            l0 += a0;
            l1 += a1;
            p[j] = pack_bf16(a0, a1);
          }
          tmem_st32(tl + colS + 32 * h, p);
        }
        l += l0 + l1;
        if (rescale && nt > 0) {
          // Softmax-state correction: O <- O * 2^(m_old - m_new).  The S
          // barrier of this tile also covers the previous P V product, and the
          // next one is issued only after the P barrier below.
#pragma unroll
          for (int cc = 0; cc < 4; ++cc) {
            uint32_t o[32];
            tmem_ld32(tl + colO + cc * 32, o);
            tmem_wait_ld_regs(o);
#pragma unroll
            for (int j = 0; j < 32; ++j) o[j] = __float_as_uint(__uint_as_float(o[j]) * alpha);
            tmem_st32(tl + colO + cc * 32, o);
          }
        }
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(bar(kBarP + ti));
        ++nt;
      }
      if (!ok) break;
      // ------------------------------------------------------------ epilogue
      const int qrow = it.qrow + ti * kT + row;
      const int64_t obase = (((int64_t)it.b * sh.S + qrow) * sh.H + it.h) * kD;
      const int64_t lidx = ((int64_t)it.b * sh.H + it.h) * sh.S + qrow;
      if (nt == 0) {
        // No visible key (a step partial): (0, -inf), in the output's format.
        if (args.step_mode) {
          float4* op = reinterpret_cast<float4*>(static_cast<float*>(args.out) + obase);
          for (int j = 0; j < kD / 4; ++j) op[j] = make_float4(0.f, 0.f, 0.f, 0.f);
        } else {
          uint4* op = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(args.out) + obase);
          for (int j = 0; j < kD / 8; ++j) op[j] = make_uint4(0u, 0u, 0u, 0u);
        }
        args.lse[lidx] = -INFINITY;
        continue;
      }
      if (!__all_sync(0xffffffffu, mbar_wait(bar(kBarO + ti), o_ph, wc))) {
        ok = false;
        break;
      }
      o_ph ^= 1;
      tc_fence_after();
      // A row with no visible key (possible only in a step partial) gets
      // (0, -inf).
      const float inv = l > 0.f ? 1.f / l : 0.f;
#pragma unroll
      for (int cc = 0; cc < 4; ++cc) {
        uint32_t o[32];
        tmem_ld32(tl + colO + cc * 32, o);
        tmem_wait_ld_regs(o);
        if (args.step_mode) {
          float4* op = reinterpret_cast<float4*>(static_cast<float*>(args.out) + obase + cc * 32);
#pragma unroll
          for (int j = 0; j < 8; ++j)
            op[j] = make_float4(__uint_as_float(o[4 * j]) * inv, __uint_as_float(o[4 * j + 1]) * inv,
                                __uint_as_float(o[4 * j + 2]) * inv,
                                __uint_as_float(o[4 * j + 3]) * inv);
        } else {
          uint4* op = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(args.out) + obase +
                                               cc * 32);
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            uint4 v;
            v.x = pack_bf16(__uint_as_float(o[8 * j + 0]) * inv, __uint_as_float(o[8 * j + 1]) * inv);
            v.y = pack_bf16(__uint_as_float(o[8 * j + 2]) * inv, __uint_as_float(o[8 * j + 3]) * inv);
            v.z = pack_bf16(__uint_as_float(o[8 * j + 4]) * inv, __uint_as_float(o[8 * j + 5]) * inv);
            v.w = pack_bf16(__uint_as_float(o[8 * j + 6]) * inv, __uint_as_float(o[8 * j + 7]) * inv);
            op[j] = v;
          }
        }
      }
      args.lse[lidx] = l > 0.f ? (m + log2f(l)) * kLn2 : -INFINITY;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  if (fn == nullptr) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  }
  return fn;
}

// [rows, heads, 128] bf16 viewed as a 3-D tensor (d, head, row), box
// (64, 1, 128) with 128-byte swizzle.
bool make_map(CUtensorMap* m, const void* ptr, int heads, int64_t rows) {
  EncodeTiledFn enc = encode_fn();
  if (enc == nullptr) return false;
  cuuint64_t dims[3] = {(cuuint64_t)kD, (cuuint64_t)heads, (cuuint64_t)rows};
  cuuint64_t strides[2] = {(cuuint64_t)kD * 2, (cuuint64_t)heads * kD * 2};
  cuuint32_t box[3] = {64, 1, (cuuint32_t)kT};
  cuuint32_t estr[3] = {1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(ptr), dims, strides, box,
             estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

bool tc_fwd_available() { return true; }

cudaError_t launch_tc_fwd(const FwdArgs& a, cudaStream_t stream) {
  const RingShape& sh = a.sh;
  const int n_items = sh.B * sh.H * (sh.S / (2 * kT));
  if (n_items == 0) return cudaSuccess;
  CUtensorMap mq, mk, mv;
  const int64_t rows = (int64_t)sh.B * sh.S;
  if (!make_map(&mq, a.q, sh.H, rows) || !make_map(&mk, a.k, sh.Hkv, rows) ||
      !make_map(&mv, a.v, sh.Hkv, rows))
    return cudaErrorInvalidValue;
  int dev = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(tc_fwd_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
  if (e != cudaSuccess) return e;
  const int grid = n_items < sms ? n_items : sms;
  tc_fwd_kernel<<<grid, kThreads, kSmemBytes, stream>>>(mq, mk, mv, a, n_items);
  return cudaGetLastError();
}

}  // namespace cpattn
