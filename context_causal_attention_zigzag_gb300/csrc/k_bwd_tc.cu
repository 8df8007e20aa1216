// Tensor-core ring backward for sm_103a (tcgen05 + TMEM + TMA): two
// persistent, warp-specialised kernels that together produce dQ, dK, dV
// without any atomic reduction.
//
// Gradients through the ring ("Context Parallelism for Long-Context
// Training", section "Prove attention equivalence"), from the saved LSE and
// Delta = rowsum(dO o O):  P = exp(s - LSE),  dS = P (dP - Delta),
// dP = dO V^T.  The tiles a query tile and a K/V tile share are those of the
// ring ("Sequence Parallelism IV", section 4): the K/V of source rank s
// reaches rank (s + t) mod cp at step t; tiles that no pair of the two sees
// (wholly in the causal future, or in another packed document) are skipped,
// and a tile that a row's window cuts (the diagonal, a document border) is
// masked element-wise for that row.
//
// dkdv kernel (K/V-major).  Work item: one 128-row K/V tile and one query
// head.  The K/V tile stays in shared memory; the query tiles that see it
// stream past (latest natural position first, see QSeq), Q and dO by TMA,
// their LSE / Delta rows by bulk copy.  Per query tile, with the tile transposed so that TMEM lanes are K/V
// rows:
//   S^T  = K Q^T   -> TMEM [0,128)       dP^T = V dO^T -> TMEM [128,256)
//   P^T  = exp2(S^T*scale*log2e - LSE*log2e)  -> bf16 over S^T
//   dS^T = scale * P^T (dP^T - Delta)         -> bf16 over dP^T
//   (dS from the float32 P, so that only dS itself is rounded to bf16; Delta
//   arrives multiplied by the scale, so dS = P (scale dP - scale Delta) is an
//   FMA and a multiply per element)
//   dV  += P^T dO  (TS)  -> TMEM [256,384)    dK += dS^T Q (TS) -> TMEM [384,512)
// MMA order per tile i: dV(i), S(i+1), dK(i), dP(i+1): the elementwise warps
// of tile i+1 overlap the tensor core's work on tile i.  At the end of the
// item the head's dK / dV partial (float32) is stored to its own slot; a
// small kernel sums the slots of the query heads sharing a kv head.  One
// item per query head keeps each TMEM accumulation chain short (the tensor
// core's float32 accumulation drifts toward zero over very long chains).
//
// dq kernel (query-major).  Work item: one 128-row query tile of one head.
// Q, dO arrive in shared memory and the elementwise warps copy them into TMEM
// as bf16 pairs at the start of the item (releasing the shared-memory copy to
// the next item's loads), so that S and dP are TS-form products, which issue
// faster than the SS form; LSE / Delta sit in registers (TMEM lane = query
// row).  The K/V tiles the item sees (earliest first, see KSeq) stream past
// through two rings of 32 KB slots, three for K and two for V (V(j)'s slot is
// free once dP(j) has read it, K(j)'s only once dQ(j) has, a tile later):
//   S = Q K^T -> TMEM [0,128)      dP = dO V^T -> TMEM [128,256)
//   dS = scale * exp2(S*scale*log2e - LSE*log2e) (dP - Delta) -> bf16 over dP
//   dQ += dS K  (TS, K read MN-major) -> TMEM [256,384)
//   Q -> TMEM [384,448), dO -> [448,512)
// MMA order per K/V tile j: S(j+1), dQ(j), dP(j+1); S is released as soon as
// the elementwise warps have read it; dP(j+1) follows dQ(j), which reads the
// dS packed over dP(j), and MMAs execute in issue order.
//
// Both kernels: CTA = 384 threads; warp 0 TMA, warp 1 TMEM owner + MMA
// issuer (the whole warp runs the issue loop, so its values stay
// warp-uniform, and one elected lane issues), warps 4-7 and 8-11 the
// elementwise work on columns [0,64) and
// [64,128) of each tile (one thread per TMEM lane), and the epilogue.  Each
// half writes its packed bf16 result over the first 32 of the 64 columns it
// read itself ([0,32) and [64,96)), so the halves never wait for each other;
// the MMA that consumes the packed tile takes its K = 16 slices from those
// two column ranges (a_col).  Every
// wait is a bounded mbarrier wait; on expiry the kernel raises the device
// error word, drains its own copies and MMAs, frees TMEM and returns.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "cpattn_internal.h"
#include "tc_ptx.cuh"

namespace cpattn {
namespace {

using namespace tc;

constexpr int kT = 128;
constexpr int kD = 128;
constexpr int kBoxBytes = kT * 64 * 2;     // 16 KB
constexpr int kTileBytes = 2 * kBoxBytes;  // 32 KB
constexpr int kThreads = 384;
constexpr int kPrefetchAhead = 4;  // tiles asked of L2 ahead of their loads
constexpr float kLog2e = 1.4426950408889634f;

constexpr uint32_t kIdescKK = idesc_bf16(128, 128, false, false);  // both K-major
constexpr uint32_t kIdescKM = idesc_bf16(128, 128, false, true);   // B MN-major

__device__ __forceinline__ int item_index(int k, int cta, int grid) {
  return k * grid + ((k & 1) ? (grid - 1 - cta) : cta);
}

// Bulk (non-tensor) copy global -> shared, completion as transaction bytes.
__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes,
                                          uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          dst),
      "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(bar)
      : "memory");
}

// TMEM column of the kk-th K = 16 slice of a packed bf16 128 x 128 tile
// written by the two elementwise halves: half h packs its 64 columns into
// [64h, 64h + 32).
__device__ __forceinline__ uint32_t a_col(int kk) {
  return (uint32_t)((kk >> 2) * 64 + (kk & 3) * 8);
}

// Location of a 128-row tile given its natural tile index.
struct TilePos {
  int chunk;  // natural chunk
  int rank;   // owning rank
  int tile;   // tile index inside the chunk
  int row;    // sharded row of the tile's first token
};

__device__ __forceinline__ TilePos tile_pos(const RingShape& sh, int knat) {
  TilePos p;
  const int nat0 = knat * kT;
  p.chunk = nat0 / sh.c;
  const int loc = nat0 - p.chunk * sh.c;
  int jj;
  if (sh.per_rank == 1 || p.chunk < sh.cp) {
    p.rank = p.chunk;
    jj = 0;
  } else {
    p.rank = 2 * sh.cp - 1 - p.chunk;
    jj = 1;
  }
  p.tile = loc / kT;
  p.row = p.rank * sh.L + jj * sh.c + loc;
  return p;
}

// Query tiles (of one head) that see a K/V tile.  The tile's keys are seen by
// the queries [lo, hi] (natural positions): under the causal rule from the
// tile's first key on, within the documents of its keys.  The walk takes
// those query tiles from the latest natural position down to the earliest,
// whichever rank holds them, so that the CTAs in flight -- K/V tiles of one
// head -- start on the same query tile and read the same Q / dO tiles at
// about the same time (one fetch from HBM serves them all through L2).  The
// ring step of each tile is reported for the census: rank r receives the
// K/V of source rank s at step (r - s) mod cp.  Query rows stay sharded in
// the all-gather schedule too (sh.kv_natural), where the order is the same.
struct QSeq {
  int cp, L, c, s, per;
  int m, m_lo;  // natural query tile, current and lowest
  int t;        // ring step of the tile last returned
  unsigned long long magic;  // RingShape::tile_magic, for chunk_of_tile

  __device__ __forceinline__ void init(const RingShape& sh, const TilePos& kv, int knat) {
    cp = sh.cp;
    per = sh.per_rank;
    L = sh.L;
    c = sh.c;
    s = kv.rank;
    int lo, hi, x;
    key_window(sh, knat * kT, lo, x);
    key_window(sh, knat * kT + kT - 1, x, hi);
    m = hi >= lo ? hi / kT : -1;
    m_lo = lo / kT;
    t = 0;
    magic = sh.tile_magic;
  }

  // qrow: sharded row of the query tile; qnat: natural position of its first row.
  __device__ __forceinline__ bool next(int& qrow, int& qnat) {
    if (m < m_lo) return false;
    qnat = m * kT;
    const int chunk = chunk_of_tile(m, magic);
    const int r = (per == 1 || chunk < cp) ? chunk : 2 * cp - 1 - chunk;
    const int slot = (per == 1 || chunk < cp) ? 0 : 1;
    qrow = r * L + slot * c + (qnat - chunk * c);
    t = ring_step_of(r, s, cp);
    --m;
    return true;
  }
};

// K/V tiles that a query tile sees.  The query tile sees the keys [lo(first
// row), hi(last row)] (natural positions; under the causal rule up to its
// own last row, so its own tile -- the diagonal, masked element-wise -- is
// the last one).  The walk takes them in natural order, earliest first,
// whichever rank holds them: the CTAs in flight hold consecutive query tiles
// of one kv head and so start on the same K/V tile and read the same K / V
// tiles at about the same time (one fetch from HBM serves them all through
// L2).  The ring step of each tile is reported for the census: rank r holds
// the K/V of source rank s at step (r - s) mod cp.  All-gather schedule
// (sh.kv_natural): the same order over the natural-order K/V rows.
struct KSeq {
  int cp, L, c, r, per;
  int m, m_hi;  // natural K/V tile, current and last
  int t;        // ring step of the tile last returned
  bool natural;
  unsigned long long magic;  // RingShape::tile_magic, for chunk_of_tile

  __device__ __forceinline__ void init(const RingShape& sh, const TilePos& q, int knat) {
    cp = sh.cp;
    per = sh.per_rank;
    L = sh.L;
    c = sh.c;
    r = q.rank;
    natural = sh.kv_natural != 0;
    const int q0 = knat * kT;
    int lo, hi, x;
    query_window(sh, q0, lo, x);
    query_window(sh, q0 + kT - 1, x, hi);
    m = lo / kT;
    m_hi = hi >= lo ? hi / kT : -1;
    t = 0;
    magic = sh.tile_magic;
  }

  // kvrow: sharded row of the K/V tile (natural row in the all-gather
  // schedule); knat: natural position of its first key.
  __device__ __forceinline__ bool next(int& kvrow, int& knat) {
    if (m > m_hi) return false;
    knat = m * kT;
    const int chunk = chunk_of_tile(m, magic);
    const int s = (per == 1 || chunk < cp) ? chunk : 2 * cp - 1 - chunk;
    const int slot = (per == 1 || chunk < cp) ? 0 : 1;
    kvrow = natural ? knat : s * L + slot * c + (knat - chunk * c);
    t = ring_step_of(r, s, cp);
    ++m;
    return true;
  }
};

// ===========================================================================
// dkdv kernel
// ===========================================================================
namespace kv {

constexpr int kOffK = 0;
constexpr int kOffV = kOffK + kTileBytes;
constexpr int kOffQ = kOffV + kTileBytes;         // [2] stages
constexpr int kOffDO = kOffQ + 2 * kTileBytes;    // [2]
constexpr int kOffLse = kOffDO + 2 * kTileBytes;  // [2][128] float (natural log)
constexpr int kOffDlt = kOffLse + 2 * kT * 4;     // [2][128] float
constexpr int kOffBar = kOffDlt + 2 * kT * 4;
constexpr int kBarKVFull = 0;
constexpr int kBarKVEmpty = 1;
constexpr int kBarQFull = 2;   // [2]
constexpr int kBarQEmpty = 4;  // [2]
constexpr int kBarS = 6;
constexpr int kBarDP = 7;
constexpr int kBarP = 8;
constexpr int kBarDS = 9;
constexpr int kBarAcc = 10;
constexpr int kBarAccFree = 11;
constexpr int kBarDrain = 12;
constexpr int kNumBars = 13;
constexpr int kOffMisc = kOffBar + kNumBars * 8;
constexpr int kSmemBytes = kOffMisc + 16 + 1024;
constexpr uint32_t kColS = 0, kColDP = 128, kColDV = 256, kColDK = 384;
constexpr uint32_t kQTx = 2 * kTileBytes + 2 * kT * 4;  // Q, dO, LSE, Delta

struct Item {
  int b, h, g, knat;
  TilePos kv;
};

// Groups are the (batch, query head) pairs, ranks the K/V tiles earliest
// first (an early tile is seen by the most query tiles), in cost bands
// (banded_item).  Consecutive items -- the CTAs running at the same time --
// share one head, so the Q / dO tiles they all stream stay in L2 (one head's
// Q and dO: 2 * S * D * 2 bytes).  Every item streams its head's Q and dO
// from its own tile to the end, so the bands keep at most about
// kMaxHeadsInFlight heads in flight.
constexpr int kMaxHeadsInFlight = 4;
__device__ __forceinline__ Item decode(const RingShape& sh, int idx) {
  const int ntiles = sh.S / kT;
  int bh, knat, sub;
  banded_item(idx, sh.B * sh.H, ntiles, 1, gridDim.x, kMaxHeadsInFlight, bh, knat, sub);
  Item it;
  it.b = bh / sh.H;
  it.h = bh - it.b * sh.H;
  it.g = it.h / (sh.H / sh.Hkv);
  it.knat = knat;
  it.kv = tile_pos(sh, knat);
  return it;
}

__global__ void __launch_bounds__(kThreads, 1)
    dkdv_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                const BwdArgs args, int n_items) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (base - raw);
  const uint32_t sK = base + kOffK, sV = base + kOffV, sQ = base + kOffQ, sDO = base + kOffDO;
  const uint32_t sLse = base + kOffLse, sDlt = base + kOffDlt;
  const float* lse_s = reinterpret_cast<const float*>(smem + kOffLse);
  const float* dlt_s = reinterpret_cast<const float*>(smem + kOffDlt);
  const uint32_t bars = base + kOffBar;
  auto bar = [&](int i) { return bars + 8u * (uint32_t)i; };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kOffMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kOffMisc + 4);

  const RingShape& sh = args.sh;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const WaitCtl wc{abort_flag, args.err};

  if (threadIdx.x == 0) {
    mbar_init(bar(kBarKVFull), 1);
    mbar_init(bar(kBarKVEmpty), 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(bar(kBarQFull + i), 1);
      mbar_init(bar(kBarQEmpty + i), 1);
    }
    mbar_init(bar(kBarS), 1);
    mbar_init(bar(kBarDP), 1);
    mbar_init(bar(kBarP), 256);
    mbar_init(bar(kBarDS), 256);
    mbar_init(bar(kBarAcc), 1);
    mbar_init(bar(kBarAccFree), 256);
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
    if (lane == 0) {
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_v);
      tma_prefetch_desc(&tm_do);
      uint32_t qi = 0, kv_armed = 0, q_armed[2] = {0, 0};
      bool ok = true;
      for (int k = 0; ok; ++k) {
        const int idx = item_index(k, blockIdx.x, gridDim.x);
        if (idx >= n_items) break;
        const Item it = decode(sh, idx);
        if (!mbar_wait(bar(kBarKVEmpty), (k & 1) ^ 1, wc)) {
          ok = false;
          break;
        }
        mbar_arrive_expect_tx(bar(kBarKVFull), 2 * kTileBytes);
        ++kv_armed;
        const int krow = it.b * sh.S + (sh.kv_natural ? it.knat * kT : it.kv.row);
        for (int half = 0; half < 2; ++half) {
          tma_load_3d(sK + half * kBoxBytes, &tm_k, bar(kBarKVFull), half * 64, it.g, krow);
          tma_load_3d(sV + half * kBoxBytes, &tm_v, bar(kBarKVFull), half * 64, it.g, krow);
        }
        QSeq seq;
        seq.init(sh, it.kv, it.knat);
        // A second walker kPrefetchAhead tiles ahead asks L2 for the Q / dO
        // tiles before their loads are issued.
        QSeq pseq = seq;
        auto prefetch_next = [&]() {
          int prow, pnat;
          if (!pseq.next(prow, pnat)) return;
          const int row = it.b * sh.S + prow;
          for (int half = 0; half < 2; ++half) {
            tma_prefetch_l2_3d(&tm_q, half * 64, it.h, row);
            tma_prefetch_l2_3d(&tm_do, half * 64, it.h, row);
          }
        };
        for (int i = 0; i < kPrefetchAhead; ++i) prefetch_next();
        int qrow, qnat;
        // Census: query tiles per (receiving rank, ring step), flushed at
        // each change of step.
        unsigned long long* census = sh.kv_natural ? nullptr : args.tiles_kv_rt;
        int c_step = -1;
        unsigned long long c_n = 0;
        while (seq.next(qrow, qnat)) {
          prefetch_next();
          if (census != nullptr) {
            if (seq.t != c_step) {
              if (c_n) atomicAdd(&census[((it.kv.rank + c_step) % sh.cp) * sh.cp + c_step], c_n);
              c_step = seq.t;
              c_n = 0;
            }
            ++c_n;
          }
          const int st = qi & 1;
          const uint32_t ph = (qi >> 1) & 1;
          if (!mbar_wait(bar(kBarQEmpty + st), ph ^ 1, wc)) {
            ok = false;
            break;
          }
          const uint32_t full = bar(kBarQFull + st);
          mbar_arrive_expect_tx(full, kQTx);
          ++q_armed[st];
          const int row = it.b * sh.S + qrow;
          for (int half = 0; half < 2; ++half) {
            tma_load_3d(sQ + st * kTileBytes + half * kBoxBytes, &tm_q, full, half * 64, it.h, row);
            tma_load_3d(sDO + st * kTileBytes + half * kBoxBytes, &tm_do, full, half * 64, it.h,
                        row);
          }
          const int64_t li = ((int64_t)it.b * sh.H + it.h) * sh.S + qrow;
          bulk_load(sLse + st * kT * 4, args.lse + li, kT * 4, full);
          bulk_load(sDlt + st * kT * 4, args.delta + li, kT * 4, full);
          ++qi;
        }
        if (census != nullptr && c_n)
          atomicAdd(&census[((it.kv.rank + c_step) % sh.cp) * sh.cp + c_step], c_n);
      }
      if (!ok) {
        if (kv_armed) mbar_drain(bar(kBarKVFull), (kv_armed - 1) & 1);
        for (int s = 0; s < 2; ++s)
          if (q_armed[s]) mbar_drain(bar(kBarQFull + s), (q_armed[s] - 1) & 1);
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
      uint32_t qi = 0, p_ph = 0, ds_ph = 0;
      bool ok = true;
      // Operand descriptors, computed once and advanced by byte offsets.
      const uint64_t d_k = sdesc_sw128(sK, 16, 1024), d_v = sdesc_sw128(sV, 16, 1024);
      const uint64_t d_q = sdesc_sw128(sQ, 16, 1024), d_do = sdesc_sw128(sDO, 16, 1024);
      const uint64_t d_q_mn = sdesc_sw128(sQ, kBoxBytes, 1024);
      const uint64_t d_do_mn = sdesc_sw128(sDO, kBoxBytes, 1024);
      auto issue_s = [&](int st) {
        if (!leader) return;
        const uint64_t b0 = sdesc_advance(d_q, st * kTileBytes);
#pragma unroll
        for (int kk = 0; kk < kD / 16; ++kk) {
          const uint32_t off = (kk >> 2) * kBoxBytes + (kk & 3) * 32;
          mma_ss(tmem + kColS, sdesc_advance(d_k, off), sdesc_advance(b0, off), kIdescKK, kk > 0);
        }
        mma_commit(bar(kBarS));
      };
      auto issue_dp = [&](int st) {
        if (!leader) return;
        const uint64_t b0 = sdesc_advance(d_do, st * kTileBytes);
#pragma unroll
        for (int kk = 0; kk < kD / 16; ++kk) {
          const uint32_t off = (kk >> 2) * kBoxBytes + (kk & 3) * 32;
          mma_ss(tmem + kColDP, sdesc_advance(d_v, off), sdesc_advance(b0, off), kIdescKK, kk > 0);
        }
        mma_commit(bar(kBarDP));
      };
      for (int k = 0; ok; ++k) {
        const int idx = item_index(k, blockIdx.x, gridDim.x);
        if (idx >= n_items) break;
        const Item it = decode(sh, idx);
        if (!wwait(bar(kBarKVFull), k & 1)) {
          ok = false;
          break;
        }
        tc_fence_after();
        QSeq seq;
        seq.init(sh, it.kv, it.knat);
        int qrow, qnat;
        bool have = seq.next(qrow, qnat);
        if (have) {
          const int st = qi & 1;
          if (!wwait(bar(kBarQFull + st), (qi >> 1) & 1)) {
            ok = false;
            break;
          }
          tc_fence_after();
          issue_s(st);
          issue_dp(st);
        }
        bool first = true;
        while (have) {
          const int st = qi & 1;
          int nqrow, nqnat;
          const bool nhave = seq.next(nqrow, nqnat);
          const int nst = (qi + 1) & 1;
          // dV += P^T dO
          if (!wwait(bar(kBarP), p_ph)) {
            ok = false;
            break;
          }
          p_ph ^= 1;
          if (first && !wwait(bar(kBarAccFree), (k & 1) ^ 1)) {
            ok = false;
            break;
          }
          tc_fence_after();
          if (leader) {
            const uint64_t b0 = sdesc_advance(d_do_mn, st * kTileBytes);
#pragma unroll
            for (int kk = 0; kk < kT / 16; ++kk)
              mma_ts(tmem + kColDV, tmem + kColS + a_col(kk), sdesc_advance(b0, kk * 2048),
                     kIdescKM, (!first || kk > 0) ? 1u : 0u);
          }
          // S for the next tile (the S^T columns are free once dV has read P^T;
          // MMAs execute in issue order).
          if (nhave) {
            if (!wwait(bar(kBarQFull + nst), ((qi + 1) >> 1) & 1)) {
              ok = false;
              break;
            }
            tc_fence_after();
            issue_s(nst);
          }
          // dK += dS^T Q
          if (!wwait(bar(kBarDS), ds_ph)) {
            ok = false;
            break;
          }
          ds_ph ^= 1;
          tc_fence_after();
          if (leader) {
            const uint64_t b0 = sdesc_advance(d_q_mn, st * kTileBytes);
#pragma unroll
            for (int kk = 0; kk < kT / 16; ++kk)
              mma_ts(tmem + kColDK, tmem + kColDP + a_col(kk), sdesc_advance(b0, kk * 2048),
                     kIdescKM, (!first || kk > 0) ? 1u : 0u);
          }
          if (leader) mma_commit(bar(kBarQEmpty + st));
          // dP for the next tile (the dP^T columns are free once dK has read dS^T).
          if (nhave) issue_dp(nst);
          first = false;
          ++qi;
          have = nhave;
        }
        if (!ok) break;
        if (first) {
          // No query tile at all (cannot happen for well-formed windows: every
          // key sees its own query): the epilogue writes zeros once the
          // previous one has been read out.
          if (!wwait(bar(kBarAccFree), (k & 1) ^ 1)) {
            ok = false;
            break;
          }
        }
        if (leader) {
          mma_commit(bar(kBarAcc));
          mma_commit(bar(kBarKVEmpty));
        }
      }
      if (!ok) {
        if (leader) mma_commit(bar(kBarDrain));
        mbar_drain(bar(kBarDrain), 0);
      }
    }
  } else if (warp >= 4) {
    // ----------------------------------------- elementwise + dK / dV epilogue
    const int half = (warp - 4) >> 2;  // columns [64*half, 64*half + 64)
    const int wq = warp & 3;
    const int row = wq * 32 + lane;    // K/V row of the tile (TMEM lane)
    const uint32_t tl = tmem + ((uint32_t)(wq * 32) << 16);
    const float sl2 = sh.scale_log2, scale = sh.scale;
    uint32_t qi = 0, s_ph = 0, dp_ph = 0;
    bool ok = true;
    for (int k = 0; ok; ++k) {
      const int idx = item_index(k, blockIdx.x, gridDim.x);
      if (idx >= n_items) break;
      const Item it = decode(sh, idx);
      QSeq seq;
      seq.init(sh, it.kv, it.knat);
      // Queries that see this thread's key (natural positions).
      int w_lo, w_hi;
      key_window(sh, it.knat * kT + row, w_lo, w_hi);
      int qrow, qnat, nq = 0;
      while (seq.next(qrow, qnat)) {
        const int st = qi & 1;
        const int c_lo = w_lo - qnat, c_hi = w_hi - qnat;  // visible query columns
        const bool cut = c_lo > 0 || c_hi < kT - 1;
        // LSE / Delta of this tile arrived with its Q / dO.
        if (!__all_sync(0xffffffffu, mbar_wait(bar(kBarQFull + st), (qi >> 1) & 1, wc))) {
          ok = false;
          break;
        }
        const float* lse = lse_s + st * kT + 64 * half;
        const float* dlt = dlt_s + st * kT + 64 * half;
        // P^T = exp2(S^T * scale*log2e - LSE*log2e), masked outside the window
        if (!__all_sync(0xffffffffu, mbar_wait(bar(kBarS), s_ph, wc))) {
          ok = false;
          break;
        }
        s_ph ^= 1;
        tc_fence_after();
        uint32_t r[64];
        tmem_ld32(tl + kColS + 64 * half, r);
        tmem_ld32(tl + kColS + 64 * half + 32, r + 32);
        tmem_wait_ld_regs(r);
        reg_fence32(r + 32);
        // P^T stays in float32 in r for dS below (the bf16 copy feeds dV only).
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          const float2 l2 = *reinterpret_cast<const float2*>(lse + 2 * j);
          r[2 * j] = __float_as_uint(ex2(fmaf(__uint_as_float(r[2 * j]), sl2, -l2.x * kLog2e)));
          r[2 * j + 1] =
              __float_as_uint(ex2(fmaf(__uint_as_float(r[2 * j + 1]), sl2, -l2.y * kLog2e)));
        }
        if (cut) {  // only on tiles the key's window cuts (diagonal, document borders)
#pragma unroll
          for (int j = 0; j < 64; ++j)
            if (64 * half + j < c_lo || 64 * half + j > c_hi) r[j] = 0u;
        }
        uint32_t pk[32];
#pragma unroll
        for (int j = 0; j < 32; ++j)
          pk[j] = pack_bf16(__uint_as_float(r[2 * j]), __uint_as_float(r[2 * j + 1]));
        tmem_st32(tl + kColS + 64 * half, pk);
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(bar(kBarP));
        // dS^T = scale * P^T (dP^T - Delta), dP^T read 32 columns at a time
        if (!__all_sync(0xffffffffu, mbar_wait(bar(kBarDP), dp_ph, wc))) {
          ok = false;
          break;
        }
        dp_ph ^= 1;
        tc_fence_after();
        uint32_t ds[32];
#pragma unroll
        for (int cc = 0; cc < 2; ++cc) {
          uint32_t d[32];
          tmem_ld32(tl + kColDP + 64 * half + 32 * cc, d);
          tmem_wait_ld_regs(d);
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const int c = 32 * cc + 2 * j;
#if CPATTN_MUTATION == 4
            const float2 dl = make_float2(0.f, 0.f);  // planted: Delta dropped from dS
#else
            const float2 dl = *reinterpret_cast<const float2*>(dlt + c);  // scale * Delta
#endif
            ds[16 * cc + j] =
                pack_bf16(__uint_as_float(r[c]) * fmaf(__uint_as_float(d[2 * j]), scale, -dl.x),
                          __uint_as_float(r[c + 1]) *
                              fmaf(__uint_as_float(d[2 * j + 1]), scale, -dl.y));
          }
        }
        tmem_st32(tl + kColDP + 64 * half, ds);
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(bar(kBarDS));
        ++qi;
        ++nq;
      }
      if (!ok) break;
      // Epilogue: this head's dK / dV partial, columns [64*half, +64).
      if (!__all_sync(0xffffffffu, mbar_wait(bar(kBarAcc), k & 1, wc))) {
        ok = false;
        break;
      }
      tc_fence_after();
      const int kv_row0 = sh.kv_natural ? it.knat * kT : it.kv.row;
      const int64_t pbase =
          (((int64_t)it.b * sh.S + kv_row0 + row) * sh.H + it.h) * kD + 64 * half;
#pragma unroll
      for (int which = 0; which < 2; ++which) {
        float* dst = (which == 0 ? args.dv_part : args.dk_part) + pbase;
        const uint32_t col = (which == 0 ? kColDV : kColDK) + 64 * half;
#pragma unroll
        for (int cc = 0; cc < 2; ++cc) {
          uint32_t d[32];
          tmem_ld32(tl + col + 32 * cc, d);
          tmem_wait_ld_regs(d);
          if (nq == 0) {
#pragma unroll
            for (int j = 0; j < 32; ++j) d[j] = 0u;
          }
#pragma unroll
          for (int u = 0; u < 8; ++u)
            *reinterpret_cast<float4*>(dst + 32 * cc + 4 * u) =
                make_float4(__uint_as_float(d[4 * u]), __uint_as_float(d[4 * u + 1]),
                            __uint_as_float(d[4 * u + 2]), __uint_as_float(d[4 * u + 3]));
        }
      }
      tc_fence_before();
      mbar_arrive(bar(kBarAccFree));
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

}  // namespace kv

// ===========================================================================
// dq kernel
// ===========================================================================
namespace qm {

// K and V tiles in rings of their own: V(j) is free once dP(j) has read it,
// K(j) only once dQ(j) has, which comes a tile later; with a ring each, V's
// copies are never held up behind K's release.
constexpr int kKSlots = 3;  // K(j) in slot j % 3
constexpr int kVSlots = 2;  // V(j) in slot j % 2
constexpr int kOffQ = 0;
constexpr int kOffDO = kOffQ + kTileBytes;
constexpr int kOffRing = kOffDO + kTileBytes;  // [kKSlots] K, then [kVSlots] V
constexpr int kOffBar = kOffRing + (kKSlots + kVSlots) * kTileBytes;
constexpr int kBarQFull = 0;
constexpr int kBarQEmpty = 1;
constexpr int kBarKFull = 2;                      // [kKSlots]
constexpr int kBarKEmpty = kBarKFull + kKSlots;   // [kKSlots]
constexpr int kBarVFull = kBarKEmpty + kKSlots;   // [kVSlots]
constexpr int kBarVEmpty = kBarVFull + kVSlots;   // [kVSlots]
constexpr int kBarS = kBarVEmpty + kVSlots;
constexpr int kBarSFree = kBarS + 1;
constexpr int kBarDP = kBarSFree + 1;
constexpr int kBarDS = kBarDP + 1;
constexpr int kBarQT = kBarDS + 1;             // Q and dO copied into TMEM
constexpr int kBarAcc = kBarQT + 1;
constexpr int kBarAccFree = kBarAcc + 1;
constexpr int kBarDrain = kBarAccFree + 1;
constexpr int kNumBars = kBarDrain + 1;
constexpr int kOffMisc = kOffBar + kNumBars * 8;
constexpr int kSmemBytes = kOffMisc + 16 + 1024;
// TMEM: S, dP (dS packed over it), the dQ accumulator, and the item's Q and
// dO tiles as bf16 pairs (the A operands of the S and dP products).
constexpr uint32_t kColS = 0, kColDP = 128, kColDQ = 256, kColQT = 384, kColDOT = 448;

struct Item {
  int b, h, g, knat;
  TilePos q;
};

// Groups are the (batch, kv head) pairs, ranks the query tiles latest first
// (a late tile sees the most K/V tiles), each rank the query heads of the kv
// head, in cost bands (banded_item): the CTAs in flight share one kv head's
// K/V through L2.
__device__ __forceinline__ Item decode(const RingShape& sh, int idx) {
  const int grp = sh.H / sh.Hkv;
  const int ntiles = sh.S / kT;
  int gi, rank, sub;
  banded_item(idx, sh.B * sh.Hkv, ntiles, grp, gridDim.x, 0, gi, rank, sub);
  const int knat = ntiles - 1 - rank;
  Item it;
  it.b = gi / sh.Hkv;
  it.g = gi - it.b * sh.Hkv;
  it.h = it.g * grp + sub;
  it.knat = knat;
  it.q = tile_pos(sh, knat);
  return it;
}

__global__ void __launch_bounds__(kThreads, 1)
    dq_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
              const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
              const BwdArgs args, int n_items) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (base - raw);
  const uint32_t sQ = base + kOffQ, sDO = base + kOffDO, sRing = base + kOffRing;
  auto kslot = [&](uint32_t j) { return sRing + (j % kKSlots) * kTileBytes; };
  auto vslot = [&](uint32_t j) { return sRing + (kKSlots + j % kVSlots) * kTileBytes; };
  const uint32_t bars = base + kOffBar;
  auto bar = [&](int i) { return bars + 8u * (uint32_t)i; };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kOffMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kOffMisc + 4);

  const RingShape& sh = args.sh;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const WaitCtl wc{abort_flag, args.err};

  if (threadIdx.x == 0) {
    mbar_init(bar(kBarQFull), 1);
    mbar_init(bar(kBarQEmpty), 256);
    for (int i = 0; i < kKSlots; ++i) {
      mbar_init(bar(kBarKFull + i), 1);
      mbar_init(bar(kBarKEmpty + i), 1);
    }
    for (int i = 0; i < kVSlots; ++i) {
      mbar_init(bar(kBarVFull + i), 1);
      mbar_init(bar(kBarVEmpty + i), 1);
    }
    mbar_init(bar(kBarDP), 1);
    mbar_init(bar(kBarS), 1);
    mbar_init(bar(kBarSFree), 256);
    mbar_init(bar(kBarDS), 256);
    mbar_init(bar(kBarQT), 256);
    mbar_init(bar(kBarAcc), 1);
    mbar_init(bar(kBarAccFree), 256);
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
    if (lane == 0) {
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_v);
      tma_prefetch_desc(&tm_do);
      uint32_t tj = 0, q_armed = 0, k_armed[kKSlots] = {0}, v_armed[kVSlots] = {0};
      bool ok = true;
      for (int k = 0; ok; ++k) {
        const int idx = item_index(k, blockIdx.x, gridDim.x);
        if (idx >= n_items) break;
        const Item it = decode(sh, idx);
        if (!mbar_wait(bar(kBarQEmpty), (k & 1) ^ 1, wc)) {
          ok = false;
          break;
        }
        mbar_arrive_expect_tx(bar(kBarQFull), 2 * kTileBytes);
        ++q_armed;
        const int qrow = it.b * sh.S + it.q.row;
        for (int half = 0; half < 2; ++half) {
          tma_load_3d(sQ + half * kBoxBytes, &tm_q, bar(kBarQFull), half * 64, it.h, qrow);
          tma_load_3d(sDO + half * kBoxBytes, &tm_do, bar(kBarQFull), half * 64, it.h, qrow);
        }
        KSeq seq;
        seq.init(sh, it.q, it.knat);
        // A second walker kPrefetchAhead tiles ahead asks L2 for the K / V
        // tiles before their loads are issued.
        KSeq pseq = seq;
        auto prefetch_next = [&]() {
          int prow, pnat;
          if (!pseq.next(prow, pnat)) return;
          const int row = it.b * sh.S + prow;
          for (int half = 0; half < 2; ++half) {
            tma_prefetch_l2_3d(&tm_k, half * 64, it.g, row);
            tma_prefetch_l2_3d(&tm_v, half * 64, it.g, row);
          }
        };
        for (int i = 0; i < kPrefetchAhead; ++i) prefetch_next();
        int kvrow, knat;
        // Census: K/V tiles per ring step (the diagonal tile arrives at step
        // 0), flushed at each change of step.
        unsigned long long* census = sh.kv_natural ? nullptr : args.tiles_q_rt;
        int c_step = -1;
        unsigned long long c_n = 0;
        while (ok && seq.next(kvrow, knat)) {
          prefetch_next();
          if (census != nullptr) {
            const int step = seq.t;
            if (step != c_step) {
              if (c_n) atomicAdd(&census[it.q.rank * sh.cp + c_step], c_n);
              c_step = step;
              c_n = 0;
            }
            ++c_n;
          }
          const int krow = it.b * sh.S + kvrow;
          const uint32_t j = tj++;
          const int ks = j % kKSlots, vs = j % kVSlots;
          if (!mbar_wait(bar(kBarKEmpty + ks), ((j / kKSlots) & 1) ^ 1, wc)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(bar(kBarKFull + ks), kTileBytes);
          ++k_armed[ks];
          for (int half = 0; half < 2; ++half)
            tma_load_3d(kslot(j) + half * kBoxBytes, &tm_k, bar(kBarKFull + ks), half * 64, it.g,
                        krow);
          if (!mbar_wait(bar(kBarVEmpty + vs), ((j / kVSlots) & 1) ^ 1, wc)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(bar(kBarVFull + vs), kTileBytes);
          ++v_armed[vs];
          for (int half = 0; half < 2; ++half)
            tma_load_3d(vslot(j) + half * kBoxBytes, &tm_v, bar(kBarVFull + vs), half * 64, it.g,
                        krow);
        }
        if (census != nullptr && c_n) atomicAdd(&census[it.q.rank * sh.cp + c_step], c_n);
      }
      if (!ok) {
        if (q_armed) mbar_drain(bar(kBarQFull), (q_armed - 1) & 1);
        for (int s = 0; s < kKSlots; ++s)
          if (k_armed[s]) mbar_drain(bar(kBarKFull + s), (k_armed[s] - 1) & 1);
        for (int s = 0; s < kVSlots; ++s)
          if (v_armed[s]) mbar_drain(bar(kBarVFull + s), (v_armed[s] - 1) & 1);
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
      // kj counts the K/V tiles this CTA has consumed.
      uint32_t kj = 0, sf_ph = 0, ds_ph = 0;
      bool ok = true;
      auto wait_k = [&](uint32_t j) {
        return wwait(bar(kBarKFull + j % kKSlots), (j / kKSlots) & 1);
      };
      auto wait_v = [&](uint32_t j) {
        return wwait(bar(kBarVFull + j % kVSlots), (j / kVSlots) & 1);
      };
      // Operand descriptors, computed once and advanced by byte offsets.
      const uint64_t d_ring = sdesc_sw128(sRing, 16, 1024);
      const uint64_t d_ring_mn = sdesc_sw128(sRing, kBoxBytes, 1024);
      auto koff = [](uint32_t j) { return (j % kKSlots) * (uint32_t)kTileBytes; };
      auto voff = [](uint32_t j) { return (kKSlots + j % kVSlots) * (uint32_t)kTileBytes; };
      // S = Q K^T and dP = dO V^T take A (Q, dO) from TMEM: the TS form.
      auto issue_s = [&](uint32_t j) {
        if (!leader) return;
        const uint64_t b0 = sdesc_advance(d_ring, koff(j));
#pragma unroll
        for (int kk = 0; kk < kD / 16; ++kk) {
          const uint32_t off = (kk >> 2) * kBoxBytes + (kk & 3) * 32;
          mma_ts(tmem + kColS, tmem + kColQT + kk * 8, sdesc_advance(b0, off), kIdescKK, kk > 0);
        }
        mma_commit(bar(kBarS));
      };
      auto issue_dp = [&](uint32_t j) {
        if (!leader) return;
        const uint64_t b0 = sdesc_advance(d_ring, voff(j));
#pragma unroll
        for (int kk = 0; kk < kD / 16; ++kk) {
          const uint32_t off = (kk >> 2) * kBoxBytes + (kk & 3) * 32;
          mma_ts(tmem + kColDP, tmem + kColDOT + kk * 8, sdesc_advance(b0, off), kIdescKK,
                 kk > 0);
        }
        mma_commit(bar(kBarDP));
        mma_commit(bar(kBarVEmpty + j % kVSlots));  // V is read only by dP
      };
      for (int k = 0; ok; ++k) {
        const int idx = item_index(k, blockIdx.x, gridDim.x);
        if (idx >= n_items) break;
        const Item it = decode(sh, idx);
        // The elementwise warps have copied the item's Q and dO into TMEM.
        if (!wwait(bar(kBarQT), k & 1)) {
          ok = false;
          break;
        }
        tc_fence_after();
        KSeq seq;
        seq.init(sh, it.q, it.knat);
        int kvrow, knat;
        bool have = seq.next(kvrow, knat);
        if (have) {
          if (!wait_k(kj)) {
            ok = false;
            break;
          }
          tc_fence_after();
          issue_s(kj);
          if (!wait_v(kj)) {
            ok = false;
            break;
          }
          tc_fence_after();
          issue_dp(kj);
        }
        bool first = true;
        while (have) {
          int nkvrow, nknat;
          const bool nhave = seq.next(nkvrow, nknat);
          if (nhave) {
            if (!wait_k(kj + 1)) {
              ok = false;
              break;
            }
            // S is released as soon as the elementwise warps have read it.
            if (!wwait(bar(kBarSFree), sf_ph)) {
              ok = false;
              break;
            }
            sf_ph ^= 1;
            tc_fence_after();
            issue_s(kj + 1);
          }
          // dQ += dS K
          if (!wwait(bar(kBarDS), ds_ph)) {
            ok = false;
            break;
          }
          ds_ph ^= 1;
          if (first && !wwait(bar(kBarAccFree), (k & 1) ^ 1)) {
            ok = false;
            break;
          }
          tc_fence_after();
          if (leader) {
            const uint64_t b0 = sdesc_advance(d_ring_mn, koff(kj));
#pragma unroll
            for (int kk = 0; kk < kT / 16; ++kk)
              mma_ts(tmem + kColDQ, tmem + kColDP + a_col(kk), sdesc_advance(b0, kk * 2048),
                     kIdescKM, (!first || kk > 0) ? 1u : 0u);
          }
          if (leader) mma_commit(bar(kBarKEmpty + kj % kKSlots));  // K is free after dQ
          if (nhave) {
            // dP of the next tile over the dS this dQ reads: MMAs execute in
            // issue order, so dQ has read dS before dP overwrites it.
            if (!wait_v(kj + 1)) {
              ok = false;
              break;
            }
            tc_fence_after();
            issue_dp(kj + 1);
          }
          first = false;
          ++kj;
          have = nhave;
        }
        if (!ok) break;
        if (first) {
          // No K/V tile at all (cannot happen for well-formed windows: every
          // query sees its own key): the epilogue writes zeros; it still
          // waits for the previous epilogue.
          if (!wwait(bar(kBarAccFree), (k & 1) ^ 1)) {
            ok = false;
            break;
          }
        } else {
          // The item's last S was read but not overwritten: take its release
          // so that the next item's first S waits on a fresh phase.
          if (!wwait(bar(kBarSFree), sf_ph)) {
            ok = false;
            break;
          }
          sf_ph ^= 1;
        }
        if (leader) mma_commit(bar(kBarAcc));
      }
      if (!ok) {
        if (leader) mma_commit(bar(kBarDrain));
        mbar_drain(bar(kBarDrain), 0);
      }
    }
  } else if (warp >= 4) {
    // ----------------------------------------------- elementwise + dQ epilogue
    const int half = (warp - 4) >> 2;  // K/V columns [64*half, 64*half + 64)
    const int wq = warp & 3;
    const int row = wq * 32 + lane;    // query row of the tile (TMEM lane)
    const uint32_t tl = tmem + ((uint32_t)(wq * 32) << 16);
    const float sl2 = sh.scale_log2, scale = sh.scale;
    uint32_t s_ph = 0, dp_ph = 0;
    bool ok = true;
    for (int k = 0; ok; ++k) {
      const int idx = item_index(k, blockIdx.x, gridDim.x);
      if (idx >= n_items) break;
      const Item it = decode(sh, idx);
      const int64_t li = ((int64_t)it.b * sh.H + it.h) * sh.S + it.q.row + row;
      const float nlse2 = -args.lse[li] * kLog2e;
      const float dlt = args.delta[li];  // scale * Delta
      // Copy the item's Q (first half) or dO (second half) tile into TMEM as
      // bf16 pairs, this thread's row: the 128-byte-swizzled TMA boxes hold
      // 16-byte chunk c of row r at chunk c ^ (r % 8).  The previous item's
      // products have all retired (its epilogue waited for them), and the
      // shared-memory copy is released to the next item's loads at once.
      if (!__all_sync(0xffffffffu, mbar_wait(bar(kBarQFull), k & 1, wc))) {
        ok = false;
        break;
      }
      {
        const uint8_t* src = smem + (half ? kOffDO : kOffQ) + row * 128;
        uint32_t w[64];
#pragma unroll
        for (int c = 0; c < 16; ++c) {
          const uint4 v = *reinterpret_cast<const uint4*>(
              src + (c >> 3) * kBoxBytes + (((c & 7) ^ (row & 7)) << 4));
          w[4 * c] = v.x;
          w[4 * c + 1] = v.y;
          w[4 * c + 2] = v.z;
          w[4 * c + 3] = v.w;
        }
        const uint32_t dst = tl + (half ? kColDOT : kColQT);
        tmem_st32(dst, w);
        tmem_st32(dst + 32, w + 32);
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(bar(kBarQT));
        mbar_arrive(bar(kBarQEmpty));
      }
      KSeq seq;
      seq.init(sh, it.q, it.knat);
      // Keys that this thread's query sees (natural positions).
      int w_lo, w_hi;
      query_window(sh, it.knat * kT + row, w_lo, w_hi);
      int kvrow, knat;
      int ntiles = 0;
      while (seq.next(kvrow, knat)) {
        const int j_lo = w_lo - knat, j_hi = w_hi - knat;  // visible key columns
        const bool cut = j_lo > 0 || j_hi < kT - 1;
        if (!__all_sync(0xffffffffu, mbar_wait(bar(kBarS), s_ph, wc))) {
          ok = false;
          break;
        }
        s_ph ^= 1;
        tc_fence_after();
        uint32_t r[64];
        tmem_ld32(tl + kColS + 64 * half, r);
        tmem_ld32(tl + kColS + 64 * half + 32, r + 32);
        tmem_wait_ld_regs(r);
        reg_fence32(r + 32);
        tc_fence_before();
        mbar_arrive(bar(kBarSFree));
        float p[64];
#pragma unroll
        for (int j = 0; j < 64; ++j) p[j] = ex2(fmaf(__uint_as_float(r[j]), sl2, nlse2));
        if (cut) {  // only on tiles the query's window cuts (diagonal, document borders)
#pragma unroll
          for (int j = 0; j < 64; ++j)
            if (64 * half + j < j_lo || 64 * half + j > j_hi) p[j] = 0.f;
        }
        if (!__all_sync(0xffffffffu, mbar_wait(bar(kBarDP), dp_ph, wc))) {
          ok = false;
          break;
        }
        dp_ph ^= 1;
        tc_fence_after();
        tmem_ld32(tl + kColDP + 64 * half, r);
        tmem_ld32(tl + kColDP + 64 * half + 32, r + 32);
        tmem_wait_ld_regs(r);
        reg_fence32(r + 32);
        uint32_t ds[32];
#pragma unroll
        for (int j = 0; j < 32; ++j)
          ds[j] = pack_bf16(p[2 * j] * fmaf(__uint_as_float(r[2 * j]), scale, -dlt),
                            p[2 * j + 1] * fmaf(__uint_as_float(r[2 * j + 1]), scale, -dlt));
        tmem_st32(tl + kColDP + 64 * half, ds);
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(bar(kBarDS));
        ++ntiles;
      }
      if (!ok) break;
      // Epilogue: dQ row, columns [64*half, +64), in the gradient dtype.
      if (!__all_sync(0xffffffffu, mbar_wait(bar(kBarAcc), k & 1, wc))) {
        ok = false;
        break;
      }
      tc_fence_after();
      const int64_t obase =
          (((int64_t)it.b * sh.S + it.q.row + row) * sh.H + it.h) * kD + 64 * half;
#pragma unroll
      for (int cc = 0; cc < 2; ++cc) {
        uint32_t d[32];
        tmem_ld32(tl + kColDQ + 64 * half + 32 * cc, d);
        tmem_wait_ld_regs(d);
        if (ntiles == 0) {
#pragma unroll
          for (int j = 0; j < 32; ++j) d[j] = 0u;
        }
        if (args.dq_f32) {
          float* dst = static_cast<float*>(args.dq) + obase + 32 * cc;
#pragma unroll
          for (int u = 0; u < 8; ++u)
            *reinterpret_cast<float4*>(dst + 4 * u) =
                make_float4(__uint_as_float(d[4 * u]), __uint_as_float(d[4 * u + 1]),
                            __uint_as_float(d[4 * u + 2]), __uint_as_float(d[4 * u + 3]));
        } else {
          __nv_bfloat16* dst = static_cast<__nv_bfloat16*>(args.dq) + obase + 32 * cc;
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            uint4 v;
            v.x = pack_bf16(__uint_as_float(d[8 * u + 0]), __uint_as_float(d[8 * u + 1]));
            v.y = pack_bf16(__uint_as_float(d[8 * u + 2]), __uint_as_float(d[8 * u + 3]));
            v.z = pack_bf16(__uint_as_float(d[8 * u + 4]), __uint_as_float(d[8 * u + 5]));
            v.w = pack_bf16(__uint_as_float(d[8 * u + 6]), __uint_as_float(d[8 * u + 7]));
            *reinterpret_cast<uint4*>(dst + 8 * u) = v;
          }
        }
      }
      tc_fence_before();
      mbar_arrive(bar(kBarAccFree));
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

}  // namespace qm

// ===========================================================================
// One-pass kernel: dK, dV and dQ from one K/V-major walk
// ===========================================================================
//
// Work item and walk as the dkdv kernel (one 128-row K/V tile x one query
// head, the query tiles that see it, latest first).  Per query tile j, with
// TMEM lanes = K/V rows for S^T, dP^T, dV, dK and lanes = features for dQ^T:
//   S^T  = K Q^T  -> X             dP^T = V dO^T -> Y
//   P^T  -> bf16 over X (TMEM)     dS^T = scale P^T (dP^T - Delta) -> bf16
//                                  into shared memory (128-byte swizzle)
//   dV  += P^T dO  (TS, A = X)     dK  += dS^T Q  (SS, A = dS^T K-major)
//   dQ^T = K^T dS^T (SS, A = K MN-major, B = dS^T MN-major) -> Y
// and the dQ^T tile (this K/V tile's share of the query tile's dQ) is read
// out of TMEM by the drain warpgroup, staged in shared memory (over dS^T,
// which the two MMAs have finished reading) and added to the float32 dQ
// accumulator [B,S,H,D] with tensor bulk reductions (cp.reduce.async.bulk
// .add), 32 query rows (16 KB) at a time through two slots.  Every K/V tile
// that a query tile sees adds its share once: 5 GEMMs per tile pair instead
// of the two-kernel path's 7, at the price of dQ's summation order, which
// follows the order the reductions reach L2 (the result is not bitwise
// reproducible from run to run; the two-kernel path is).
//
// CTA = 512 threads: warp 0 TMA, warp 1 TMEM owner + MMA issuer (warps 0-3:
// 104 registers), warps 4-11 the elementwise halves ([0,64) and [64,128) of
// the query columns) and the dK / dV epilogue (152 registers), warps 12-15
// the dQ drain (104 registers; thread = feature lane).  The split uses the
// whole 512 x 128 registers of the launch and leaves ptxas nothing to
// spill.  Shared memory: K, V, two Q / dO stages, dS^T (= the dQ staging),
// LSE / Delta rows: 226 KB.
namespace fz {

constexpr int kThreadsF = 512;
constexpr int kOffK = 0;
constexpr int kOffV = kOffK + kTileBytes;
constexpr int kOffQ = kOffV + kTileBytes;         // [2] stages
constexpr int kOffDO = kOffQ + 2 * kTileBytes;    // [2]
constexpr int kOffDS = kOffDO + 2 * kTileBytes;   // dS^T, then the two dQ staging slots
constexpr int kOffLse = kOffDS + kTileBytes;      // [2][128] float (natural log)
constexpr int kOffDlt = kOffLse + 2 * kT * 4;     // [2][128] float
constexpr int kOffBar = kOffDlt + 2 * kT * 4;
constexpr int kBarKVFull = 0;
constexpr int kBarKVEmpty = 1;
constexpr int kBarQFull = 2;       // [2]
constexpr int kBarQEmpty = 4;      // [2]
constexpr int kBarS = 6;
constexpr int kBarDP = 7;
constexpr int kBarP = 8;
constexpr int kBarDS = 9;
constexpr int kBarDQ = 10;
constexpr int kBarYFree = 11;
constexpr int kBarDSFree = 12;
constexpr int kBarStageFull = 13;  // [2]
constexpr int kBarStageFree = 15;  // [2]
constexpr int kBarAcc = 17;
constexpr int kBarAccFree = 18;
constexpr int kBarDrain = 19;
constexpr int kNumBars = 20;
constexpr int kOffMisc = kOffBar + kNumBars * 8;
// The dynamic shared memory starts on a 1024-byte boundary (checked at run
// time; the kernel refuses to run otherwise), so no alignment slack.
constexpr int kSmemBytes = kOffMisc + 16;
constexpr uint32_t kColX = 0, kColY = 128, kColDV = 256, kColDK = 384;
constexpr uint32_t kQTx = 2 * kTileBytes + 2 * kT * 4;  // Q, dO, LSE, Delta
constexpr uint32_t kIdescMM = idesc_bf16(128, 128, true, true);  // A and B MN-major
constexpr int kStageRows = 32;                       // query rows per reduction
constexpr int kStageBytes = kStageRows * kD * 4;     // 16 KB of float32
// Registers per thread for the three roles (setmaxnreg); the launch gives
// 512 threads x 128.
constexpr int kRegCtl = 104, kRegEw = 152, kRegDrain = 104;
static_assert(128 * (kRegCtl + 2 * kRegEw + kRegDrain) <= 512 * 128, "register split");
static_assert(kSmemBytes <= 232448, "shared memory");

template <int N>
__device__ __forceinline__ void reg_dec() {
  asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(N));
}
template <int N>
__device__ __forceinline__ void reg_inc() {
  asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(N));
}
__device__ __forceinline__ void fence_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
// Adds a [32 rows][128] float32 box of shared memory into the accumulator at
// (feature 0, head h, row); completion tracked as a bulk group.
__device__ __forceinline__ void tma_reduce_add_3d(const CUtensorMap* map, uint32_t src, int h,
                                                  int row) {
  asm volatile(
      "cp.reduce.async.bulk.tensor.3d.global.shared::cta.add.tile.bulk_group "
      "[%0, {%1, %2, %3}], [%4];" ::"l"(reinterpret_cast<uint64_t>(map)),
      "r"(0), "r"(h), "r"(row), "r"(src)
      : "memory");
}
__device__ __forceinline__ void bulk_commit() {
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
template <int N>
__device__ __forceinline__ void bulk_wait_read() {
  asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}
__device__ __forceinline__ void bulk_wait_all() {
  asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}

using kv::Item;
using kv::decode;

__global__ void __launch_bounds__(kThreadsF, 1)
    dkdvq_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                 const __grid_constant__ CUtensorMap tm_v,
                 const __grid_constant__ CUtensorMap tm_do,
                 const __grid_constant__ CUtensorMap tm_dq, const BwdArgs args, int n_items) {
  extern __shared__ __align__(1024) uint8_t smem_fz[];
  const uint32_t base = smem_u32(smem_fz);
  if ((base & 1023u) != 0) {  // uniform: every thread leaves before any wait
    if (threadIdx.x == 0) atomicExch(args.err, kErrLaunch);
    return;
  }
  uint8_t* smem = smem_fz;
  const uint32_t sK = base + kOffK, sV = base + kOffV, sQ = base + kOffQ, sDO = base + kOffDO;
  const uint32_t sDS = base + kOffDS, sLse = base + kOffLse, sDlt = base + kOffDlt;
  const float* lse_s = reinterpret_cast<const float*>(smem + kOffLse);
  const float* dlt_s = reinterpret_cast<const float*>(smem + kOffDlt);
  const uint32_t bars = base + kOffBar;
  auto bar = [&](int i) { return bars + 8u * (uint32_t)i; };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kOffMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kOffMisc + 4);

  const RingShape& sh = args.sh;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const WaitCtl wc{abort_flag, args.err};

  if (threadIdx.x == 0) {
    mbar_init(bar(kBarKVFull), 1);
    mbar_init(bar(kBarKVEmpty), 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(bar(kBarQFull + i), 1);
      mbar_init(bar(kBarQEmpty + i), 1);
      mbar_init(bar(kBarStageFull + i), 128);
      mbar_init(bar(kBarStageFree + i), 1);
    }
    mbar_init(bar(kBarS), 1);
    mbar_init(bar(kBarDP), 1);
    mbar_init(bar(kBarP), 256);
    mbar_init(bar(kBarDS), 256);
    mbar_init(bar(kBarDQ), 1);
    mbar_init(bar(kBarYFree), 128);
    mbar_init(bar(kBarDSFree), 1);
    mbar_init(bar(kBarAcc), 1);
    mbar_init(bar(kBarAccFree), 256);
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

  if (warp < 4) {
    reg_dec<kRegCtl>();
  }
  if (warp == 0) {
    // ------------------------------------------------------------------ TMA
    if (lane == 0) {
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_v);
      tma_prefetch_desc(&tm_do);
      uint32_t qi = 0, kv_armed = 0, q_armed[2] = {0, 0};
      bool ok = true;
      for (int k = 0; ok; ++k) {
        const int idx = item_index(k, blockIdx.x, gridDim.x);
        if (idx >= n_items) break;
        const Item it = decode(sh, idx);
        if (!mbar_wait(bar(kBarKVEmpty), (k & 1) ^ 1, wc)) {
          ok = false;
          break;
        }
        mbar_arrive_expect_tx(bar(kBarKVFull), 2 * kTileBytes);
        ++kv_armed;
        const int krow = it.b * sh.S + (sh.kv_natural ? it.knat * kT : it.kv.row);
        for (int half = 0; half < 2; ++half) {
          tma_load_3d(sK + half * kBoxBytes, &tm_k, bar(kBarKVFull), half * 64, it.g, krow);
          tma_load_3d(sV + half * kBoxBytes, &tm_v, bar(kBarKVFull), half * 64, it.g, krow);
        }
        QSeq seq;
        seq.init(sh, it.kv, it.knat);
        int qrow, qnat;
        unsigned long long* census = sh.kv_natural ? nullptr : args.tiles_kv_rt;
        unsigned long long* census_q = sh.kv_natural ? nullptr : args.tiles_q_rt;
        int c_step = -1;
        unsigned long long c_n = 0;
        while (seq.next(qrow, qnat)) {
          if (census != nullptr) {
            if (seq.t != c_step) {
              if (c_n) {
                const int cell = ((it.kv.rank + c_step) % sh.cp) * sh.cp + c_step;
                atomicAdd(&census[cell], c_n);
                if (census_q != nullptr) atomicAdd(&census_q[cell], c_n);
              }
              c_step = seq.t;
              c_n = 0;
            }
            ++c_n;
          }
          const int st = qi & 1;
          const uint32_t ph = (qi >> 1) & 1;
          if (!mbar_wait(bar(kBarQEmpty + st), ph ^ 1, wc)) {
            ok = false;
            break;
          }
          const uint32_t full = bar(kBarQFull + st);
          mbar_arrive_expect_tx(full, kQTx);
          ++q_armed[st];
          const int row = it.b * sh.S + qrow;
          for (int half = 0; half < 2; ++half) {
            tma_load_3d(sQ + st * kTileBytes + half * kBoxBytes, &tm_q, full, half * 64, it.h, row);
            tma_load_3d(sDO + st * kTileBytes + half * kBoxBytes, &tm_do, full, half * 64, it.h,
                        row);
          }
          const int64_t li = ((int64_t)it.b * sh.H + it.h) * sh.S + qrow;
          bulk_load(sLse + st * kT * 4, args.lse + li, kT * 4, full);
          bulk_load(sDlt + st * kT * 4, args.delta + li, kT * 4, full);
          ++qi;
        }
        if (census != nullptr && c_n) {
          const int cell = ((it.kv.rank + c_step) % sh.cp) * sh.cp + c_step;
          atomicAdd(&census[cell], c_n);
          if (census_q != nullptr) atomicAdd(&census_q[cell], c_n);
        }
      }
      if (!ok) {
        if (kv_armed) mbar_drain(bar(kBarKVFull), (kv_armed - 1) & 1);
        for (int s = 0; s < 2; ++s)
          if (q_armed[s]) mbar_drain(bar(kBarQFull + s), (q_armed[s] - 1) & 1);
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
      uint32_t qi = 0, p_ph = 0, ds_ph = 0;
      bool ok = true;
      // Operand descriptors, computed once and advanced by byte offsets.
      const uint64_t d_k = sdesc_sw128(sK, 16, 1024), d_v = sdesc_sw128(sV, 16, 1024);
      const uint64_t d_q = sdesc_sw128(sQ, 16, 1024), d_do = sdesc_sw128(sDO, 16, 1024);
      const uint64_t d_q_mn = sdesc_sw128(sQ, kBoxBytes, 1024);
      const uint64_t d_do_mn = sdesc_sw128(sDO, kBoxBytes, 1024);
      const uint64_t d_k_mn = sdesc_sw128(sK, kBoxBytes, 1024);
      const uint64_t d_ds_mn = sdesc_sw128(sDS, kBoxBytes, 1024);
      auto issue_s = [&](int st) {
        if (!leader) return;
        const uint64_t b0 = sdesc_advance(d_q, st * kTileBytes);
#pragma unroll
        for (int kk = 0; kk < kD / 16; ++kk) {
          const uint32_t off = (kk >> 2) * kBoxBytes + (kk & 3) * 32;
          mma_ss(tmem + kColX, sdesc_advance(d_k, off), sdesc_advance(b0, off), kIdescKK, kk > 0);
        }
        mma_commit(bar(kBarS));
      };
      auto issue_dp = [&](int st) {
        if (!leader) return;
        const uint64_t b0 = sdesc_advance(d_do, st * kTileBytes);
#pragma unroll
        for (int kk = 0; kk < kD / 16; ++kk) {
          const uint32_t off = (kk >> 2) * kBoxBytes + (kk & 3) * 32;
          mma_ss(tmem + kColY, sdesc_advance(d_v, off), sdesc_advance(b0, off), kIdescKK, kk > 0);
        }
        mma_commit(bar(kBarDP));
      };
      for (int k = 0; ok; ++k) {
        const int idx = item_index(k, blockIdx.x, gridDim.x);
        if (idx >= n_items) break;
        const Item it = decode(sh, idx);
        if (!wwait(bar(kBarKVFull), k & 1)) {
          ok = false;
          break;
        }
        tc_fence_after();
        QSeq seq;
        seq.init(sh, it.kv, it.knat);
        int qrow, qnat;
        bool have = seq.next(qrow, qnat);
        if (have) {
          const int st = qi & 1;
          if (!wwait(bar(kBarQFull + st), (qi >> 1) & 1)) {
            ok = false;
            break;
          }
          tc_fence_after();
          issue_s(st);
          // Y holds the previous tile's dQ^T until the drain has read it.
          if (!wwait(bar(kBarYFree), (qi & 1) ^ 1)) {
            ok = false;
            break;
          }
          tc_fence_after();
          issue_dp(st);
        }
        bool first = true;
        while (have) {
          const int st = qi & 1;
          int nqrow, nqnat;
          const bool nhave = seq.next(nqrow, nqnat);
          const int nst = (qi + 1) & 1;
          // dV += P^T dO
          if (!wwait(bar(kBarP), p_ph)) {
            ok = false;
            break;
          }
          p_ph ^= 1;
          if (first && !wwait(bar(kBarAccFree), (k & 1) ^ 1)) {
            ok = false;
            break;
          }
          tc_fence_after();
          if (leader) {
            const uint64_t b0 = sdesc_advance(d_do_mn, st * kTileBytes);
#pragma unroll
            for (int kk = 0; kk < kT / 16; ++kk)
              mma_ts(tmem + kColDV, tmem + kColX + a_col(kk), sdesc_advance(b0, kk * 2048),
                     kIdescKM, (!first || kk > 0) ? 1u : 0u);
          }
          // dK += dS^T Q (A = the bf16 dS^T the elementwise warps packed into
          // Y), then dQ^T = K^T dS^T (both operands in shared memory) over Y:
          // MMAs run in order, so dK has read Y before dQ^T writes it.
          if (!wwait(bar(kBarDS), ds_ph)) {
            ok = false;
            break;
          }
          ds_ph ^= 1;
          tc_fence_after();
          if (leader) {
            const uint64_t b0 = sdesc_advance(d_q_mn, st * kTileBytes);
#pragma unroll
            for (int kk = 0; kk < kT / 16; ++kk)
              mma_ts(tmem + kColDK, tmem + kColY + a_col(kk), sdesc_advance(b0, kk * 2048),
                     kIdescKM, (!first || kk > 0) ? 1u : 0u);
            mma_commit(bar(kBarQEmpty + st));  // Q, dO of this tile read for the last time
#pragma unroll
            for (int kk = 0; kk < kT / 16; ++kk)
              mma_ss(tmem + kColY, sdesc_advance(d_k_mn, kk * 2048),
                     sdesc_advance(d_ds_mn, kk * 2048), kIdescMM, kk > 0 ? 1u : 0u);
            mma_commit(bar(kBarDQ));
          }
          if (nhave) {
            // S of the next tile over X (dV has read P^T; MMAs run in order).
            if (!wwait(bar(kBarQFull + nst), ((qi + 1) >> 1) & 1)) {
              ok = false;
              break;
            }
            tc_fence_after();
            issue_s(nst);
            // dP of the next tile once the drain has read this tile's dQ^T.
            if (!wwait(bar(kBarYFree), ((qi + 1) & 1) ^ 1)) {
              ok = false;
              break;
            }
            tc_fence_after();
            issue_dp(nst);
          }
          first = false;
          ++qi;
          have = nhave;
        }
        if (!ok) break;
        if (first) {
          if (!wwait(bar(kBarAccFree), (k & 1) ^ 1)) {
            ok = false;
            break;
          }
        }
        if (leader) {
          mma_commit(bar(kBarAcc));
          mma_commit(bar(kBarKVEmpty));
        }
      }
      if (!ok) {
        if (leader) mma_commit(bar(kBarDrain));
        mbar_drain(bar(kBarDrain), 0);
      }
    }
  } else if (warp < 4) {
    // warps 2-3: no role
  } else if (warp < 12) {
    // ------------------------------------------------ elementwise + dK / dV
    reg_inc<kRegEw>();
    const int half = (warp - 4) >> 2;  // query columns [64*half, 64*half + 64)
    const int wq = warp & 3;
    const int row = wq * 32 + lane;    // K/V row of the tile (TMEM lane)
    const uint32_t tl = tmem + ((uint32_t)(wq * 32) << 16);
    const float sl2 = sh.scale_log2, scale = sh.scale;
    // This thread's 128-byte row of its half's dS^T box (128-byte swizzle).
    const uint32_t ds_row = sDS + half * kBoxBytes + row * 128;
    uint32_t qi = 0, s_ph = 0, dp_ph = 0;
    bool ok = true;
    for (int k = 0; ok; ++k) {
      const int idx = item_index(k, blockIdx.x, gridDim.x);
      if (idx >= n_items) break;
      const Item it = decode(sh, idx);
      QSeq seq;
      seq.init(sh, it.kv, it.knat);
      int w_lo, w_hi;
      key_window(sh, it.knat * kT + row, w_lo, w_hi);
      int qrow, qnat, nq = 0;
      while (seq.next(qrow, qnat)) {
        const int st = qi & 1;
        const int c_lo = w_lo - qnat, c_hi = w_hi - qnat;  // visible query columns
        const bool cut = c_lo > 0 || c_hi < kT - 1;
        if (!__all_sync(0xffffffffu, mbar_wait(bar(kBarQFull + st), (qi >> 1) & 1, wc))) {
          ok = false;
          break;
        }
        const float* lse = lse_s + st * kT + 64 * half;
        const float* dlt = dlt_s + st * kT + 64 * half;
        if (!__all_sync(0xffffffffu, mbar_wait(bar(kBarS), s_ph, wc))) {
          ok = false;
          break;
        }
        s_ph ^= 1;
        tc_fence_after();
        uint32_t r[64];
        tmem_ld32(tl + kColX + 64 * half, r);
        tmem_ld32(tl + kColX + 64 * half + 32, r + 32);
        tmem_wait_ld_regs(r);
        reg_fence32(r + 32);
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          const float2 l2 = *reinterpret_cast<const float2*>(lse + 2 * j);
          r[2 * j] = __float_as_uint(ex2(fmaf(__uint_as_float(r[2 * j]), sl2, -l2.x * kLog2e)));
          r[2 * j + 1] =
              __float_as_uint(ex2(fmaf(__uint_as_float(r[2 * j + 1]), sl2, -l2.y * kLog2e)));
        }
        if (cut) {
#pragma unroll
          for (int j = 0; j < 64; ++j)
            if (64 * half + j < c_lo || 64 * half + j > c_hi) r[j] = 0u;
        }
        uint32_t pk[32];
#pragma unroll
        for (int j = 0; j < 32; ++j)
          pk[j] = pack_bf16(__uint_as_float(r[2 * j]), __uint_as_float(r[2 * j + 1]));
        tmem_st32(tl + kColX + 64 * half, pk);
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(bar(kBarP));
        // dS^T = scale * P^T (dP^T - Delta), dP^T read 32 columns at a time
        if (!__all_sync(0xffffffffu, mbar_wait(bar(kBarDP), dp_ph, wc))) {
          ok = false;
          break;
        }
        dp_ph ^= 1;
        tc_fence_after();
        uint32_t ds[32];
#pragma unroll
        for (int cc = 0; cc < 2; ++cc) {
          uint32_t d[32];
          tmem_ld32(tl + kColY + 64 * half + 32 * cc, d);
          tmem_wait_ld_regs(d);
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const int c = 32 * cc + 2 * j;
            const float2 dl = *reinterpret_cast<const float2*>(dlt + c);  // scale * Delta
            ds[16 * cc + j] =
                pack_bf16(__uint_as_float(r[c]) * fmaf(__uint_as_float(d[2 * j]), scale, -dl.x),
                          __uint_as_float(r[c + 1]) *
                              fmaf(__uint_as_float(d[2 * j + 1]), scale, -dl.y));
          }
        }
        // The dS^T buffer doubles as the previous tile's dQ staging: wait
        // until the drain's last reduction of that tile has read it.
        if (!__all_sync(0xffffffffu, mbar_wait(bar(kBarDSFree), (qi & 1) ^ 1, wc))) {
          ok = false;
          break;
        }
        // dS^T twice: packed over the first 32 of this half's dP^T columns in
        // TMEM (dK's A operand), and into its shared-memory box (dQ^T's B).
        tmem_st32(tl + kColY + 64 * half, ds);
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          const uint32_t addr = ds_row + ((uint32_t)(c ^ (row & 7)) << 4);
          asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(ds[4 * c]),
                       "r"(ds[4 * c + 1]), "r"(ds[4 * c + 2]), "r"(ds[4 * c + 3])
                       : "memory");
        }
        fence_async_smem();  // generic-proxy writes -> the tensor core's reads
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(bar(kBarDS));
        ++qi;
        ++nq;
      }
      if (!ok) break;
      // Epilogue: this head's dK / dV partial, columns [64*half, +64).
      if (!__all_sync(0xffffffffu, mbar_wait(bar(kBarAcc), k & 1, wc))) {
        ok = false;
        break;
      }
      tc_fence_after();
      const int kv_row0 = sh.kv_natural ? it.knat * kT : it.kv.row;
      const int64_t pbase =
          (((int64_t)it.b * sh.S + kv_row0 + row) * sh.H + it.h) * kD + 64 * half;
#pragma unroll
      for (int which = 0; which < 2; ++which) {
        float* dst = (which == 0 ? args.dv_part : args.dk_part) + pbase;
        const uint32_t col = (which == 0 ? kColDV : kColDK) + 64 * half;
#pragma unroll
        for (int cc = 0; cc < 2; ++cc) {
          uint32_t d[32];
          tmem_ld32(tl + col + 32 * cc, d);
          tmem_wait_ld_regs(d);
          if (nq == 0) {
#pragma unroll
            for (int j = 0; j < 32; ++j) d[j] = 0u;
          }
#pragma unroll
          for (int u = 0; u < 8; ++u)
            *reinterpret_cast<float4*>(dst + 32 * cc + 4 * u) =
                make_float4(__uint_as_float(d[4 * u]), __uint_as_float(d[4 * u + 1]),
                            __uint_as_float(d[4 * u + 2]), __uint_as_float(d[4 * u + 3]));
        }
      }
      tc_fence_before();
      mbar_arrive(bar(kBarAccFree));
    }
  } else {
    // -------------------------------------------------------------- dQ drain
    // Thread = feature lane d of dQ^T (TMEM lane); four rounds of 32 query
    // columns per tile, staged as [32 rows][128] float32 in two 16 KB slots
    // over the dS^T buffer, each added to the accumulator by one bulk
    // reduction issued by the leader thread.
    reg_dec<kRegDrain>();
    const int wq = warp & 3;
    const int dl = wq * 32 + lane;
    const uint32_t tl = tmem + ((uint32_t)(wq * 32) << 16);
    const bool leader = warp == 12 && lane == 0;
    uint32_t qi = 0;
    bool ok = true;
    auto stage = [&](int slot, const uint32_t* v) {
      const uint32_t dst = sDS + slot * kStageBytes + dl * 4;
#pragma unroll
      for (int i = 0; i < 32; ++i)
        asm volatile("st.shared.b32 [%0], %1;" ::"r"(dst + i * (kD * 4)), "r"(v[i]) : "memory");
      fence_async_smem();
      mbar_arrive(bar(kBarStageFull + slot));
    };
    for (int k = 0; ok; ++k) {
      const int idx = item_index(k, blockIdx.x, gridDim.x);
      if (idx >= n_items) break;
      const Item it = decode(sh, idx);
      QSeq seq;
      seq.init(sh, it.kv, it.knat);
      int qrow, qnat;
      while (seq.next(qrow, qnat)) {
        const int row0 = it.b * sh.S + qrow;
        if (!__all_sync(0xffffffffu, mbar_wait(bar(kBarDQ), qi & 1, wc))) {
          ok = false;
          break;
        }
        tc_fence_after();
        uint32_t v[64];
        tmem_ld32(tl + kColY, v);
        tmem_ld32(tl + kColY + 32, v + 32);
        tmem_wait_ld_regs(v);
        reg_fence32(v + 32);
        stage(0, v);
        stage(1, v + 32);
        tmem_ld32(tl + kColY + 64, v);
        tmem_ld32(tl + kColY + 96, v + 32);
        tmem_wait_ld_regs(v);
        reg_fence32(v + 32);
        tc_fence_before();
        mbar_arrive(bar(kBarYFree));  // Y is free for the next tile's dP^T
        if (leader) {
          for (int s = 0; s < 2 && ok; ++s) {
            if (!mbar_wait(bar(kBarStageFull + s), 0u, wc)) {
              ok = false;
              break;
            }
            tma_reduce_add_3d(&tm_dq, sDS + s * kStageBytes, it.h, row0 + s * kStageRows);
            bulk_commit();
          }
          if (ok) {
            bulk_wait_read<1>();
            mbar_arrive(bar(kBarStageFree + 0));
            bulk_wait_read<0>();
            mbar_arrive(bar(kBarStageFree + 1));
          }
        }
        if (!__all_sync(0xffffffffu, ok)) {
          ok = false;
          break;
        }
        for (int s = 0; s < 2; ++s) {
          if (!__all_sync(0xffffffffu, mbar_wait(bar(kBarStageFree + s), qi & 1, wc))) {
            ok = false;
            break;
          }
          stage(s, v + 32 * s);
        }
        if (!ok) break;
        if (leader) {
          for (int s = 0; s < 2 && ok; ++s) {
            if (!mbar_wait(bar(kBarStageFull + s), 1u, wc)) {
              ok = false;
              break;
            }
            tma_reduce_add_3d(&tm_dq, sDS + s * kStageBytes, it.h,
                              row0 + (2 + s) * kStageRows);
            bulk_commit();
          }
          if (ok) {
            bulk_wait_read<0>();
            mbar_arrive(bar(kBarDSFree));  // dS^T of the next tile may overwrite the slots
          }
        }
        if (!__all_sync(0xffffffffu, ok)) {
          ok = false;
          break;
        }
        ++qi;
      }
    }
    if (leader) bulk_wait_all();  // every reduction complete before the CTA ends
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

}  // namespace fz

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

// The float32 dQ accumulator [rows][heads][128] as a 3-D tensor, box of 32
// rows x 1 head x 128 features (16 KB, no swizzle): the bulk reductions'
// destination.
bool make_map_dq(CUtensorMap* m, const float* ptr, int heads, int64_t rows) {
  EncodeTiledFn enc = encode_fn();
  if (enc == nullptr) return false;
  cuuint64_t dims[3] = {(cuuint64_t)kD, (cuuint64_t)heads, (cuuint64_t)rows};
  cuuint64_t strides[2] = {(cuuint64_t)kD * 4, (cuuint64_t)heads * kD * 4};
  cuuint32_t box[3] = {(cuuint32_t)kD, 1, (cuuint32_t)fz::kStageRows};
  cuuint32_t estr[3] = {1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<float*>(ptr), dims, strides, box,
             estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

bool tc_bwd_available() { return true; }

cudaError_t launch_tc_bwd_onepass(const BwdArgs& a, cudaStream_t stream) {
  const RingShape& sh = a.sh;
  const int n_items = sh.B * sh.H * (sh.S / kT);
  if (n_items == 0) return cudaSuccess;
  CUtensorMap mq, mk, mv, mdo, mdq;
  const int64_t rows = (int64_t)sh.B * sh.S;
  if (!make_map(&mq, a.q, sh.H, rows) || !make_map(&mk, a.k, sh.Hkv, rows) ||
      !make_map(&mv, a.v, sh.Hkv, rows) || !make_map(&mdo, a.dout, sh.H, rows) ||
      !make_map_dq(&mdq, a.dq_acc, sh.H, rows))
    return cudaErrorInvalidValue;
  int dev = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(fz::dkdvq_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           fz::kSmemBytes);
  if (e != cudaSuccess) return e;
  const int grid = n_items < sms ? n_items : sms;
  fz::dkdvq_kernel<<<grid, fz::kThreadsF, fz::kSmemBytes, stream>>>(mq, mk, mv, mdo, mdq, a,
                                                                    n_items);
  return cudaGetLastError();
}

cudaError_t launch_tc_bwd(const BwdArgs& a, cudaStream_t stream) {
  const RingShape& sh = a.sh;
  const int n_items = sh.B * sh.H * (sh.S / kT);
  if (n_items == 0) return cudaSuccess;
  CUtensorMap mq, mk, mv, mdo;
  const int64_t rows = (int64_t)sh.B * sh.S;
  if (!make_map(&mq, a.q, sh.H, rows) || !make_map(&mk, a.k, sh.Hkv, rows) ||
      !make_map(&mv, a.v, sh.Hkv, rows) || !make_map(&mdo, a.dout, sh.H, rows))
    return cudaErrorInvalidValue;
  int dev = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(kv::dkdv_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           kv::kSmemBytes);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(qm::dq_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           qm::kSmemBytes);
  if (e != cudaSuccess) return e;
  const int grid = n_items < sms ? n_items : sms;
  kv::dkdv_kernel<<<grid, kThreads, kv::kSmemBytes, stream>>>(mq, mk, mv, mdo, a, n_items);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  qm::dq_kernel<<<grid, kThreads, qm::kSmemBytes, stream>>>(mq, mk, mv, mdo, a, n_items);
  return cudaGetLastError();
}

}  // namespace cpattn
