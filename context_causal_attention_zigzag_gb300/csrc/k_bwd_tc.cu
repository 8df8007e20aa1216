// Tensor-core ring backward for sm_103a (tcgen05 + TMEM + TMA), persistent,
// warp-specialised, KV-major.
//
// Gradients through the ring ("Context Parallelism for Long-Context
// Training", section "Prove attention equivalence"): a work item is one
// 128-row K/V tile of one (batch, query head).  It stays in shared memory
// while the query tiles that see it stream past, in the order of the ring
// steps t = 0..cp-1 that carry this K/V to rank (s + t) mod cp ("Sequence
// Parallelism IV", section 4), tiles wholly in the causal past of the query
// skipped, the diagonal tile masked.  Per query tile:
//
//   S^T  = K Q^T                 (SS, 128x128x128)          -> TMEM cols [0,128)
//   dP^T = V dO^T                (SS)                        -> TMEM cols [128,256)
//   P^T  = exp2(S^T*scale*log2e - LSE*log2e)   (elementwise warps, bf16 back
//          over S^T in TMEM)
//   dV  += P^T dO                (TS: P^T from TMEM, dO MN-major) -> cols [256,384)
//   dS^T = scale * P^T (dP^T - Delta)          (elementwise warps, bf16 into
//          shared memory in the 128-byte-swizzled layout)
//   dK  += dS^T Q                (SS: dS^T K-major, Q MN-major)   -> cols [384,512)
//   dQ_t = dS K                  (SS: dS^T read MN-major, K MN-major) -> cols [128,256)
//   dQ  += dQ_t                  (dQ warps: float4 atomic adds into the float32
//          accumulator in HBM)
// At the end of the item the dK / dV partials of this query head are added
// (float4 atomics) into float32 accumulators shared by the heads of the group.
// One item per query head, rather than per kv head, bounds the number of
// MMA steps that accumulate into one TMEM sum (the tensor core's float32
// accumulation drifts toward zero over very long chains).
//
// CTA = 384 threads: warp 0 TMA (K, V once per item; Q and dO per query tile
// into a 2-stage ring), warp 1 TMEM owner + MMA issuer, warps 4-7 elementwise
// (one thread per K/V row = TMEM lane), warps 8-11 dQ reduction and the dK /
// dV epilogue.  LSE and Delta of the current query tile sit in shared memory,
// written by the elementwise warps (prefetched one tile ahead in registers);
// the warps hand that buffer over with two mbarriers, so every wait of the
// kernel stays bounded.
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

constexpr int kOffK = 0;
constexpr int kOffV = kOffK + kTileBytes;
constexpr int kOffQ = kOffV + kTileBytes;        // 2 stages
constexpr int kOffDO = kOffQ + 2 * kTileBytes;   // 2 stages
constexpr int kOffDS = kOffDO + 2 * kTileBytes;  // dS^T, bf16
constexpr int kOffLse = kOffDS + kTileBytes;     // 128 floats (log2 domain)
constexpr int kOffDlt = kOffLse + kT * 4;        // 128 floats
constexpr int kOffBar = kOffDlt + kT * 4;
constexpr int kBarKVFull = 0;
constexpr int kBarKVEmpty = 1;
constexpr int kBarQFull = 2;   // [2]
constexpr int kBarQEmpty = 4;  // [2]
constexpr int kBarS = 6;
constexpr int kBarDP = 7;
constexpr int kBarP = 8;
constexpr int kBarDS = 9;
constexpr int kBarDSFree = 10;
constexpr int kBarDQ = 11;
constexpr int kBarDQFree = 12;
constexpr int kBarAcc = 13;
constexpr int kBarAccFree = 14;
constexpr int kBarDrain = 15;
constexpr int kBarLseReady = 16;  // the elementwise warps staged this tile's LSE / Delta
constexpr int kBarLseFree = 17;   // ... and are done reading them
constexpr int kNumBars = 18;
constexpr int kOffMisc = kOffBar + kNumBars * 8;
constexpr int kSmemBytes = kOffMisc + 16 + 1024;

constexpr uint32_t kColS = 0, kColDP = 128, kColDV = 256, kColDK = 384;

constexpr uint32_t kIdescKK = idesc_bf16(128, 128, false, false);  // both K-major
constexpr uint32_t kIdescKM = idesc_bf16(128, 128, false, true);   // A K-major, B MN-major
constexpr uint32_t kIdescMM = idesc_bf16(128, 128, true, true);    // both MN-major

constexpr float kLog2e = 1.4426950408889634f;

struct Item {
  int b, h, g, s, kc, kt, kvrow;  // kc: natural chunk of the K/V tile, kt: its tile in the chunk
};

// Items in order of decreasing cost: earliest natural K/V tile first (it is
// seen by the most query tiles), (batch, query head) innermost so that the
// heads sharing one K/V tile run side by side.
__device__ __forceinline__ Item decode_item(const RingShape& sh, int idx) {
  const int BH = sh.B * sh.H;
  const int knat = idx / BH;
  const int bh = idx - knat * BH;
  Item it;
  it.b = bh / sh.H;
  it.h = bh - it.b * sh.H;
  it.g = it.h / (sh.H / sh.Hkv);
  const int nat0 = knat * kT;
  it.kc = nat0 / sh.c;
  const int loc = nat0 - it.kc * sh.c;
  int jj;
  if (sh.per_rank == 1 || it.kc < sh.cp) {
    it.s = it.kc;
    jj = 0;
  } else {
    it.s = 2 * sh.cp - 1 - it.kc;
    jj = 1;
  }
  it.kt = loc / kT;
  it.kvrow = it.s * sh.L + jj * sh.c + loc;
  return it;
}

// Query tiles of one head that see one K/V tile: ring steps t = 0..cp-1
// (receiving rank (s + t) mod cp), then that rank's chunks.
struct QSeq {
  int cp, per, L, c, ctiles, causal, s, kc, kt;
  int t, jq, qt;

  __device__ __forceinline__ void init(const RingShape& sh, const Item& it) {
    cp = sh.cp;
    per = sh.per_rank;
    L = sh.L;
    c = sh.c;
    ctiles = sh.c / kT;
    causal = sh.causal;
    s = it.s;
    kc = it.kc;
    kt = it.kt;
    t = 0;
    jq = 0;
    qt = 0;
  }

  __device__ __forceinline__ bool next(int& qrow, bool& diag) {
    while (t < cp) {
      const int r = (s + t) % cp;
      while (jq < per) {
        const int qc = (per == 1 || jq == 0) ? r : 2 * cp - 1 - r;
        int lo = 0, hi = ctiles;
        if (causal && qc == kc)
          lo = kt;  // from the diagonal tile on
        else if (causal && qc < kc)
          hi = 0;   // the whole chunk precedes this K/V: skipped
        if (qt < lo) qt = lo;
        if (qt < hi) {
          qrow = r * L + jq * c + qt * kT;
          diag = causal && qc == kc && qt == kt;
          ++qt;
          return true;
        }
        ++jq;
        qt = 0;
      }
      ++t;
      jq = 0;
    }
    return false;
  }
};

__device__ __forceinline__ int item_index(int k, int cta, int grid) {
  return k * grid + ((k & 1) ? (grid - 1 - cta) : cta);
}

__device__ __forceinline__ void fence_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__global__ void __launch_bounds__(kThreads, 1)
    tc_bwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                  const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                  const BwdArgs args, int n_items) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (base - raw);
  const uint32_t sK = base + kOffK, sV = base + kOffV, sQ = base + kOffQ, sDO = base + kOffDO;
  const uint32_t sDS = base + kOffDS;
  float* lse_s = reinterpret_cast<float*>(smem + kOffLse);
  float* dlt_s = reinterpret_cast<float*>(smem + kOffDlt);
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
    mbar_init(bar(kBarP), 128);
    mbar_init(bar(kBarDS), 128);
    mbar_init(bar(kBarDSFree), 1);
    mbar_init(bar(kBarDQ), 1);
    mbar_init(bar(kBarDQFree), 128);
    mbar_init(bar(kBarAcc), 1);
    mbar_init(bar(kBarAccFree), 128);
    mbar_init(bar(kBarDrain), 1);
    mbar_init(bar(kBarLseReady), 128);
    mbar_init(bar(kBarLseFree), 128);
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
        const Item it = decode_item(sh, idx);
        if (!mbar_wait(bar(kBarKVEmpty), (k & 1) ^ 1, wc)) {
          ok = false;
          break;
        }
        mbar_arrive_expect_tx(bar(kBarKVFull), 2 * kTileBytes);
        ++kv_armed;
        const int krow = it.b * sh.S + it.kvrow;
        for (int half = 0; half < 2; ++half) {
          tma_load_3d(sK + half * kBoxBytes, &tm_k, bar(kBarKVFull), half * 64, it.g, krow);
          tma_load_3d(sV + half * kBoxBytes, &tm_v, bar(kBarKVFull), half * 64, it.g, krow);
        }
        QSeq seq;
        seq.init(sh, it);
        const int h = it.h;
        int qrow;
        bool diag;
        while (seq.next(qrow, diag)) {
          const int st = qi & 1;
          const uint32_t ph = (qi >> 1) & 1;
          if (!mbar_wait(bar(kBarQEmpty + st), ph ^ 1, wc)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(bar(kBarQFull + st), 2 * kTileBytes);
          ++q_armed[st];
          const int row = it.b * sh.S + qrow;
          for (int half = 0; half < 2; ++half) {
            tma_load_3d(sQ + st * kTileBytes + half * kBoxBytes, &tm_q, bar(kBarQFull + st),
                        half * 64, h, row);
            tma_load_3d(sDO + st * kTileBytes + half * kBoxBytes, &tm_do, bar(kBarQFull + st),
                        half * 64, h, row);
          }
          ++qi;
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
    if (lane == 0) {
      uint32_t qi = 0, p_ph = 0, ds_ph = 0, dqf_ph = 1;
      bool ok = true;
      for (int k = 0; ok; ++k) {
        const int idx = item_index(k, blockIdx.x, gridDim.x);
        if (idx >= n_items) break;
        const Item it = decode_item(sh, idx);
        if (!mbar_wait(bar(kBarKVFull), k & 1, wc)) {
          ok = false;
          break;
        }
        tc_fence_after();
        QSeq seq;
        seq.init(sh, it);
        int qrow;
        bool diag;
        bool first = true;
        while (seq.next(qrow, diag)) {
          const int st = qi & 1;
          const uint32_t ph = (qi >> 1) & 1;
          const uint32_t q_s = sQ + st * kTileBytes, do_s = sDO + st * kTileBytes;
          if (!mbar_wait(bar(kBarQFull + st), ph, wc)) {
            ok = false;
            break;
          }
          tc_fence_after();
          // S^T = K Q^T
          for (int kk = 0; kk < kD / 16; ++kk) {
            const uint32_t off = (kk >> 2) * kBoxBytes + (kk & 3) * 32;
            mma_ss(tmem + kColS, sdesc_sw128(sK + off, 16, 1024), sdesc_sw128(q_s + off, 16, 1024),
                   kIdescKK, kk > 0);
          }
          mma_commit(bar(kBarS));
          // dP^T = V dO^T, once the previous dQ has left those columns.
          if (!mbar_wait(bar(kBarDQFree), dqf_ph, wc)) {
            ok = false;
            break;
          }
          dqf_ph ^= 1;
          tc_fence_after();
          for (int kk = 0; kk < kD / 16; ++kk) {
            const uint32_t off = (kk >> 2) * kBoxBytes + (kk & 3) * 32;
            mma_ss(tmem + kColDP, sdesc_sw128(sV + off, 16, 1024),
                   sdesc_sw128(do_s + off, 16, 1024), kIdescKK, kk > 0);
          }
          mma_commit(bar(kBarDP));
          // dV += P^T dO
          if (!mbar_wait(bar(kBarP), p_ph, wc)) {
            ok = false;
            break;
          }
          p_ph ^= 1;
          if (first && !mbar_wait(bar(kBarAccFree), (k & 1) ^ 1, wc)) {
            ok = false;
            break;
          }
          tc_fence_after();
          for (int kk = 0; kk < kT / 16; ++kk)
            mma_ts(tmem + kColDV, tmem + kColS + kk * 8,
                   sdesc_sw128(do_s + kk * 2048, kBoxBytes, 1024), kIdescKM,
                   (!first || kk > 0) ? 1u : 0u);
          // dK += dS^T Q ; dQ_t = dS K
          if (!mbar_wait(bar(kBarDS), ds_ph, wc)) {
            ok = false;
            break;
          }
          ds_ph ^= 1;
          tc_fence_after();
          for (int kk = 0; kk < kT / 16; ++kk) {
            const uint32_t off = (kk >> 2) * kBoxBytes + (kk & 3) * 32;
            mma_ss(tmem + kColDK, sdesc_sw128(sDS + off, 16, 1024),
                   sdesc_sw128(q_s + kk * 2048, kBoxBytes, 1024), kIdescKM,
                   (!first || kk > 0) ? 1u : 0u);
          }
          for (int kk = 0; kk < kT / 16; ++kk)
            mma_ss(tmem + kColDP, sdesc_sw128(sDS + kk * 2048, kBoxBytes, 1024),
                   sdesc_sw128(sK + kk * 2048, kBoxBytes, 1024), kIdescMM, kk > 0);
          mma_commit(bar(kBarDQ));
          mma_commit(bar(kBarQEmpty + st));
          mma_commit(bar(kBarDSFree));
          first = false;
          ++qi;
        }
        if (!ok) break;
        mma_commit(bar(kBarAcc));
        mma_commit(bar(kBarKVEmpty));
      }
      if (!ok) {
        mma_commit(bar(kBarDrain));
        mbar_drain(bar(kBarDrain), 0);
      }
    }
  } else if (warp >= 4 && warp < 8) {
    // ---------------------------------------------------------- elementwise
    const int wq = warp & 3;
    const int row = wq * 32 + lane;  // K/V row of the tile (TMEM lane); also the
                                     // query column whose LSE / Delta it stages
    const uint32_t tl = tmem + ((uint32_t)(wq * 32) << 16);
    const float sl2 = sh.scale_log2, scale = sh.scale;
    uint32_t s_ph = 0, dp_ph = 0, dsf_ph = 1, lr_ph = 0, lf_ph = 1;
    bool ok = true;
    for (int k = 0; ok; ++k) {
      const int idx = item_index(k, blockIdx.x, gridDim.x);
      if (idx >= n_items) break;
      const Item it = decode_item(sh, idx);
      QSeq seq;
      seq.init(sh, it);
      const int h = it.h;
      int qrow;
      bool diag;
      bool have = seq.next(qrow, diag);
      float cur_l = 0.f, cur_d = 0.f;
      if (have) {
        const int64_t li = ((int64_t)it.b * sh.H + h) * sh.S + qrow + row;
        cur_l = args.lse[li] * kLog2e;
        cur_d = args.delta[li];
      }
      while (have) {
        int nqrow = 0;
        bool ndiag = false;
        const bool nhave = seq.next(nqrow, ndiag);
        // Everyone is done with the previous tile's LSE / Delta ...
        if (!__all_sync(0xffffffffu, mbar_wait(bar(kBarLseFree), lf_ph, wc))) {
          ok = false;
          break;
        }
        lf_ph ^= 1;
        lse_s[row] = cur_l;
        dlt_s[row] = cur_d;
        // ... and everyone has staged this tile's.
        mbar_arrive(bar(kBarLseReady));
        if (!__all_sync(0xffffffffu, mbar_wait(bar(kBarLseReady), lr_ph, wc))) {
          ok = false;
          break;
        }
        lr_ph ^= 1;
        float nl = 0.f, nd = 0.f;
        if (nhave) {
          const int64_t li = ((int64_t)it.b * sh.H + h) * sh.S + nqrow + row;
          nl = args.lse[li] * kLog2e;
          nd = args.delta[li];
        }
        // P^T = exp2(S^T * scale*log2e - LSE*log2e), masked on the diagonal.
        if (!__all_sync(0xffffffffu, mbar_wait(bar(kBarS), s_ph, wc))) {
          ok = false;
          break;
        }
        s_ph ^= 1;
        tc_fence_after();
        uint32_t r[128];
        tmem_ld32(tl + kColS + 0, r + 0);
        tmem_ld32(tl + kColS + 32, r + 32);
        tmem_ld32(tl + kColS + 64, r + 64);
        tmem_ld32(tl + kColS + 96, r + 96);
        tmem_wait_ld_regs(r);
        reg_fence32(r + 32);
        reg_fence32(r + 64);
        reg_fence32(r + 96);
        uint32_t pk[64];
#pragma unroll
        for (int j = 0; j < 64; ++j) {
          const float2 l2 = *reinterpret_cast<const float2*>(lse_s + 2 * j);
          float p0 = ex2(fmaf(__uint_as_float(r[2 * j]), sl2, -l2.x));
          float p1 = ex2(fmaf(__uint_as_float(r[2 * j + 1]), sl2, -l2.y));
          if (diag) {
            if (2 * j < row) p0 = 0.f;
            if (2 * j + 1 < row) p1 = 0.f;
          }
          pk[j] = pack_bf16(p0, p1);
        }
        tmem_st32(tl + kColS + 0, pk);
        tmem_st32(tl + kColS + 32, pk + 32);
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(bar(kBarP));
        // dS^T = scale * P^T (dP^T - Delta) -> shared memory (bf16, swizzled)
        if (!__all_sync(0xffffffffu, mbar_wait(bar(kBarDP), dp_ph, wc))) {
          ok = false;
          break;
        }
        dp_ph ^= 1;
        if (!__all_sync(0xffffffffu, mbar_wait(bar(kBarDSFree), dsf_ph, wc))) {
          ok = false;
          break;
        }
        dsf_ph ^= 1;
        tc_fence_after();
        uint8_t* ds_row = smem + kOffDS + row * 128;
#pragma unroll
        for (int cc = 0; cc < 4; ++cc) {
          uint32_t d[32];
          tmem_ld32(tl + kColDP + cc * 32, d);
          tmem_wait_ld_regs(d);
          uint32_t w[16];
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const int col = cc * 32 + 2 * j;
            const float2 p = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&pk[col / 2]));
            const float2 dl = *reinterpret_cast<const float2*>(dlt_s + col);
            w[j] = pack_bf16(scale * p.x * (__uint_as_float(d[2 * j]) - dl.x),
                             scale * p.y * (__uint_as_float(d[2 * j + 1]) - dl.y));
          }
          const int box = cc >> 1;
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const int cb = (cc & 1) * 4 + u;  // 16-byte chunk within the 128-byte row
            uint4 v = make_uint4(w[4 * u], w[4 * u + 1], w[4 * u + 2], w[4 * u + 3]);
            *reinterpret_cast<uint4*>(ds_row + box * kBoxBytes + ((cb ^ (row & 7)) << 4)) = v;
          }
        }
        fence_async_smem();
        tc_fence_before();
        mbar_arrive(bar(kBarDS));
        mbar_arrive(bar(kBarLseFree));
        cur_l = nl;
        cur_d = nd;
        qrow = nqrow;
        diag = ndiag;
        have = nhave;
      }
    }
  } else if (warp >= 8) {
    // ------------------------------------------------ dQ reduction, dK / dV
    const int wq = warp & 3;
    const int lrow = wq * 32 + lane;  // TMEM lane: query row of dQ_t, K/V row of dK / dV
    const uint32_t tl = tmem + ((uint32_t)(wq * 32) << 16);
    uint32_t dq_ph = 0;
    bool ok = true;
    for (int k = 0; ok; ++k) {
      const int idx = item_index(k, blockIdx.x, gridDim.x);
      if (idx >= n_items) break;
      const Item it = decode_item(sh, idx);
      QSeq seq;
      seq.init(sh, it);
      const int h = it.h;
      int qrow;
      bool diag;
      while (seq.next(qrow, diag)) {
        if (!__all_sync(0xffffffffu, mbar_wait(bar(kBarDQ), dq_ph, wc))) {
          ok = false;
          break;
        }
        dq_ph ^= 1;
        tc_fence_after();
        float* dst = args.dq_acc + (((int64_t)it.b * sh.S + qrow + lrow) * sh.H + h) * kD;
#pragma unroll
        for (int cc = 0; cc < 4; ++cc) {
          uint32_t d[32];
          tmem_ld32(tl + kColDP + cc * 32, d);
          tmem_wait_ld_regs(d);
#pragma unroll
          for (int u = 0; u < 8; ++u)
            atomicAdd(reinterpret_cast<float4*>(dst + cc * 32 + 4 * u),
                      make_float4(__uint_as_float(d[4 * u]), __uint_as_float(d[4 * u + 1]),
                                  __uint_as_float(d[4 * u + 2]), __uint_as_float(d[4 * u + 3])));
        }
        tc_fence_before();
        mbar_arrive(bar(kBarDQFree));
      }
      if (!ok) break;
      if (!__all_sync(0xffffffffu, mbar_wait(bar(kBarAcc), k & 1, wc))) {
        ok = false;
        break;
      }
      tc_fence_after();
      const int64_t kbase = (((int64_t)it.b * sh.S + it.kvrow + lrow) * sh.Hkv + it.g) * kD;
#pragma unroll
      for (int which = 0; which < 2; ++which) {
        float* dst = (which == 0 ? args.dv_acc : args.dk_acc) + kbase;
        const uint32_t col = which == 0 ? kColDV : kColDK;
#pragma unroll
        for (int cc = 0; cc < 4; ++cc) {
          uint32_t d[32];
          tmem_ld32(tl + col + cc * 32, d);
          tmem_wait_ld_regs(d);
#pragma unroll
          for (int u = 0; u < 8; ++u)
            atomicAdd(reinterpret_cast<float4*>(dst + cc * 32 + 4 * u),
                      make_float4(__uint_as_float(d[4 * u]), __uint_as_float(d[4 * u + 1]),
                                  __uint_as_float(d[4 * u + 2]), __uint_as_float(d[4 * u + 3])));
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

}  // namespace

bool tc_bwd_available() { return true; }

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
  e = cudaFuncSetAttribute(tc_bwd_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
  if (e != cudaSuccess) return e;
  const int grid = n_items < sms ? n_items : sms;
  tc_bwd_kernel<<<grid, kThreads, kSmemBytes, stream>>>(mq, mk, mv, mdo, a, n_items);
  return cudaGetLastError();
}

}  // namespace cpattn
