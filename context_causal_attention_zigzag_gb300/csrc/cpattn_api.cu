// C-ABI layer of libcpattn: argument validation, kernel selection, the
// closed-form work census and the device error word.  Declarations and the
// meaning of every argument are in include/cpattn.h.
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>
#include <string.h>

#include "cpattn.h"
#include "cpattn_internal.h"

using namespace cpattn;

namespace {

// One error word per device, written by kernels whose bounded waits give up.
__device__ int g_device_error;

constexpr int kMaxDevices = 64;
int* g_err_ptr[kMaxDevices] = {nullptr};

int* device_error_word() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  if (g_err_ptr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_device_error) != cudaSuccess) return nullptr;
    g_err_ptr[dev] = static_cast<int*>(p);
  }
  return g_err_ptr[dev];
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

int chunks_per_rank(int layout) { return layout == CPATTN_LAYOUT_ZIGZAG ? 2 : 1; }

// Fills a RingShape; returns CPATTN_OK or CPATTN_ERR_INVALID_ARG.
int make_shape(int B, int H, int Hkv, int S, int D, int cp, int layout, int causal,
               float softmax_scale, RingShape* sh) {
  if (B < 0 || H < 1 || Hkv < 1 || S < 0 || cp < 1) return CPATTN_ERR_INVALID_ARG;
  if (H % Hkv != 0) return CPATTN_ERR_INVALID_ARG;
  if (D != 64 && D != 128) return CPATTN_ERR_INVALID_ARG;
  if (layout != CPATTN_LAYOUT_CONTIGUOUS && layout != CPATTN_LAYOUT_ZIGZAG)
    return CPATTN_ERR_INVALID_ARG;
  if (causal != 0 && causal != 1) return CPATTN_ERR_INVALID_ARG;
  const int per = chunks_per_rank(layout);
  if (S % (cp * per) != 0) return CPATTN_ERR_INVALID_ARG;
  if (!(softmax_scale <= 0.f) && !isfinite(softmax_scale)) return CPATTN_ERR_INVALID_ARG;
  sh->B = B;
  sh->H = H;
  sh->Hkv = Hkv;
  sh->S = S;
  sh->D = D;
  sh->cp = cp;
  sh->layout = layout;
  sh->causal = causal;
  sh->per_rank = per;
  sh->L = S / cp;
  sh->c = sh->L / per;
  sh->scale = softmax_scale > 0.f ? softmax_scale : 1.0f / sqrtf((float)D);
  sh->scale_log2 = sh->scale * 1.4426950408889634f;
  sh->docs = nullptr;
  sh->kv_natural = 0;
  const unsigned long long tpc = (unsigned long long)(sh->c / kTcTile);
  sh->tile_magic = (sh->c > 0 && sh->c % kTcTile == 0) ? ((1ull << 32) + tpc - 1) / tpc : 0;
  return CPATTN_OK;
}

// Document bounds as the kernels read them; NULL passes through, a pointer
// must be 8-byte aligned.
bool doc_ptr(const int32_t* bounds, const int2** out) {
  if (bounds != nullptr && (reinterpret_cast<uintptr_t>(bounds) & 7) != 0) return false;
  *out = reinterpret_cast<const int2*>(bounds);
  return true;
}

bool device_is_sm103() {
  int dev = 0, major = 0, minor = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return false;
  if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess)
    return false;
  if (cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
    return false;
  return major == 10 && minor == 3;
}

// Tensor-core forward: bf16, D = 128, every chunk a whole number of 256-row
// query pairs (two 128-row tiles share each K/V tile).  Both tensor-core
// paths take S < 2^23 (their tile walks find a tile's chunk with a multiply
// by RingShape::tile_magic, exact below that).
constexpr int kTcMaxS = 1 << 23;
bool tc_fwd_eligible(const RingShape& sh, int dtype) {
  return dtype == CPATTN_BF16 && sh.D == 128 && sh.c % (2 * kTcTile) == 0 && sh.S < kTcMaxS;
}
bool tc_bwd_eligible(const RingShape& sh, int dtype) {
  return dtype == CPATTN_BF16 && sh.D == 128 && sh.c % kTcTile == 0 && sh.S < kTcMaxS;
}

int fwd_common(const void* q, const void* k, const void* v, void* out, float* lse, int B, int H,
               int Hkv, int S, int D, int cp, int layout, int causal, int dtype,
               float softmax_scale, int t_begin, int t_end, int step_mode,
               unsigned long long* tiles_rt, const int2* docs, int kv_natural,
               cudaStream_t stream) {
  RingShape sh;
  int rc = make_shape(B, H, Hkv, S, D, cp, layout, causal, softmax_scale, &sh);
  if (rc != CPATTN_OK) return rc;
  sh.docs = docs;
  sh.kv_natural = kv_natural;
  if (dtype != CPATTN_F32 && dtype != CPATTN_BF16) return CPATTN_ERR_INVALID_ARG;
  if ((long long)B * S == 0) return CPATTN_OK;
  if (!q || !k || !v || !out || !lse) return CPATTN_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out) || !aligned16(lse))
    return CPATTN_ERR_INVALID_ARG;
  int* err = device_error_word();
  if (err == nullptr) return CPATTN_ERR_CUDA;
  FwdArgs a;
  a.sh = sh;
  a.q = q;
  a.k = k;
  a.v = v;
  a.out = out;
  a.lse = lse;
  a.t_begin = t_begin;
  a.t_end = t_end;
  a.step_mode = step_mode;
  a.tiles_rt = tiles_rt;
  a.err = err;
  cudaError_t e;
  if (tc_fwd_eligible(sh, dtype) && tc_fwd_available() && device_is_sm103())
    e = launch_tc_fwd(a, stream);
  else
    e = launch_simt_fwd(a, dtype, stream);
  return e == cudaSuccess ? CPATTN_OK : CPATTN_ERR_CUDA;
}

int plan_common(int B, int H, int Hkv, int S, int D, int cp, int layout, int causal, int dtype,
                bool fwd, int* path, int* tile) {
  RingShape sh;
  int rc = make_shape(B, H, Hkv, S, D, cp, layout, causal, 0.f, &sh);
  if (rc != CPATTN_OK) return rc;
  dtype &= fwd ? ~0 : ~kDtypeFlags;
  if (dtype != CPATTN_F32 && dtype != CPATTN_BF16) return CPATTN_ERR_INVALID_ARG;
  bool tc = fwd ? (tc_fwd_eligible(sh, dtype) && tc_fwd_available())
                : (tc_bwd_eligible(sh, dtype) && tc_bwd_available());
  if (path) *path = tc ? CPATTN_PATH_TCGEN05 : CPATTN_PATH_SIMT;
  if (tile) *tile = tc ? kTcTile : kSimtTile;
  return CPATTN_OK;
}

size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

// Sharded tensor [outer, S, inner]; natural tensor [outer, S_nat, inner].
int permute_common(const void* in, void* out, int64_t outer, int64_t S, int64_t S_nat,
                   int64_t inner_bytes, int cp_size, int layout, bool inverse,
                   cudaStream_t stream) {
  if (outer < 0 || S < 0 || S_nat < 0 || S_nat > S || inner_bytes < 1 || cp_size < 1)
    return CPATTN_ERR_INVALID_ARG;
  if (layout != CPATTN_LAYOUT_CONTIGUOUS && layout != CPATTN_LAYOUT_ZIGZAG)
    return CPATTN_ERR_INVALID_ARG;
  const int per = chunks_per_rank(layout);
  if (S % ((int64_t)cp_size * per) != 0 || S > INT32_MAX) return CPATTN_ERR_INVALID_ARG;
  if (outer * S == 0) return CPATTN_OK;
  if (!in || !out) return CPATTN_ERR_INVALID_ARG;
  const char* a = static_cast<const char*>(in);
  const char* b = static_cast<const char*>(out);
  const int64_t in_bytes = outer * (inverse ? S : S_nat) * inner_bytes;
  const int64_t out_bytes = outer * (inverse ? S_nat : S) * inner_bytes;
  if (a < b + out_bytes && b < a + in_bytes) return CPATTN_ERR_INVALID_ARG;
  RingShape sh;
  memset(&sh, 0, sizeof(sh));
  sh.cp = cp_size;
  sh.per_rank = per;
  sh.S = (int)S;
  sh.L = (int)(S / cp_size);
  sh.c = sh.L / per;
  cudaError_t e = launch_permute(in, out, outer, S, S_nat, inner_bytes, sh, inverse, stream);
  return e == cudaSuccess ? CPATTN_OK : CPATTN_ERR_CUDA;
}

}  // namespace

extern "C" {

int cpattn_zigzag_permute(const void* in, void* out, int64_t outer, int64_t S,
                          int64_t inner_bytes, int cp_size, int layout, cpattn_stream_t stream) {
  return permute_common(in, out, outer, S, S, inner_bytes, cp_size, layout, false,
                        (cudaStream_t)stream);
}

int cpattn_zigzag_unpermute(const void* in, void* out, int64_t outer, int64_t S,
                            int64_t inner_bytes, int cp_size, int layout, cpattn_stream_t stream) {
  return permute_common(in, out, outer, S, S, inner_bytes, cp_size, layout, true,
                        (cudaStream_t)stream);
}

int cpattn_zigzag_permute_pad(const void* in, void* out, int64_t outer, int64_t S_real,
                              int64_t S, int64_t inner_bytes, int cp_size, int layout,
                              cpattn_stream_t stream) {
  return permute_common(in, out, outer, S, S_real, inner_bytes, cp_size, layout, false,
                        (cudaStream_t)stream);
}

int cpattn_zigzag_unpermute_pad(const void* in, void* out, int64_t outer, int64_t S_real,
                                int64_t S, int64_t inner_bytes, int cp_size, int layout,
                                cpattn_stream_t stream) {
  return permute_common(in, out, outer, S, S_real, inner_bytes, cp_size, layout, true,
                        (cudaStream_t)stream);
}

int cpattn_ring_fwd(const void* q, const void* k, const void* v, void* out, float* lse, int B,
                    int H, int Hkv, int S, int D, int cp_size, int layout, int causal, int dtype,
                    float softmax_scale, cpattn_stream_t stream) {
  return fwd_common(q, k, v, out, lse, B, H, Hkv, S, D, cp_size, layout, causal, dtype,
                    softmax_scale, 0, cp_size, 0, nullptr, nullptr, 0, (cudaStream_t)stream);
}

int cpattn_doc_bounds(const int32_t* cu_seqlens, int ndocs, int S, int32_t* bounds,
                      cpattn_stream_t stream) {
  if (S < 0 || ndocs < 1 || ndocs > (S > 0 ? S : 1)) return CPATTN_ERR_INVALID_ARG;
  if (S == 0) return CPATTN_OK;
  if (!cu_seqlens || !bounds || (reinterpret_cast<uintptr_t>(bounds) & 7) != 0 ||
      (reinterpret_cast<uintptr_t>(cu_seqlens) & 3) != 0)
    return CPATTN_ERR_INVALID_ARG;
  int* err = device_error_word();
  if (err == nullptr) return CPATTN_ERR_CUDA;
  cudaError_t e = launch_doc_bounds(cu_seqlens, ndocs, S, reinterpret_cast<int2*>(bounds), err,
                                    (cudaStream_t)stream);
  return e == cudaSuccess ? CPATTN_OK : CPATTN_ERR_CUDA;
}

int cpattn_ring_fwd_docs(const void* q, const void* k, const void* v, void* out, float* lse,
                         int B, int H, int Hkv, int S, int D, int cp_size, int layout, int causal,
                         int dtype, float softmax_scale, const int32_t* doc_bounds,
                         unsigned long long* tiles_rt, cpattn_stream_t stream) {
  const int2* docs = nullptr;
  if (doc_bounds == nullptr || !doc_ptr(doc_bounds, &docs)) return CPATTN_ERR_INVALID_ARG;
  return fwd_common(q, k, v, out, lse, B, H, Hkv, S, D, cp_size, layout, causal, dtype,
                    softmax_scale, 0, cp_size, 0, tiles_rt, docs, 0, (cudaStream_t)stream);
}

int64_t cpattn_padded_length(int64_t S, int cp_size, int layout) {
  if (S < 0 || cp_size < 1) return -1;
  if (layout != CPATTN_LAYOUT_CONTIGUOUS && layout != CPATTN_LAYOUT_ZIGZAG) return -1;
  const int64_t unit = (int64_t)cp_size * chunks_per_rank(layout) * 2 * kTcTile;
  return (S + unit - 1) / unit * unit;
}

int cpattn_ring_fwd_census(const void* q, const void* k, const void* v, void* out, float* lse,
                           int B, int H, int Hkv, int S, int D, int cp_size, int layout,
                           int causal, int dtype, float softmax_scale,
                           unsigned long long* tiles_rt, cpattn_stream_t stream) {
  if (tiles_rt == nullptr) return CPATTN_ERR_INVALID_ARG;
  return fwd_common(q, k, v, out, lse, B, H, Hkv, S, D, cp_size, layout, causal, dtype,
                    softmax_scale, 0, cp_size, 0, tiles_rt, nullptr, 0, (cudaStream_t)stream);
}

int cpattn_ring_fwd_plan(int B, int H, int Hkv, int S, int D, int cp_size, int layout,
                         int causal, int dtype, int* path, int* tile) {
  return plan_common(B, H, Hkv, S, D, cp_size, layout, causal, dtype, true, path, tile);
}

int cpattn_ring_bwd_plan(int B, int H, int Hkv, int S, int D, int cp_size, int layout,
                         int causal, int dtype, int* path, int* tile) {
  return plan_common(B, H, Hkv, S, D, cp_size, layout, causal, dtype, false, path, tile);
}

int cpattn_ring_fwd_step(const void* q, const void* k, const void* v, int B, int H, int Hkv,
                         int S, int D, int cp_size, int layout, int causal, int dtype,
                         float softmax_scale, int step, float* o_part, float* lse_part,
                         cpattn_stream_t stream) {
  if (step < 0 || step >= cp_size) return CPATTN_ERR_INVALID_ARG;
  return fwd_common(q, k, v, o_part, lse_part, B, H, Hkv, S, D, cp_size, layout, causal, dtype,
                    softmax_scale, step, step + 1, 1, nullptr, nullptr, 0, (cudaStream_t)stream);
}

int cpattn_lse_merge(const float* o_a, const float* lse_a, const float* o_b, const float* lse_b,
                     float* o_out, float* lse_out, int B, int S, int H, int D,
                     cpattn_stream_t stream) {
  if (B < 0 || S < 0 || H < 0 || (D != 64 && D != 128)) return CPATTN_ERR_INVALID_ARG;
  if ((long long)B * S * H == 0) return CPATTN_OK;
  if (!o_a || !lse_a || !o_b || !lse_b || !o_out || !lse_out) return CPATTN_ERR_INVALID_ARG;
  if (!aligned16(o_a) || !aligned16(o_b) || !aligned16(o_out)) return CPATTN_ERR_INVALID_ARG;
  cudaError_t e = launch_lse_merge(o_a, lse_a, o_b, lse_b, o_out, lse_out, B, S, H, D,
                                   (cudaStream_t)stream);
  return e == cudaSuccess ? CPATTN_OK : CPATTN_ERR_CUDA;
}

size_t cpattn_ring_bwd_workspace_bytes(int B, int H, int Hkv, int S, int D, int dtype) {
  (void)dtype;
  if (B < 0 || H < 0 || Hkv < 0 || S < 0 || D < 0) return 0;
  (void)Hkv;
  const size_t q = (size_t)B * S * H * D * sizeof(float);
  const size_t delta = (size_t)B * H * S * sizeof(float);
  return 3 * align256(q) + align256(delta);
}

}  // extern "C"

namespace {

int bwd_common(const void* q, const void* k, const void* v, const void* out, const void* dout,
               const float* lse, void* dq, void* dk, void* dv, int B, int H, int Hkv, int S,
               int D, int cp_size, int layout, int causal, int dtype, float softmax_scale,
               const int2* docs, int kv_natural, void* workspace, size_t workspace_bytes,
               cudaStream_t st, unsigned long long* tiles_kv_rt = nullptr,
               unsigned long long* tiles_q_rt = nullptr) {
  RingShape sh;
  int rc = make_shape(B, H, Hkv, S, D, cp_size, layout, causal, softmax_scale, &sh);
  if (rc != CPATTN_OK) return rc;
  sh.docs = docs;
  sh.kv_natural = kv_natural;
  const int in_dtype = dtype & ~kDtypeFlags;
  if (in_dtype != CPATTN_F32 && in_dtype != CPATTN_BF16) return CPATTN_ERR_INVALID_ARG;
  const int out_dtype = (dtype & CPATTN_GRAD_F32) ? CPATTN_F32 : in_dtype;
  if ((long long)B * S == 0) return CPATTN_OK;
  if (!q || !k || !v || !out || !dout || !lse || !dq || !dk || !dv) return CPATTN_ERR_INVALID_ARG;
  const void* ptrs[] = {q, k, v, out, dout, lse, dq, dk, dv};
  for (const void* p : ptrs)
    if (!aligned16(p)) return CPATTN_ERR_INVALID_ARG;
  const size_t need = cpattn_ring_bwd_workspace_bytes(B, H, Hkv, S, D, dtype);
  if (workspace == nullptr || workspace_bytes < need ||
      (reinterpret_cast<uintptr_t>(workspace) & 255) != 0)
    return CPATTN_ERR_WORKSPACE;
  int* err = device_error_word();
  if (err == nullptr) return CPATTN_ERR_CUDA;
  const int64_t n_q = (int64_t)B * S * H * D, n_kv = (int64_t)B * S * Hkv * D;
  // Workspace: three float32 regions of n_q elements, then Delta [B,H,S].
  // Tensor cores: the per-query-head dK / dV partials, and the one-pass
  // kernel's dQ accumulator for non-float32 outputs.  CUDA cores: the dQ,
  // dK, dV accumulators.
  char* ws = static_cast<char*>(workspace);
  float* reg_a = reinterpret_cast<float*>(ws);
  ws += align256((size_t)n_q * sizeof(float));
  float* reg_b = reinterpret_cast<float*>(ws);
  ws += align256((size_t)n_q * sizeof(float));
  float* reg_c = reinterpret_cast<float*>(ws);
  ws += align256((size_t)n_q * sizeof(float));
  float* delta = reinterpret_cast<float*>(ws);
  const bool tc = tc_bwd_eligible(sh, in_dtype) && tc_bwd_available() && device_is_sm103();
  BwdArgs a;
  memset(&a, 0, sizeof(a));
  a.sh = sh;
  a.q = q;
  a.k = k;
  a.v = v;
  a.dout = dout;
  a.lse = lse;
  a.delta = delta;
  a.err = err;
  a.tiles_kv_rt = tiles_kv_rt;
  a.tiles_q_rt = tiles_q_rt;
  cudaError_t e;
  if (tc && (dtype & CPATTN_BWD_ONEPASS)) {
    // One pass: Delta and a zeroed float32 dQ accumulator (the output itself
    // for float32 gradients), the one-pass kernel, the per-group sum of
    // dK / dV, and for bf16 gradients the conversion of dQ.
    float* dq_acc = out_dtype == CPATTN_F32 ? static_cast<float*>(dq) : reg_c;
    e = launch_bwd_prep(out, dout, delta, dq_acc, nullptr, nullptr, 0, B, S, H, D, in_dtype,
                        sh.scale, st);
    if (e != cudaSuccess) return CPATTN_ERR_CUDA;
    a.dk_part = reg_a;
    a.dv_part = reg_b;
    a.dq_acc = dq_acc;
    e = launch_tc_bwd_onepass(a, st);
    if (e != cudaSuccess) return CPATTN_ERR_CUDA;
    e = launch_grad_reduce(reg_a, reg_b, dk, dv, B, S, H, Hkv, D, out_dtype, st);
    if (e != cudaSuccess) return CPATTN_ERR_CUDA;
    if (out_dtype != CPATTN_F32)
      e = launch_grad_convert(dq_acc, nullptr, nullptr, dq, nullptr, nullptr, n_q, 0, out_dtype,
                              st);
    return e == cudaSuccess ? CPATTN_OK : CPATTN_ERR_CUDA;
  }
  if (tc) {
    // Tensor cores: Delta only, then the dK/dV and dQ kernels (every output
    // element written exactly once), then the per-group sum of dK / dV.
    e = launch_bwd_prep(out, dout, delta, nullptr, nullptr, nullptr, 0, B, S, H, D, in_dtype,
                        sh.scale, st);
    if (e != cudaSuccess) return CPATTN_ERR_CUDA;
    a.dk_part = reg_a;
    a.dv_part = reg_b;
    a.dq = dq;
    a.dq_f32 = out_dtype == CPATTN_F32;
    e = launch_tc_bwd(a, st);
    if (e != cudaSuccess) return CPATTN_ERR_CUDA;
    e = launch_grad_reduce(reg_a, reg_b, dk, dv, B, S, H, Hkv, D, out_dtype, st);
    return e == cudaSuccess ? CPATTN_OK : CPATTN_ERR_CUDA;
  }
  // CUDA cores: Delta, the dK/dV and dQ kernels (every accumulator element
  // written once), the conversion.
  e = launch_bwd_prep(out, dout, delta, nullptr, nullptr, nullptr, 0, B, S, H, D, in_dtype, 1.f,
                      st);
  if (e != cudaSuccess) return CPATTN_ERR_CUDA;
  a.dq_acc = reg_a;
  a.dk_acc = reg_b;
  a.dv_acc = reg_c;
  e = launch_simt_bwd(a, in_dtype, st);
  if (e != cudaSuccess) return CPATTN_ERR_CUDA;
  e = launch_grad_convert(reg_a, reg_b, reg_c, dq, dk, dv, n_q, n_kv, out_dtype, st);
  return e == cudaSuccess ? CPATTN_OK : CPATTN_ERR_CUDA;
}

// Sequence <-> head all-to-all schedules.  The hierarchical (a2a+p2p)
// schedule has level sizes [A, P], cp = A * P: an all-to-all inside groups
// of A consecutive ranks, then the ring of the second level over the P
// groups.  The Ulysses variant is its one-level case [cp, 1] (the ring is
// then a single rank attending to the whole sequence).
struct A2aPlan {
  RingShape sh;     // the sequence owners: cp = A * P ranks, the caller's layout
  RingShape inner;  // the second level's order on the head owners' side
  int A, P;
  int hc, nkv;      // query heads and kv heads per head owner
  int inner_layout;
};

int a2a_plan(int B, int H, int Hkv, int S, int D, int A, int P, int layout, A2aPlan* pl) {
  if (A < 1 || P < 1 || (long long)A * P > (1 << 20)) return CPATTN_ERR_INVALID_ARG;
  int rc = make_shape(B, H, Hkv, S, D, A * P, layout, 1, 0.f, &pl->sh);
  if (rc != CPATTN_OK) return rc;
  if (H % A != 0) return CPATTN_ERR_INVALID_ARG;
  const int h = H / A, grp = H / Hkv;
  if (h % grp != 0 && grp % h != 0) return CPATTN_ERR_INVALID_ARG;
  // With one group of the second level the ring is one rank: keep the
  // sequence in natural order.
  pl->inner_layout = P == 1 ? CPATTN_LAYOUT_CONTIGUOUS : layout;
  rc = make_shape(B, H, Hkv, S, D, P, pl->inner_layout, 1, 0.f, &pl->inner);
  if (rc != CPATTN_OK) return rc;
  pl->A = A;
  pl->P = P;
  pl->hc = h;
  pl->nkv = h >= grp ? h / grp : 1;
  return CPATTN_OK;
}

A2aShape a2a_shape(const A2aPlan& pl, int B, int H, int Hkv, bool kv) {
  A2aShape a;
  a.sh = pl.sh;
  a.inner = pl.inner;
  a.ranks = pl.A;
  a.B = B;
  a.D = pl.sh.D;
  a.X = kv ? Hkv : H;
  a.nx = kv ? pl.nkv : pl.hc;
  a.x_num = pl.hc;
  a.x_den = kv ? H / Hkv : 1;
  return a;
}

struct A2aWs {
  size_t q, kv, lse, grad_q, grad_kv, inner, total;
};

A2aWs a2a_ws(const A2aPlan& pl, int B, int H, int S, int D, int dtype, bool backward) {
  A2aWs w;
  const int in_dtype = dtype & ~kDtypeFlags;
  const size_t elt = in_dtype == CPATTN_BF16 ? 2 : 4;
  const size_t gelt = (dtype & CPATTN_GRAD_F32) ? 4 : elt;
  const size_t rows = (size_t)pl.A * B * S;
  w.q = align256(rows * pl.hc * D * elt);
  w.kv = align256(rows * pl.nkv * D * elt);
  w.lse = align256((size_t)B * H * S * sizeof(float));
  w.grad_q = backward ? align256(rows * pl.hc * D * gelt) : 0;
  w.grad_kv = backward ? align256(rows * pl.nkv * D * gelt) : 0;
  w.inner = backward ? align256(cpattn_ring_bwd_workspace_bytes(pl.A * B, pl.hc, pl.nkv, S, D,
                                                                dtype))
                     : 0;
  // q-like: q, o (+ dO, dQ); kv-like: k, v (+ dK, dV)
  w.total = (backward ? 3 : 2) * w.q + 2 * w.kv + w.lse + w.grad_q + 2 * w.grad_kv + w.inner;
  return w;
}

int a2a_copy(const void* in, void* out, int B, int S, int H, int Hkv, int D, int A, int P,
             int layout, int kv_heads, int to_seq, int dtype, cudaStream_t stream) {
  A2aPlan pl;
  int rc = a2a_plan(B, H, Hkv, S, D, A, P, layout, &pl);
  if (rc != CPATTN_OK) return rc;
  if ((dtype != CPATTN_F32 && dtype != CPATTN_BF16) || (kv_heads != 0 && kv_heads != 1) ||
      (to_seq != 0 && to_seq != 1))
    return CPATTN_ERR_INVALID_ARG;
  if ((long long)B * S == 0) return CPATTN_OK;
  if (!in || !out || !aligned16(in) || !aligned16(out)) return CPATTN_ERR_INVALID_ARG;
  const A2aShape a = a2a_shape(pl, B, H, Hkv, kv_heads != 0);
  const size_t elt = dtype == CPATTN_BF16 ? 2 : 4;
  const size_t big = (size_t)A * B * S * a.nx * D * elt;
  const size_t small = (size_t)B * S * a.X * D * elt;
  const char* x = static_cast<const char*>(in);
  const char* y = static_cast<const char*>(out);
  const size_t in_b = to_seq ? big : small, out_b = to_seq ? small : big;
  if (x < y + out_b && y < x + in_b) return CPATTN_ERR_INVALID_ARG;
  cudaError_t e = launch_a2a(in, out, a, to_seq != 0, dtype, stream);
  return e == cudaSuccess ? CPATTN_OK : CPATTN_ERR_CUDA;
}

int a2a_lse_copy(const float* in, float* out, int B, int S, int H, int A, int P, int layout,
                 int to_seq, cudaStream_t stream) {
  A2aPlan pl;
  int rc = a2a_plan(B, H, H, S, 64, A, P, layout, &pl);
  if (rc != CPATTN_OK) return rc;
  if (to_seq != 0 && to_seq != 1) return CPATTN_ERR_INVALID_ARG;
  if ((long long)B * S == 0) return CPATTN_OK;
  if (!in || !out) return CPATTN_ERR_INVALID_ARG;
  const size_t bytes = (size_t)B * H * S * sizeof(float);
  const char* x = reinterpret_cast<const char*>(in);
  const char* y = reinterpret_cast<const char*>(out);
  if (x < y + bytes && y < x + bytes) return CPATTN_ERR_INVALID_ARG;
  cudaError_t e = launch_lse_a2a(in, out, pl.sh, pl.inner, A, B, H, to_seq != 0, stream);
  return e == cudaSuccess ? CPATTN_OK : CPATTN_ERR_CUDA;
}

size_t a2a_workspace_bytes(int B, int H, int Hkv, int S, int D, int A, int P, int layout,
                           int dtype, int backward) {
  A2aPlan pl;
  if (a2a_plan(B, H, Hkv, S, D, A, P, layout, &pl) != CPATTN_OK) return 0;
  return a2a_ws(pl, B, H, S, D, dtype, backward != 0).total;
}

// All-to-all to the head owners, the ring of the second level on every head
// owner's slice in ONE launch of the ring kernels (the head owners stacked
// along the batch axis, cp = P), all-to-all back.
int a2a_fwd(const void* q, const void* k, const void* v, void* out, float* lse, int B, int H,
            int Hkv, int S, int D, int A, int P, int layout, int causal, int dtype,
            float softmax_scale, const int32_t* doc_bounds, void* workspace,
            size_t workspace_bytes, cudaStream_t st) {
  A2aPlan pl;
  int rc = a2a_plan(B, H, Hkv, S, D, A, P, layout, &pl);
  if (rc != CPATTN_OK) return rc;
  if (dtype != CPATTN_F32 && dtype != CPATTN_BF16) return CPATTN_ERR_INVALID_ARG;
  if (causal != 0 && causal != 1) return CPATTN_ERR_INVALID_ARG;
  if ((long long)B * S == 0) return CPATTN_OK;
  if (!q || !k || !v || !out || !lse) return CPATTN_ERR_INVALID_ARG;
  const int2* docs = nullptr;
  if (!doc_ptr(doc_bounds, &docs)) return CPATTN_ERR_INVALID_ARG;
  const A2aWs w = a2a_ws(pl, B, H, S, D, dtype, false);
  if (workspace == nullptr || workspace_bytes < w.total ||
      (reinterpret_cast<uintptr_t>(workspace) & 255) != 0)
    return CPATTN_ERR_WORKSPACE;
  char* p = static_cast<char*>(workspace);
  void* wq = p;
  void* wo = p + w.q;
  void* wk = p + 2 * w.q;
  void* wv = p + 2 * w.q + w.kv;
  float* wl = reinterpret_cast<float*>(p + 2 * w.q + 2 * w.kv);
  rc = a2a_copy(q, wq, B, S, H, Hkv, D, A, P, layout, 0, 0, dtype, st);
  if (rc == CPATTN_OK) rc = a2a_copy(k, wk, B, S, H, Hkv, D, A, P, layout, 1, 0, dtype, st);
  if (rc == CPATTN_OK) rc = a2a_copy(v, wv, B, S, H, Hkv, D, A, P, layout, 1, 0, dtype, st);
  if (rc != CPATTN_OK) return rc;
  rc = fwd_common(wq, wk, wv, wo, wl, A * B, pl.hc, pl.nkv, S, D, P, pl.inner_layout, causal,
                  dtype, softmax_scale, 0, P, 0, nullptr, docs, 0, st);
  if (rc != CPATTN_OK) return rc;
  rc = a2a_copy(wo, out, B, S, H, Hkv, D, A, P, layout, 0, 1, dtype, st);
  if (rc != CPATTN_OK) return rc;
  return a2a_lse_copy(wl, lse, B, S, H, A, P, layout, 1, st);
}

int a2a_bwd(const void* q, const void* k, const void* v, const void* out, const void* dout,
            const float* lse, void* dq, void* dk, void* dv, int B, int H, int Hkv, int S, int D,
            int A, int P, int layout, int causal, int dtype, float softmax_scale,
            const int32_t* doc_bounds, void* workspace, size_t workspace_bytes,
            cudaStream_t st) {
  A2aPlan pl;
  int rc = a2a_plan(B, H, Hkv, S, D, A, P, layout, &pl);
  if (rc != CPATTN_OK) return rc;
  const int in_dtype = dtype & ~kDtypeFlags;
  if (in_dtype != CPATTN_F32 && in_dtype != CPATTN_BF16) return CPATTN_ERR_INVALID_ARG;
  const int out_dtype = (dtype & CPATTN_GRAD_F32) ? CPATTN_F32 : in_dtype;
  if (causal != 0 && causal != 1) return CPATTN_ERR_INVALID_ARG;
  if ((long long)B * S == 0) return CPATTN_OK;
  if (!q || !k || !v || !out || !dout || !lse || !dq || !dk || !dv) return CPATTN_ERR_INVALID_ARG;
  const int2* docs = nullptr;
  if (!doc_ptr(doc_bounds, &docs)) return CPATTN_ERR_INVALID_ARG;
  const A2aWs w = a2a_ws(pl, B, H, S, D, dtype, true);
  if (workspace == nullptr || workspace_bytes < w.total ||
      (reinterpret_cast<uintptr_t>(workspace) & 255) != 0)
    return CPATTN_ERR_WORKSPACE;
  char* p = static_cast<char*>(workspace);
  void* wq = p;
  void* wo = p + w.q;
  void* wdo = p + 2 * w.q;
  void* wk = p + 3 * w.q;
  void* wv = p + 3 * w.q + w.kv;
  float* wl = reinterpret_cast<float*>(p + 3 * w.q + 2 * w.kv);
  char* g = p + 3 * w.q + 2 * w.kv + w.lse;
  void* wdq = g;
  void* wdk = g + w.grad_q;
  void* wdv = g + w.grad_q + w.grad_kv;
  void* inner = g + w.grad_q + 2 * w.grad_kv;
  const void* src_q[3] = {q, out, dout};
  void* dst_q[3] = {wq, wo, wdo};
  for (int i = 0; i < 3 && rc == CPATTN_OK; ++i)
    rc = a2a_copy(src_q[i], dst_q[i], B, S, H, Hkv, D, A, P, layout, 0, 0, in_dtype, st);
  if (rc == CPATTN_OK) rc = a2a_copy(k, wk, B, S, H, Hkv, D, A, P, layout, 1, 0, in_dtype, st);
  if (rc == CPATTN_OK) rc = a2a_copy(v, wv, B, S, H, Hkv, D, A, P, layout, 1, 0, in_dtype, st);
  if (rc == CPATTN_OK) rc = a2a_lse_copy(lse, wl, B, S, H, A, P, layout, 0, st);
  if (rc != CPATTN_OK) return rc;
  rc = bwd_common(wq, wk, wv, wo, wdo, wl, wdq, wdk, wdv, A * B, pl.hc, pl.nkv, S, D, P,
                  pl.inner_layout, causal, dtype, softmax_scale, docs, 0, inner, w.inner, st);
  if (rc != CPATTN_OK) return rc;
  // Back to the sequence owners; a kv head held by several head owners gets
  // the sum of their dK / dV.
  rc = a2a_copy(wdq, dq, B, S, H, Hkv, D, A, P, layout, 0, 1, out_dtype, st);
  if (rc == CPATTN_OK) rc = a2a_copy(wdk, dk, B, S, H, Hkv, D, A, P, layout, 1, 1, out_dtype, st);
  if (rc == CPATTN_OK) rc = a2a_copy(wdv, dv, B, S, H, Hkv, D, A, P, layout, 1, 1, out_dtype, st);
  return rc;
}

}  // namespace

extern "C" {

int cpattn_ulysses_a2a(const void* in, void* out, int B, int S, int H, int Hkv, int D,
                       int cp_size, int layout, int kv_heads, int to_seq, int dtype,
                       cpattn_stream_t stream) {
  return a2a_copy(in, out, B, S, H, Hkv, D, cp_size, 1, layout, kv_heads, to_seq, dtype,
                  (cudaStream_t)stream);
}

int cpattn_ulysses_lse_a2a(const float* in, float* out, int B, int S, int H, int cp_size,
                           int layout, int to_seq, cpattn_stream_t stream) {
  return a2a_lse_copy(in, out, B, S, H, cp_size, 1, layout, to_seq, (cudaStream_t)stream);
}

size_t cpattn_ulysses_workspace_bytes(int B, int H, int Hkv, int S, int D, int cp_size,
                                      int layout, int dtype, int backward) {
  return a2a_workspace_bytes(B, H, Hkv, S, D, cp_size, 1, layout, dtype, backward);
}

int cpattn_ulysses_fwd(const void* q, const void* k, const void* v, void* out, float* lse,
                       int B, int H, int Hkv, int S, int D, int cp_size, int layout, int causal,
                       int dtype, float softmax_scale, const int32_t* doc_bounds,
                       void* workspace, size_t workspace_bytes, cpattn_stream_t stream) {
  return a2a_fwd(q, k, v, out, lse, B, H, Hkv, S, D, cp_size, 1, layout, causal, dtype,
                 softmax_scale, doc_bounds, workspace, workspace_bytes, (cudaStream_t)stream);
}

int cpattn_ulysses_bwd(const void* q, const void* k, const void* v, const void* out,
                       const void* dout, const float* lse, void* dq, void* dk, void* dv, int B,
                       int H, int Hkv, int S, int D, int cp_size, int layout, int causal,
                       int dtype, float softmax_scale, const int32_t* doc_bounds,
                       void* workspace, size_t workspace_bytes, cpattn_stream_t stream) {
  return a2a_bwd(q, k, v, out, dout, lse, dq, dk, dv, B, H, Hkv, S, D, cp_size, 1, layout,
                 causal, dtype, softmax_scale, doc_bounds, workspace, workspace_bytes,
                 (cudaStream_t)stream);
}

int cpattn_hier_a2a(const void* in, void* out, int B, int S, int H, int Hkv, int D, int cp_a2a,
                    int cp_p2p, int layout, int kv_heads, int to_seq, int dtype,
                    cpattn_stream_t stream) {
  return a2a_copy(in, out, B, S, H, Hkv, D, cp_a2a, cp_p2p, layout, kv_heads, to_seq, dtype,
                  (cudaStream_t)stream);
}

int cpattn_hier_lse_a2a(const float* in, float* out, int B, int S, int H, int cp_a2a,
                        int cp_p2p, int layout, int to_seq, cpattn_stream_t stream) {
  return a2a_lse_copy(in, out, B, S, H, cp_a2a, cp_p2p, layout, to_seq, (cudaStream_t)stream);
}

size_t cpattn_hier_workspace_bytes(int B, int H, int Hkv, int S, int D, int cp_a2a, int cp_p2p,
                                   int layout, int dtype, int backward) {
  return a2a_workspace_bytes(B, H, Hkv, S, D, cp_a2a, cp_p2p, layout, dtype, backward);
}

int cpattn_hier_fwd(const void* q, const void* k, const void* v, void* out, float* lse, int B,
                    int H, int Hkv, int S, int D, int cp_a2a, int cp_p2p, int layout, int causal,
                    int dtype, float softmax_scale, const int32_t* doc_bounds, void* workspace,
                    size_t workspace_bytes, cpattn_stream_t stream) {
  return a2a_fwd(q, k, v, out, lse, B, H, Hkv, S, D, cp_a2a, cp_p2p, layout, causal, dtype,
                 softmax_scale, doc_bounds, workspace, workspace_bytes, (cudaStream_t)stream);
}

int cpattn_hier_bwd(const void* q, const void* k, const void* v, const void* out,
                    const void* dout, const float* lse, void* dq, void* dk, void* dv, int B,
                    int H, int Hkv, int S, int D, int cp_a2a, int cp_p2p, int layout, int causal,
                    int dtype, float softmax_scale, const int32_t* doc_bounds, void* workspace,
                    size_t workspace_bytes, cpattn_stream_t stream) {
  return a2a_bwd(q, k, v, out, dout, lse, dq, dk, dv, B, H, Hkv, S, D, cp_a2a, cp_p2p, layout,
                 causal, dtype, softmax_scale, doc_bounds, workspace, workspace_bytes,
                 (cudaStream_t)stream);
}

int cpattn_ring_bwd(const void* q, const void* k, const void* v, const void* out,
                    const void* dout, const float* lse, void* dq, void* dk, void* dv, int B,
                    int H, int Hkv, int S, int D, int cp_size, int layout, int causal, int dtype,
                    float softmax_scale, void* workspace, size_t workspace_bytes,
                    cpattn_stream_t stream) {
  return bwd_common(q, k, v, out, dout, lse, dq, dk, dv, B, H, Hkv, S, D, cp_size, layout, causal,
                    dtype, softmax_scale, nullptr, 0, workspace, workspace_bytes,
                    (cudaStream_t)stream);
}

int cpattn_ring_bwd_census(const void* q, const void* k, const void* v, const void* out,
                           const void* dout, const float* lse, void* dq, void* dk, void* dv,
                           int B, int H, int Hkv, int S, int D, int cp_size, int layout,
                           int causal, int dtype, float softmax_scale, void* workspace,
                           size_t workspace_bytes, unsigned long long* tiles_kv_rt,
                           unsigned long long* tiles_q_rt, cpattn_stream_t stream) {
  if (tiles_kv_rt == nullptr || tiles_q_rt == nullptr) return CPATTN_ERR_INVALID_ARG;
  return bwd_common(q, k, v, out, dout, lse, dq, dk, dv, B, H, Hkv, S, D, cp_size, layout, causal,
                    dtype, softmax_scale, nullptr, 0, workspace, workspace_bytes,
                    (cudaStream_t)stream, tiles_kv_rt, tiles_q_rt);
}

int cpattn_ring_bwd_docs(const void* q, const void* k, const void* v, const void* out,
                         const void* dout, const float* lse, void* dq, void* dk, void* dv, int B,
                         int H, int Hkv, int S, int D, int cp_size, int layout, int causal,
                         int dtype, float softmax_scale, const int32_t* doc_bounds,
                         void* workspace, size_t workspace_bytes, cpattn_stream_t stream) {
  const int2* docs = nullptr;
  if (doc_bounds == nullptr || !doc_ptr(doc_bounds, &docs)) return CPATTN_ERR_INVALID_ARG;
  return bwd_common(q, k, v, out, dout, lse, dq, dk, dv, B, H, Hkv, S, D, cp_size, layout, causal,
                    dtype, softmax_scale, docs, 0, workspace, workspace_bytes,
                    (cudaStream_t)stream);
}

int cpattn_allgather_fwd(const void* q, const void* k_full, const void* v_full, void* out,
                         float* lse, int B, int H, int Hkv, int S, int D, int cp_size, int layout,
                         int causal, int dtype, float softmax_scale, const int32_t* doc_bounds,
                         unsigned long long* tiles_rt, cpattn_stream_t stream) {
  const int2* docs = nullptr;
  if (!doc_ptr(doc_bounds, &docs)) return CPATTN_ERR_INVALID_ARG;
  return fwd_common(q, k_full, v_full, out, lse, B, H, Hkv, S, D, cp_size, layout, causal, dtype,
                    softmax_scale, 0, cp_size, 0, tiles_rt, docs, 1, (cudaStream_t)stream);
}

int cpattn_allgather_bwd(const void* q, const void* k_full, const void* v_full, const void* out,
                         const void* dout, const float* lse, void* dq, void* dk_full,
                         void* dv_full, int B, int H, int Hkv, int S, int D, int cp_size,
                         int layout, int causal, int dtype, float softmax_scale,
                         const int32_t* doc_bounds, void* workspace, size_t workspace_bytes,
                         cpattn_stream_t stream) {
  const int2* docs = nullptr;
  if (!doc_ptr(doc_bounds, &docs)) return CPATTN_ERR_INVALID_ARG;
  return bwd_common(q, k_full, v_full, out, dout, lse, dq, dk_full, dv_full, B, H, Hkv, S, D,
                    cp_size, layout, causal, dtype, softmax_scale, docs, 1, workspace,
                    workspace_bytes, (cudaStream_t)stream);
}

int cpattn_tile_counts(int64_t S, int cp_size, int layout, int causal, int64_t tile,
                       uint64_t* tiles_rt, uint64_t* pairs_rt) {
  if (S < 0 || cp_size < 1 || tile < 1) return CPATTN_ERR_INVALID_ARG;
  if (layout != CPATTN_LAYOUT_CONTIGUOUS && layout != CPATTN_LAYOUT_ZIGZAG)
    return CPATTN_ERR_INVALID_ARG;
  const int per = chunks_per_rank(layout);
  if (S % ((int64_t)cp_size * per) != 0) return CPATTN_ERR_INVALID_ARG;
  const int64_t c = S / ((int64_t)cp_size * per);
  if (c % tile != 0) return CPATTN_ERR_INVALID_ARG;
  const uint64_t n = (uint64_t)(c / tile);
  const uint64_t cc = (uint64_t)c;
  // Chunk-pair arithmetic: a key chunk earlier than the query chunk is fully
  // visible (n^2 tiles, c^2 pairs), the same chunk is a triangle with its
  // diagonal (n(n+1)/2 tiles, c(c+1)/2 pairs), a later chunk is skipped.
  for (int r = 0; r < cp_size; ++r) {
    for (int t = 0; t < cp_size; ++t) {
      int s = ((r - t) % cp_size + cp_size) % cp_size;
      uint64_t tiles = 0, pairs = 0;
      for (int jq = 0; jq < per; ++jq) {
        int qc = (per == 1 || jq == 0) ? r : 2 * cp_size - 1 - r;
        for (int jk = 0; jk < per; ++jk) {
          int kc = (per == 1 || jk == 0) ? s : 2 * cp_size - 1 - s;
          if (!causal || kc < qc) {
            tiles += n * n;
            pairs += cc * cc;
          } else if (kc == qc) {
            tiles += n * (n + 1) / 2;
            pairs += cc * (cc + 1) / 2;
          }
        }
      }
      if (tiles_rt) tiles_rt[r * cp_size + t] = tiles;
      if (pairs_rt) pairs_rt[r * cp_size + t] = pairs;
    }
  }
  return CPATTN_OK;
}

int cpattn_wait_probe(int64_t limit_ns, cpattn_stream_t stream) {
  if (limit_ns < 1 || limit_ns > 2000000000LL) return CPATTN_ERR_INVALID_ARG;
  int* err = device_error_word();
  if (err == nullptr) return CPATTN_ERR_CUDA;
  cudaError_t e = launch_wait_probe(err, (uint64_t)limit_ns, (cudaStream_t)stream);
  return e == cudaSuccess ? CPATTN_OK : CPATTN_ERR_CUDA;
}

int cpattn_device_status(cpattn_stream_t stream) {
  cudaError_t e = cudaStreamSynchronize((cudaStream_t)stream);
  if (e != cudaSuccess) return CPATTN_ERR_CUDA;
  int* err = device_error_word();
  if (err == nullptr) return CPATTN_ERR_CUDA;
  int host = 0;
  if (cudaMemcpy(&host, err, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess)
    return CPATTN_ERR_CUDA;
  if (host != 0) {
    int zero = 0;
    if (cudaMemcpy(err, &zero, sizeof(int), cudaMemcpyHostToDevice) != cudaSuccess)
      return CPATTN_ERR_CUDA;
    if (host == kErrBadDocs) return CPATTN_ERR_INVALID_ARG;
    if (host == kErrLaunch) return CPATTN_ERR_UNSUPPORTED;
    return CPATTN_ERR_DEVICE_TIMEOUT;
  }
  return CPATTN_OK;
}

const char* cpattn_status_string(int status) {
  switch (status) {
    case CPATTN_OK:
      return "ok";
    case CPATTN_ERR_INVALID_ARG:
      return "invalid argument";
    case CPATTN_ERR_UNSUPPORTED:
      return "unsupported";
    case CPATTN_ERR_CUDA:
      return "CUDA error";
    case CPATTN_ERR_DEVICE_TIMEOUT:
      return "device-side wait timed out";
    case CPATTN_ERR_WORKSPACE:
      return "workspace missing or too small";
    default:
      return "unknown status";
  }
}

}  // extern "C"
