// End-to-end entry point on host buffers: natural-order inputs in host
// memory, natural-order results back to host memory, the whole path on the
// device in between.
//
// The zigzag permutation is folded into the copies: natural chunk nc of
// batch row b is one contiguous run on both sides (host: natural position
// nc*c; device: the sharded position of that chunk), so each tensor moves as
// B * 2*cp (zigzag) or B * cp (contiguous) cudaMemcpyAsync calls.  LSE, whose
// sequence axis is innermost, is unpermuted by the device kernel and copied
// back in one piece.
//
// Overlap: dO goes up on a side stream while the forward runs, and O / LSE
// come down on the side stream while the backward runs.  The side stream
// and its events are created once per device on first use; the caller's
// stream waits for the side stream before the call's last operation, so the
// call is complete when the caller's stream reaches that point.
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>
#include <string.h>

#include <mutex>

#include "cpattn.h"
#include "cpattn_internal.h"

using namespace cpattn;

namespace {

constexpr int kMaxDevices = 64;
struct SideStream {
  cudaStream_t stream = nullptr;
  cudaEvent_t ev_a = nullptr, ev_b = nullptr, ev_c = nullptr;
};
SideStream g_side[kMaxDevices];
std::mutex g_side_mutex;

// The side stream of the current device (created on first use).
SideStream* side_stream() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(g_side_mutex);
  SideStream& s = g_side[dev];
  if (s.stream == nullptr) {
    cudaStream_t st = nullptr;
    if (cudaStreamCreateWithFlags(&st, cudaStreamNonBlocking) != cudaSuccess) return nullptr;
    cudaEvent_t e[3] = {nullptr, nullptr, nullptr};
    for (auto& ev : e)
      if (cudaEventCreateWithFlags(&ev, cudaEventDisableTiming) != cudaSuccess) return nullptr;
    s.ev_a = e[0];
    s.ev_b = e[1];
    s.ev_c = e[2];
    s.stream = st;
  }
  return &s;
}

size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

struct HostPlan {
  int B, S, cp, per, c, L;
  size_t elt, gelt;
  size_t q, kv, lse, gq, gkv, bwd, total;
};

bool plan_host(int B, int H, int Hkv, int S, int D, int cp, int layout, int dtype, bool backward,
               HostPlan* p) {
  if (B < 0 || H < 1 || Hkv < 1 || S < 0 || cp < 1 || (D != 64 && D != 128)) return false;
  if (layout != CPATTN_LAYOUT_CONTIGUOUS && layout != CPATTN_LAYOUT_ZIGZAG) return false;
  const int in_dtype = dtype & ~CPATTN_GRAD_F32;
  if (in_dtype != CPATTN_F32 && in_dtype != CPATTN_BF16) return false;
  const int per = layout == CPATTN_LAYOUT_ZIGZAG ? 2 : 1;
  if (S % (cp * per) != 0) return false;
  p->B = B;
  p->S = S;
  p->cp = cp;
  p->per = per;
  p->L = S / cp;
  p->c = p->L / per;
  p->elt = in_dtype == CPATTN_BF16 ? 2 : 4;
  p->gelt = (dtype & CPATTN_GRAD_F32) ? 4 : p->elt;
  const size_t rows = (size_t)B * S;
  p->q = align256(rows * H * D * p->elt);
  p->kv = align256(rows * Hkv * D * p->elt);
  p->lse = align256((size_t)B * H * S * sizeof(float));
  p->gq = backward ? align256(rows * H * D * p->gelt) : 0;
  p->gkv = backward ? align256(rows * Hkv * D * p->gelt) : 0;
  p->bwd = backward ? align256(cpattn_ring_bwd_workspace_bytes(B, H, Hkv, S, D, dtype)) : 0;
  // q, k, v, (dO), out, lse sharded, lse natural, (dq, dk, dv), backward workspace
  p->total = (backward ? 3 : 2) * p->q + 2 * p->kv + 2 * p->lse + p->gq + 2 * p->gkv + p->bwd;
  return true;
}

// Sharded row of the first token of natural chunk nc.
int64_t chunk_row(const HostPlan& p, int nc) {
  if (p.per == 1) return (int64_t)nc * p.c;
  const int r = nc < p.cp ? nc : 2 * p.cp - 1 - nc;
  return (int64_t)r * p.L + (nc < p.cp ? 0 : p.c);
}

// Copies a [B, S, row_bytes] tensor between natural-order host memory and
// sharded-order device memory, one contiguous chunk per cudaMemcpyAsync.
cudaError_t copy_chunks(const HostPlan& p, const void* src, void* dst, size_t row_bytes,
                        bool to_device, cudaStream_t st) {
  const int nchunk = p.cp * p.per;
  const size_t chunk_bytes = (size_t)p.c * row_bytes;
  for (int b = 0; b < p.B; ++b)
    for (int nc = 0; nc < nchunk; ++nc) {
      const size_t nat = ((size_t)b * p.S + (size_t)nc * p.c) * row_bytes;
      const size_t shd = ((size_t)b * p.S + (size_t)chunk_row(p, nc)) * row_bytes;
      const char* s = static_cast<const char*>(src) + (to_device ? nat : shd);
      char* d = static_cast<char*>(dst) + (to_device ? shd : nat);
      cudaError_t e = cudaMemcpyAsync(d, s, chunk_bytes,
                                      to_device ? cudaMemcpyHostToDevice : cudaMemcpyDeviceToHost,
                                      st);
      if (e != cudaSuccess) return e;
    }
  return cudaSuccess;
}

}  // namespace

extern "C" {

size_t cpattn_attention_host_workspace_bytes(int B, int H, int Hkv, int S, int D, int cp_size,
                                             int layout, int dtype, int backward) {
  HostPlan p;
  if (!plan_host(B, H, Hkv, S, D, cp_size, layout, dtype, backward != 0, &p)) return 0;
  return p.total;
}

int cpattn_attention_host(const void* q, const void* k, const void* v, const void* dout,
                          void* out, float* lse, void* dq, void* dk, void* dv, int B, int H,
                          int Hkv, int S, int D, int cp_size, int layout, int causal, int dtype,
                          float softmax_scale, void* workspace, size_t workspace_bytes,
                          cpattn_stream_t stream) {
  const bool backward = dout != nullptr;
  HostPlan p;
  if (!plan_host(B, H, Hkv, S, D, cp_size, layout, dtype, backward, &p))
    return CPATTN_ERR_INVALID_ARG;
  if ((long long)B * S == 0) return CPATTN_OK;
  if (!q || !k || !v || !out || !lse) return CPATTN_ERR_INVALID_ARG;
  if (backward && (!dq || !dk || !dv)) return CPATTN_ERR_INVALID_ARG;
  if (workspace == nullptr || workspace_bytes < p.total ||
      (reinterpret_cast<uintptr_t>(workspace) & 255) != 0)
    return CPATTN_ERR_WORKSPACE;
  const int in_dtype = dtype & ~CPATTN_GRAD_F32;
  cudaStream_t st = (cudaStream_t)stream;
  char* w = static_cast<char*>(workspace);
  void* qs = w;
  w += p.q;
  void* os = w;
  w += p.q;
  void* dos = nullptr;
  if (backward) {
    dos = w;
    w += p.q;
  }
  void* ks = w;
  w += p.kv;
  void* vs = w;
  w += p.kv;
  float* lse_s = reinterpret_cast<float*>(w);
  w += p.lse;
  float* lse_n = reinterpret_cast<float*>(w);
  w += p.lse;
  void* dqs = w;
  w += p.gq;
  void* dks = w;
  w += p.gkv;
  void* dvs = w;
  w += p.gkv;
  void* bws = w;

  const size_t qrow = (size_t)H * D * p.elt, kvrow = (size_t)Hkv * D * p.elt;
  const size_t gqrow = (size_t)H * D * p.gelt, gkvrow = (size_t)Hkv * D * p.gelt;
  SideStream* side = backward ? side_stream() : nullptr;
  if (backward && side == nullptr) return CPATTN_ERR_CUDA;
  int rc = CPATTN_OK;
#define CPATTN_TRY(x)                                 \
  do {                                                \
    if ((x) != cudaSuccess) return CPATTN_ERR_CUDA;   \
  } while (0)
  if (backward) {
    // dO goes up on the side stream, once the caller's stream is here.
    CPATTN_TRY(cudaEventRecord(side->ev_a, st));
    CPATTN_TRY(cudaStreamWaitEvent(side->stream, side->ev_a, 0));
    CPATTN_TRY(copy_chunks(p, dout, dos, qrow, true, side->stream));
    CPATTN_TRY(cudaEventRecord(side->ev_b, side->stream));
  }
  CPATTN_TRY(copy_chunks(p, q, qs, qrow, true, st));
  CPATTN_TRY(copy_chunks(p, k, ks, kvrow, true, st));
  CPATTN_TRY(copy_chunks(p, v, vs, kvrow, true, st));
  rc = cpattn_ring_fwd(qs, ks, vs, os, lse_s, B, H, Hkv, S, D, cp_size, layout, causal, in_dtype,
                       softmax_scale, stream);
  if (rc != CPATTN_OK) return rc;
  rc = cpattn_zigzag_unpermute(lse_s, lse_n, (int64_t)B * H, S, sizeof(float), cp_size, layout,
                               stream);
  if (rc != CPATTN_OK) return rc;
  if (!backward) {
    CPATTN_TRY(copy_chunks(p, os, out, qrow, false, st));
    CPATTN_TRY(cudaMemcpyAsync(lse, lse_n, (size_t)B * H * S * sizeof(float),
                               cudaMemcpyDeviceToHost, st));
    return CPATTN_OK;
  }
  // O and LSE come down on the side stream while the backward runs.
  CPATTN_TRY(cudaEventRecord(side->ev_c, st));
  CPATTN_TRY(cudaStreamWaitEvent(side->stream, side->ev_c, 0));
  CPATTN_TRY(copy_chunks(p, os, out, qrow, false, side->stream));
  CPATTN_TRY(cudaMemcpyAsync(lse, lse_n, (size_t)B * H * S * sizeof(float),
                             cudaMemcpyDeviceToHost, side->stream));
  CPATTN_TRY(cudaEventRecord(side->ev_a, side->stream));
  CPATTN_TRY(cudaStreamWaitEvent(st, side->ev_b, 0));  // dO is on the device
  rc = cpattn_ring_bwd(qs, ks, vs, os, dos, lse_s, dqs, dks, dvs, B, H, Hkv, S, D, cp_size, layout,
                       causal, dtype, softmax_scale, bws, p.bwd, stream);
  if (rc != CPATTN_OK) return rc;
  CPATTN_TRY(copy_chunks(p, dqs, dq, gqrow, false, st));
  CPATTN_TRY(copy_chunks(p, dks, dk, gkvrow, false, st));
  CPATTN_TRY(copy_chunks(p, dvs, dv, gkvrow, false, st));
  CPATTN_TRY(cudaStreamWaitEvent(st, side->ev_a, 0));  // O and LSE are on the host
#undef CPATTN_TRY
  return CPATTN_OK;
}

}  // extern "C"
