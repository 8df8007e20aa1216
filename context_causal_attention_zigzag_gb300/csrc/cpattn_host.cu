// End-to-end entry point on host buffers: natural-order inputs in host
// memory, natural-order results back to host memory, the whole path on the
// device in between.
//
// Parts: the heads are split into `parts` groups of whole kv-head groups
// (part p: query heads [p*Hp, (p+1)*Hp), kv heads [p*Hkvp, (p+1)*Hkvp)).
// Each part has contiguous device tensors [B, S, Hp, D] of its own, filled
// by copies that gather the part's heads out of the natural host rows and
// fold the zigzag permutation in (natural chunk nc of batch row b is one
// run of rows on both sides: one 2-D copy per chunk and batch row).  The
// attention of a head does not depend on the other heads, so each part runs
// the ring forward and backward unchanged on its own tensors and the
// results are, bit for bit, those of one call over all heads.
//
// Overlap, three streams:
//   up stream       Q_p, K_p, V_p of every part in turn, then dO_p;
//   caller stream   forward(p) once part p is up, then backward(p) once dO_p
//                   is up;
//   down stream     O_p and LSE_p once forward(p) is done, dQ_p, dK_p, dV_p
//                   once backward(p) is done.
// Only the first part's upload and the last part's download are not hidden
// behind computation.  The two side streams and their events are created
// once per device on first use; the caller's stream waits for both before
// the call's last operation, so the call is complete when the caller's
// stream reaches that point.
#include <cuda_runtime.h>
#include <limits.h>
#include <stddef.h>
#include <stdint.h>
#include <string.h>

#include <mutex>

#include "cpattn.h"
#include "cpattn_internal.h"

using namespace cpattn;

namespace {

constexpr int kMaxDevices = 64;
constexpr int kMaxParts = 8;

struct SideStreams {
  bool ready = false;
  cudaStream_t up = nullptr, down = nullptr;
  cudaEvent_t start = nullptr, up_end = nullptr, down_end = nullptr;
  cudaEvent_t qkv[kMaxParts], dout[kMaxParts], fwd[kMaxParts], bwd[kMaxParts];
  // Pinned staging of document offsets; `cu_copied` marks the copy that
  // last read it (a later call waits for it before rewriting the buffer).
  int32_t* cu_host = nullptr;
  size_t cu_cap = 0;
  cudaEvent_t cu_copied = nullptr;
  bool cu_pending = false;
};
SideStreams g_side[kMaxDevices];
std::mutex g_side_mutex;

// The side streams of the current device (created on first use).
SideStreams* side_streams() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(g_side_mutex);
  SideStreams& s = g_side[dev];
  if (s.ready) return &s;
  SideStreams n;
  bool ok = cudaStreamCreateWithFlags(&n.up, cudaStreamNonBlocking) == cudaSuccess &&
            cudaStreamCreateWithFlags(&n.down, cudaStreamNonBlocking) == cudaSuccess;
  cudaEvent_t* evs[4 + 4 * kMaxParts];
  int ne = 0;
  evs[ne++] = &n.cu_copied;
  evs[ne++] = &n.start;
  evs[ne++] = &n.up_end;
  evs[ne++] = &n.down_end;
  for (int p = 0; p < kMaxParts; ++p) {
    evs[ne++] = &n.qkv[p];
    evs[ne++] = &n.dout[p];
    evs[ne++] = &n.fwd[p];
    evs[ne++] = &n.bwd[p];
  }
  for (int i = 0; i < ne; ++i) *evs[i] = nullptr;
  for (int i = 0; i < ne && ok; ++i)
    ok = cudaEventCreateWithFlags(evs[i], cudaEventDisableTiming) == cudaSuccess;
  if (!ok) {
    for (int i = 0; i < ne; ++i)
      if (*evs[i]) cudaEventDestroy(*evs[i]);
    if (n.up) cudaStreamDestroy(n.up);
    if (n.down) cudaStreamDestroy(n.down);
    return nullptr;
  }
  n.ready = true;
  s = n;
  return &s;
}

size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

// Device bytes reserved for a tensor of `full` bytes split into up to
// kMaxParts 256-byte-aligned parts.
size_t reserve(size_t full) { return align256(full) + (size_t)kMaxParts * 256; }

struct HostPlan {
  int B, S, S_real, H, Hkv, D, cp, per, c, L;  // S: device (padded) length
  int n, Hp, Hkvp;  // parts, query / kv heads per part
  bool docs;        // document rule (bounds table in the workspace)
  size_t elt, gelt;
  // bytes of one part's tensor (slot = 256-aligned stride between parts)
  size_t q, kv, lse, gq, gkv;
  size_t q_slot, kv_slot, lse_slot, gq_slot, gkv_slot;
  size_t bwd;    // backward workspace of one part
  size_t cu_bytes, bounds_bytes;
  size_t total;  // workspace bound, independent of the number of parts
};

// Parts chosen when the caller passes 0: the largest of 8, 4, 2 that
// divides Hkv and leaves each part at least 64 MiB of bf16 queries, else 1
// (S=131072, 32 heads, 8 kv heads: 8 parts, 491 ms per step from host
// buffers against 502 ms with 4 parts and 514 ms with 1 on one GB300).
int auto_parts(int B, int S, int H, int Hkv, int D) {
  const double q_bytes = (double)B * S * H * D * 2.0;
  for (int n = 8; n >= 2; n /= 2)
    if (Hkv % n == 0 && q_bytes / n >= 64.0 * 1024 * 1024) return n;
  return 1;
}

// S_real tokens on the host; S tokens on the device (S = S_real, or the
// padded length under the document rule).
bool plan_host(int B, int H, int Hkv, int S_real, int S, int D, int cp, int layout, int dtype,
               bool backward, int parts, bool docs, HostPlan* p) {
  if (B < 0 || H < 1 || Hkv < 1 || S_real < 0 || S < S_real || cp < 1 || (D != 64 && D != 128))
    return false;
  if (H % Hkv != 0) return false;
  if (layout != CPATTN_LAYOUT_CONTIGUOUS && layout != CPATTN_LAYOUT_ZIGZAG) return false;
  const int in_dtype = dtype & ~kDtypeFlags;
  if (in_dtype != CPATTN_F32 && in_dtype != CPATTN_BF16) return false;
  const int per = layout == CPATTN_LAYOUT_ZIGZAG ? 2 : 1;
  if (S % (cp * per) != 0) return false;
  if (parts == 0) parts = auto_parts(B, S, H, Hkv, D);
  if (parts < 1 || parts > kMaxParts || Hkv % parts != 0) return false;
  p->B = B;
  p->S = S;
  p->S_real = S_real;
  p->H = H;
  p->Hkv = Hkv;
  p->D = D;
  p->cp = cp;
  p->per = per;
  p->L = S / cp;
  p->c = p->L / per;
  p->n = parts;
  p->Hp = H / parts;
  p->Hkvp = Hkv / parts;
  p->docs = docs;
  p->elt = in_dtype == CPATTN_BF16 ? 2 : 4;
  p->gelt = (dtype & CPATTN_GRAD_F32) ? 4 : p->elt;
  const size_t rows = (size_t)B * S;
  p->q = rows * p->Hp * D * p->elt;
  p->kv = rows * p->Hkvp * D * p->elt;
  p->lse = (size_t)B * p->Hp * S * sizeof(float);
  p->gq = rows * p->Hp * D * p->gelt;
  p->gkv = rows * p->Hkvp * D * p->gelt;
  p->q_slot = align256(p->q);
  p->kv_slot = align256(p->kv);
  p->lse_slot = align256(p->lse);
  p->gq_slot = align256(p->gq);
  p->gkv_slot = align256(p->gkv);
  p->bwd = backward ? cpattn_ring_bwd_workspace_bytes(B, p->Hp, p->Hkvp, S, D, dtype) : 0;
  // offsets of up to S_real documents plus the padding, and the bounds table
  p->cu_bytes = docs ? align256(((size_t)S_real + 2) * sizeof(int32_t)) : 0;
  p->bounds_bytes = docs ? align256((size_t)S * 2 * sizeof(int32_t)) : 0;
  // q, out, (dO); k, v; lse sharded, lse natural; (dq, dk, dv); backward
  // workspace -- each reserved for any number of parts up to kMaxParts.
  const size_t fq = rows * H * D * p->elt, fkv = rows * Hkv * D * p->elt;
  const size_t flse = (size_t)B * H * S * sizeof(float);
  const size_t fgq = rows * H * D * p->gelt, fgkv = rows * Hkv * D * p->gelt;
  p->total = (backward ? 3 : 2) * reserve(fq) + 2 * reserve(fkv) + 2 * reserve(flse) +
             p->cu_bytes + p->bounds_bytes;
  if (backward)
    p->total += reserve(fgq) + 2 * reserve(fgkv) +
                align256(cpattn_ring_bwd_workspace_bytes(B, H, Hkv, S, D, dtype));
  return true;
}

// Sharded row of the first token of natural chunk nc.
int64_t chunk_row(const HostPlan& p, int nc) {
  if (p.per == 1) return (int64_t)nc * p.c;
  const int r = nc < p.cp ? nc : 2 * p.cp - 1 - nc;
  return (int64_t)r * p.L + (nc < p.cp ? 0 : p.c);
}

// Copies the heads of part `part` of a [B, S_real, X, D] tensor (X heads,
// elt bytes each) from src to dst: natural-order host memory to the part's
// sharded device tensor [B, S, X / n, D] (to_device), or back.  One copy per
// natural chunk and batch row, 2-D (a run of rows, each the part's slice of
// a host row) when the part is not the whole row.  Only real tokens move;
// on the way in, the device rows of padding tokens are zeroed.
cudaError_t copy_part(const HostPlan& p, const void* src, void* dst, int X, size_t elt, int part,
                      bool to_device, cudaStream_t st) {
  const size_t hpitch = (size_t)X * p.D * elt;  // a natural host row
  const size_t dpitch = hpitch / p.n;            // a row of the part's device tensor
  const size_t hoff = (size_t)part * dpitch;     // the part's heads within a host row
  const int nchunk = p.cp * p.per;
  char* host = static_cast<char*>(to_device ? const_cast<void*>(src) : dst);
  char* dev = static_cast<char*>(to_device ? dst : const_cast<void*>(src));
  for (int b = 0; b < p.B; ++b)
    for (int nc = 0; nc < nchunk; ++nc) {
      const int64_t nat0 = (int64_t)nc * p.c;
      const int64_t real = nat0 >= p.S_real ? 0 : (p.S_real - nat0 < p.c ? p.S_real - nat0 : p.c);
      char* h = host + ((size_t)b * p.S_real + (size_t)nat0) * hpitch + hoff;
      char* d = dev + ((size_t)b * p.S + (size_t)chunk_row(p, nc)) * dpitch;
      cudaError_t e = cudaSuccess;
      if (real > 0) {
        if (p.n == 1)
          e = to_device
                  ? cudaMemcpyAsync(d, h, (size_t)real * dpitch, cudaMemcpyHostToDevice, st)
                  : cudaMemcpyAsync(h, d, (size_t)real * dpitch, cudaMemcpyDeviceToHost, st);
        else
          e = to_device ? cudaMemcpy2DAsync(d, dpitch, h, hpitch, dpitch, (size_t)real,
                                            cudaMemcpyHostToDevice, st)
                        : cudaMemcpy2DAsync(h, hpitch, d, dpitch, dpitch, (size_t)real,
                                            cudaMemcpyDeviceToHost, st);
      }
      if (e == cudaSuccess && to_device && real < p.c)
        e = cudaMemsetAsync(d + (size_t)real * dpitch, 0, (size_t)(p.c - real) * dpitch, st);
      if (e != cudaSuccess) return e;
    }
  return cudaSuccess;
}

// LSE of part `part` ([B, Hp, S_real], natural order on the device) into the
// host's [B, H, S_real].
cudaError_t copy_lse_part(const HostPlan& p, const float* dev, float* host, int part,
                          cudaStream_t st) {
  const size_t width = (size_t)p.Hp * p.S_real * sizeof(float);
  const size_t hpitch = (size_t)p.H * p.S_real * sizeof(float);
  char* h = reinterpret_cast<char*>(host) + (size_t)part * width;
  if (p.n == 1) return cudaMemcpyAsync(h, dev, (size_t)p.B * width, cudaMemcpyDeviceToHost, st);
  return cudaMemcpy2DAsync(h, hpitch, dev, width, width, p.B, cudaMemcpyDeviceToHost, st);
}

// Document offsets on the host: 0 = cu[0] < ... < cu[ndocs] = S_real.
bool valid_offsets(const int32_t* cu, int ndocs, int S_real) {
  if (ndocs < 1 || ndocs > S_real || cu[0] != 0 || cu[ndocs] != S_real) return false;
  for (int d = 0; d < ndocs; ++d)
    if (cu[d + 1] <= cu[d]) return false;
  return true;
}

// The path shared by both entry points.  cu / ndocs: host document offsets
// over the real tokens when p.docs (NULL: one document).
int host_common(const HostPlan& p, const void* q, const void* k, const void* v, const void* dout,
                void* out, float* lse, void* dq, void* dk, void* dv, int layout, int causal,
                int dtype, float softmax_scale, const int32_t* cu, int ndocs, void* workspace,
                size_t workspace_bytes, cpattn_stream_t stream) {
  const bool backward = dout != nullptr;
  const int B = p.B, S = p.S, H = p.H, Hkv = p.Hkv, D = p.D, cp_size = p.cp;
  if ((long long)B * p.S_real == 0) return CPATTN_OK;
  if (!q || !k || !v || !out || !lse) return CPATTN_ERR_INVALID_ARG;
  if (backward && (!dq || !dk || !dv)) return CPATTN_ERR_INVALID_ARG;
  if (p.docs && cu != nullptr && !valid_offsets(cu, ndocs, p.S_real)) return CPATTN_ERR_INVALID_ARG;
  if (workspace == nullptr || workspace_bytes < p.total ||
      (reinterpret_cast<uintptr_t>(workspace) & 255) != 0)
    return CPATTN_ERR_WORKSPACE;
  const int in_dtype = dtype & ~kDtypeFlags;
  cudaStream_t st = (cudaStream_t)stream;
  SideStreams* ss = side_streams();
  if (ss == nullptr) return CPATTN_ERR_CUDA;

  // Workspace regions, one 256-byte-aligned slot per part in each.
  char* w = static_cast<char*>(workspace);
  const size_t fq = (size_t)B * S * H * D * p.elt, fkv = (size_t)B * S * Hkv * D * p.elt;
  const size_t flse = (size_t)B * H * S * sizeof(float);
  char* qs = w;
  w += reserve(fq);
  char* os = w;
  w += reserve(fq);
  char* dos = nullptr;
  if (backward) {
    dos = w;
    w += reserve(fq);
  }
  char* ks = w;
  w += reserve(fkv);
  char* vs = w;
  w += reserve(fkv);
  char* lse_s = w;
  w += reserve(flse);
  char* lse_n = w;
  w += reserve(flse);
  int32_t* cu_dev = reinterpret_cast<int32_t*>(w);
  w += p.cu_bytes;
  int32_t* bounds = p.docs ? reinterpret_cast<int32_t*>(w) : nullptr;
  w += p.bounds_bytes;
  char *dqs = nullptr, *dks = nullptr, *dvs = nullptr, *bws = nullptr;
  if (backward) {
    dqs = w;
    w += reserve((size_t)B * S * H * D * p.gelt);
    dks = w;
    w += reserve((size_t)B * S * Hkv * D * p.gelt);
    dvs = w;
    w += reserve((size_t)B * S * Hkv * D * p.gelt);
    bws = w;
  }

  // Document offsets of the device sequence: the caller's (or one
  // document), and the padding as one more document, staged in pinned
  // memory for an asynchronous copy.
  size_t ncu = 0;
  if (p.docs) {
    const size_t need = (size_t)(cu != nullptr ? ndocs : 1) + 2;
    if (ss->cu_pending && cudaEventSynchronize(ss->cu_copied) != cudaSuccess)
      return CPATTN_ERR_CUDA;
    ss->cu_pending = false;
    if (ss->cu_cap < need) {
      if (ss->cu_host != nullptr) cudaFreeHost(ss->cu_host);
      ss->cu_host = nullptr;
      ss->cu_cap = 0;
      if (cudaHostAlloc(reinterpret_cast<void**>(&ss->cu_host), need * sizeof(int32_t),
                        cudaHostAllocDefault) != cudaSuccess)
        return CPATTN_ERR_CUDA;
      ss->cu_cap = need;
    }
    if (cu != nullptr) {
      memcpy(ss->cu_host, cu, ((size_t)ndocs + 1) * sizeof(int32_t));
      ncu = (size_t)ndocs + 1;
    } else {
      ss->cu_host[0] = 0;
      ss->cu_host[1] = p.S_real;
      ncu = 2;
    }
    if (S > p.S_real) ss->cu_host[ncu++] = S;
  }

  // From here on every exit makes the caller's stream wait for both side
  // streams, so nothing the call enqueued outlives it unseen.
  if (cudaEventRecord(ss->start, st) != cudaSuccess ||
      cudaStreamWaitEvent(ss->up, ss->start, 0) != cudaSuccess ||
      cudaStreamWaitEvent(ss->down, ss->start, 0) != cudaSuccess)
    return CPATTN_ERR_CUDA;
  int rc = CPATTN_OK;
  auto cuda = [&](cudaError_t e) {
    if (e != cudaSuccess && rc == CPATTN_OK) rc = CPATTN_ERR_CUDA;
    return rc == CPATTN_OK;
  };
  auto lib = [&](int r) {
    if (r != CPATTN_OK && rc == CPATTN_OK) rc = r;
    return rc == CPATTN_OK;
  };
  const int n = p.n;
  if (p.docs) {
    cuda(cudaMemcpyAsync(cu_dev, ss->cu_host, ncu * sizeof(int32_t), cudaMemcpyHostToDevice,
                         st)) &&
        cuda(cudaEventRecord(ss->cu_copied, st)) &&
        lib(cpattn_doc_bounds(cu_dev, (int)ncu - 1, S, bounds, stream));
    ss->cu_pending = true;
  }
  // Part by part: Q, K, V up, then the forward (which waits for them) and
  // the part's O and LSE down behind it.  The host enqueues in this order so
  // that the first forward is queued before the later parts' copies.
  for (int i = 0; i < n && rc == CPATTN_OK; ++i) {
    cuda(copy_part(p, q, qs + i * p.q_slot, H, p.elt, i, true, ss->up)) &&
        cuda(copy_part(p, k, ks + i * p.kv_slot, Hkv, p.elt, i, true, ss->up)) &&
        cuda(copy_part(p, v, vs + i * p.kv_slot, Hkv, p.elt, i, true, ss->up)) &&
        cuda(cudaEventRecord(ss->qkv[i], ss->up));
    if (rc != CPATTN_OK) break;
    void* o_i = os + i * p.q_slot;
    float* ls_i = reinterpret_cast<float*>(lse_s + i * p.lse_slot);
    float* ln_i = reinterpret_cast<float*>(lse_n + i * p.lse_slot);
    const char* q_i = qs + i * p.q_slot;
    const char* k_i = ks + i * p.kv_slot;
    const char* v_i = vs + i * p.kv_slot;
    cuda(cudaStreamWaitEvent(st, ss->qkv[i], 0)) &&
        lib(p.docs ? cpattn_ring_fwd_docs(q_i, k_i, v_i, o_i, ls_i, B, p.Hp, p.Hkvp, S, D,
                                          cp_size, layout, causal, in_dtype, softmax_scale,
                                          bounds, nullptr, stream)
                   : cpattn_ring_fwd(q_i, k_i, v_i, o_i, ls_i, B, p.Hp, p.Hkvp, S, D, cp_size,
                                     layout, causal, in_dtype, softmax_scale, stream)) &&
        lib(cpattn_zigzag_unpermute_pad(ls_i, ln_i, (int64_t)B * p.Hp, p.S_real, S,
                                        sizeof(float), cp_size, layout, stream)) &&
        cuda(cudaEventRecord(ss->fwd[i], st)) &&
        cuda(cudaStreamWaitEvent(ss->down, ss->fwd[i], 0)) &&
        cuda(copy_part(p, o_i, out, H, p.elt, i, false, ss->down)) &&
        cuda(copy_lse_part(p, ln_i, lse, i, ss->down));
  }
  // dO up part by part (behind the last Q, K, V, while the forwards run).
  for (int i = 0; backward && i < n && rc == CPATTN_OK; ++i) {
    cuda(copy_part(p, dout, dos + i * p.q_slot, H, p.elt, i, true, ss->up)) &&
        cuda(cudaEventRecord(ss->dout[i], ss->up));
  }
  // Backward part by part; each part's gradients go down behind it.
  for (int i = 0; backward && i < n && rc == CPATTN_OK; ++i) {
    void* dq_i = dqs + i * p.gq_slot;
    void* dk_i = dks + i * p.gkv_slot;
    void* dv_i = dvs + i * p.gkv_slot;
    const char* q_i = qs + i * p.q_slot;
    const char* k_i = ks + i * p.kv_slot;
    const char* v_i = vs + i * p.kv_slot;
    const char* o_i = os + i * p.q_slot;
    const char* do_i = dos + i * p.q_slot;
    const float* ls_i = reinterpret_cast<const float*>(lse_s + i * p.lse_slot);
    cuda(cudaStreamWaitEvent(st, ss->dout[i], 0)) &&
        lib(p.docs ? cpattn_ring_bwd_docs(q_i, k_i, v_i, o_i, do_i, ls_i, dq_i, dk_i, dv_i, B,
                                          p.Hp, p.Hkvp, S, D, cp_size, layout, causal, dtype,
                                          softmax_scale, bounds, bws, p.bwd, stream)
                   : cpattn_ring_bwd(q_i, k_i, v_i, o_i, do_i, ls_i, dq_i, dk_i, dv_i, B, p.Hp,
                                     p.Hkvp, S, D, cp_size, layout, causal, dtype, softmax_scale,
                                     bws, p.bwd, stream)) &&
        cuda(cudaEventRecord(ss->bwd[i], st)) &&
        cuda(cudaStreamWaitEvent(ss->down, ss->bwd[i], 0)) &&
        cuda(copy_part(p, dq_i, dq, H, p.gelt, i, false, ss->down)) &&
        cuda(copy_part(p, dk_i, dk, Hkv, p.gelt, i, false, ss->down)) &&
        cuda(copy_part(p, dv_i, dv, Hkv, p.gelt, i, false, ss->down));
  }
  // The caller's stream waits for both side streams.
  const bool joined = cudaEventRecord(ss->up_end, ss->up) == cudaSuccess &&
                      cudaEventRecord(ss->down_end, ss->down) == cudaSuccess &&
                      cudaStreamWaitEvent(st, ss->up_end, 0) == cudaSuccess &&
                      cudaStreamWaitEvent(st, ss->down_end, 0) == cudaSuccess;
  if (!joined && rc == CPATTN_OK) rc = CPATTN_ERR_CUDA;
  return rc;
}

}  // namespace

extern "C" {

size_t cpattn_attention_host_workspace_bytes(int B, int H, int Hkv, int S, int D, int cp_size,
                                             int layout, int dtype, int backward) {
  HostPlan p;
  if (!plan_host(B, H, Hkv, S, S, D, cp_size, layout, dtype, backward != 0, 1, false, &p))
    return 0;
  return p.total;
}

int cpattn_attention_host_parts(int B, int H, int Hkv, int S, int D) {
  if (B < 0 || H < 1 || Hkv < 1 || S < 0 || H % Hkv != 0) return 1;
  return auto_parts(B, S, H, Hkv, D);
}

int cpattn_attention_host(const void* q, const void* k, const void* v, const void* dout,
                          void* out, float* lse, void* dq, void* dk, void* dv, int B, int H,
                          int Hkv, int S, int D, int cp_size, int layout, int causal, int dtype,
                          float softmax_scale, int parts, void* workspace, size_t workspace_bytes,
                          cpattn_stream_t stream) {
  HostPlan p;
  if (!plan_host(B, H, Hkv, S, S, D, cp_size, layout, dtype, dout != nullptr, parts, false, &p))
    return CPATTN_ERR_INVALID_ARG;
  return host_common(p, q, k, v, dout, out, lse, dq, dk, dv, layout, causal, dtype, softmax_scale,
                     nullptr, 0, workspace, workspace_bytes, stream);
}

size_t cpattn_attention_host_docs_workspace_bytes(int B, int H, int Hkv, int S, int D,
                                                  int cp_size, int layout, int dtype,
                                                  int backward) {
  const int64_t Sp = cpattn_padded_length(S, cp_size, layout);
  if (Sp < 0 || Sp > INT32_MAX) return 0;
  HostPlan p;
  if (!plan_host(B, H, Hkv, S, (int)Sp, D, cp_size, layout, dtype, backward != 0, 1, true, &p))
    return 0;
  return p.total;
}

int cpattn_attention_host_docs(const void* q, const void* k, const void* v, const void* dout,
                               void* out, float* lse, void* dq, void* dk, void* dv, int B, int H,
                               int Hkv, int S, int D, int cp_size, int layout, int causal,
                               int dtype, float softmax_scale, const int32_t* cu_seqlens,
                               int ndocs, int parts, void* workspace, size_t workspace_bytes,
                               cpattn_stream_t stream) {
  const int64_t Sp = cpattn_padded_length(S, cp_size, layout);
  if (Sp < 0 || Sp > INT32_MAX) return CPATTN_ERR_INVALID_ARG;
  HostPlan p;
  if (!plan_host(B, H, Hkv, S, (int)Sp, D, cp_size, layout, dtype, dout != nullptr, parts, true,
                 &p))
    return CPATTN_ERR_INVALID_ARG;
  return host_common(p, q, k, v, dout, out, lse, dq, dk, dv, layout, causal, dtype, softmax_scale,
                     cu_seqlens, ndocs, workspace, workspace_bytes, stream);
}

}  // extern "C"
