/*
 * cpattn.h -- C ABI of libcpattn: context-parallel blockwise causal attention
 * with the zigzag (load-balanced) layout, run on ONE GPU with the cp_size
 * context-parallel ranks held as logical shards of that device's memory.
 *
 * What is computed, and where it is defined:
 *   "Sequence Parallelism IV: Megatron Context Parallel and Load-Balanced
 *   Rings" (section 3: the sequence is cut into 2*cp_size chunks and rank r
 *   owns chunks r and 2*cp_size-1-r; section 4: local Q stays, K/V blocks
 *   move around the ring, each arriving block gives a partial output and the
 *   online-softmax state keeps the result exact, causal sub-blocks that are
 *   entirely in the future are skipped; section 5: softmax-state correction
 *   per ring step), and "Context Parallelism for Long-Context Training"
 *   (section "Prove attention equivalence": the result, and its gradients,
 *   equal unsharded attention).
 *
 * Conventions shared by every call
 *   - Tensors are row-major.  Q, O, dQ, dO: [B, S, H, D]; K, V, dK, dV:
 *     [B, S, Hkv, D]; LSE: [B, H, S] float32, natural log of the softmax
 *     normaliser including the scale.  Query head h reads kv head
 *     h / (H / Hkv).
 *   - Attention calls take tensors in SHARDED order along S: the shards of
 *     ranks 0..cp_size-1 one after another.  With CPATTN_LAYOUT_ZIGZAG rank r's
 *     shard is [chunk r, chunk 2*cp_size-1-r] (chunk length S / (2*cp_size));
 *     with CPATTN_LAYOUT_CONTIGUOUS rank r's shard is chunk r (length
 *     S / cp_size), i.e. sharded order equals natural order.  The causal mask
 *     is always taken on natural positions (key j is visible to query i iff
 *     j <= i).  cpattn_zigzag_permute / _unpermute convert between orders.
 *   - Ring: at step t = 0..cp_size-1 rank r holds the K/V shard of rank
 *     (r - t) mod cp_size.
 *   - Every pointer marked "device" must be device memory of the current
 *     device; the caller owns every buffer.  The library allocates nothing
 *     per call; it holds one static device error word per device.
 *   - Calls are asynchronous on `stream` (NULL = legacy default stream)
 *     unless stated.  Arguments are validated before anything is launched; a
 *     call that returns an error launched nothing.
 *   - dtype CPATTN_F32: float32 inputs/outputs, computed with fp32 FMA.
 *     dtype CPATTN_BF16: bf16 inputs/outputs, fp32 accumulation (tensor
 *     cores on sm_103a when D == 128 and every chunk is a multiple of 256
 *     tokens; otherwise the fp32 CUDA-core kernels).
 *   - softmax_scale <= 0 selects 1/sqrt(D).
 */
#ifndef CPATTN_H
#define CPATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define CPATTN_API __attribute__((visibility("default")))
#else
#define CPATTN_API
#endif

/* Same type as cudaStream_t. */
typedef struct CUstream_st* cpattn_stream_t;

enum cpattn_status_code {
  CPATTN_OK = 0,
  CPATTN_ERR_INVALID_ARG = -1,    /* shape, pointer, alignment or enum out of range */
  CPATTN_ERR_UNSUPPORTED = -2,    /* valid request this build cannot run (e.g. no sm_103 device) */
  CPATTN_ERR_CUDA = -3,           /* a CUDA runtime call or launch failed */
  CPATTN_ERR_DEVICE_TIMEOUT = -4, /* a bounded device-side wait gave up (reported by cpattn_device_status) */
  CPATTN_ERR_WORKSPACE = -5       /* workspace missing or smaller than required */
};

enum cpattn_layout { CPATTN_LAYOUT_CONTIGUOUS = 0, CPATTN_LAYOUT_ZIGZAG = 1 };
enum cpattn_dtype {
  CPATTN_F32 = 0,
  CPATTN_BF16 = 1,
  /* Flag for the backward calls (OR it into dtype): dq, dk, dv are written
   * as float32 whatever the input dtype.  A bf16 gradient element of
   * magnitude >= 8 carries a rounding error of up to 2^-5; float32 output
   * keeps the gradients at their float32 accumulation accuracy. */
  CPATTN_GRAD_F32 = 0x10,
  /* Flag for the ring backward (OR it into dtype): on the tensor-core path,
   * compute dK, dV and dQ in one pass over the K/V tiles (five tile
   * products per tile pair instead of seven), each K/V tile adding its share
   * of dQ to a float32 accumulator with bulk reductions.  The order of
   * those additions varies from run to run, so dQ is not bitwise
   * reproducible (it stays within the same tolerance); without the flag the
   * backward is deterministic.  Ignored on the CUDA-core path. */
  CPATTN_BWD_ONEPASS = 0x20
};
enum cpattn_path { CPATTN_PATH_SIMT = 0, CPATTN_PATH_TCGEN05 = 1 };

/*
 * Reorders a tensor along its sequence axis.  The tensor is viewed as
 * [outer, S, inner_bytes] bytes (Q: outer = B, inner_bytes = H*D*elt; LSE:
 * outer = B*H, inner_bytes = 4).
 *   permute:   out[o, p, :] = in[o, natural(p), :]   (natural -> sharded)
 *   unpermute: out[o, natural(p), :] = in[o, p, :]   (sharded -> natural)
 * where natural(p) is the natural position of sharded position p
 * ("Sequence Parallelism IV ...", section 3).  in, out: device, must not
 * overlap.  Requires S % (2*cp_size) == 0 (zigzag) or S % cp_size == 0
 * (contiguous).  Bytes move in 16-byte vectors when alignment allows.
 */
CPATTN_API int cpattn_zigzag_permute(const void* in, void* out, int64_t outer, int64_t S,
                          int64_t inner_bytes, int cp_size, int layout, cpattn_stream_t stream);
CPATTN_API int cpattn_zigzag_unpermute(const void* in, void* out, int64_t outer, int64_t S,
                            int64_t inner_bytes, int cp_size, int layout, cpattn_stream_t stream);

/*
 * The same reorderings with padding ("Context Parallelism for Long-Context
 * Training", section "Test sequence divisibility and padding"): a sequence of
 * S_real tokens that does not split into the ring's chunks is padded at its
 * end to S tokens (S_real <= S, S as the permute above requires, e.g. from
 * cpattn_padded_length).  The padding belongs to whichever ranks own the last
 * natural positions (with zigzag: rank 0's second chunk first).
 *   permute_pad:   in [outer, S_real, inner] natural -> out [outer, S, inner]
 *                  sharded; natural positions >= S_real are written as zeros.
 *   unpermute_pad: in [outer, S, inner] sharded -> out [outer, S_real, inner]
 *                  natural; the padded positions are dropped.
 * Pair the padded tensors with a document whose range is [S_real, S) (see
 * cpattn_doc_bounds) so that no real token sees the padding.
 */
CPATTN_API int cpattn_zigzag_permute_pad(const void* in, void* out, int64_t outer, int64_t S_real,
                                         int64_t S, int64_t inner_bytes, int cp_size, int layout,
                                         cpattn_stream_t stream);
CPATTN_API int cpattn_zigzag_unpermute_pad(const void* in, void* out, int64_t outer,
                                           int64_t S_real, int64_t S, int64_t inner_bytes,
                                           int cp_size, int layout, cpattn_stream_t stream);

/*
 * Ring forward ("Sequence Parallelism IV ...", sections 4-5): for every
 * virtual rank r, its query shard attends to the K/V shards arriving at ring
 * steps t = 0..cp_size-1; tiles wholly in the causal future are skipped,
 * diagonal tiles are masked, and the online-softmax correction merges the
 * steps exactly.
 *   q [B,S,H,D], k/v [B,S,Hkv,D] (device, sharded order, dtype);
 *   out [B,S,H,D] (device, dtype) receives softmax(QK^T*scale) V;
 *   lse [B,H,S] (device, float32) receives the natural-log normaliser.
 * Requires H % Hkv == 0, D in {64, 128}, cp_size >= 1, the S divisibility
 * above, and 16-byte aligned q/k/v/out.
 */
CPATTN_API int cpattn_ring_fwd(const void* q, const void* k, const void* v, void* out, float* lse, int B,
                    int H, int Hkv, int S, int D, int cp_size, int layout, int causal, int dtype,
                    float softmax_scale, cpattn_stream_t stream);

/*
 * Same computation, and additionally adds to tiles_rt[r * cp_size + t]
 * (device, uint64, caller zeroes it) the number of (query tile, key tile)
 * pairs the kernel actually processed for virtual rank r at ring step t,
 * summed over batch and heads.  The tile edge is the one
 * cpattn_ring_fwd_plan reports.
 */
CPATTN_API int cpattn_ring_fwd_census(const void* q, const void* k, const void* v, void* out, float* lse,
                           int B, int H, int Hkv, int S, int D, int cp_size, int layout,
                           int causal, int dtype, float softmax_scale,
                           unsigned long long* tiles_rt, cpattn_stream_t stream);

/*
 * Which kernel cpattn_ring_fwd / cpattn_ring_bwd would run for these
 * arguments (host only, no GPU work): *path is a cpattn_path, *tile the tile
 * edge in tokens.  Either output pointer may be NULL.  The tensor-core path
 * takes bf16 inputs, D = 128, S < 2^23 and chunks (S / (2 cp_size) tokens
 * zigzag, S / cp_size contiguous) of whole 128-token tiles, whole 256-token
 * pairs of them for the forward, on an sm_103 device; everything else runs
 * on CUDA cores.
 */
CPATTN_API int cpattn_ring_fwd_plan(int B, int H, int Hkv, int S, int D, int cp_size, int layout,
                         int causal, int dtype, int* path, int* tile);
CPATTN_API int cpattn_ring_bwd_plan(int B, int H, int Hkv, int S, int D, int cp_size, int layout,
                         int causal, int dtype, int* path, int* tile);

/*
 * One ring step as its own partial ("each arriving K/V block gives a partial
 * output", section 4): for every rank r, the normalised partial attention of
 * r's queries over the K/V shard of rank (r - step) mod cp_size only.
 *   o_part [B,S,H,D] float32 (device), lse_part [B,H,S] float32 (device);
 *   a row with no visible key gets o = 0 and lse = -inf.
 * Merging the cp_size partials with cpattn_lse_merge gives cpattn_ring_fwd.
 */
CPATTN_API int cpattn_ring_fwd_step(const void* q, const void* k, const void* v, int B, int H, int Hkv,
                         int S, int D, int cp_size, int layout, int causal, int dtype,
                         float softmax_scale, int step, float* o_part, float* lse_part,
                         cpattn_stream_t stream);

/*
 * Exact merge of two normalised partials (the softmax-state correction,
 * section 5):  L = log(e^La + e^Lb),  O = e^(La-L) O_a + e^(Lb-L) O_b,
 * with (0, -inf) as the neutral element.
 *   o_a, o_b, o_out: [B,S,H,D] float32 (device); lse_a, lse_b, lse_out:
 *   [B,H,S] float32 (device).  o_out may alias o_a or o_b and lse_out may
 *   alias lse_a or lse_b (in-place merge); other overlaps are not allowed.
 * Requires D in {64, 128} and 16-byte aligned O pointers.
 */
CPATTN_API int cpattn_lse_merge(const float* o_a, const float* lse_a, const float* o_b, const float* lse_b,
                     float* o_out, float* lse_out, int B, int S, int H, int D,
                     cpattn_stream_t stream);

/* Device workspace cpattn_ring_bwd needs, in bytes (host only). */
CPATTN_API size_t cpattn_ring_bwd_workspace_bytes(int B, int H, int Hkv, int S, int D, int dtype);

/*
 * Ring backward (gradients through the ring, "Context Parallelism for
 * Long-Context Training", section "Prove attention equivalence"): from the
 * saved out and lse of cpattn_ring_fwd and the upstream gradient dout,
 *   Delta_i = dout_i . out_i,  P_ij = exp(s_ij - lse_i),
 *   dS_ij = P_ij (dout_i . v_j - Delta_i),
 *   dq_i = scale sum_j dS_ij k_j,  dk_j = scale sum_i dS_ij q_i,
 *   dv_j = sum_i P_ij dout_i  (dk, dv summed over the heads sharing kv head j).
 * The K/V tiles of source rank s visit ranks (s + t) mod cp_size, t =
 * 0..cp_size-1, in the ring's order.
 *   q, out, dout, dq: [B,S,H,D]; k, v, dk, dv: [B,S,Hkv,D]; lse [B,H,S]
 *   float32; all device, sharded order, dtype (lse float32; dq, dk, dv
 *   float32 when dtype carries CPATTN_GRAD_F32).
 *   workspace: device, at least cpattn_ring_bwd_workspace_bytes, 256-byte
 *   aligned; its contents are scratch (no state kept between calls): float32
 *   accumulators for dQ, dK, dV and the Delta rows.
 */
CPATTN_API int cpattn_ring_bwd(const void* q, const void* k, const void* v, const void* out,
                    const void* dout, const float* lse, void* dq, void* dk, void* dv, int B,
                    int H, int Hkv, int S, int D, int cp_size, int layout, int causal, int dtype,
                    float softmax_scale, void* workspace, size_t workspace_bytes,
                    cpattn_stream_t stream);

/*
 * The same backward, and additionally the device census of the tiles its
 * kernels visit ("Sequence Parallelism IV ...", sections 3-4: per-iteration
 * work of each rank, future sub-blocks skipped): tiles_kv_rt[r * cp_size +
 * t] += the (query tile, key tile) pairs the K/V-major walk (dK, dV) handled
 * for receiving rank r at ring step t, tiles_q_rt likewise for the
 * query-major walk (dQ); summed over batch and heads, tile edge as
 * cpattn_ring_bwd_plan reports.  Both device, uint64 [cp_size * cp_size],
 * zeroed by the caller, non-NULL (else CPATTN_ERR_INVALID_ARG).  Each must
 * equal the forward's census and the closed form of cpattn_tile_counts.
 */
CPATTN_API int cpattn_ring_bwd_census(const void* q, const void* k, const void* v,
                                      const void* out, const void* dout, const float* lse,
                                      void* dq, void* dk, void* dv, int B, int H, int Hkv, int S,
                                      int D, int cp_size, int layout, int causal, int dtype,
                                      float softmax_scale, void* workspace,
                                      size_t workspace_bytes, unsigned long long* tiles_kv_rt,
                                      unsigned long long* tiles_q_rt, cpattn_stream_t stream);

/*
 * cpattn_ring_bwd without a workspace argument.  The pages describe no such
 * call; it exists for callers that cannot allocate device memory -- code
 * running under a memory manager that owns the whole device (a framework's
 * caching allocator, a serving runtime that reserves HBM at start-up) or on
 * a latency-critical loop where cudaMalloc / cudaFree would synchronise the
 * device.  The caller still passes every input and output exactly as for
 * cpattn_ring_bwd.
 *   Scratch: a 64 MiB array inside the library's device image (a static
 *   __device__ array), held by every GPU that loads the library until the
 *   process exits.  Problems whose cpattn_ring_bwd_workspace_bytes exceeds
 *   64 MiB (67108864 bytes) are rejected with CPATTN_ERR_WORKSPACE before
 *   anything is launched.
 *   The first call on a device looks the array's device address up
 *   (cudaGetSymbolAddress with that device current); make that first call
 *   before any stream capture.  Nothing is allocated, by this call or later.
 *   Every call on a device shares the one array, which keeps the last call's
 *   contents (each call re-zeroes what must start at zero): calls whose
 *   execution overlaps on the GPU -- on different streams, or from different
 *   host threads -- race on it and give wrong results.  Serialise them.
 */
CPATTN_API int cpattn_ring_bwd_noalloc(const void* q, const void* k, const void* v,
                                       const void* out, const void* dout, const float* lse,
                                       void* dq, void* dk, void* dv, int B, int H, int Hkv, int S,
                                       int D, int cp_size, int layout, int causal, int dtype,
                                       float softmax_scale, cpattn_stream_t stream);

/*
 * Packed documents and padding ("Context Parallelism for Long-Context
 * Training", section "Prove attention equivalence": document masks, like the
 * causal mask, must give the unsharded result; section "Test sequence
 * divisibility and padding": padded tokens must not change any real token's
 * output).  The sequence holds ndocs documents back to back: document d
 * covers the natural positions [cu_seqlens[d], cu_seqlens[d+1]), and a token
 * sees only tokens of its own document (with causal = 1, only the earlier
 * ones and itself).  The same documents apply to every batch row.  Padding is
 * one more document at the end: no real token sees it, and a zero dout on it
 * gives it no gradient and makes it contribute none.
 *
 * cpattn_doc_bounds turns the offsets into per-position bounds, computed once
 * and passed to the *_docs calls: bounds[2p] = first position and
 * bounds[2p+1] = one past the last position of the document holding natural
 * position p.
 *   cu_seqlens: device int32 [ndocs + 1]: 0, strictly increasing, ending at S.
 *   bounds: device int32 [S][2], 8-byte aligned.
 * Requires 1 <= ndocs <= S.  Offsets that break the rule above are reported
 * as CPATTN_ERR_INVALID_ARG by the next cpattn_device_status; the bounds are
 * still written (each position's range contains the position), so the calls
 * that read them stay within their buffers, but their results are undefined.
 */
CPATTN_API int cpattn_doc_bounds(const int32_t* cu_seqlens, int ndocs, int S, int32_t* bounds,
                                 cpattn_stream_t stream);

/*
 * cpattn_ring_fwd under the document rule.  doc_bounds: from
 * cpattn_doc_bounds for this S (device, natural positions).  Tiles that hold
 * no visible pair -- causal future or other documents -- are skipped, so a
 * packed sequence costs about the sum of its documents' own costs.
 * tiles_rt: NULL, or the census of cpattn_ring_fwd_census (tiles with at
 * least one visible pair under the document rule).
 */
CPATTN_API int cpattn_ring_fwd_docs(const void* q, const void* k, const void* v, void* out,
                                    float* lse, int B, int H, int Hkv, int S, int D, int cp_size,
                                    int layout, int causal, int dtype, float softmax_scale,
                                    const int32_t* doc_bounds, unsigned long long* tiles_rt,
                                    cpattn_stream_t stream);

/*
 * cpattn_ring_bwd under the document rule; out and lse from
 * cpattn_ring_fwd_docs with the same doc_bounds.  Workspace as
 * cpattn_ring_bwd (cpattn_ring_bwd_workspace_bytes).
 */
CPATTN_API int cpattn_ring_bwd_docs(const void* q, const void* k, const void* v, const void* out,
                                    const void* dout, const float* lse, void* dq, void* dk,
                                    void* dv, int B, int H, int Hkv, int S, int D, int cp_size,
                                    int layout, int causal, int dtype, float softmax_scale,
                                    const int32_t* doc_bounds, void* workspace,
                                    size_t workspace_bytes, cpattn_stream_t stream);

/*
 * The all-gather K/V schedule ("Context Parallelism in MegaDLMs", key-value
 * communication patterns: the ranks exchange K/V before attention so that
 * each holds the whole context).  Every virtual rank attends its own query
 * shard to the WHOLE K/V in one pass, walking it chunk by chunk in natural
 * order; there are no ring steps and no partials to merge.  On one GPU the
 * all-gather itself is cpattn_zigzag_unpermute of the sharded K and V into
 * k_full / v_full (one copy serves every rank), and the reduce-scatter that
 * returns gathered gradients to their owners is cpattn_zigzag_permute of
 * dk_full / dv_full (the sum over ranks happens inside the backward).
 *   q, out, lse, dout, dq: SHARDED order, as for cpattn_ring_fwd / _bwd;
 *   k_full, v_full, dk_full, dv_full: [B,S,Hkv,D] in NATURAL order.
 *   doc_bounds: NULL (one document) or from cpattn_doc_bounds.
 *   tiles_rt: NULL or the census of cpattn_ring_fwd_census, each tile
 *   attributed to the ring step at which its chunk's owner would deliver it
 *   (so the counts equal the ring's).
 * Shapes, dtypes, workspace and errors as cpattn_ring_fwd / cpattn_ring_bwd.
 */
CPATTN_API int cpattn_allgather_fwd(const void* q, const void* k_full, const void* v_full,
                                    void* out, float* lse, int B, int H, int Hkv, int S, int D,
                                    int cp_size, int layout, int causal, int dtype,
                                    float softmax_scale, const int32_t* doc_bounds,
                                    unsigned long long* tiles_rt, cpattn_stream_t stream);
CPATTN_API int cpattn_allgather_bwd(const void* q, const void* k_full, const void* v_full,
                                    const void* out, const void* dout, const float* lse, void* dq,
                                    void* dk_full, void* dv_full, int B, int H, int Hkv, int S,
                                    int D, int cp_size, int layout, int causal, int dtype,
                                    float softmax_scale, const int32_t* doc_bounds,
                                    void* workspace, size_t workspace_bytes,
                                    cpattn_stream_t stream);

/*
 * The Ulysses variant ("Sequence Parallelism IV", section 7): an all-to-all
 * moves sequence ownership to head ownership, so that rank r holds ALL
 * tokens of a head slice and computes full attention for it; the inverse
 * all-to-all returns the results to the token owners.  Rank r's query heads
 * are the r-th of cp_size equal slices (H % cp_size == 0); its kv heads are
 * the ones those query heads read, h / (H / Hkv): whole kv groups when a
 * slice holds them, else one kv head shared with the other ranks of its
 * group (so H/cp_size and H/Hkv must divide one another).  No zigzag is
 * needed for balance (every rank does the same work); `layout` only says how
 * the sequence is sharded in the inputs and outputs.
 *
 * cpattn_ulysses_a2a: one all-to-all on one GPU.
 *   to_seq = 0 (sequence -> head): in [B,S,X,D] sharded order ->
 *     out [cp][B,S,nx,D], rank r's heads of every token in natural order;
 *   to_seq = 1 (head -> sequence): the inverse; a kv head held by several
 *     ranks receives the sum of their rows (the gradient reduction).
 *   kv_heads = 0: query-head tensors (X = H, nx = H/cp_size); 1: kv-head
 *   tensors (X = Hkv, nx = kv heads per rank).  dtype CPATTN_F32 or
 *   CPATTN_BF16 (the element type).  16-byte aligned, non-overlapping.
 * cpattn_ulysses_lse_a2a: the same for LSE, [B,H,S] sharded <->
 *   [cp][B,H/cp,S] natural (float32).
 * cpattn_ulysses_fwd / _bwd: the whole variant on sharded-order tensors
 *   (shapes, dtypes and outputs as cpattn_ring_fwd / cpattn_ring_bwd):
 *   all-to-all of the inputs into the workspace, attention for every rank
 *   in one launch (ranks stacked along the batch), all-to-all back.
 *   doc_bounds: NULL or from cpattn_doc_bounds.  workspace: device, at least
 *   cpattn_ulysses_workspace_bytes(..., backward), 256-byte aligned, scratch.
 */
CPATTN_API int cpattn_ulysses_a2a(const void* in, void* out, int B, int S, int H, int Hkv, int D,
                                  int cp_size, int layout, int kv_heads, int to_seq, int dtype,
                                  cpattn_stream_t stream);
CPATTN_API int cpattn_ulysses_lse_a2a(const float* in, float* out, int B, int S, int H,
                                      int cp_size, int layout, int to_seq,
                                      cpattn_stream_t stream);
CPATTN_API size_t cpattn_ulysses_workspace_bytes(int B, int H, int Hkv, int S, int D,
                                                 int cp_size, int layout, int dtype,
                                                 int backward);
CPATTN_API int cpattn_ulysses_fwd(const void* q, const void* k, const void* v, void* out,
                                  float* lse, int B, int H, int Hkv, int S, int D, int cp_size,
                                  int layout, int causal, int dtype, float softmax_scale,
                                  const int32_t* doc_bounds, void* workspace,
                                  size_t workspace_bytes, cpattn_stream_t stream);
CPATTN_API int cpattn_ulysses_bwd(const void* q, const void* k, const void* v, const void* out,
                                  const void* dout, const float* lse, void* dq, void* dk,
                                  void* dv, int B, int H, int Hkv, int S, int D, int cp_size,
                                  int layout, int causal, int dtype, float softmax_scale,
                                  const int32_t* doc_bounds, void* workspace,
                                  size_t workspace_bytes, cpattn_stream_t stream);

/*
 * Hierarchical context parallelism, the a2a+p2p type ("Context Parallelism
 * in MegaDLMs", sections "Hierarchical Context Parallelism": a list of level
 * sizes such as [2, 2] splits the context group over two levels, and
 * "Key-Value Communication Patterns": a2a+p2p combines the all-to-all and
 * the point-to-point ring).  Level sizes [cp_a2a, cp_p2p], cp = cp_a2a *
 * cp_p2p virtual ranks; global rank r = p * cp_a2a + a is member a of group
 * p (groups are cp_a2a consecutive ranks).  The sequence is sharded over
 * all cp ranks with `layout` (zigzag: 2*cp chunks, rank r holding chunks r
 * and 2cp-1-r), so group p holds exactly shard p of the second level (for
 * zigzag: chunks p and 2*cp_p2p-1-p of 2*cp_p2p).  The first-level
 * all-to-all gives member a head slice a of its group's tokens (heads as
 * for the Ulysses variant with cp_a2a ranks), ordered as that second-level
 * shard; the members a of all groups then run the ring of cpattn_ring_fwd /
 * _bwd with cp_size = cp_p2p and the same layout on their head slice; the
 * inverse all-to-all returns the results to the token owners.
 * [cp, 1] is the Ulysses variant, [1, cp] the plain ring (through the copy).
 *
 * cpattn_hier_a2a: the first-level all-to-all on one GPU.
 *   to_seq = 0: in [B,S,X,D] sharded over cp ranks -> out
 *     [cp_a2a][B,S,nx,D]; block a holds member a's head slice, rows
 *     [p*S/cp_p2p, (p+1)*S/cp_p2p) being what member a of group p holds, in
 *     the second level's sharded order;
 *   to_seq = 1: the inverse; a kv head held by several members receives the
 *     sum of their rows.  kv_heads, dtype, alignment as cpattn_ulysses_a2a.
 * cpattn_hier_lse_a2a: the same for LSE, [B,H,S] <-> [cp_a2a][B,H/cp_a2a,S].
 * cpattn_hier_fwd / _bwd: the whole schedule on sharded-order tensors
 *   (shapes, dtypes and outputs as cpattn_ring_fwd / cpattn_ring_bwd): the
 *   all-to-all into the workspace, the second-level ring for every member in
 *   one launch (members stacked along the batch), the all-to-all back.
 *   doc_bounds: NULL or from cpattn_doc_bounds.  workspace: device, at least
 *   cpattn_hier_workspace_bytes(..., backward), 256-byte aligned, scratch.
 * Errors: CPATTN_ERR_INVALID_ARG for level sizes < 1, H % cp_a2a != 0, head
 * slices that do not divide the kv groups (or the reverse), S not split into
 * whole chunks at cp = cp_a2a * cp_p2p; CPATTN_ERR_WORKSPACE for a short or
 * misaligned workspace; otherwise as cpattn_ring_fwd / _bwd.
 */
CPATTN_API int cpattn_hier_a2a(const void* in, void* out, int B, int S, int H, int Hkv, int D,
                               int cp_a2a, int cp_p2p, int layout, int kv_heads, int to_seq,
                               int dtype, cpattn_stream_t stream);
CPATTN_API int cpattn_hier_lse_a2a(const float* in, float* out, int B, int S, int H, int cp_a2a,
                                   int cp_p2p, int layout, int to_seq, cpattn_stream_t stream);
CPATTN_API size_t cpattn_hier_workspace_bytes(int B, int H, int Hkv, int S, int D, int cp_a2a,
                                              int cp_p2p, int layout, int dtype, int backward);
CPATTN_API int cpattn_hier_fwd(const void* q, const void* k, const void* v, void* out,
                               float* lse, int B, int H, int Hkv, int S, int D, int cp_a2a,
                               int cp_p2p, int layout, int causal, int dtype,
                               float softmax_scale, const int32_t* doc_bounds, void* workspace,
                               size_t workspace_bytes, cpattn_stream_t stream);
CPATTN_API int cpattn_hier_bwd(const void* q, const void* k, const void* v, const void* out,
                               const void* dout, const float* lse, void* dq, void* dk, void* dv,
                               int B, int H, int Hkv, int S, int D, int cp_a2a, int cp_p2p,
                               int layout, int causal, int dtype, float softmax_scale,
                               const int32_t* doc_bounds, void* workspace,
                               size_t workspace_bytes, cpattn_stream_t stream);

/*
 * Sequence length to pad a sequence of S tokens to (host only): the smallest
 * multiple of cp_size * 256 (contiguous) or 2 * cp_size * 256 (zigzag) that
 * is >= S, so that every chunk is a whole number of 256-token query pairs
 * and the tensor-core kernels take the problem.  With zigzag the padding
 * lands in the last chunks (rank 0's second chunk first).  Returns -1 for
 * S < 0, cp_size < 1 or an unknown layout.
 */
CPATTN_API int64_t cpattn_padded_length(int64_t S, int cp_size, int layout);

/*
 * The whole path from HOST memory to HOST memory: natural-order q, k, v (and
 * dout) in host buffers, natural-order out, lse (and dq, dk, dv) written back
 * to host buffers; in between, on the device, the sharded layout, the ring
 * forward (cpattn_ring_fwd) and, when dout is not NULL, the ring backward
 * (cpattn_ring_bwd).  The zigzag permutation happens in the copies (one copy
 * per chunk and batch row).
 *   parts: the heads are processed in `parts` groups of whole kv-head groups
 *   (parts must divide Hkv; 1..8; 0 = the library's choice: the largest of
 *   8, 4, 2 that divides Hkv and leaves each part at least 64 MiB of bf16
 *   queries, else 1).  A part's
 *   inputs upload while the previous part computes and its results download
 *   while the next one computes, on two side streams (upload, download) the
 *   library creates once per device; only the first part's upload and the
 *   last part's download are exposed.  Results are bit for bit those of
 *   parts = 1 (heads are independent).
 *   The caller's stream waits for both side streams, so the call has
 *   finished when `stream` reaches that point.
 *   Host buffers: pinned memory for asynchronous copies (pageable memory
 *   works, synchronously); they must stay valid until `stream` gets there.
 *   dtype: as cpattn_ring_bwd (CPATTN_GRAD_F32 for float32 gradients).
 *   workspace: device, at least cpattn_attention_host_workspace_bytes (with
 *   backward = dout != NULL; the size covers every value of parts),
 *   256-byte aligned, scratch.  Calls that share a workspace, or that run on
 *   one device from several host threads at once (they share the side
 *   streams), must be serialised by the caller.
 *   Errors: CPATTN_ERR_INVALID_ARG for shapes as cpattn_ring_fwd, a parts
 *   value that does not divide Hkv or is outside 0..8, or a NULL buffer;
 *   CPATTN_ERR_WORKSPACE; CPATTN_ERR_CUDA when a copy or launch fails (the
 *   caller's stream still waits for what was enqueued).
 */
CPATTN_API size_t cpattn_attention_host_workspace_bytes(int B, int H, int Hkv, int S, int D,
                                                        int cp_size, int layout, int dtype,
                                                        int backward);
/* The number of parts cpattn_attention_host takes for parts = 0 (host only;
 * 1 for shapes it would reject). */
CPATTN_API int cpattn_attention_host_parts(int B, int H, int Hkv, int S, int D);
CPATTN_API int cpattn_attention_host(const void* q, const void* k, const void* v,
                                     const void* dout, void* out, float* lse, void* dq, void* dk,
                                     void* dv, int B, int H, int Hkv, int S, int D, int cp_size,
                                     int layout, int causal, int dtype, float softmax_scale,
                                     int parts, void* workspace, size_t workspace_bytes,
                                     cpattn_stream_t stream);

/*
 * cpattn_attention_host for packed documents and any sequence length: q, k,
 * v (and dout), out, lse (and dq, dk, dv) hold S real tokens in natural
 * order on the host ([B, S, H, D], lse [B, H, S]); on the device the
 * sequence is padded to cpattn_padded_length(S, cp_size, layout) (the
 * padding is one more document, zero on the device and never copied back)
 * and the ring runs under the document rule (cpattn_ring_fwd_docs /
 * cpattn_ring_bwd_docs).
 *   cu_seqlens: HOST int32 [ndocs + 1], 0 = cu[0] < ... < cu[ndocs] = S
 *   (checked here: CPATTN_ERR_INVALID_ARG otherwise), or NULL for one
 *   document.  Read before the call returns.
 *   workspace: at least cpattn_attention_host_docs_workspace_bytes.
 *   Everything else as cpattn_attention_host.
 */
CPATTN_API size_t cpattn_attention_host_docs_workspace_bytes(int B, int H, int Hkv, int S, int D,
                                                             int cp_size, int layout, int dtype,
                                                             int backward);
CPATTN_API int cpattn_attention_host_docs(const void* q, const void* k, const void* v,
                                          const void* dout, void* out, float* lse, void* dq,
                                          void* dk, void* dv, int B, int H, int Hkv, int S,
                                          int D, int cp_size, int layout, int causal, int dtype,
                                          float softmax_scale, const int32_t* cu_seqlens,
                                          int ndocs, int parts, void* workspace,
                                          size_t workspace_bytes, cpattn_stream_t stream);

/*
 * Closed-form work census of the ring (host only): for every rank r and
 * step t, the number of tile x tile blocks with at least one visible
 * (query, key) pair, tiles_rt[r*cp_size + t], and the number of visible
 * pairs, pairs_rt[r*cp_size + t], per (batch, head).  Either output may be
 * NULL.  Requires the chunk length to be a multiple of `tile`.
 * ("Sequence Parallelism IV ...", sections 3-4: the per-iteration balance
 * the zigzag layout is built for.)
 */
CPATTN_API int cpattn_tile_counts(int64_t S, int cp_size, int layout, int causal, int64_t tile,
                       uint64_t* tiles_rt, uint64_t* pairs_rt);

/*
 * Waits for `stream`, then reads and clears this device's error word.
 * Returns CPATTN_ERR_DEVICE_TIMEOUT if a kernel's bounded wait gave up since
 * the last call, CPATTN_ERR_INVALID_ARG if cpattn_doc_bounds found broken
 * document offsets since the last call, CPATTN_ERR_CUDA if the stream
 * reports a CUDA error, else CPATTN_OK.  Synchronous.
 */
CPATTN_API int cpattn_device_status(cpattn_stream_t stream);

/*
 * Checks the device-side failure path without faulting the GPU: launches one
 * CTA that waits, with the same bounded wait the attention kernels use, on an
 * mbarrier phase that never completes.  After limit_ns nanoseconds (1 ..
 * 2e9) the wait gives up, raises the device error word and the kernel
 * returns; the next cpattn_device_status reports CPATTN_ERR_DEVICE_TIMEOUT
 * (and clears it), and the context stays usable.  (The attention kernels'
 * waits give up after 2 s.)  The pages describe no such call.
 */
CPATTN_API int cpattn_wait_probe(int64_t limit_ns, cpattn_stream_t stream);

/* Static description of a status code (never NULL). */
CPATTN_API const char* cpattn_status_string(int status);

#ifdef __cplusplus
}
#endif

#endif /* CPATTN_H */
