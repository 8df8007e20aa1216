/*
 * cpattn_oracle.c -- plain, slow, fp64 CPU oracle for context-parallel
 * zigzag causal attention.
 *
 * TEST INFRASTRUCTURE ONLY.  Only tests/, __graft_entry__.smoke() and the
 * CPU-baseline leg of bench.py may load this library.  The product path
 * (libcpattn and its Python binding) never links, loads or calls it, and this
 * file includes no header and shares no helper with the CUDA path.
 *
 * What it computes and where that is defined:
 *
 *  - Softmax attention itself (the "unsharded reference"): "Context
 *    Parallelism for Long-Context Training", section "Prove attention
 *    equivalence" -- the sharded result must agree with CP=1, outputs and
 *    gradients, under causal masks.  Written out here from its plain
 *    definition: s_ij = scale * q_i . k_j over the valid set V(i) (j <= i when
 *    causal, all j otherwise), LSE_i = ln sum_j exp(s_ij),
 *    O_i = sum_j exp(s_ij - LSE_i) v_j.
 *  - The zigzag / load-balanced chunk placement: "Sequence Parallelism IV:
 *    Megatron Context Parallel and Load-Balanced Rings", section 3 -- the
 *    sequence is cut into 2*cp chunks and rank r holds chunks r and 2cp-1-r
 *    (the cp=4 assignment printed there is a golden fixture).  The contiguous
 *    placement (rank r holds tokens [r*S/cp, (r+1)*S/cp)) is the naive ring of
 *    the same section and the shard function of the runnable artifact on
 *    "Context Parallelism for Long-Context Training".
 *  - The ring: same page, section 4 -- Q stays on its rank, K/V blocks move
 *    around the group; each arriving block gives a partial output for the
 *    local query chunks; online-softmax state keeps the result exact.  Here:
 *    at ring step t rank r holds the K/V of rank (r - t) mod cp, each step
 *    gives a normalised partial (O_rt, L_rt) over that source's tokens (masked
 *    on natural positions), and the partials are merged with an exact
 *    log-add-exp (section 5, "update the online softmax state").
 *  - Gradients: the plain derivative of the definition above for a loss whose
 *    gradient with respect to O is dO: with Delta_i = dO_i . O_i and
 *    P_ij = exp(s_ij - LSE_i), dS_ij = P_ij (dO_i . v_j - Delta_i),
 *    dQ_i = scale sum_j dS_ij k_j, dK_j = scale sum_i dS_ij q_i,
 *    dV_j = sum_i P_ij dO_i (sums over i also run over the query heads that
 *    share kv head j).
 *  - Document (packed-sequence) masks: "Context Parallelism for Long-Context
 *    Training", sections "Prove attention equivalence" (causal and document
 *    masks must agree with CP=1) and "Test sequence divisibility and padding".
 *    Documents are the ranges [cu[d], cu[d+1]); the valid set V(i) above
 *    keeps only keys of i's own document.  Padding is read as one more
 *    document, so no real token sees a padded one.  The *_docs entry points
 *    take cu; the others use one document (cu = NULL).
 *  - Hierarchical context parallelism (a2a+p2p): "Context Parallelism in
 *    MegaDLMs", sections "Hierarchical Context Parallelism" and "Key-Value
 *    Communication Patterns" -- an all-to-all inside groups of A consecutive
 *    ranks, then the ring of the second level over the P groups (cp = A*P);
 *    see oracle_hier_a2a below for the reading.
 *
 * Readings where the pages are silent: tensors are [B, S, H, D] row-major,
 * LSE is [B, H, S] in natural log; query head h uses kv head h / (H / Hkv);
 * the ring direction is "rank r receives from r - 1"; inside a rank's shard
 * the early chunk comes first.
 *
 * Inputs are float32 arrays (they hold bf16- or fp32-valued data exactly) and
 * every sum is taken in double precision.
 *
 * Pins (tests/test_oracle.py): pure-Python brute force at S <= 16, the printed
 * cp=4 zigzag assignment, shard coverage, cp=1 equals the definition, ring
 * result independent of cp / layout / merge order, constant V gives V, Q = 0
 * gives the closed-form uniform average, row 0 gives v_0, central finite
 * differences for every gradient, the sum rules sum_j dV_j = sum_i dO_i and
 * sum_j dK_j = 0, closed-form tile / pair counts, and for documents: brute
 * force and finite differences with documents, one token per document in
 * closed form, packed documents equal to each document alone, one document
 * equal to the plain mask, the ring under documents equal to the definition,
 * and per-rank pair counts; the hierarchical all-to-all against the two
 * levels' token lists and the hierarchical schedule against the definition;
 * dK / dV on listed key rows against finite differences and the sum rules.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* Planted mistakes, compiled in only by the mutation tests (never by the
 * regular build).  Each one must make at least one pin fail. */
#ifndef ORACLE_MUTATION
#define ORACLE_MUTATION 0
#endif

enum { LAYOUT_CONTIGUOUS = 0, LAYOUT_ZIGZAG = 1 };

void oracle_set_threads(int n) {
#ifdef _OPENMP
  if (n > 0) omp_set_num_threads(n);
#else
  (void)n;
#endif
}

int oracle_get_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

/* ------------------------------------------------------------------------ */
/* Chunk placement                                                           */
/* ------------------------------------------------------------------------ */

/* Natural chunk ids held by rank r, in the order they sit in its shard.
 * Zigzag: chunks r and 2cp-1-r (early one first).  Contiguous: chunk r.
 * Returns the number of chunks per rank. */
static int rank_chunks(int r, int cp, int layout, int* out) {
  if (layout == LAYOUT_ZIGZAG) {
    out[0] = r;
    out[1] = 2 * cp - 1 - r;
#if ORACLE_MUTATION == 1
    out[1] = 2 * cp - 2 - r + (r == cp - 1 ? cp : 0); /* wrong pairing */
#endif
    return 2;
  }
  out[0] = r;
  return 1;
}

/* Fills nat_of_sharded[p] = natural token position of sharded position p, by
 * appending each rank's chunks in rank order.  Returns 0, or -1 if S does not
 * split into whole chunks. */
int oracle_shard_order(long S, int cp, int layout, long* nat_of_sharded) {
  if (cp < 1) return -1;
  int per_rank = (layout == LAYOUT_ZIGZAG) ? 2 : 1;
  long nchunk = (long)cp * per_rank;
  if (S % nchunk != 0) return -1;
  long c = S / nchunk;
  long p = 0;
  for (int r = 0; r < cp; ++r) {
    int ch[2];
    int n = rank_chunks(r, cp, layout, ch);
    for (int a = 0; a < n; ++a)
      for (long o = 0; o < c; ++o) nat_of_sharded[p++] = (long)ch[a] * c + o;
  }
  return 0;
}

/* Natural positions of every token held by rank s (its K/V, or its Q). */
static long rank_tokens(long S, int cp, int layout, int s, long* out) {
  int per_rank = (layout == LAYOUT_ZIGZAG) ? 2 : 1;
  long c = S / ((long)cp * per_rank);
  int ch[2];
  int n = rank_chunks(s, cp, layout, ch);
  long m = 0;
  for (int a = 0; a < n; ++a)
    for (long o = 0; o < c; ++o) out[m++] = (long)ch[a] * c + o;
  return m;
}

/* ------------------------------------------------------------------------ */
/* Softmax attention over an explicit key set                                */
/* ------------------------------------------------------------------------ */

static inline long idx4(long b, long s, long h, long d, long S, long H, long D) {
  return ((b * S + s) * H + h) * D + d;
}

static inline int kv_head_of(int h, int H, int Hkv) {
#if ORACLE_MUTATION == 2
  return h % Hkv; /* interleaved instead of consecutive grouping */
#else
  return h / (H / Hkv);
#endif
}

static inline int is_valid(long i, long j, int causal) {
#if ORACLE_MUTATION == 3
  return !causal || j < i; /* mask seam off by one: diagonal dropped */
#else
  return !causal || j <= i;
#endif
}

/* Which keys a query sees.  The causal rule above, and -- when cu is not NULL
 * -- the document rule of a packed sequence: documents are the position
 * ranges [cu[d], cu[d+1]), d = 0..ndocs-1, with cu[0] = 0 and cu[ndocs] = S,
 * and a token sees only tokens of its own document ("Context Parallelism for
 * Long-Context Training", "Prove attention equivalence": test causal and
 * document masks; "Test sequence divisibility and padding": padding is a
 * document of its own, so real tokens never see it). */
typedef struct {
  int causal;
  const long* cu;
  long ndocs;
} Mask;

static long doc_of(const Mask* m, long p) {
  for (long d = 0; d < m->ndocs; ++d)
#if ORACLE_MUTATION == 7
    if (p <= m->cu[d + 1]) return d;
#else
    if (p < m->cu[d + 1]) return d;
#endif
  return m->ndocs - 1;
}

static int visible(const Mask* m, long i, long j) {
  if (!is_valid(i, j, m->causal)) return 0;
  if (m->cu != NULL && doc_of(m, i) != doc_of(m, j)) return 0;
  return 1;
}

/* Normalised partial of query row (b, h, natural i) against the keys at the
 * natural positions keys[0..nk): o[0..D) and *l (natural-log LSE).  A row
 * with no valid key gives o = 0, l = -inf.  s_buf holds nk doubles. */
static void partial_row(const float* q, const float* k, const float* v, long B, int H,
                        int Hkv, long S, int D, const Mask* msk, double scale, long b, int h,
                        long i, const long* keys, long nk, double* s_buf, double* o,
                        double* l) {
  (void)B;
  int g = kv_head_of(h, H, Hkv);
  const float* qi = q + idx4(b, i, h, 0, S, H, D);
  double mx = -INFINITY;
  for (long a = 0; a < nk; ++a) {
    long j = keys[a];
    if (!visible(msk, i, j)) {
      s_buf[a] = -INFINITY;
      continue;
    }
    const float* kj = k + idx4(b, j, g, 0, S, Hkv, D);
    double dot = 0.0;
    for (int d = 0; d < D; ++d) dot += (double)qi[d] * (double)kj[d];
#if ORACLE_MUTATION == 4
    s_buf[a] = dot; /* softmax scale dropped */
#else
    s_buf[a] = scale * dot;
#endif
    if (s_buf[a] > mx) mx = s_buf[a];
  }
  for (int d = 0; d < D; ++d) o[d] = 0.0;
  if (mx == -INFINITY) {
    *l = -INFINITY;
    return;
  }
  double sum = 0.0;
  for (long a = 0; a < nk; ++a) {
    if (s_buf[a] == -INFINITY) continue;
    double w = exp(s_buf[a] - mx);
    sum += w;
    const float* vj = v + idx4(b, keys[a], g, 0, S, Hkv, D);
    for (int d = 0; d < D; ++d) o[d] += w * (double)vj[d];
  }
  for (int d = 0; d < D; ++d) o[d] /= sum;
  *l = mx + log(sum);
}

/* Full attention (the definition), natural order.  out [B,S,H,D], lse [B,H,S]. */
static void attn_fwd_m(const float* q, const float* k, const float* v, long B, int H, int Hkv,
                       long S, int D, const Mask* msk, double scale, double* out, double* lse) {
  long nrows = B * (long)H * S;
#pragma omp parallel
  {
    long* keys = (long*)malloc(sizeof(long) * S);
    double* sb = (double*)malloc(sizeof(double) * S);
    for (long j = 0; j < S; ++j) keys[j] = j;
#pragma omp for schedule(dynamic, 16)
    for (long row = 0; row < nrows; ++row) {
      long b = row / ((long)H * S);
      int h = (int)((row / S) % H);
      long i = row % S;
      double l;
      partial_row(q, k, v, B, H, Hkv, S, D, msk, scale, b, h, i, keys, S, sb,
                  out + idx4(b, i, h, 0, S, H, D), &l);
      lse[(b * H + h) * S + i] = l;
    }
    free(keys);
    free(sb);
  }
}

void oracle_attn_fwd(const float* q, const float* k, const float* v, long B, int H, int Hkv,
                     long S, int D, int causal, double scale, double* out, double* lse) {
  const Mask msk = {causal, NULL, 0};
  attn_fwd_m(q, k, v, B, H, Hkv, S, D, &msk, scale, out, lse);
}

/* The definition under the document rule (documents cu[0..ndocs]). */
void oracle_attn_fwd_docs(const float* q, const float* k, const float* v, long B, int H, int Hkv,
                          long S, int D, int causal, double scale, const long* cu, long ndocs,
                          double* out, double* lse) {
  const Mask msk = {causal, cu, ndocs};
  attn_fwd_m(q, k, v, B, H, Hkv, S, D, &msk, scale, out, lse);
}

/* The definition evaluated on a list of rows: rows[3*n + {0,1,2}] = (b, h, i)
 * natural.  out [n, D], lse [n]. */
static void attn_fwd_rows_m(const float* q, const float* k, const float* v, long B, int H,
                            int Hkv, long S, int D, const Mask* msk, double scale,
                            const long* rows, long n, double* out, double* lse) {
#pragma omp parallel
  {
    long* keys = (long*)malloc(sizeof(long) * S);
    double* sb = (double*)malloc(sizeof(double) * S);
    for (long j = 0; j < S; ++j) keys[j] = j;
#pragma omp for schedule(dynamic, 1)
    for (long a = 0; a < n; ++a) {
      partial_row(q, k, v, B, H, Hkv, S, D, msk, scale, rows[3 * a], (int)rows[3 * a + 1],
                  rows[3 * a + 2], keys, S, sb, out + a * D, lse + a);
    }
    free(keys);
    free(sb);
  }
}

void oracle_attn_fwd_rows(const float* q, const float* k, const float* v, long B, int H,
                          int Hkv, long S, int D, int causal, double scale, const long* rows,
                          long n, double* out, double* lse) {
  const Mask msk = {causal, NULL, 0};
  attn_fwd_rows_m(q, k, v, B, H, Hkv, S, D, &msk, scale, rows, n, out, lse);
}

void oracle_attn_fwd_rows_docs(const float* q, const float* k, const float* v, long B, int H,
                               int Hkv, long S, int D, int causal, double scale, const long* cu,
                               long ndocs, const long* rows, long n, double* out, double* lse) {
  const Mask msk = {causal, cu, ndocs};
  attn_fwd_rows_m(q, k, v, B, H, Hkv, S, D, &msk, scale, rows, n, out, lse);
}

/* ------------------------------------------------------------------------ */
/* Exact merge of two normalised partials                                    */
/* ------------------------------------------------------------------------ */

/* (o_a, l_a) (+) (o_b, l_b): L = log(e^La + e^Lb) taken as Lmax + log1p(e^(Lmin-Lmax)),
 * O = e^(La-L) O_a + e^(Lb-L) O_b.  An empty side (l = -inf) leaves the other
 * unchanged.  o may alias o_a or o_b. */
void oracle_lse_merge(const double* o_a, double l_a, const double* o_b, double l_b, int D,
                      double* o, double* l) {
  if (l_b == -INFINITY) {
    for (int d = 0; d < D; ++d) o[d] = o_a[d];
    *l = l_a;
    return;
  }
  if (l_a == -INFINITY) {
    for (int d = 0; d < D; ++d) o[d] = o_b[d];
    *l = l_b;
    return;
  }
  double hi = l_a > l_b ? l_a : l_b;
  double lo = l_a > l_b ? l_b : l_a;
  double L = hi + log1p(exp(lo - hi));
  double wa = exp(l_a - L), wb = exp(l_b - L);
#if ORACLE_MUTATION == 5
  wb = 0.0; /* dropped merge term */
#endif
  for (int d = 0; d < D; ++d) o[d] = wa * o_a[d] + wb * o_b[d];
  *l = L;
}

/* Array form used by the merge tests: O [B,S,H,D] doubles, LSE [B,H,S]. */
void oracle_lse_merge_arrays(const double* o_a, const double* l_a, const double* o_b,
                             const double* l_b, long B, long S, int H, int D, double* o,
                             double* l) {
#pragma omp parallel for schedule(static)
  for (long row = 0; row < B * S * H; ++row) {
    long b = row / (S * H), s = (row / H) % S;
    int h = (int)(row % H);
    long li = (b * H + h) * S + s;
    double lo;
    oracle_lse_merge(o_a + row * D, l_a[li], o_b + row * D, l_b[li], D, o + row * D, &lo);
    l[li] = lo;
  }
}

/* ------------------------------------------------------------------------ */
/* Sequential ring                                                           */
/* ------------------------------------------------------------------------ */

static int ring_source(int r, int t, int cp) {
#if ORACLE_MUTATION == 6
  return (r + t) % cp; /* ring turned the other way */
#else
  return ((r - t) % cp + cp) % cp;
#endif
}

/* Partial of ring step t for every rank: for each natural query row i, owned
 * by rank r, the normalised partial against the tokens of rank
 * (r - t) mod cp.  o_part [B,S,H,D], l_part [B,H,S], natural order. */
int oracle_ring_step(const float* q, const float* k, const float* v, long B, int H, int Hkv,
                     long S, int D, int cp, int layout, int causal, double scale, int t,
                     double* o_part, double* l_part) {
  int per_rank = (layout == LAYOUT_ZIGZAG) ? 2 : 1;
  if (cp < 1 || S % ((long)cp * per_rank) != 0 || t < 0 || t >= cp) return -1;
  const Mask msk = {causal, NULL, 0};
  long L = S / cp;
  for (int r = 0; r < cp; ++r) {
    long* qpos = (long*)malloc(sizeof(long) * L);
    long* kpos = (long*)malloc(sizeof(long) * L);
    rank_tokens(S, cp, layout, r, qpos);
    rank_tokens(S, cp, layout, ring_source(r, t, cp), kpos);
    long n = B * (long)H * L;
#pragma omp parallel
    {
      double* sb = (double*)malloc(sizeof(double) * L);
#pragma omp for schedule(dynamic, 16)
      for (long a = 0; a < n; ++a) {
        long b = a / ((long)H * L);
        int h = (int)((a / L) % H);
        long i = qpos[a % L];
        double l;
        partial_row(q, k, v, B, H, Hkv, S, D, &msk, scale, b, h, i, kpos, L, sb,
                    o_part + idx4(b, i, h, 0, S, H, D), &l);
        l_part[(b * H + h) * S + i] = l;
      }
      free(sb);
    }
    free(qpos);
    free(kpos);
  }
  return 0;
}

/* The whole ring: cp steps of partials, merged per row.  merge_order 0: t =
 * 0, 1, ..., cp-1 (left fold); 1: t = cp-1, ..., 0; 2: pairwise tree over t.
 * out [B,S,H,D], lse [B,H,S], natural order.  Returns 0 or -1 on bad
 * arguments. */
static int ring_fwd_m(const float* q, const float* k, const float* v, long B, int H, int Hkv,
                      long S, int D, int cp, int layout, const Mask* msk, double scale,
                      int merge_order, double* out, double* lse) {
  int per_rank = (layout == LAYOUT_ZIGZAG) ? 2 : 1;
  if (cp < 1 || S % ((long)cp * per_rank) != 0) return -1;
  long L = S / cp;
  long* qpos = (long*)malloc(sizeof(long) * L);
  long* kpos = (long*)malloc(sizeof(long) * L * cp);
  for (int r = 0; r < cp; ++r) {
    rank_tokens(S, cp, layout, r, qpos);
    for (int t = 0; t < cp; ++t) rank_tokens(S, cp, layout, ring_source(r, t, cp), kpos + t * L);
    long n = B * (long)H * L;
#pragma omp parallel
    {
      double* sb = (double*)malloc(sizeof(double) * L);
      double* po = (double*)malloc(sizeof(double) * D * cp);
      double* pl = (double*)malloc(sizeof(double) * cp);
#pragma omp for schedule(dynamic, 16)
      for (long a = 0; a < n; ++a) {
        long b = a / ((long)H * L);
        int h = (int)((a / L) % H);
        long i = qpos[a % L];
        for (int t = 0; t < cp; ++t)
          partial_row(q, k, v, B, H, Hkv, S, D, msk, scale, b, h, i, kpos + t * L, L, sb,
                      po + t * D, pl + t);
        if (merge_order == 2) {
          for (int w = 1; w < cp; w *= 2)
            for (int t = 0; t + w < cp; t += 2 * w)
              oracle_lse_merge(po + t * D, pl[t], po + (t + w) * D, pl[t + w], D, po + t * D,
                               pl + t);
        } else if (merge_order == 1) {
          for (int t = cp - 2; t >= 0; --t)
            oracle_lse_merge(po + (cp - 1) * D, pl[cp - 1], po + t * D, pl[t], D,
                             po + (cp - 1) * D, pl + cp - 1);
          memcpy(po, po + (cp - 1) * D, sizeof(double) * D);
          pl[0] = pl[cp - 1];
        } else {
          for (int t = 1; t < cp; ++t)
            oracle_lse_merge(po, pl[0], po + t * D, pl[t], D, po, pl);
        }
        memcpy(out + idx4(b, i, h, 0, S, H, D), po, sizeof(double) * D);
        lse[(b * H + h) * S + i] = pl[0];
      }
      free(sb);
      free(po);
      free(pl);
    }
  }
  free(qpos);
  free(kpos);
  return 0;
}

int oracle_ring_fwd(const float* q, const float* k, const float* v, long B, int H, int Hkv,
                    long S, int D, int cp, int layout, int causal, double scale,
                    int merge_order, double* out, double* lse) {
  const Mask msk = {causal, NULL, 0};
  return ring_fwd_m(q, k, v, B, H, Hkv, S, D, cp, layout, &msk, scale, merge_order, out, lse);
}

/* The ring under the document rule: a step whose keys hold nothing of a
 * query's document gives that query the neutral partial (0, -inf). */
int oracle_ring_fwd_docs(const float* q, const float* k, const float* v, long B, int H, int Hkv,
                         long S, int D, int cp, int layout, int causal, double scale,
                         const long* cu, long ndocs, int merge_order, double* out, double* lse) {
  const Mask msk = {causal, cu, ndocs};
  return ring_fwd_m(q, k, v, B, H, Hkv, S, D, cp, layout, &msk, scale, merge_order, out, lse);
}

/* ------------------------------------------------------------------------ */
/* The all-gather schedule                                                   */
/* ------------------------------------------------------------------------ */

/* Sharded <-> natural copies of a [B, S, X, D] float tensor with the chunker
 * above: natural[b, nat[p]] = sharded[b, p]. */
static void unshard_f(const float* sh, float* nat, const long* nat_of, long B, long S, long X,
                      int D) {
  for (long b = 0; b < B; ++b)
    for (long p = 0; p < S; ++p)
      memcpy(nat + idx4(b, nat_of[p], 0, 0, S, X, D), sh + idx4(b, p, 0, 0, S, X, D),
             sizeof(float) * X * D);
}

/* The all-gather variant of context parallelism ("Context Parallelism in
 * MegaDLMs", key-value communication patterns: the ranks exchange K/V before
 * attention so that each holds the whole context).  Inputs are in sharded
 * order, as the ranks hold them.  Step 1, all-gather: every rank r builds the
 * whole K/V in natural order from all ranks' shards (shard s lands on the
 * natural positions of s's chunks).  Step 2: r's own query tokens attend to
 * the gathered K/V in one pass -- no ring steps, no partials to merge.  Out
 * and LSE are written at r's own (sharded) positions.  Returns 0, or -1 if S
 * does not split into chunks. */
static int allgather_fwd_m(const float* q_sh, const float* k_sh, const float* v_sh, long B, int H,
                           int Hkv, long S, int D, int cp, int layout, const Mask* msk,
                           double scale, double* out_sh, double* lse_sh) {
  long* nat_of = (long*)malloc(sizeof(long) * (S > 0 ? S : 1));
  if (oracle_shard_order(S, cp, layout, nat_of) != 0) {
    free(nat_of);
    return -1;
  }
  float* qn = (float*)malloc(sizeof(float) * B * S * H * D + 1);
  float* kn = (float*)malloc(sizeof(float) * B * S * Hkv * D + 1);
  float* vn = (float*)malloc(sizeof(float) * B * S * Hkv * D + 1);
  unshard_f(q_sh, qn, nat_of, B, S, H, D);  /* only to index r's own queries */
  unshard_f(k_sh, kn, nat_of, B, S, Hkv, D); /* the all-gather of K */
  unshard_f(v_sh, vn, nat_of, B, S, Hkv, D); /* and of V */
  const long L = S / cp;
  for (int r = 0; r < cp; ++r) {
#pragma omp parallel
    {
      long* keys = (long*)malloc(sizeof(long) * S);
      double* sb = (double*)malloc(sizeof(double) * S);
      for (long j = 0; j < S; ++j) keys[j] = j;
#pragma omp for schedule(dynamic, 16)
      for (long a = 0; a < B * H * L; ++a) {
        long b = a / (H * L);
        int h = (int)((a / L) % H);
        long p = r * L + a % L; /* r's sharded position */
        partial_row(qn, kn, vn, B, H, Hkv, S, D, msk, scale, b, h, nat_of[p], keys, S, sb,
                    out_sh + idx4(b, p, h, 0, S, H, D), lse_sh + (b * H + h) * S + p);
      }
      free(keys);
      free(sb);
    }
  }
  free(qn);
  free(kn);
  free(vn);
  free(nat_of);
  return 0;
}

int oracle_allgather_fwd(const float* q_sh, const float* k_sh, const float* v_sh, long B, int H,
                         int Hkv, long S, int D, int cp, int layout, int causal, double scale,
                         const long* cu, long ndocs, double* out_sh, double* lse_sh) {
  const Mask msk = {causal, cu, ndocs};
  return allgather_fwd_m(q_sh, k_sh, v_sh, B, H, Hkv, S, D, cp, layout, &msk, scale, out_sh,
                         lse_sh);
}

/* ------------------------------------------------------------------------ */
/* The Ulysses (all-to-all) variant                                          */
/* ------------------------------------------------------------------------ */

/* Heads of rank r after the sequence-to-head all-to-all ("Sequence
 * Parallelism IV", section 7: after the transpose a rank has all tokens for
 * a head slice).  Query heads: the r-th of cp equal slices, H/cp heads.  KV
 * heads: those the slice's query heads read (query head h reads kv head
 * h / (H/Hkv)); when a slice holds fewer query heads than a kv group, one kv
 * head, shared with the other ranks of the group. */
static void ulysses_heads(int r, int cp, int H, int Hkv, int* q0, int* nq, int* g0, int* ng) {
  const int hc = H / cp, grp = H / Hkv;
  *q0 = r * hc;
  *nq = hc;
  *g0 = (r * hc) / grp;
#if ORACLE_MUTATION == 9
  *g0 = (((r + 1) % cp) * hc) / grp; /* kv slice of the wrong rank */
#endif
  *ng = hc >= grp ? hc / grp : 1;
}

/* The sequence-to-head all-to-all for one rank: from sharded [B,S,X,D]
 * (rank s holds sharded rows [s*L, (s+1)*L)) to rank r's [B,S,nx,D] holding
 * heads x0..x0+nx-1 of every token in natural order. */
static void a2a_to_rank(const float* sh, float* out, const long* nat_of, long B, long S, int X,
                        int x0, int nx, int D) {
  for (long b = 0; b < B; ++b)
    for (long p = 0; p < S; ++p)
      memcpy(out + idx4(b, nat_of[p], 0, 0, S, nx, D), sh + idx4(b, p, x0, 0, S, X, D),
             sizeof(float) * nx * D);
}

/* The all-to-all itself, as an entry point: out is [cp][B,S,nx,D], rank r's
 * head slice (query heads when kv = 0, its kv heads when kv = 1). */
int oracle_ulysses_a2a(const float* sh, long B, long S, int H, int Hkv, int D, int cp, int layout,
                       int kv, float* out) {
  if (cp < 1 || H % cp != 0 || H % Hkv != 0) return -1;
  const int hc = H / cp, grp = H / Hkv;
  if (hc % grp != 0 && grp % hc != 0) return -1;
  long* nat_of = (long*)malloc(sizeof(long) * (S > 0 ? S : 1));
  if (oracle_shard_order(S, cp, layout, nat_of) != 0) {
    free(nat_of);
    return -1;
  }
  for (int r = 0; r < cp; ++r) {
    int q0, nq, g0, ng;
    ulysses_heads(r, cp, H, Hkv, &q0, &nq, &g0, &ng);
    const int X = kv ? Hkv : H, x0 = kv ? g0 : q0, nx = kv ? ng : nq;
    a2a_to_rank(sh, out + (long)r * B * S * nx * D, nat_of, B, S, X, x0, nx, D);
  }
  free(nat_of);
  return 0;
}

/* Ulysses attention ("Sequence Parallelism IV", section 7), sharded order in
 * and out: the all-to-all gives each rank all tokens of its head slice; each
 * rank computes full attention (the definition) over the whole sequence for
 * those heads; the inverse all-to-all returns out and LSE to the sequence
 * owners. */
static int ulysses_fwd_m(const float* q_sh, const float* k_sh, const float* v_sh, long B, int H,
                         int Hkv, long S, int D, int cp, int layout, const Mask* msk,
                         double scale, double* out_sh, double* lse_sh) {
  if (cp < 1 || H % cp != 0 || H % Hkv != 0) return -1;
  const int hc = H / cp, grp = H / Hkv;
  if (hc % grp != 0 && grp % hc != 0) return -1;
  long* nat_of = (long*)malloc(sizeof(long) * (S > 0 ? S : 1));
  if (oracle_shard_order(S, cp, layout, nat_of) != 0) {
    free(nat_of);
    return -1;
  }
  for (int r = 0; r < cp; ++r) {
    int q0, nq, g0, ng;
    ulysses_heads(r, cp, H, Hkv, &q0, &nq, &g0, &ng);
    float* qr = (float*)malloc(sizeof(float) * B * S * nq * D + 1);
    float* kr = (float*)malloc(sizeof(float) * B * S * ng * D + 1);
    float* vr = (float*)malloc(sizeof(float) * B * S * ng * D + 1);
    double* orr = (double*)malloc(sizeof(double) * B * S * nq * D + 1);
    double* lr = (double*)malloc(sizeof(double) * B * nq * S + 1);
    a2a_to_rank(q_sh, qr, nat_of, B, S, H, q0, nq, D);
    a2a_to_rank(k_sh, kr, nat_of, B, S, Hkv, g0, ng, D);
    a2a_to_rank(v_sh, vr, nat_of, B, S, Hkv, g0, ng, D);
    attn_fwd_m(qr, kr, vr, B, nq, ng, S, D, msk, scale, orr, lr);
    /* Inverse all-to-all: rank r's heads go back to the token owners. */
    for (long b = 0; b < B; ++b)
      for (long p = 0; p < S; ++p) {
        const long n = nat_of[p];
        memcpy(out_sh + idx4(b, p, q0, 0, S, H, D), orr + idx4(b, n, 0, 0, S, nq, D),
               sizeof(double) * nq * D);
        for (int h = 0; h < nq; ++h)
          lse_sh[(b * H + q0 + h) * S + p] = lr[(b * nq + h) * S + n];
      }
    free(qr);
    free(kr);
    free(vr);
    free(orr);
    free(lr);
  }
  free(nat_of);
  return 0;
}

int oracle_ulysses_fwd(const float* q_sh, const float* k_sh, const float* v_sh, long B, int H,
                       int Hkv, long S, int D, int cp, int layout, int causal, double scale,
                       const long* cu, long ndocs, double* out_sh, double* lse_sh) {
  const Mask msk = {causal, cu, ndocs};
  return ulysses_fwd_m(q_sh, k_sh, v_sh, B, H, Hkv, S, D, cp, layout, &msk, scale, out_sh,
                       lse_sh);
}

static void attn_bwd_m(const float* q, const float* k, const float* v, const float* dout,
                       long B, int H, int Hkv, long S, int D, const Mask* msk, double scale,
                       double* dq, double* dk, double* dv);

/* Ulysses backward, sharded order in and out: dO follows the all-to-all to
 * the head owners, each rank takes the gradients of full attention for its
 * heads, and the inverse all-to-all returns dQ, dK, dV to the token owners;
 * a kv head held by several ranks receives the sum of their dK / dV. */
static int ulysses_bwd_m(const float* q_sh, const float* k_sh, const float* v_sh,
                         const float* do_sh, long B, int H, int Hkv, long S, int D, int cp,
                         int layout, const Mask* msk, double scale, double* dq_sh, double* dk_sh,
                         double* dv_sh) {
  if (cp < 1 || H % cp != 0 || H % Hkv != 0) return -1;
  const int hc = H / cp, grp = H / Hkv;
  if (hc % grp != 0 && grp % hc != 0) return -1;
  long* nat_of = (long*)malloc(sizeof(long) * (S > 0 ? S : 1));
  if (oracle_shard_order(S, cp, layout, nat_of) != 0) {
    free(nat_of);
    return -1;
  }
  memset(dk_sh, 0, sizeof(double) * B * S * Hkv * D);
  memset(dv_sh, 0, sizeof(double) * B * S * Hkv * D);
  for (int r = 0; r < cp; ++r) {
    int q0, nq, g0, ng;
    ulysses_heads(r, cp, H, Hkv, &q0, &nq, &g0, &ng);
    float* qr = (float*)malloc(sizeof(float) * B * S * nq * D + 1);
    float* dor = (float*)malloc(sizeof(float) * B * S * nq * D + 1);
    float* kr = (float*)malloc(sizeof(float) * B * S * ng * D + 1);
    float* vr = (float*)malloc(sizeof(float) * B * S * ng * D + 1);
    double* dqr = (double*)malloc(sizeof(double) * B * S * nq * D + 1);
    double* dkr = (double*)malloc(sizeof(double) * B * S * ng * D + 1);
    double* dvr = (double*)malloc(sizeof(double) * B * S * ng * D + 1);
    a2a_to_rank(q_sh, qr, nat_of, B, S, H, q0, nq, D);
    a2a_to_rank(do_sh, dor, nat_of, B, S, H, q0, nq, D);
    a2a_to_rank(k_sh, kr, nat_of, B, S, Hkv, g0, ng, D);
    a2a_to_rank(v_sh, vr, nat_of, B, S, Hkv, g0, ng, D);
    attn_bwd_m(qr, kr, vr, dor, B, nq, ng, S, D, msk, scale, dqr, dkr, dvr);
    for (long b = 0; b < B; ++b)
      for (long p = 0; p < S; ++p) {
        const long n = nat_of[p];
        memcpy(dq_sh + idx4(b, p, q0, 0, S, H, D), dqr + idx4(b, n, 0, 0, S, nq, D),
               sizeof(double) * nq * D);
        for (long x = 0; x < (long)ng * D; ++x) {
          dk_sh[idx4(b, p, g0, 0, S, Hkv, D) + x] += dkr[idx4(b, n, 0, 0, S, ng, D) + x];
          dv_sh[idx4(b, p, g0, 0, S, Hkv, D) + x] += dvr[idx4(b, n, 0, 0, S, ng, D) + x];
        }
      }
    free(qr);
    free(dor);
    free(kr);
    free(vr);
    free(dqr);
    free(dkr);
    free(dvr);
  }
  free(nat_of);
  return 0;
}

int oracle_ulysses_bwd(const float* q_sh, const float* k_sh, const float* v_sh,
                       const float* do_sh, long B, int H, int Hkv, long S, int D, int cp,
                       int layout, int causal, double scale, const long* cu, long ndocs,
                       double* dq_sh, double* dk_sh, double* dv_sh) {
  const Mask msk = {causal, cu, ndocs};
  return ulysses_bwd_m(q_sh, k_sh, v_sh, do_sh, B, H, Hkv, S, D, cp, layout, &msk, scale, dq_sh,
                       dk_sh, dv_sh);
}

/* ------------------------------------------------------------------------ */
/* Hierarchical context parallelism: all-to-all inside groups, ring across   */
/* ------------------------------------------------------------------------ */

/* "Context Parallelism in MegaDLMs", sections "Hierarchical Context
 * Parallelism" (a list of level sizes such as [2, 2] splits the context
 * group over two levels) and "Key-Value Communication Patterns" (the
 * a2a+p2p type combines the all-to-all and the point-to-point ring).
 * Reading: the sizes are [A, P] with cp = A * P; the first level is an
 * all-to-all among A consecutive ranks (a group), the second a ring among
 * the P groups.  Global rank r = p * A + a is member a of group p.  The
 * sequence is sharded over all cp ranks with the chosen layout (zigzag:
 * 2*cp chunks).  The all-to-all gives member a of group p head slice a
 * (ulysses_heads with A slices) of every token its group holds, ordered as
 * shard p of the second level (zigzag: level-two chunks p and 2P-1-p of
 * 2P); the members a of all P groups then run the ring of the second level
 * on that head slice, and the inverse all-to-all returns out, LSE and the
 * gradients to the token owners. */
static int hier_rank(int p, int a, int A, int P) {
#if ORACLE_MUTATION == 11
  (void)A;
  return a * P + p; /* groups of strided ranks: the wrong level */
#else
  (void)P;
  return p * A + a;
#endif
}

/* The first-level all-to-all, as an entry point: sh [B,S,X,D] sharded over
 * cp = A*P ranks -> out [A][B][S][nx][D]; block a holds member a's head
 * slice, rows [p*S/P, (p+1)*S/P) being what member a of group p holds, in
 * the order of level-two shard p.  Returns -1 on bad arguments or when a
 * group does not hold exactly the tokens of its level-two shard. */
int oracle_hier_a2a(const float* sh, long B, long S, int H, int Hkv, int D, int A, int P,
                    int layout, int kv, float* out) {
  if (A < 1 || P < 1 || H % A != 0 || H % Hkv != 0) return -1;
  const int hc = H / A, grp = H / Hkv;
  if (hc % grp != 0 && grp % hc != 0) return -1;
  const int cp = A * P;
  long* nat_of = (long*)malloc(sizeof(long) * (S > 0 ? S : 1));
  long* slot = (long*)malloc(sizeof(long) * (S > 0 ? S : 1));
  long* tok = (long*)malloc(sizeof(long) * (S > 0 ? S : 1));
  int rc = 0;
  if (oracle_shard_order(S, cp, layout, nat_of) != 0 || oracle_shard_order(S, P, layout, tok))
    rc = -1;
  const long L = S / cp, LP = S / P;
  for (int p = 0; p < P && rc == 0; ++p) {
    /* Where each token of the group sits in the cp-level sharded tensor. */
    for (long n = 0; n < S; ++n) slot[n] = -1;
    for (int a = 0; a < A; ++a) {
      const long r = hier_rank(p, a, A, P);
      for (long o = 0; o < L; ++o) slot[nat_of[r * L + o]] = r * L + o;
    }
    rank_tokens(S, P, layout, p, tok); /* level-two shard p, in its order */
    for (long m = 0; m < LP; ++m)
      if (slot[tok[m]] < 0) rc = -1;
    for (int a = 0; a < A && rc == 0; ++a) {
      int q0, nq, g0, ng;
      ulysses_heads(a, A, H, Hkv, &q0, &nq, &g0, &ng);
      const int X = kv ? Hkv : H, x0 = kv ? g0 : q0, nx = kv ? ng : nq;
      for (long b = 0; b < B; ++b)
        for (long m = 0; m < LP; ++m)
          memcpy(out + (((long)a * B + b) * S + p * LP + m) * nx * D,
                 sh + idx4(b, slot[tok[m]], x0, 0, S, X, D), sizeof(float) * nx * D);
    }
  }
  free(nat_of);
  free(slot);
  free(tok);
  return rc;
}

/* Member a's head slice of every token in natural order, from the
 * all-to-all's block a (level-two sharded order). */
static void hier_block_natural(const float* blk, float* nat, long B, long S, int nx, int D, int P,
                               int layout, long* tmp) {
  oracle_shard_order(S, P, layout, tmp);
  for (long b = 0; b < B; ++b)
    for (long m = 0; m < S; ++m)
      memcpy(nat + idx4(b, tmp[m], 0, 0, S, nx, D), blk + ((b * S + m) * nx) * D,
             sizeof(float) * nx * D);
}

/* Hierarchical forward, sharded order in and out: the all-to-all, the ring
 * of the second level (P ranks) on each member's head slice, the inverse
 * all-to-all. */
static int hier_fwd_m(const float* q_sh, const float* k_sh, const float* v_sh, long B, int H,
                      int Hkv, long S, int D, int A, int P, int layout, const Mask* msk,
                      double scale, double* out_sh, double* lse_sh) {
  if (A < 1 || P < 1 || H % A != 0 || H % Hkv != 0) return -1;
  const int hc = H / A, grp = H / Hkv;
  if (hc % grp != 0 && grp % hc != 0) return -1;
  const int nkv = hc >= grp ? hc / grp : 1;
  long* nat_of = (long*)malloc(sizeof(long) * (S > 0 ? S : 1));
  long* tmp = (long*)malloc(sizeof(long) * (S > 0 ? S : 1));
  float* qa = (float*)malloc(sizeof(float) * A * B * S * hc * D + 1);
  float* ka = (float*)malloc(sizeof(float) * A * B * S * nkv * D + 1);
  float* va = (float*)malloc(sizeof(float) * A * B * S * nkv * D + 1);
  float* qn = (float*)malloc(sizeof(float) * B * S * hc * D + 1);
  float* kn = (float*)malloc(sizeof(float) * B * S * nkv * D + 1);
  float* vn = (float*)malloc(sizeof(float) * B * S * nkv * D + 1);
  double* on = (double*)malloc(sizeof(double) * B * S * hc * D + 1);
  double* ln = (double*)malloc(sizeof(double) * B * hc * S + 1);
  int rc = oracle_shard_order(S, A * P, layout, nat_of);
  if (rc == 0) rc = oracle_hier_a2a(q_sh, B, S, H, Hkv, D, A, P, layout, 0, qa);
  if (rc == 0) rc = oracle_hier_a2a(k_sh, B, S, H, Hkv, D, A, P, layout, 1, ka);
  if (rc == 0) rc = oracle_hier_a2a(v_sh, B, S, H, Hkv, D, A, P, layout, 1, va);
  for (int a = 0; a < A && rc == 0; ++a) {
    int q0, nq, g0, ng;
    ulysses_heads(a, A, H, Hkv, &q0, &nq, &g0, &ng);
    hier_block_natural(qa + (long)a * B * S * hc * D, qn, B, S, hc, D, P, layout, tmp);
    hier_block_natural(ka + (long)a * B * S * nkv * D, kn, B, S, nkv, D, P, layout, tmp);
    hier_block_natural(va + (long)a * B * S * nkv * D, vn, B, S, nkv, D, P, layout, tmp);
    rc = ring_fwd_m(qn, kn, vn, B, nq, ng, S, D, P, layout, msk, scale, 0, on, ln);
    for (long b = 0; b < B && rc == 0; ++b)
      for (long p = 0; p < S; ++p) {
        const long n = nat_of[p];
        memcpy(out_sh + idx4(b, p, q0, 0, S, H, D), on + idx4(b, n, 0, 0, S, nq, D),
               sizeof(double) * nq * D);
        for (int h = 0; h < nq; ++h) lse_sh[(b * H + q0 + h) * S + p] = ln[(b * nq + h) * S + n];
      }
  }
  free(nat_of);
  free(tmp);
  free(qa);
  free(ka);
  free(va);
  free(qn);
  free(kn);
  free(vn);
  free(on);
  free(ln);
  return rc;
}

int oracle_hier_fwd(const float* q_sh, const float* k_sh, const float* v_sh, long B, int H,
                    int Hkv, long S, int D, int A, int P, int layout, int causal, double scale,
                    const long* cu, long ndocs, double* out_sh, double* lse_sh) {
  const Mask msk = {causal, cu, ndocs};
  return hier_fwd_m(q_sh, k_sh, v_sh, B, H, Hkv, S, D, A, P, layout, &msk, scale, out_sh,
                    lse_sh);
}

/* Hierarchical backward, sharded order in and out: dO follows the
 * all-to-all; each member takes the gradients of attention on its head
 * slice (the ring of the second level reaches the same sums); the inverse
 * all-to-all returns dQ, dK, dV to the token owners, a kv head held by
 * several members receiving the sum of their dK / dV. */
static int hier_bwd_m(const float* q_sh, const float* k_sh, const float* v_sh,
                      const float* do_sh, long B, int H, int Hkv, long S, int D, int A, int P,
                      int layout, const Mask* msk, double scale, double* dq_sh, double* dk_sh,
                      double* dv_sh) {
  if (A < 1 || P < 1 || H % A != 0 || H % Hkv != 0) return -1;
  const int hc = H / A, grp = H / Hkv;
  if (hc % grp != 0 && grp % hc != 0) return -1;
  const int nkv = hc >= grp ? hc / grp : 1;
  long* nat_of = (long*)malloc(sizeof(long) * (S > 0 ? S : 1));
  long* tmp = (long*)malloc(sizeof(long) * (S > 0 ? S : 1));
  float* qa = (float*)malloc(sizeof(float) * A * B * S * hc * D + 1);
  float* da = (float*)malloc(sizeof(float) * A * B * S * hc * D + 1);
  float* ka = (float*)malloc(sizeof(float) * A * B * S * nkv * D + 1);
  float* va = (float*)malloc(sizeof(float) * A * B * S * nkv * D + 1);
  float* qn = (float*)malloc(sizeof(float) * B * S * hc * D + 1);
  float* dn = (float*)malloc(sizeof(float) * B * S * hc * D + 1);
  float* kn = (float*)malloc(sizeof(float) * B * S * nkv * D + 1);
  float* vn = (float*)malloc(sizeof(float) * B * S * nkv * D + 1);
  double* dqn = (double*)malloc(sizeof(double) * B * S * hc * D + 1);
  double* dkn = (double*)malloc(sizeof(double) * B * S * nkv * D + 1);
  double* dvn = (double*)malloc(sizeof(double) * B * S * nkv * D + 1);
  int rc = oracle_shard_order(S, A * P, layout, nat_of);
  if (rc == 0) rc = oracle_hier_a2a(q_sh, B, S, H, Hkv, D, A, P, layout, 0, qa);
  if (rc == 0) rc = oracle_hier_a2a(do_sh, B, S, H, Hkv, D, A, P, layout, 0, da);
  if (rc == 0) rc = oracle_hier_a2a(k_sh, B, S, H, Hkv, D, A, P, layout, 1, ka);
  if (rc == 0) rc = oracle_hier_a2a(v_sh, B, S, H, Hkv, D, A, P, layout, 1, va);
  if (rc == 0) {
    memset(dk_sh, 0, sizeof(double) * B * S * Hkv * D);
    memset(dv_sh, 0, sizeof(double) * B * S * Hkv * D);
  }
  for (int a = 0; a < A && rc == 0; ++a) {
    int q0, nq, g0, ng;
    ulysses_heads(a, A, H, Hkv, &q0, &nq, &g0, &ng);
    hier_block_natural(qa + (long)a * B * S * hc * D, qn, B, S, hc, D, P, layout, tmp);
    hier_block_natural(da + (long)a * B * S * hc * D, dn, B, S, hc, D, P, layout, tmp);
    hier_block_natural(ka + (long)a * B * S * nkv * D, kn, B, S, nkv, D, P, layout, tmp);
    hier_block_natural(va + (long)a * B * S * nkv * D, vn, B, S, nkv, D, P, layout, tmp);
    attn_bwd_m(qn, kn, vn, dn, B, nq, ng, S, D, msk, scale, dqn, dkn, dvn);
    for (long b = 0; b < B; ++b)
      for (long p = 0; p < S; ++p) {
        const long n = nat_of[p];
        memcpy(dq_sh + idx4(b, p, q0, 0, S, H, D), dqn + idx4(b, n, 0, 0, S, nq, D),
               sizeof(double) * nq * D);
        for (long x = 0; x < (long)ng * D; ++x) {
          dk_sh[idx4(b, p, g0, 0, S, Hkv, D) + x] += dkn[idx4(b, n, 0, 0, S, ng, D) + x];
          dv_sh[idx4(b, p, g0, 0, S, Hkv, D) + x] += dvn[idx4(b, n, 0, 0, S, ng, D) + x];
        }
      }
  }
  free(nat_of);
  free(tmp);
  free(qa);
  free(da);
  free(ka);
  free(va);
  free(qn);
  free(dn);
  free(kn);
  free(vn);
  free(dqn);
  free(dkn);
  free(dvn);
  return rc;
}

int oracle_hier_bwd(const float* q_sh, const float* k_sh, const float* v_sh, const float* do_sh,
                    long B, int H, int Hkv, long S, int D, int A, int P, int layout, int causal,
                    double scale, const long* cu, long ndocs, double* dq_sh, double* dk_sh,
                    double* dv_sh) {
  const Mask msk = {causal, cu, ndocs};
  return hier_bwd_m(q_sh, k_sh, v_sh, do_sh, B, H, Hkv, S, D, A, P, layout, &msk, scale, dq_sh,
                    dk_sh, dv_sh);
}

/* ------------------------------------------------------------------------ */
/* Gradients                                                                 */
/* ------------------------------------------------------------------------ */

static double dot_f(const float* a, const float* b, int D) {
  double s = 0.0;
  for (int d = 0; d < D; ++d) s += (double)a[d] * (double)b[d];
  return s;
}

/* dQ, dK, dV of the definition for the upstream gradient dout = dL/dO.
 * All natural order, dq [B,S,H,D], dk/dv [B,S,Hkv,D]. */
static void attn_bwd_m(const float* q, const float* k, const float* v, const float* dout,
                       long B, int H, int Hkv, long S, int D, const Mask* msk, double scale,
                       double* dq, double* dk, double* dv) {
  double* o = (double*)malloc(sizeof(double) * B * S * H * D);
  double* lse = (double*)malloc(sizeof(double) * B * H * S);
  double* delta = (double*)malloc(sizeof(double) * B * H * S);
  attn_fwd_m(q, k, v, B, H, Hkv, S, D, msk, scale, o, lse);
#pragma omp parallel for schedule(static)
  for (long row = 0; row < B * S * H; ++row) {
    long b = row / (S * H), i = (row / H) % S;
    int h = (int)(row % H);
    double s = 0.0;
    for (int d = 0; d < D; ++d) s += (double)dout[row * D + d] * o[row * D + d];
    delta[(b * H + h) * S + i] = s;
  }
  /* dQ: one query row at a time. */
#pragma omp parallel for schedule(dynamic, 16)
  for (long row = 0; row < B * S * H; ++row) {
    long b = row / (S * H), i = (row / H) % S;
    int h = (int)(row % H);
    int g = kv_head_of(h, H, Hkv);
    const float* qi = q + row * D;
    const float* doi = dout + row * D;
    double l = lse[(b * H + h) * S + i], dl = delta[(b * H + h) * S + i];
    double* dqi = dq + row * D;
    for (int d = 0; d < D; ++d) dqi[d] = 0.0;
    for (long j = 0; j < S; ++j) {
      if (!visible(msk, i, j)) continue;
      const float* kj = k + idx4(b, j, g, 0, S, Hkv, D);
      const float* vj = v + idx4(b, j, g, 0, S, Hkv, D);
      double p = exp(scale * dot_f(qi, kj, D) - l);
      double ds = p * (dot_f(doi, vj, D) - dl);
      for (int d = 0; d < D; ++d) dqi[d] += scale * ds * (double)kj[d];
    }
  }
  /* dK, dV: one key row at a time, summed over the query heads sharing it. */
  int grp = H / Hkv;
#pragma omp parallel for schedule(dynamic, 16)
  for (long krow = 0; krow < B * S * Hkv; ++krow) {
    long b = krow / (S * Hkv), j = (krow / Hkv) % S;
    int g = (int)(krow % Hkv);
    const float* kj = k + krow * D;
    const float* vj = v + krow * D;
    double* dkj = dk + krow * D;
    double* dvj = dv + krow * D;
    for (int d = 0; d < D; ++d) dkj[d] = dvj[d] = 0.0;
    for (int h = 0; h < H; ++h) {
      if (kv_head_of(h, H, Hkv) != g) continue;
      for (long i = 0; i < S; ++i) {
        if (!visible(msk, i, j)) continue;
        const float* qi = q + idx4(b, i, h, 0, S, H, D);
        const float* doi = dout + idx4(b, i, h, 0, S, H, D);
        double p = exp(scale * dot_f(qi, kj, D) - lse[(b * H + h) * S + i]);
        double ds = p * (dot_f(doi, vj, D) - delta[(b * H + h) * S + i]);
        for (int d = 0; d < D; ++d) {
          dkj[d] += scale * ds * (double)qi[d];
          dvj[d] += p * (double)doi[d];
        }
      }
    }
    (void)grp;
  }
  free(o);
  free(lse);
  free(delta);
}

/* Backward of the all-gather schedule, inputs and outputs in sharded order.
 * Each rank r, from its own query tokens only: dQ of those tokens, and a
 * contribution to dK / dV of every gathered key.  The contributions of all
 * ranks are then summed and each rank keeps its own shard (the
 * reduce-scatter that returns gathered gradients to their owners). */
static int allgather_bwd_m(const float* q_sh, const float* k_sh, const float* v_sh,
                           const float* do_sh, long B, int H, int Hkv, long S, int D, int cp,
                           int layout, const Mask* msk, double scale, double* dq_sh,
                           double* dk_sh, double* dv_sh) {
  long* nat_of = (long*)malloc(sizeof(long) * (S > 0 ? S : 1));
  if (oracle_shard_order(S, cp, layout, nat_of) != 0) {
    free(nat_of);
    return -1;
  }
  const long nq = B * S * H * D, nkv = B * S * Hkv * D;
  float* qn = (float*)malloc(sizeof(float) * nq + 1);
  float* kn = (float*)malloc(sizeof(float) * nkv + 1);
  float* vn = (float*)malloc(sizeof(float) * nkv + 1);
  float* don = (float*)malloc(sizeof(float) * nq + 1);
  unshard_f(q_sh, qn, nat_of, B, S, H, D);
  unshard_f(k_sh, kn, nat_of, B, S, Hkv, D);
  unshard_f(v_sh, vn, nat_of, B, S, Hkv, D);
  unshard_f(do_sh, don, nat_of, B, S, H, D);
  long* rank_of = (long*)malloc(sizeof(long) * (S > 0 ? S : 1));
  const long L = S / cp;
  for (long p = 0; p < S; ++p) rank_of[nat_of[p]] = p / L;
  /* Forward state of every query row, natural order. */
  double* o = (double*)malloc(sizeof(double) * nq + 1);
  double* lse = (double*)malloc(sizeof(double) * B * H * S + 1);
  double* delta = (double*)malloc(sizeof(double) * B * H * S + 1);
  attn_fwd_m(qn, kn, vn, B, H, Hkv, S, D, msk, scale, o, lse);
  for (long row = 0; row < B * S * H; ++row) {
    long b = row / (S * H), i = (row / H) % S;
    int h = (int)(row % H);
    double t = 0.0;
    for (int d = 0; d < D; ++d) t += (double)don[row * D + d] * o[row * D + d];
    delta[(b * H + h) * S + i] = t;
  }
  /* dQ of every query token (each rank computes its own). */
  double* dqn = (double*)calloc((size_t)nq + 1, sizeof(double));
#pragma omp parallel for schedule(dynamic, 16)
  for (long row = 0; row < B * S * H; ++row) {
    long b = row / (S * H), i = (row / H) % S;
    int h = (int)(row % H);
    int g = kv_head_of(h, H, Hkv);
    const float* qi = qn + row * D;
    const float* doi = don + row * D;
    const double l = lse[(b * H + h) * S + i], dl = delta[(b * H + h) * S + i];
    for (long j = 0; j < S; ++j) {
      if (!visible(msk, i, j)) continue;
      const float* kj = kn + idx4(b, j, g, 0, S, Hkv, D);
      const float* vj = vn + idx4(b, j, g, 0, S, Hkv, D);
      double pr = exp(scale * dot_f(qi, kj, D) - l);
      double ds = pr * (dot_f(doi, vj, D) - dl);
      for (int d = 0; d < D; ++d) dqn[row * D + d] += scale * ds * (double)kj[d];
    }
  }
  /* Per-rank contributions to the gathered dK / dV: rank r's queries only,
   * for every key, natural order. */
  double* part_k = (double*)calloc((size_t)cp * nkv + 1, sizeof(double));
  double* part_v = (double*)calloc((size_t)cp * nkv + 1, sizeof(double));
#pragma omp parallel for schedule(dynamic, 16)
  for (long krow = 0; krow < B * S * Hkv; ++krow) {
    long b = krow / (S * Hkv), j = (krow / Hkv) % S;
    int g = (int)(krow % Hkv);
    const float* kj = kn + krow * D;
    const float* vj = vn + krow * D;
    for (int h = 0; h < H; ++h) {
      if (kv_head_of(h, H, Hkv) != g) continue;
      for (long i = 0; i < S; ++i) {
        if (!visible(msk, i, j)) continue;
        const long r = rank_of[i];
        const float* qi = qn + idx4(b, i, h, 0, S, H, D);
        const float* doi = don + idx4(b, i, h, 0, S, H, D);
        double pr = exp(scale * dot_f(qi, kj, D) - lse[(b * H + h) * S + i]);
        double ds = pr * (dot_f(doi, vj, D) - delta[(b * H + h) * S + i]);
        double* pk = part_k + r * nkv + krow * D;
        double* pv = part_v + r * nkv + krow * D;
        for (int d = 0; d < D; ++d) {
          pk[d] += scale * ds * (double)qi[d];
          pv[d] += pr * (double)doi[d];
        }
      }
    }
  }
  /* Reduce over ranks, scatter to the owners (sharded order). */
  for (long b = 0; b < B; ++b)
    for (long p = 0; p < S; ++p) {
      const long j = nat_of[p];
      for (long x = 0; x < (long)Hkv * D; ++x) {
        double sk = 0.0, sv = 0.0;
        for (int r = 0; r < cp; ++r) {
#if ORACLE_MUTATION == 8
          if (r == cp - 1 && cp > 1) continue; /* one rank's contribution dropped */
#endif
          sk += part_k[r * nkv + idx4(b, j, 0, 0, S, Hkv, D) + x];
          sv += part_v[r * nkv + idx4(b, j, 0, 0, S, Hkv, D) + x];
        }
        dk_sh[idx4(b, p, 0, 0, S, Hkv, D) + x] = sk;
        dv_sh[idx4(b, p, 0, 0, S, Hkv, D) + x] = sv;
      }
      memcpy(dq_sh + idx4(b, p, 0, 0, S, H, D), dqn + idx4(b, j, 0, 0, S, H, D),
             sizeof(double) * H * D);
    }
  free(qn);
  free(kn);
  free(vn);
  free(don);
  free(rank_of);
  free(o);
  free(lse);
  free(delta);
  free(part_k);
  free(part_v);
  free(dqn);
  free(nat_of);
  return 0;
}

int oracle_allgather_bwd(const float* q_sh, const float* k_sh, const float* v_sh,
                         const float* do_sh, long B, int H, int Hkv, long S, int D, int cp,
                         int layout, int causal, double scale, const long* cu, long ndocs,
                         double* dq_sh, double* dk_sh, double* dv_sh) {
  const Mask msk = {causal, cu, ndocs};
  return allgather_bwd_m(q_sh, k_sh, v_sh, do_sh, B, H, Hkv, S, D, cp, layout, &msk, scale,
                         dq_sh, dk_sh, dv_sh);
}

void oracle_attn_bwd(const float* q, const float* k, const float* v, const float* dout,
                     long B, int H, int Hkv, long S, int D, int causal, double scale,
                     double* dq, double* dk, double* dv) {
  const Mask msk = {causal, NULL, 0};
  attn_bwd_m(q, k, v, dout, B, H, Hkv, S, D, &msk, scale, dq, dk, dv);
}

/* The gradients under the document rule (documents cu[0..ndocs]). */
void oracle_attn_bwd_docs(const float* q, const float* k, const float* v, const float* dout,
                          long B, int H, int Hkv, long S, int D, int causal, double scale,
                          const long* cu, long ndocs, double* dq, double* dk, double* dv) {
  const Mask msk = {causal, cu, ndocs};
  attn_bwd_m(q, k, v, dout, B, H, Hkv, S, D, &msk, scale, dq, dk, dv);
}

/* dQ of the definition on a list of query rows (b, h, i): each row needs only
 * its own softmax row, so this is exact for any dout.  dq [n, D]. */
static void attn_bwd_dq_rows_m(const float* q, const float* k, const float* v,
                               const float* dout, long B, int H, int Hkv, long S, int D,
                               const Mask* msk, double scale, const long* rows, long n,
                               double* dq) {
  (void)B;
#pragma omp parallel
  {
    long* keys = (long*)malloc(sizeof(long) * S);
    double* sb = (double*)malloc(sizeof(double) * S);
    double* o = (double*)malloc(sizeof(double) * D);
    for (long j = 0; j < S; ++j) keys[j] = j;
#pragma omp for schedule(dynamic, 1)
    for (long a = 0; a < n; ++a) {
      long b = rows[3 * a], i = rows[3 * a + 2];
      int h = (int)rows[3 * a + 1];
      int g = kv_head_of(h, H, Hkv);
      double l;
      partial_row(q, k, v, B, H, Hkv, S, D, msk, scale, b, h, i, keys, S, sb, o, &l);
      const float* qi = q + idx4(b, i, h, 0, S, H, D);
      const float* doi = dout + idx4(b, i, h, 0, S, H, D);
      double dl = 0.0;
      for (int d = 0; d < D; ++d) dl += (double)doi[d] * o[d];
      double* dqi = dq + a * D;
      for (int d = 0; d < D; ++d) dqi[d] = 0.0;
      for (long j = 0; j < S; ++j) {
        if (!visible(msk, i, j)) continue;
        const float* kj = k + idx4(b, j, g, 0, S, Hkv, D);
        const float* vj = v + idx4(b, j, g, 0, S, Hkv, D);
        double p = exp(scale * dot_f(qi, kj, D) - l);
        double ds = p * (dot_f(doi, vj, D) - dl);
        for (int d = 0; d < D; ++d) dqi[d] += scale * ds * (double)kj[d];
      }
    }
    free(keys);
    free(sb);
    free(o);
  }
}

void oracle_attn_bwd_dq_rows(const float* q, const float* k, const float* v, const float* dout,
                             long B, int H, int Hkv, long S, int D, int causal, double scale,
                             const long* rows, long n, double* dq) {
  const Mask msk = {causal, NULL, 0};
  attn_bwd_dq_rows_m(q, k, v, dout, B, H, Hkv, S, D, &msk, scale, rows, n, dq);
}

void oracle_attn_bwd_dq_rows_docs(const float* q, const float* k, const float* v,
                                  const float* dout, long B, int H, int Hkv, long S, int D,
                                  int causal, double scale, const long* cu, long ndocs,
                                  const long* rows, long n, double* dq) {
  const Mask msk = {causal, cu, ndocs};
  attn_bwd_dq_rows_m(q, k, v, dout, B, H, Hkv, S, D, &msk, scale, rows, n, dq);
}

/* dK, dV of the definition on a list of key rows (b, g, j), for an upstream
 * gradient that is zero on every query row except the natural positions
 * qrows[0..nq) (all batches, all heads).  Rows with dO_i = 0 have
 * Delta_i = 0 and hence dS_ij = 0 and P_ij dO_i = 0, so the sums over i may
 * be restricted to qrows: the result is the exact definition for such a
 * dout.  dk, dv [n, D]. */
static void attn_bwd_dkdv_rows_sparse_m(const float* q, const float* k, const float* v,
                                        const float* dout, long B, int H, int Hkv, long S, int D,
                                        const Mask* msk, double scale, const long* qrows,
                                        long nq, const long* krows, long n, double* dk,
                                        double* dv) {
  /* Softmax state of the needed query rows, every (b, h). */
  double* lse = (double*)malloc(sizeof(double) * B * H * nq);
  double* delta = (double*)malloc(sizeof(double) * B * H * nq);
#pragma omp parallel
  {
    long* keys = (long*)malloc(sizeof(long) * S);
    double* sb = (double*)malloc(sizeof(double) * S);
    double* o = (double*)malloc(sizeof(double) * D);
    for (long j = 0; j < S; ++j) keys[j] = j;
#pragma omp for schedule(dynamic, 1)
    for (long a = 0; a < B * H * nq; ++a) {
      long b = a / (H * nq);
      int h = (int)((a / nq) % H);
      long i = qrows[a % nq];
      partial_row(q, k, v, B, H, Hkv, S, D, msk, scale, b, h, i, keys, S, sb, o, lse + a);
      const float* doi = dout + idx4(b, i, h, 0, S, H, D);
      double dl = 0.0;
      for (int d = 0; d < D; ++d) dl += (double)doi[d] * o[d];
      delta[a] = dl;
    }
    free(keys);
    free(sb);
    free(o);
  }
#pragma omp parallel for schedule(dynamic, 1)
  for (long a = 0; a < n; ++a) {
    long b = krows[3 * a], j = krows[3 * a + 2];
    int g = (int)krows[3 * a + 1];
    const float* kj = k + idx4(b, j, g, 0, S, Hkv, D);
    const float* vj = v + idx4(b, j, g, 0, S, Hkv, D);
    double* dkj = dk + a * D;
    double* dvj = dv + a * D;
    for (int d = 0; d < D; ++d) dkj[d] = dvj[d] = 0.0;
    for (int h = 0; h < H; ++h) {
      if (kv_head_of(h, H, Hkv) != g) continue;
      for (long x = 0; x < nq; ++x) {
        long i = qrows[x];
        if (!visible(msk, i, j)) continue;
        const float* qi = q + idx4(b, i, h, 0, S, H, D);
        const float* doi = dout + idx4(b, i, h, 0, S, H, D);
        long si = (b * H + h) * nq + x;
        double p = exp(scale * dot_f(qi, kj, D) - lse[si]);
        double ds = p * (dot_f(doi, vj, D) - delta[si]);
        for (int d = 0; d < D; ++d) {
          dkj[d] += scale * ds * (double)qi[d];
          dvj[d] += p * (double)doi[d];
        }
      }
    }
  }
  free(lse);
  free(delta);
}

void oracle_attn_bwd_dkdv_rows_sparse(const float* q, const float* k, const float* v,
                                      const float* dout, long B, int H, int Hkv, long S, int D,
                                      int causal, double scale, const long* qrows, long nq,
                                      const long* krows, long n, double* dk, double* dv) {
  const Mask msk = {causal, NULL, 0};
  attn_bwd_dkdv_rows_sparse_m(q, k, v, dout, B, H, Hkv, S, D, &msk, scale, qrows, nq, krows, n,
                              dk, dv);
}

void oracle_attn_bwd_dkdv_rows_sparse_docs(const float* q, const float* k, const float* v,
                                           const float* dout, long B, int H, int Hkv, long S,
                                           int D, int causal, double scale, const long* cu,
                                           long ndocs, const long* qrows, long nq,
                                           const long* krows, long n, double* dk, double* dv) {
  const Mask msk = {causal, cu, ndocs};
  attn_bwd_dkdv_rows_sparse_m(q, k, v, dout, B, H, Hkv, S, D, &msk, scale, qrows, nq, krows, n,
                              dk, dv);
}

/* dK, dV of the definition on a list of key rows (b, g, j) for ANY upstream
 * gradient dout, given the definition's output and LSE of every query row
 * (out [B,S,H,D] and lse [B,H,S] as oracle_attn_fwd returns them):
 * Delta_i = dout_i . out_i, P_ij = exp(s_ij - lse_i),
 * dS_ij = P_ij (dout_i . v_j - Delta_i), dK_j = scale sum_h sum_i dS_ij q_i,
 * dV_j = sum_h sum_i P_ij dout_i, the sums running over the query heads h
 * that read kv head g and over every query row i that sees key j.  This is
 * the key-row half of the gradients above with the forward state handed in,
 * so that a long sequence's forward is computed once for many key rows.
 * dk, dv [n, D]. */
void oracle_attn_bwd_dkdv_rows(const float* q, const float* k, const float* v,
                               const float* dout, long B, int H, int Hkv, long S, int D,
                               int causal, double scale, const double* out, const double* lse,
                               const long* krows, long n, double* dk, double* dv) {
  const Mask msk = {causal, NULL, 0};
  double* delta = (double*)malloc(sizeof(double) * B * H * S);
#pragma omp parallel for schedule(static)
  for (long row = 0; row < B * S * H; ++row) {
    long b = row / (S * H), i = (row / H) % S;
    int h = (int)(row % H);
    double s = 0.0;
    for (int d = 0; d < D; ++d) s += (double)dout[row * D + d] * out[row * D + d];
    delta[(b * H + h) * S + i] = s;
  }
#pragma omp parallel for schedule(dynamic, 1)
  for (long a = 0; a < n; ++a) {
    long b = krows[3 * a], j = krows[3 * a + 2];
    int g = (int)krows[3 * a + 1];
    const float* kj = k + idx4(b, j, g, 0, S, Hkv, D);
    const float* vj = v + idx4(b, j, g, 0, S, Hkv, D);
    double* dkj = dk + a * D;
    double* dvj = dv + a * D;
    for (int d = 0; d < D; ++d) dkj[d] = dvj[d] = 0.0;
    for (int h = 0; h < H; ++h) {
      if (kv_head_of(h, H, Hkv) != g) continue;
#if ORACLE_MUTATION == 10
      if (h != g * (H / Hkv)) continue; /* only the first query head of the group */
#endif
      for (long i = 0; i < S; ++i) {
        if (!visible(&msk, i, j)) continue;
        const float* qi = q + idx4(b, i, h, 0, S, H, D);
        const float* doi = dout + idx4(b, i, h, 0, S, H, D);
        long si = (b * H + h) * S + i;
        double p = exp(scale * dot_f(qi, kj, D) - lse[si]);
        double ds = p * (dot_f(doi, vj, D) - delta[si]);
        for (int d = 0; d < D; ++d) {
          dkj[d] += scale * ds * (double)qi[d];
          dvj[d] += p * (double)doi[d];
        }
      }
    }
  }
  free(delta);
}

/* ------------------------------------------------------------------------ */
/* Work census of the ring                                                   */
/* ------------------------------------------------------------------------ */

/* For every rank r and ring step t: the number of T x T tiles that hold at
 * least one valid (query, key) pair, and (if pairs_rt is not NULL) the number
 * of valid pairs, per (batch, head).  Tiles are T consecutive tokens of a
 * rank's shard (query side) and of the source rank's shard (key side), each
 * inside one chunk; T must divide the chunk length.  Found by enumeration
 * over tiles (and, for pairs, over every pair of every live tile). */
static int tile_counts_m(long S, int cp, int layout, const Mask* msk, long T, uint64_t* tiles_rt,
                         uint64_t* pairs_rt) {
  int per_rank = (layout == LAYOUT_ZIGZAG) ? 2 : 1;
  if (cp < 1 || T < 1 || S % ((long)cp * per_rank) != 0) return -1;
  long L = S / cp, c = L / per_rank;
  if (c % T != 0) return -1;
  long* qpos = (long*)malloc(sizeof(long) * L);
  long* kpos = (long*)malloc(sizeof(long) * L);
  for (int r = 0; r < cp; ++r) {
    rank_tokens(S, cp, layout, r, qpos);
    for (int t = 0; t < cp; ++t) {
      rank_tokens(S, cp, layout, ring_source(r, t, cp), kpos);
      uint64_t tiles = 0, pairs = 0;
      for (long qa = 0; qa < L; qa += T) {
        for (long kb = 0; kb < L; kb += T) {
          int any = 0;
          if (msk->cu == NULL) {
            /* j <= i is monotone, so some pair of the tile is valid exactly
             * when the latest query and the earliest key form a valid pair. */
            long qmax = qpos[qa], kmin = kpos[kb];
            for (long x = 1; x < T; ++x) qmax = qpos[qa + x] > qmax ? qpos[qa + x] : qmax;
            for (long y = 1; y < T; ++y) kmin = kpos[kb + y] < kmin ? kpos[kb + y] : kmin;
            any = visible(msk, qmax, kmin);
          } else {
            for (long x = 0; x < T && !any; ++x)
              for (long y = 0; y < T && !any; ++y) any = visible(msk, qpos[qa + x], kpos[kb + y]);
          }
          tiles += (uint64_t)any;
          if (pairs_rt && any)
            for (long x = 0; x < T; ++x)
              for (long y = 0; y < T; ++y)
                pairs += (uint64_t)visible(msk, qpos[qa + x], kpos[kb + y]);
        }
      }
      tiles_rt[r * cp + t] = tiles;
      if (pairs_rt) pairs_rt[r * cp + t] = pairs;
    }
  }
  free(qpos);
  free(kpos);
  return 0;
}

int oracle_tile_counts(long S, int cp, int layout, int causal, long T, uint64_t* tiles_rt,
                       uint64_t* pairs_rt) {
  const Mask msk = {causal, NULL, 0};
  return tile_counts_m(S, cp, layout, &msk, T, tiles_rt, pairs_rt);
}

/* The census under the document rule (documents cu[0..ndocs]). */
int oracle_tile_counts_docs(long S, int cp, int layout, int causal, const long* cu, long ndocs,
                            long T, uint64_t* tiles_rt, uint64_t* pairs_rt) {
  const Mask msk = {causal, cu, ndocs};
  return tile_counts_m(S, cp, layout, &msk, T, tiles_rt, pairs_rt);
}
