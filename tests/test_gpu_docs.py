"""GPU parity of packed documents and padding ("Context Parallelism for
Long-Context Training", sections "Prove attention equivalence" -- causal and
document masks must give the unsharded result -- and "Test sequence
divisibility and padding" -- padded tokens must not change any real token).

libcpattn (through its C ABI) against the fp64 CPU oracle's document rule,
with the same bars as the plain mask: float32 O <= 1e-4, LSE <= 1e-5,
gradients <= 1e-4; bf16 O, dQ, dK, dV <= 2e-2, LSE <= 1e-3; document bounds
and the tile census bit-exact.

Gradients of bf16 inputs are compared as float32 outputs (the backward's
float32-gradient flag): short documents give rows with few keys, so dV of a
document's first keys reaches 4 to 10, where storing one bf16 value alone
costs up to 0.0156 of the 0.02 bar.  The bf16 outputs are then checked to be
exactly the float32 outputs rounded to nearest even.
"""
import numpy as np
import pytest
import torch

import oracle
import context_causal_attention_zigzag_gb300 as cpa
from context_causal_attention_zigzag_gb300 import inputs

pytestmark = pytest.mark.gpu

TOL = {torch.float32: dict(o=1e-4, lse=1e-5, grad=1e-4),
       torch.bfloat16: dict(o=2e-2, lse=1e-3, grad=2e-2)}
DEV = "cuda"


def make(B, H, Hkv, S, D, dtype, seed, dout=False):
    w = inputs.Workload("docs", B, H, Hkv, S, D, 1, inputs.ZIGZAG, True, dtype, seed=seed)
    return inputs.generate(w, with_dout=dout)


def f32(x):
    return inputs.to_f32_numpy(x)


def maxerr(gpu, ref):
    g = gpu.detach().to("cpu", torch.float64).numpy() if torch.is_tensor(gpu) else gpu
    return float(np.max(np.abs(g - ref))) if g.size else 0.0


def bounds_ref(cu):
    """(first, one past last) of each position's document, by expansion."""
    out = []
    for a, b in zip(cu[:-1], cu[1:]):
        out.extend([(a, b)] * (b - a))
    return np.array(out, dtype=np.int32)


# Hand-placed borders: a one-token document, borders inside tiles, on tile
# edges and on zigzag chunk edges; then generated mixes.
CU_2048 = [0, 1, 130, 256, 700, 1024, 1029, 1535, 2048]

DOC_CASES = [
    # B, H, Hkv, S, D, cp, layout, causal, dtype, cu
    (1, 4, 2, 2048, 128, 2, cpa.ZIGZAG, True, torch.bfloat16, CU_2048),
    (1, 4, 2, 2048, 128, 4, cpa.ZIGZAG, True, torch.bfloat16,
     inputs.packed_doc_offsets(2048, 300, 11)),
    (2, 4, 1, 1536, 128, 3, cpa.ZIGZAG, True, torch.bfloat16,
     inputs.packed_doc_offsets(1536, 200, 12)),
    (1, 2, 1, 2048, 128, 2, cpa.CONTIGUOUS, True, torch.bfloat16, CU_2048),
    (1, 2, 2, 2048, 128, 4, cpa.CONTIGUOUS, False, torch.bfloat16,
     inputs.packed_doc_offsets(2048, 500, 13)),
    (1, 2, 2, 2048, 128, 2, cpa.ZIGZAG, False, torch.bfloat16, CU_2048),
    (1, 2, 2, 256, 64, 2, cpa.ZIGZAG, True, torch.float32, [0, 1, 17, 64, 65, 200, 256]),
    (2, 4, 2, 320, 64, 4, cpa.ZIGZAG, False, torch.float32,
     inputs.packed_doc_offsets(320, 40, 14)),
    (1, 2, 1, 640, 128, 2, cpa.ZIGZAG, True, torch.bfloat16,
     inputs.packed_doc_offsets(640, 90, 15)),                     # padded to 1024
    (1, 2, 2, 384, 64, 3, cpa.ZIGZAG, True, torch.bfloat16,
     inputs.packed_doc_offsets(384, 50, 16)),                     # bf16, D 64: CUDA cores
]


def case_id(c):
    return "B{}H{}K{}S{}D{}cp{}L{}c{}{}n{}".format(
        *c[:8], "f32" if c[8] == torch.float32 else "bf16", len(c[9]) - 1)


def test_doc_bounds_bit_exact():
    for S, cu in ((2048, CU_2048), (64, [0, 64]), (7, list(range(8))),
                  (131072, inputs.DOC_WORKLOADS["docs_bf16_s131072_fwdbwd"].doc_offsets())):
        got = cpa.doc_bounds(cu, S).cpu().numpy()
        assert np.array_equal(got, bounds_ref(cu)), S
    assert cpa.device_status() == 0


def test_doc_bounds_reports_broken_offsets():
    # Not increasing, wrong start, wrong end: reported as an invalid argument
    # by the next status read; the bounds still hold each position.
    S = 64
    for cu in ([0, 10, 10, 64], [1, 10, 64], [0, 10, 63], [0, 40, 20, 64]):
        b = cpa.doc_bounds(cu, S).cpu().numpy()
        assert cpa.device_status() == cpa._binding.ERR_INVALID_ARG, cu
        pos = np.arange(S)
        assert (b[:, 0] <= pos).all() and (b[:, 1] > pos).all() and (b[:, 1] <= S).all()
    assert cpa.device_status() == 0


@pytest.mark.parametrize("case", DOC_CASES, ids=case_id)
def test_forward_docs_matches_oracle(case):
    B, H, Hkv, S, D, cp, layout, causal, dtype, cu = case
    q, k, v, _ = make(B, H, Hkv, S, D, dtype, seed=3000 + S + cp)
    out, lse = cpa.attention_docs(q.to(DEV), k.to(DEV), v.to(DEV), cp, cu, layout, causal)
    ro, rl = oracle.attn_fwd_docs(f32(q), f32(k), f32(v), cu, causal=causal)
    tol = TOL[dtype]
    assert maxerr(out, ro) <= tol["o"], maxerr(out, ro)
    assert maxerr(lse, rl) <= tol["lse"], maxerr(lse, rl)
    assert cpa.device_status() == 0


@pytest.mark.parametrize("case", DOC_CASES, ids=case_id)
def test_backward_docs_matches_oracle(case):
    B, H, Hkv, S, D, cp, layout, causal, dtype, cu = case
    q, k, v, do = (x.to(DEV) for x in make(B, H, Hkv, S, D, dtype, seed=4000 + S + cp,
                                             dout=True))
    _, _, dq, dk, dv = cpa.attention_docs_fwd_bwd(q, k, v, do, cp, cu, layout, causal,
                                                  grad_dtype=torch.float32)
    rq, rk, rv = oracle.attn_bwd_docs(f32(q), f32(k), f32(v), f32(do), cu, causal=causal)
    tol = TOL[dtype]["grad"]
    for name, got, ref in (("dq", dq, rq), ("dk", dk, rk), ("dv", dv, rv)):
        assert maxerr(got, ref) <= tol, (name, maxerr(got, ref))
    if dtype == torch.bfloat16:
        # Both backward paths write every gradient element once (no atomics),
        # so bf16 gradients are the float32 ones rounded, bit for bit.
        _, _, bq, bk, bv = cpa.attention_docs_fwd_bwd(q, k, v, do, cp, cu, layout, causal)
        for a, b in ((bq, dq), (bk, dk), (bv, dv)):
            assert a.dtype == torch.bfloat16 and torch.equal(a, b.to(torch.bfloat16))
    assert cpa.device_status() == 0


@pytest.mark.parametrize("case", [c for c in DOC_CASES if c[0] * c[1] <= 4], ids=case_id)
def test_census_docs_bit_exact(case):
    # Tiles the kernel processed per (rank, step) = tiles holding at least one
    # visible pair under the document rule, summed over batch and heads.
    B, H, Hkv, S, D, cp, layout, causal, dtype, cu = case
    _, tile = cpa.plan(B, H, Hkv, S, D, cp, layout, causal, dtype)
    c = S // (cp * (2 if layout == cpa.ZIGZAG else 1))
    if c % tile:
        pytest.skip("census needs whole tiles per chunk")
    q, k, v, _ = make(B, H, Hkv, S, D, dtype, seed=5000 + S)
    qs, ks, vs = (cpa.zigzag_permute(x.to(DEV), cp, layout) for x in (q, k, v))
    bounds = cpa.doc_bounds(cu, S)
    _, _, counts = cpa.ring_fwd_docs_census(qs, ks, vs, cp, bounds, layout, causal)
    ref, _ = oracle.tile_counts_docs(S, cp, layout, causal, cu, tile)
    assert np.array_equal(counts.cpu().numpy(), ref.astype(np.int64) * B * H)


def test_one_document_equals_plain_path():
    # cu = [0, S]: the document path gives the plain path's bits.
    B, H, Hkv, S, D, cp = 1, 4, 2, 2048, 128, 4
    q, k, v, do = (x.to(DEV) for x in make(B, H, Hkv, S, D, torch.bfloat16, seed=61, dout=True))
    qs, ks, vs, dos = (cpa.zigzag_permute(x, cp) for x in (q, k, v, do))
    o1, l1 = cpa.ring_fwd(qs, ks, vs, cp)
    bounds = cpa.doc_bounds([0, S], S)
    o2, l2 = cpa.ring_fwd_docs(qs, ks, vs, cp, bounds)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
    g1 = cpa.ring_bwd(qs, ks, vs, o1, dos, l1, cp)
    g2 = cpa.ring_bwd_docs(qs, ks, vs, o2, dos, l2, cp, bounds)
    for a, b in zip(g1, g2):
        assert torch.equal(a, b)


# ---------------------------------------------------------------------------
# padding
# ---------------------------------------------------------------------------

PAD_CASES = [
    # B, H, Hkv, S_real, D, cp, layout, causal, dtype, cu (None: one document)
    (1, 4, 2, 1000, 128, 2, cpa.ZIGZAG, True, torch.bfloat16, [0, 300, 301, 1000]),
    (1, 2, 1, 777, 128, 4, cpa.ZIGZAG, True, torch.bfloat16, None),
    (1, 2, 2, 3000, 128, 3, cpa.CONTIGUOUS, True, torch.bfloat16, None),
    (1, 2, 2, 1300, 128, 2, cpa.ZIGZAG, False, torch.bfloat16, [0, 650, 1300]),
    (1, 2, 1, 250, 64, 2, cpa.ZIGZAG, True, torch.float32, [0, 100, 250]),
]


@pytest.mark.parametrize("case", PAD_CASES, ids=lambda c: "S{}cp{}L{}c{}".format(*c[3:4], *c[5:8]))
def test_padding_leaves_real_tokens_unchanged(case):
    # Awkward lengths: padded to cpattn_padded_length, the padding its own
    # document; the real tokens must equal the oracle on the unpadded input.
    B, H, Hkv, S_real, D, cp, layout, causal, dtype, cu = case
    S = cpa.padded_length(S_real, cp, layout)
    assert S > S_real
    q, k, v, do = make(B, H, Hkv, S_real, D, dtype, seed=6000 + S_real, dout=True)
    o, lse, dq, dk, dv = cpa.attention_docs_fwd_bwd(q.to(DEV), k.to(DEV), v.to(DEV), do.to(DEV),
                                                    cp, cu, layout, causal,
                                                    grad_dtype=torch.float32)
    assert o.shape[1] == S_real and lse.shape[2] == S_real
    cuo = cu if cu is not None else [0, S_real]
    ro, rl = oracle.attn_fwd_docs(f32(q), f32(k), f32(v), cuo, causal=causal)
    rq, rk, rv = oracle.attn_bwd_docs(f32(q), f32(k), f32(v), f32(do), cuo, causal=causal)
    tol = TOL[dtype]
    assert maxerr(o, ro) <= tol["o"] and maxerr(lse, rl) <= tol["lse"]
    for name, got, ref in (("dq", dq, rq), ("dk", dk, rk), ("dv", dv, rv)):
        assert maxerr(got, ref) <= tol["grad"], (name, maxerr(got, ref))
    assert cpa.device_status() == 0


def test_permute_pad_bit_exact():
    g = torch.Generator().manual_seed(9)
    for layout in (cpa.ZIGZAG, cpa.CONTIGUOUS):
        for cp, S_real in ((2, 1000), (4, 777), (3, 1), (1, 500)):
            S = cpa.padded_length(S_real, cp, layout)
            order = torch.as_tensor(oracle.shard_order(S, cp, layout))
            for shape, seq_dim, dtype in [((2, S_real, 3, 8), 1, torch.bfloat16),
                                          ((2, 3, S_real), 2, torch.float32),
                                          ((1, S_real, 5), 1, torch.uint8)]:
                x = torch.randint(1, 255, shape, generator=g).to(dtype)
                padded = torch.cat([x, torch.zeros_like(x).narrow(seq_dim, 0, 1)
                                    .expand(*[S - S_real if d == seq_dim else n
                                              for d, n in enumerate(x.shape)])], dim=seq_dim)
                ref = torch.index_select(padded, seq_dim, order)
                y = cpa.zigzag_permute_pad(x.to(DEV), cp, S, layout, seq_dim=seq_dim)
                assert torch.equal(y.cpu(), ref)
                z = cpa.zigzag_unpermute_pad(y, cp, S_real, layout, seq_dim=seq_dim)
                assert torch.equal(z.cpu(), x)
    assert cpa.device_status() == 0


# ---------------------------------------------------------------------------
# the S=131072 packed-document workload at full size
# ---------------------------------------------------------------------------

def test_docs_full_size_forward_backward():
    w = inputs.DOC_WORKLOADS["docs_bf16_s131072_fwdbwd"]
    cu = w.doc_offsets()
    q, k, v, do = inputs.generate(w)
    qd, kd, vd, dod = (x.to(DEV) for x in (q, k, v, do))
    path, _ = cpa.plan(w.B, w.H, w.Hkv, w.S, w.D, w.cp, w.layout, w.causal, w.dtype)
    assert path == cpa.PATH_TCGEN05
    o, lse, dq, dk, dv = cpa.attention_docs_fwd_bwd(qd, kd, vd, dod, w.cp, cu, w.layout, w.causal,
                                                    grad_dtype=torch.float32)
    assert cpa.device_status() == 0
    rng = np.random.default_rng(17)
    # Sampled rows: every document's first and last row, both sides of every
    # zigzag chunk border, and random rows, on every head.
    c = w.S // (2 * w.cp)
    base = set(cu[:-1]) | {x - 1 for x in cu[1:]}
    base |= {m * c for m in range(2 * w.cp)} | {m * c - 1 for m in range(1, 2 * w.cp)}
    rows = []
    for h in range(w.H):
        pick = sorted(base | set(rng.integers(0, w.S, 24).tolist()))
        rows += [(0, h, i) for i in pick]
    rows = np.array(rows)
    fq, fk, fv, fdo = f32(q), f32(k), f32(v), f32(do)
    ro, rl = oracle.attn_fwd_rows_docs(fq, fk, fv, rows, cu)
    got_o = o[0, rows[:, 2], rows[:, 1]]
    got_l = lse[0, rows[:, 1], rows[:, 2]]
    assert maxerr(got_o, ro) <= 2e-2 and maxerr(got_l, rl) <= 1e-3
    sub = rows[rng.choice(len(rows), 256, replace=False)]
    rdq = oracle.attn_bwd_dq_rows_docs(fq, fk, fv, fdo, sub, cu)
    assert maxerr(dq[0, sub[:, 2], sub[:, 1]], rdq) <= 2e-2
    # Per-document sum rules (each softmax row sums to one within its
    # document): sum of dV over a document = sum of dO over it per kv group,
    # sum of dK over a document = 0.
    grp = w.H // w.Hkv
    d64 = dod.double().view(1, w.S, w.Hkv, grp, w.D).sum(3)
    for a, b in zip(cu[:-1], cu[1:]):
        bound = 4e-3 * np.sqrt(b - a) + 1e-3
        e_v = (dv[0, a:b].double().sum(0) - d64[0, a:b].sum(0)).abs().max().item()
        e_k = dk[0, a:b].double().sum(0).abs().max().item()
        assert e_v <= bound and e_k <= bound, (a, b, e_v, e_k)
    del dq, dk, dv
    # dK / dV rows: a second backward with dO zero outside a few query rows
    # (document borders among them); the oracle's sums over those rows are exact.
    qrows = np.array(sorted(({cu[1] - 1, cu[1], cu[2], w.S - 1, c - 1, c}
                             | set(rng.integers(0, w.S, 8).tolist()))))
    sparse = torch.zeros_like(do)
    sparse[:, qrows] = do[:, qrows]
    _, _, _, dk2, dv2 = cpa.attention_docs_fwd_bwd(qd, kd, vd, sparse.to(DEV), w.cp, cu, w.layout,
                                                   w.causal, grad_dtype=torch.float32)
    kj = sorted(set(qrows.tolist()) | {cu[1] - 2, cu[2] - 1, 0}
                | set(rng.integers(0, w.S, 16).tolist()))
    krows = np.array([(0, g, j) for g in range(w.Hkv) for j in kj], dtype=np.int64)
    rdk, rdv = oracle.attn_bwd_dkdv_rows_sparse_docs(fq, fk, fv, f32(sparse), qrows, krows, cu)
    assert maxerr(dk2[0, krows[:, 2], krows[:, 1]], rdk) <= 2e-2
    assert maxerr(dv2[0, krows[:, 2], krows[:, 1]], rdv) <= 2e-2
    assert cpa.device_status() == 0


def test_many_short_documents_s32768():
    # 32768 tokens packed with 320 documents of mean length 100: most tiles
    # hold no visible pair and most visited tiles are cut by a border.
    # Forward rows and dQ rows against the oracle (every document's first
    # and last row of one head, random rows of every head), and dK / dV of
    # whole documents against the oracle run on each document alone
    # (documents are independent, so that is exact).
    B, H, Hkv, S, D, cp = 1, 8, 2, 32768, 128, 8
    cu = inputs.packed_doc_offsets(S, 100, seed=77)
    q, k, v, do = make(B, H, Hkv, S, D, torch.bfloat16, seed=7700, dout=True)
    qd, kd, vd, dod = (x.to(DEV) for x in (q, k, v, do))
    o, lse, dq, dk, dv = cpa.attention_docs_fwd_bwd(qd, kd, vd, dod, cp, cu, cpa.ZIGZAG, True,
                                                    grad_dtype=torch.float32)
    assert cpa.device_status() == 0
    rng = np.random.default_rng(78)
    rows = [(0, 3, i) for i in sorted(set(cu[:-1]) | {x - 1 for x in cu[1:]})]
    rows += [(0, h, int(i)) for h in range(H) for i in rng.integers(0, S, 128)]
    rows = np.array(rows, dtype=np.int64)
    fq, fk, fv, fdo = f32(q), f32(k), f32(v), f32(do)
    ro, rl = oracle.attn_fwd_rows_docs(fq, fk, fv, rows, cu)
    assert maxerr(o[0, rows[:, 2], rows[:, 1]], ro) <= 2e-2
    assert maxerr(lse[0, rows[:, 1], rows[:, 2]], rl) <= 1e-3
    rdq = oracle.attn_bwd_dq_rows_docs(fq, fk, fv, fdo, rows, cu)
    assert maxerr(dq[0, rows[:, 2], rows[:, 1]], rdq) <= 2e-2
    ndoc = len(cu) - 1
    picks = sorted({0, ndoc - 1} | set(rng.choice(ndoc, 24, replace=False).tolist()))
    for d in picks:
        a, b = cu[d], cu[d + 1]
        _, rk, rv = oracle.attn_bwd(fq[:, a:b], fk[:, a:b], fv[:, a:b], fdo[:, a:b], causal=True)
        assert maxerr(dk[:, a:b], rk) <= 2e-2, ("dk", d, maxerr(dk[:, a:b], rk))
        assert maxerr(dv[:, a:b], rv) <= 2e-2, ("dv", d, maxerr(dv[:, a:b], rv))
    assert cpa.device_status() == 0
