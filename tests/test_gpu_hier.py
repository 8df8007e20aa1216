"""GPU parity of hierarchical context parallelism, the a2a+p2p type
("Context Parallelism in MegaDLMs", sections "Hierarchical Context
Parallelism" and "Key-Value Communication Patterns"): level sizes
[cp_a2a, cp_p2p], an all-to-all inside groups of cp_a2a consecutive ranks,
then the zigzag ring over the cp_p2p groups on each head slice, against the
oracle's two-level schedule on the same sharded inputs.

Bars: the all-to-all bit-exact (it only moves bytes; the head -> sequence
direction of shared kv heads sums in float32, compared with the exact sum
rounded once); attention as for the ring: float32 O <= 1e-4, LSE <= 1e-5,
gradients <= 1e-4; bf16 O <= 2e-2, LSE <= 1e-3, gradients (float32 outputs)
<= 2e-2.  The one-level splits are checked bit for bit against the paths
they reduce to: [1, cp] is the plain ring, [cp, 1] the Ulysses variant.
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
    w = inputs.Workload("hier", B, H, Hkv, S, D, 1, inputs.ZIGZAG, True, dtype, seed=seed)
    return inputs.generate(w, with_dout=dout)


def f32(x):
    return inputs.to_f32_numpy(x)


def maxerr(gpu, ref):
    g = gpu.detach().to("cpu", torch.float64).numpy() if torch.is_tensor(gpu) else gpu
    return float(np.max(np.abs(g - ref))) if g.size else 0.0


@pytest.mark.parametrize("A,P", [(2, 2), (2, 4), (4, 2), (4, 4), (8, 2)])
@pytest.mark.parametrize("layout", [cpa.ZIGZAG, cpa.CONTIGUOUS])
def test_a2a_bit_exact(A, P, layout):
    B, D, H = 2, 64, 8
    S = 64 * A * P
    g = torch.Generator().manual_seed(A * 100 + P)
    order = oracle.shard_order(S, A * P, layout)
    for Hkv in (2, 8):
        for dtype in (torch.bfloat16, torch.float32):
            for kv in (False, True):
                X = Hkv if kv else H
                x = torch.randn((B, S, X, D), generator=g).to(dtype)
                xs = x[:, torch.as_tensor(order)].contiguous()
                y = cpa.hier_a2a(xs.to(DEV), A, P, H, Hkv, layout, kv_heads=kv)
                ref = oracle.hier_a2a(f32(xs), H, Hkv, A, P, layout, kv)
                assert np.array_equal(f32(y), ref)
                back = cpa.hier_a2a(y, A, P, H, Hkv, layout, kv_heads=kv, to_seq=True)
                if not kv or (H // A) >= (H // Hkv):
                    assert torch.equal(back.cpu(), xs)      # one owner per head: a copy
                else:
                    share = (H // Hkv) // (H // A)          # members holding each kv head
                    acc = torch.zeros_like(xs, dtype=torch.float32)
                    for _ in range(share):
                        acc = acc + xs.float()
                    assert torch.equal(back.cpu(), acc.to(dtype))
    assert cpa.device_status() == 0


CASES = [
    # B, H, Hkv, S, D, A, P, layout, causal, dtype, cu (None: one document)
    (1, 8, 2, 2048, 128, 2, 2, cpa.ZIGZAG, True, torch.bfloat16, None),     # the pages' [2, 2]
    (1, 8, 2, 4096, 128, 2, 4, cpa.ZIGZAG, True, torch.bfloat16, None),
    (1, 8, 2, 4096, 128, 4, 2, cpa.ZIGZAG, True, torch.bfloat16, None),     # shared kv heads
    (1, 8, 4, 2048, 128, 2, 2, cpa.CONTIGUOUS, True, torch.bfloat16, None),
    (2, 4, 4, 2048, 128, 2, 2, cpa.ZIGZAG, False, torch.bfloat16, None),
    (1, 8, 2, 4096, 128, 2, 4, cpa.ZIGZAG, True, torch.bfloat16, [0, 1, 130, 256, 1700, 4096]),
    (1, 4, 2, 512, 64, 2, 2, cpa.ZIGZAG, True, torch.float32, None),
    (1, 4, 1, 640, 64, 2, 2, cpa.CONTIGUOUS, True, torch.float32, [0, 17, 300, 640]),
]


def case_id(c):
    return "B{}H{}K{}S{}D{}a{}p{}L{}c{}{}{}".format(
        *c[:9], "f32" if c[9] == torch.float32 else "bf16", "" if c[10] is None else "docs")


@pytest.mark.parametrize("case", CASES, ids=case_id)
def test_hier_forward_backward_match_oracle(case):
    B, H, Hkv, S, D, A, P, layout, causal, dtype, cu = case
    q, k, v, do = make(B, H, Hkv, S, D, dtype, seed=8200 + S + A * P, dout=True)
    order = oracle.shard_order(S, A * P, layout)
    idx = torch.as_tensor(order)
    qs, ks, vs, dos = (x[:, idx].contiguous().to(DEV) for x in (q, k, v, do))
    bounds = cpa.doc_bounds(cu, S) if cu is not None else None
    o, lse = cpa.hier_fwd(qs, ks, vs, A, P, layout, causal, bounds=bounds)
    fq, fk, fv, fdo = (f32(x)[:, order] for x in (q, k, v, do))
    ro, rl = oracle.hier_fwd(fq, fk, fv, A, P, layout, causal, cu_seqlens=cu)
    tol = TOL[dtype]
    assert maxerr(o, ro) <= tol["o"], maxerr(o, ro)
    assert maxerr(lse, rl) <= tol["lse"], maxerr(lse, rl)
    dq, dk, dv = cpa.hier_bwd(qs, ks, vs, o, dos, lse, A, P, layout, causal, bounds=bounds,
                              grad_dtype=torch.float32)
    rq, rk, rv = oracle.hier_bwd(fq, fk, fv, fdo, A, P, layout, causal, cu_seqlens=cu)
    for name, got, ref in (("dq", dq, rq), ("dk", dk, rk), ("dv", dv, rv)):
        assert maxerr(got, ref) <= tol["grad"], (name, maxerr(got, ref))
    assert cpa.device_status() == 0


def test_one_level_splits_reduce_to_ring_and_ulysses():
    B, H, Hkv, S, D, cp = 1, 8, 2, 4096, 128, 4
    q, k, v, do = make(B, H, Hkv, S, D, torch.bfloat16, seed=8301, dout=True)
    qs, ks, vs, dos = (cpa.zigzag_permute(x.to(DEV), cp, cpa.ZIGZAG) for x in (q, k, v, do))
    # [1, cp]: the all-to-all is a copy and the second level is the ring itself.
    o, lse = cpa.hier_fwd(qs, ks, vs, 1, cp)
    ro, rl = cpa.ring_fwd(qs, ks, vs, cp)
    assert torch.equal(o, ro) and torch.equal(lse, rl)
    g = cpa.hier_bwd(qs, ks, vs, o, dos, lse, 1, cp, grad_dtype=torch.float32)
    rg = cpa.ring_bwd(qs, ks, vs, ro, dos, rl, cp, grad_dtype=torch.float32)
    assert all(torch.equal(a, b) for a, b in zip(g, rg))
    # [cp, 1]: the Ulysses variant.
    o, lse = cpa.hier_fwd(qs, ks, vs, cp, 1)
    uo, ul = cpa.ulysses_fwd(qs, ks, vs, cp)
    assert torch.equal(o, uo) and torch.equal(lse, ul)
    g = cpa.hier_bwd(qs, ks, vs, o, dos, lse, cp, 1, grad_dtype=torch.float32)
    ug = cpa.ulysses_bwd(qs, ks, vs, uo, dos, ul, cp, grad_dtype=torch.float32)
    assert all(torch.equal(a, b) for a, b in zip(g, ug))
    assert cpa.device_status() == 0


def test_hier_rejects_splits_it_cannot_make():
    q = torch.zeros((1, 1024, 6, 64), device=DEV, dtype=torch.bfloat16)
    k = torch.zeros((1, 1024, 2, 64), device=DEV, dtype=torch.bfloat16)
    with pytest.raises(cpa.CpattnError):
        cpa.hier_fwd(q, k, k, 4, 2)   # 6 query heads over 4 members
    with pytest.raises(cpa.CpattnError):
        cpa.hier_fwd(q, k, k, 2, 0)   # empty second level
    q2 = torch.zeros((1, 1004, 8, 64), device=DEV, dtype=torch.bfloat16)
    k2 = torch.zeros((1, 1004, 2, 64), device=DEV, dtype=torch.bfloat16)
    with pytest.raises(cpa.CpattnError):
        cpa.hier_fwd(q2, k2, k2, 2, 2)   # 1004 tokens do not split into 8 chunks
    assert cpa.device_status() == 0


@pytest.mark.parametrize("A,P", [(4, 4), (2, 8)])
def test_hier_full_size(A, P):
    # The S=131072 workload (cp = 16) through the hierarchical schedule:
    # sampled rows against the oracle's definition, dQ on a subset, and the
    # sum rules of dK / dV over the whole tensors.
    w = inputs.WORKLOADS["c5_bf16_s131072_fwdbwd"]
    assert A * P == w.cp
    q, k, v, do = inputs.generate(w)
    qd, kd, vd, dod = (x.to(DEV) for x in (q, k, v, do))
    o, lse, dq, dk, dv = cpa.attention_hier_fwd_bwd(qd, kd, vd, dod, A, P, w.layout, w.causal,
                                                    grad_dtype=torch.float32)
    assert cpa.device_status() == 0
    rng = np.random.default_rng(31 + A)
    c = w.S // (2 * w.cp)
    cP = w.S // (2 * P)
    edges = sorted({m * c for m in range(2 * w.cp)} | {m * c - 1 for m in range(1, 2 * w.cp)}
                   | {m * cP for m in range(2 * P)})
    rows = np.array([(0, h, i) for h in range(w.H)
                     for i in edges[h % 4::4] + rng.integers(0, w.S, 48).tolist()])
    fq, fk, fv, fdo = f32(q), f32(k), f32(v), f32(do)
    ro, rl = oracle.attn_fwd_rows(fq, fk, fv, rows)
    assert maxerr(o[0, rows[:, 2], rows[:, 1]], ro) <= 2e-2
    assert maxerr(lse[0, rows[:, 1], rows[:, 2]], rl) <= 1e-3
    sub = rows[rng.choice(len(rows), 128, replace=False)]
    rdq = oracle.attn_bwd_dq_rows(fq, fk, fv, fdo, sub)
    assert maxerr(dq[0, sub[:, 2], sub[:, 1]], rdq) <= 2e-2
    grp = w.H // w.Hkv
    bound = 4e-3 * np.sqrt(w.S)
    sdo = dod.double().sum(dim=1)[0].view(w.Hkv, grp, w.D).sum(1)
    assert (dv.double().sum(dim=1)[0] - sdo).abs().max().item() <= bound
    assert dk.double().sum(dim=1).abs().max().item() <= bound
