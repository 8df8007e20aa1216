"""GPU parity of the Ulysses variant ("Sequence Parallelism IV", section 7:
an all-to-all from sequence to head ownership, after which a rank has all
tokens of a head slice) against the oracle's Ulysses variant on the same
sharded inputs.

Bars: the all-to-all bit-exact (it only moves bytes; the head -> sequence
direction of shared kv heads sums in float32, compared with the oracle's
exact sum at float32 rounding); attention as for the ring: float32 O <= 1e-4,
LSE <= 1e-5, gradients <= 1e-4; bf16 O <= 2e-2, LSE <= 1e-3, gradients
(float32 outputs) <= 2e-2.
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
    w = inputs.Workload("ul", B, H, Hkv, S, D, 1, inputs.ZIGZAG, True, dtype, seed=seed)
    return inputs.generate(w, with_dout=dout)


def f32(x):
    return inputs.to_f32_numpy(x)


def maxerr(gpu, ref):
    g = gpu.detach().to("cpu", torch.float64).numpy() if torch.is_tensor(gpu) else gpu
    return float(np.max(np.abs(g - ref))) if g.size else 0.0


@pytest.mark.parametrize("H,Hkv,cp", [(8, 2, 4), (8, 4, 2), (8, 8, 8), (4, 1, 1), (16, 2, 16)])
@pytest.mark.parametrize("layout", [cpa.ZIGZAG, cpa.CONTIGUOUS])
def test_a2a_bit_exact(H, Hkv, cp, layout):
    B, S, D = 2, 64 * cp, 64
    g = torch.Generator().manual_seed(H * 100 + cp)
    order = oracle.shard_order(S, cp, layout)
    for dtype in (torch.bfloat16, torch.float32):
        for kv in (False, True):
            X = Hkv if kv else H
            x = torch.randn((B, S, X, D), generator=g).to(dtype)
            xs = x[:, torch.as_tensor(order)].contiguous()
            y = cpa.ulysses_a2a(xs.to(DEV), cp, H, Hkv, layout, kv_heads=kv)
            ref = oracle.ulysses_a2a(f32(xs), H, Hkv, cp, layout, kv)
            assert np.array_equal(f32(y), ref)
            back = cpa.ulysses_a2a(y, cp, H, Hkv, layout, kv_heads=kv, to_seq=True)
            if not kv or (H // cp) >= (H // Hkv):
                assert torch.equal(back.cpu(), xs)        # one owner per head: a copy
            else:
                share = (H // Hkv) // (H // cp)           # ranks holding each kv head
                acc = torch.zeros_like(xs, dtype=torch.float32)
                for _ in range(share):                    # float32 sum, then one rounding
                    acc = acc + xs.float()
                assert torch.equal(back.cpu(), acc.to(dtype))
    assert cpa.device_status() == 0


CASES = [
    # B, H, Hkv, S, D, cp, layout, causal, dtype, cu (None: one document)
    (1, 8, 2, 2048, 128, 4, cpa.ZIGZAG, True, torch.bfloat16, None),       # shared kv heads
    (1, 8, 4, 2048, 128, 2, cpa.CONTIGUOUS, True, torch.bfloat16, None),   # 2 kv heads / rank
    (2, 4, 4, 1024, 128, 2, cpa.ZIGZAG, False, torch.bfloat16, None),
    (1, 8, 2, 2048, 128, 8, cpa.ZIGZAG, True, torch.bfloat16, [0, 1, 130, 256, 700, 2048]),
    (1, 4, 2, 256, 64, 2, cpa.ZIGZAG, True, torch.float32, None),
    (1, 4, 1, 320, 64, 4, cpa.CONTIGUOUS, True, torch.float32, [0, 17, 100, 320]),
]


def case_id(c):
    return "B{}H{}K{}S{}D{}cp{}L{}c{}{}{}".format(
        *c[:8], "f32" if c[8] == torch.float32 else "bf16", "" if c[9] is None else "docs")


@pytest.mark.parametrize("case", CASES, ids=case_id)
def test_ulysses_forward_backward_match_oracle(case):
    B, H, Hkv, S, D, cp, layout, causal, dtype, cu = case
    q, k, v, do = make(B, H, Hkv, S, D, dtype, seed=8000 + S + cp, dout=True)
    order = oracle.shard_order(S, cp, layout)
    idx = torch.as_tensor(order)
    qs, ks, vs, dos = (x[:, idx].contiguous().to(DEV) for x in (q, k, v, do))
    bounds = cpa.doc_bounds(cu, S) if cu is not None else None
    o, lse = cpa.ulysses_fwd(qs, ks, vs, cp, layout, causal, bounds=bounds)
    fq, fk, fv, fdo = (f32(x)[:, order] for x in (q, k, v, do))
    ro, rl = oracle.ulysses_fwd(fq, fk, fv, cp, layout, causal, cu_seqlens=cu)
    tol = TOL[dtype]
    assert maxerr(o, ro) <= tol["o"], maxerr(o, ro)
    assert maxerr(lse, rl) <= tol["lse"], maxerr(lse, rl)
    dq, dk, dv = cpa.ulysses_bwd(qs, ks, vs, o, dos, lse, cp, layout, causal, bounds=bounds,
                                 grad_dtype=torch.float32)
    rq, rk, rv = oracle.ulysses_bwd(fq, fk, fv, fdo, cp, layout, causal, cu_seqlens=cu)
    for name, got, ref in (("dq", dq, rq), ("dk", dk, rk), ("dv", dv, rv)):
        assert maxerr(got, ref) <= tol["grad"], (name, maxerr(got, ref))
    assert cpa.device_status() == 0


def test_ulysses_rejects_head_counts_it_cannot_split():
    q = torch.zeros((1, 384, 6, 64), device=DEV, dtype=torch.bfloat16)
    k = torch.zeros((1, 384, 2, 64), device=DEV, dtype=torch.bfloat16)
    with pytest.raises(cpa.CpattnError):
        cpa.ulysses_fwd(q, k, k, 4)   # 6 query heads over 4 ranks
    with pytest.raises(cpa.CpattnError):
        cpa.ulysses_fwd(q, k, k, 3)   # 2 query heads per rank, kv groups of 3
    assert cpa.device_status() == 0


def test_ulysses_full_size():
    # The S=131072 workload through the Ulysses variant (16 ranks, 2 query
    # heads each, each kv head shared by 2 ranks): sampled rows against the
    # oracle and the sum rules of the gradients.
    w = inputs.WORKLOADS["c5_bf16_s131072_fwdbwd"]
    q, k, v, do = inputs.generate(w)
    qd, kd, vd, dod = (x.to(DEV) for x in (q, k, v, do))
    o, lse, dq, dk, dv = cpa.attention_ulysses_fwd_bwd(qd, kd, vd, dod, w.cp, w.layout, w.causal,
                                                       grad_dtype=torch.float32)
    assert cpa.device_status() == 0
    rng = np.random.default_rng(29)
    c = w.S // (2 * w.cp)
    edges = sorted({m * c for m in range(2 * w.cp)} | {m * c - 1 for m in range(1, 2 * w.cp)})
    rows = np.array([(0, h, i) for h in range(w.H)
                     for i in edges[h % 4::4] + rng.integers(0, w.S, 60).tolist()])
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
