"""GPU parity of the all-gather K/V schedule ("Context Parallelism in
MegaDLMs", key-value communication patterns: every rank holds the whole K/V
before attention) against the oracle's all-gather schedule, which works on
the same sharded inputs.

Bars as for the ring: float32 O <= 1e-4, LSE <= 1e-5, gradients <= 1e-4;
bf16 O <= 2e-2, LSE <= 1e-3, gradients (written as float32, as for the ring's
long workloads) <= 2e-2; tile census bit-exact and equal to the ring's.
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
    w = inputs.Workload("ag", B, H, Hkv, S, D, 1, inputs.ZIGZAG, True, dtype, seed=seed)
    return inputs.generate(w, with_dout=dout)


def f32(x):
    return inputs.to_f32_numpy(x)


def maxerr(gpu, ref):
    g = gpu.detach().to("cpu", torch.float64).numpy() if torch.is_tensor(gpu) else gpu
    return float(np.max(np.abs(g - ref))) if g.size else 0.0


CASES = [
    # B, H, Hkv, S, D, cp, layout, causal, dtype, cu (None: one document)
    (1, 4, 2, 2048, 128, 4, cpa.ZIGZAG, True, torch.bfloat16, None),
    (2, 4, 1, 1536, 128, 3, cpa.ZIGZAG, True, torch.bfloat16, None),
    (1, 2, 2, 2048, 128, 2, cpa.CONTIGUOUS, True, torch.bfloat16, None),
    (1, 2, 1, 2048, 128, 4, cpa.CONTIGUOUS, False, torch.bfloat16, None),
    (1, 4, 2, 2048, 128, 2, cpa.ZIGZAG, True, torch.bfloat16, [0, 1, 130, 256, 700, 1024, 2048]),
    (1, 2, 2, 256, 64, 2, cpa.ZIGZAG, True, torch.float32, None),
    (2, 4, 2, 320, 64, 4, cpa.ZIGZAG, False, torch.float32, [0, 17, 100, 101, 320]),
    (1, 2, 1, 640, 128, 2, cpa.ZIGZAG, True, torch.bfloat16, None),  # chunk 160: CUDA cores
]


def case_id(c):
    return "B{}H{}K{}S{}D{}cp{}L{}c{}{}{}".format(
        *c[:8], "f32" if c[8] == torch.float32 else "bf16", "" if c[9] is None else "docs")


def shard(x, cp, layout):
    return cpa.zigzag_permute(x.to(DEV), cp, layout)


@pytest.mark.parametrize("case", CASES, ids=case_id)
def test_allgather_forward_backward_match_oracle(case):
    B, H, Hkv, S, D, cp, layout, causal, dtype, cu = case
    q, k, v, do = make(B, H, Hkv, S, D, dtype, seed=7000 + S + cp, dout=True)
    qs, ks, vs, dos = (shard(x, cp, layout) for x in (q, k, v, do))
    kf, vf = cpa.kv_allgather(ks, vs, cp, layout)
    assert torch.equal(kf, k.to(DEV)) and torch.equal(vf, v.to(DEV))
    bounds = cpa.doc_bounds(cu, S) if cu is not None else None
    o, lse = cpa.allgather_fwd(qs, kf, vf, cp, layout, causal, bounds=bounds)
    order = oracle.shard_order(S, cp, layout)
    fq, fk, fv, fdo = (f32(x)[:, order] for x in (q, k, v, do))
    ro, rl = oracle.allgather_fwd(fq, fk, fv, cp, layout, causal, cu_seqlens=cu)
    tol = TOL[dtype]
    assert maxerr(o, ro) <= tol["o"], maxerr(o, ro)
    assert maxerr(lse, rl) <= tol["lse"], maxerr(lse, rl)
    dq, dkf, dvf = cpa.allgather_bwd(qs, kf, vf, o, dos, lse, cp, layout, causal, bounds=bounds,
                                     grad_dtype=torch.float32)
    # The reduce-scatter: each rank keeps its shard of the summed dK / dV.
    dks, dvs = shard(dkf, cp, layout), shard(dvf, cp, layout)
    rq, rk, rv = oracle.allgather_bwd(fq, fk, fv, fdo, cp, layout, causal, cu_seqlens=cu)
    for name, got, ref in (("dq", dq, rq), ("dk", dks, rk), ("dv", dvs, rv)):
        assert maxerr(got, ref) <= tol["grad"], (name, maxerr(got, ref))
    assert cpa.device_status() == 0


@pytest.mark.parametrize("case", [c for c in CASES if c[0] * c[1] <= 4], ids=case_id)
def test_allgather_census_equals_ring(case):
    # Each tile is attributed to the ring step at which its chunk would have
    # arrived, so the all-gather census equals the ring's, tile for tile.
    B, H, Hkv, S, D, cp, layout, causal, dtype, cu = case
    _, tile = cpa.plan(B, H, Hkv, S, D, cp, layout, causal, dtype)
    if (S // (cp * (2 if layout == cpa.ZIGZAG else 1))) % tile:
        pytest.skip("census needs whole tiles per chunk")
    q, k, v, _ = make(B, H, Hkv, S, D, dtype, seed=7100 + S)
    qs, ks, vs = (shard(x, cp, layout) for x in (q, k, v))
    kf, vf = cpa.kv_allgather(ks, vs, cp, layout)
    bounds = cpa.doc_bounds(cu if cu is not None else [0, S], S)
    counts = torch.zeros((cp, cp), device=DEV, dtype=torch.int64)
    cpa.allgather_fwd(qs, kf, vf, cp, layout, causal, bounds=bounds, tiles_rt=counts)
    _, _, ring = cpa.ring_fwd_docs_census(qs, ks, vs, cp, bounds, layout, causal)
    assert torch.equal(counts, ring)
    ref, _ = oracle.tile_counts_docs(S, cp, layout, causal, cu if cu is not None else [0, S], tile)
    assert np.array_equal(counts.cpu().numpy(), ref.astype(np.int64) * B * H)


def test_allgather_agrees_with_ring_natural_order():
    # The natural-order convenience through the all-gather schedule against
    # the ring's, on the same inputs.
    B, H, Hkv, S, D, cp = 1, 4, 2, 4096, 128, 4
    q, k, v, do = (x.to(DEV) for x in make(B, H, Hkv, S, D, torch.bfloat16, seed=71, dout=True))
    a = cpa.attention_allgather_fwd_bwd(q, k, v, do, cp, grad_dtype=torch.float32)
    b = cpa.attention_fwd_bwd(q, k, v, do, cp, grad_dtype=torch.float32)
    for name, x, y in zip(("o", "lse", "dq", "dk", "dv"), a, b):
        err = (x.double() - y.double()).abs().max().item()
        assert err <= (1e-3 if name == "lse" else 2e-2), (name, err)
    assert cpa.device_status() == 0


def test_allgather_full_size():
    # The S=131072 workload through the all-gather schedule: sampled rows
    # against the oracle, and the sum rules of the gathered gradients.
    w = inputs.WORKLOADS["c5_bf16_s131072_fwdbwd"]
    q, k, v, do = inputs.generate(w)
    qd, kd, vd, dod = (x.to(DEV) for x in (q, k, v, do))
    o, lse, dq, dk, dv = cpa.attention_allgather_fwd_bwd(qd, kd, vd, dod, w.cp, w.layout, w.causal,
                                                         grad_dtype=torch.float32)
    assert cpa.device_status() == 0
    rng = np.random.default_rng(23)
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
