"""Seeded random sweep of small problems through the natural-order calls,
forward and backward, each against the oracle.

Every case draws: batch, kv heads and group size (GQA), head dim, input
precision, ring size, layout, causal or full attention, a sequence length
that is either a whole number of chunks or arbitrary (padded by the
document path), and, for some, packed documents with random lengths.  The
bars are those of the other parity files (float32 O <= 1e-4, LSE <= 1e-5,
gradients <= 1e-4; bf16 O <= 2e-2, LSE <= 1e-3, float32 gradients
<= 2e-2).  The draw is fixed by the case number, so a failure names a
reproducible problem.  The draws with plain lengths also go through the
hierarchical a2a+p2p schedule (when the ring splits into two levels) and the
one-pass backward (when the tensor-core backward takes them).
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
N_CASES = 64


def draw(i):
    rng = np.random.default_rng(7100 + i)
    dtype = torch.bfloat16 if rng.random() < 0.7 else torch.float32
    D = 128 if rng.random() < 0.75 else 64
    Hkv = int(rng.choice([1, 2, 4]))
    grp = int(rng.choice([1, 2, 4]))
    if Hkv * grp > 8:
        grp = 8 // Hkv
    B = int(rng.choice([1, 2]))
    cp = int(rng.choice([1, 2, 3, 4, 8]))
    layout = int(rng.choice([cpa.ZIGZAG, cpa.CONTIGUOUS]))
    causal = bool(rng.random() < 0.75)
    per = 2 if layout == cpa.ZIGZAG else 1
    if rng.random() < 0.5:
        # whole chunks of 128-token tiles (the tensor-core kernels take bf16, D=128)
        unit = cp * per * 128
        S = unit * int(rng.integers(1, max(2, 2048 // unit) + 1))
        padded = False
    else:
        S = int(rng.integers(1, 2049))
        padded = True
    cu = None
    if rng.random() < 0.4 and S > 1:
        ncut = int(rng.integers(1, min(6, S - 1) + 1))
        cuts = np.sort(rng.choice(np.arange(1, S), size=ncut, replace=False))
        cu = [0] + [int(c) for c in cuts] + [S]
    return dict(B=B, H=Hkv * grp, Hkv=Hkv, S=S, D=D, cp=cp, layout=layout, causal=causal,
                dtype=dtype, padded=padded, cu=cu, seed=7100 + i)


def case_id(i):
    c = draw(i)
    return "{}-B{B}H{H}K{Hkv}S{S}D{D}cp{cp}L{layout}c{c}{dt}{docs}".format(
        i, c=int(c["causal"]), dt="f32" if c["dtype"] == torch.float32 else "bf16",
        docs="docs" if c["cu"] else "", **{k: c[k] for k in ("B", "H", "Hkv", "S", "D", "cp",
                                                                "layout")})


def maxerr(gpu, ref):
    g = gpu.detach().to("cpu", torch.float64).numpy()
    return float(np.max(np.abs(g - ref))) if g.size else 0.0


@pytest.mark.parametrize("i", range(N_CASES), ids=case_id)
def test_random_case_matches_oracle(i):
    c = draw(i)
    w = inputs.Workload("sweep", c["B"], c["H"], c["Hkv"], c["S"], c["D"], c["cp"], c["layout"],
                        c["causal"], c["dtype"], seed=c["seed"])
    q, k, v, do = inputs.generate(w, with_dout=True)
    dev = [x.to(DEV) for x in (q, k, v, do)]
    f = [inputs.to_f32_numpy(x) for x in (q, k, v, do)]
    if c["padded"] or c["cu"] is not None:
        res = cpa.attention_docs_fwd_bwd(*dev, c["cp"], c["cu"], c["layout"], c["causal"],
                                         grad_dtype=torch.float32)
        cu = c["cu"] if c["cu"] is not None else [0, c["S"]]
        ro, rl = oracle.attn_fwd_docs(f[0], f[1], f[2], cu, causal=c["causal"])
        rg = oracle.attn_bwd_docs(*f, cu, causal=c["causal"])
    else:
        res = cpa.attention_fwd_bwd(*dev, c["cp"], c["layout"], c["causal"],
                                    grad_dtype=torch.float32)
        ro, rl = oracle.attn_fwd(f[0], f[1], f[2], causal=c["causal"])
        rg = oracle.attn_bwd(*f, causal=c["causal"])
    out, lse, dq, dk, dv = res
    tol = TOL[c["dtype"]]
    assert maxerr(out, ro) <= tol["o"], ("out", maxerr(out, ro))
    assert maxerr(lse, rl) <= tol["lse"], ("lse", maxerr(lse, rl))
    for name, got, ref in zip(("dq", "dk", "dv"), (dq, dk, dv), rg):
        assert maxerr(got, ref) <= tol["grad"], (name, maxerr(got, ref))
    assert cpa.device_status() == 0


def hier_split(c):
    """A two-level split [A, P] of the case's ring (A > 1, P > 1) whose head
    slices divide the kv groups (or the reverse), or None."""
    H, Hkv, cp = c["H"], c["Hkv"], c["cp"]
    for A in (2, 4):
        if cp % A or cp // A < 2 or H % A:
            continue
        hc, grp = H // A, H // Hkv
        if hc % grp == 0 or grp % hc == 0:
            return A, cp // A
    return None


@pytest.mark.parametrize("i", range(N_CASES), ids=case_id)
def test_random_case_other_routes(i):
    # The same draw through the hierarchical a2a+p2p schedule (when the ring
    # splits in two levels) and through the one-pass backward (when the
    # tensor-core backward takes the case), against the same oracle values.
    c = draw(i)
    if c["padded"] or c["cu"] is not None:
        pytest.skip("plain sequence lengths only")
    split = hier_split(c)
    onepass = (c["dtype"] == torch.bfloat16 and c["D"] == 128 and
               cpa.plan(c["B"], c["H"], c["Hkv"], c["S"], c["D"], c["cp"], c["layout"],
                        c["causal"], c["dtype"], backward=True)[0] == cpa.PATH_TCGEN05)
    if split is None and not onepass:
        pytest.skip("no second route for this draw")
    w = inputs.Workload("sweep", c["B"], c["H"], c["Hkv"], c["S"], c["D"], c["cp"], c["layout"],
                        c["causal"], c["dtype"], seed=c["seed"])
    q, k, v, do = inputs.generate(w, with_dout=True)
    dev = [x.to(DEV) for x in (q, k, v, do)]
    f = [inputs.to_f32_numpy(x) for x in (q, k, v, do)]
    ro, rl = oracle.attn_fwd(f[0], f[1], f[2], causal=c["causal"])
    rg = oracle.attn_bwd(*f, causal=c["causal"])
    tol = TOL[c["dtype"]]
    routes = []
    if split is not None:
        routes.append(cpa.attention_hier_fwd_bwd(*dev, split[0], split[1], c["layout"],
                                                 c["causal"], grad_dtype=torch.float32))
    if onepass:
        routes.append(cpa.attention_fwd_bwd(*dev, c["cp"], c["layout"], c["causal"],
                                            grad_dtype=torch.float32, onepass=True))
    for out, lse, dq, dk, dv in routes:
        assert maxerr(out, ro) <= tol["o"], ("out", maxerr(out, ro))
        assert maxerr(lse, rl) <= tol["lse"], ("lse", maxerr(lse, rl))
        for name, got, ref in zip(("dq", "dk", "dv"), (dq, dk, dv), rg):
            assert maxerr(got, ref) <= tol["grad"], (name, maxerr(got, ref))
    assert cpa.device_status() == 0
