"""GPU parity of the one-pass tensor-core backward (CPATTN_BWD_ONEPASS).

One K/V-major walk computes dK, dV and dQ ("Context Parallelism for
Long-Context Training", section "Prove attention equivalence": the gradients
of the sharded computation equal the unsharded ones); each K/V tile adds its
share of dQ to a float32 accumulator with bulk reductions, so dQ's summation
order follows the order the reductions arrive and is not bitwise
reproducible.  Bars: the oracle at the parity tests' tolerances (bf16
inputs: 2e-2 on every gradient), dK and dV bit-identical to the two-kernel
path (the same products accumulated in the same order), dQ within float32
reordering error of the two-kernel path's, the tile census bit-exact, and at
S=131072 the stored fp64 values of one kv group with the dense dO.
"""
import json
import os

import numpy as np
import pytest
import torch

import oracle
import context_causal_attention_zigzag_gb300 as cpa
from context_causal_attention_zigzag_gb300 import inputs

pytestmark = pytest.mark.gpu
DEV = "cuda"
GOLDEN_C5 = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden",
                         "c5_kvgroup5_s131072.npz")


def f32(x):
    return inputs.to_f32_numpy(x)


def maxerr(gpu, ref):
    g = gpu.detach().to("cpu", torch.float64).numpy() if torch.is_tensor(gpu) else gpu
    return float(np.max(np.abs(g - ref))) if g.size else 0.0


CASES = [
    # B, H, Hkv, S, cp, layout, causal, grad dtype
    (1, 4, 2, 1024, 4, cpa.ZIGZAG, True, torch.bfloat16),
    (1, 4, 2, 1024, 4, cpa.ZIGZAG, True, torch.float32),
    (1, 4, 1, 2048, 2, cpa.CONTIGUOUS, True, torch.float32),
    (1, 2, 2, 1024, 2, cpa.ZIGZAG, False, torch.float32),
    (1, 2, 1, 768, 3, cpa.ZIGZAG, True, torch.float32),
    (2, 8, 4, 4096, 4, cpa.ZIGZAG, True, torch.float32),
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "B{}H{}K{}S{}cp{}L{}c{}{}".format(
    *c[:7], "f32" if c[7] == torch.float32 else "bf16"))
def test_onepass_matches_oracle_and_two_kernel_path(case):
    B, H, Hkv, S, cp, layout, causal, gdt = case
    w = inputs.Workload("onepass", B, H, Hkv, S, 128, cp, layout, causal, torch.bfloat16,
                        seed=7000 + S + cp)
    q, k, v, do = inputs.generate(w, with_dout=True)
    assert cpa.plan(B, H, Hkv, S, 128, cp, layout, causal, torch.bfloat16,
                    backward=True)[0] == cpa.PATH_TCGEN05
    qs, ks, vs, dos = (cpa.zigzag_permute(x.to(DEV), cp, layout) for x in (q, k, v, do))
    o, lse = cpa.ring_fwd(qs, ks, vs, cp, layout, causal)
    one = cpa.ring_bwd(qs, ks, vs, o, dos, lse, cp, layout, causal, grad_dtype=gdt, onepass=True)
    two = cpa.ring_bwd(qs, ks, vs, o, dos, lse, cp, layout, causal, grad_dtype=gdt)
    assert torch.equal(one[1], two[1]) and torch.equal(one[2], two[2])   # dK, dV
    dq_gap = (one[0].double() - two[0].double()).abs().max().item()
    assert dq_gap <= (1e-3 if gdt == torch.float32 else 2 ** -7), dq_gap
    rq, rk, rv = oracle.attn_bwd(f32(q), f32(k), f32(v), f32(do), causal=causal)
    for got, ref in zip(one, (rq, rk, rv)):
        nat = cpa.zigzag_unpermute(got, cp, layout)
        assert maxerr(nat, ref) <= 2e-2, maxerr(nat, ref)
    assert cpa.device_status() == 0


def test_onepass_census_bit_exact():
    B, H, Hkv, S, cp = 2, 4, 2, 8192, 8
    for layout in (cpa.ZIGZAG, cpa.CONTIGUOUS):
        w = inputs.Workload("census", B, H, Hkv, S, 128, cp, layout, True, torch.bfloat16,
                            seed=7100 + layout)
        q, k, v, do = inputs.generate(w, with_dout=True)
        qs, ks, vs, dos = (cpa.zigzag_permute(x.to(DEV), cp, layout) for x in (q, k, v, do))
        o, lse = cpa.ring_fwd(qs, ks, vs, cp, layout, True)
        kv_rt = torch.zeros((cp, cp), device=DEV, dtype=torch.int64)
        q_rt = torch.zeros((cp, cp), device=DEV, dtype=torch.int64)
        cpa.ring_bwd(qs, ks, vs, o, dos, lse, cp, layout, True, tiles_kv_rt=kv_rt,
                     tiles_q_rt=q_rt, onepass=True)
        closed, _ = cpa.tile_counts(S, cp, layout, True, 128)
        for got in (kv_rt, q_rt):
            assert np.array_equal(got.cpu().numpy().astype(np.uint64), closed * (B * H))
    assert cpa.device_status() == 0


def test_onepass_documents_match_oracle():
    B, H, Hkv, S, cp = 1, 4, 2, 2048, 4
    cu = [0, 1, 300, 1024, 1500, 2048]
    w = inputs.Workload("onepass_docs", B, H, Hkv, S, 128, cp, cpa.ZIGZAG, True,
                        torch.bfloat16, seed=7200)
    q, k, v, do = inputs.generate(w, with_dout=True)
    _, _, dq, dk, dv = cpa.attention_docs_fwd_bwd(q.to(DEV), k.to(DEV), v.to(DEV), do.to(DEV), cp,
                                                  cu, cpa.ZIGZAG, True,
                                                  grad_dtype=torch.float32, onepass=True)
    rq, rk, rv = oracle.attn_bwd_docs(f32(q), f32(k), f32(v), f32(do), cu, causal=True)
    for got, ref in ((dq, rq), (dk, rk), (dv, rv)):
        assert maxerr(got, ref) <= 2e-2, maxerr(got, ref)
    assert cpa.device_status() == 0


def test_onepass_c5_full_size_against_stored_values():
    # The S=131072 workload (cp 16, zigzag, B1 H32 Hkv8, bf16, float32
    # gradients) through the one-pass backward; kv group 5 carries the
    # counter-based draws whose fp64 oracle values are stored.
    w = inputs.WORKLOADS["c5_bf16_s131072_fwdbwd"]
    q, k, v, do = inputs.generate(w)
    gold = np.load(GOLDEN_C5)
    meta = json.loads(str(gold["meta"]))
    g = meta["group"]
    group = inputs.group_inputs(w, g)
    assert inputs.digest(*group) == meta["input_sha256"], "kv group draw differs from the stored"
    inputs.embed_group(w, g, (q, k, v, do), group)
    dod = do.to(DEV)
    _, lse, dq, dk, dv = cpa.attention_fwd_bwd(q.to(DEV), k.to(DEV), v.to(DEV), dod, w.cp,
                                               w.layout, w.causal, grad_dtype=torch.float32,
                                               onepass=True)
    assert cpa.device_status() == 0
    heads = meta["query_heads"]
    assert maxerr(lse[0, heads], gold["lse"]) <= 1e-3
    qrows = torch.as_tensor(gold["dq_rows"]).to(DEV)
    gdq = dq[0, qrows][:, heads].double().cpu().numpy().transpose(1, 0, 2)
    assert np.max(np.abs(gdq - gold["dq"])) <= 2e-2, np.max(np.abs(gdq - gold["dq"]))
    krows = torch.as_tensor(gold["k_rows"]).to(DEV)
    assert maxerr(dk[0, krows, g], gold["dk"]) <= 2e-2, maxerr(dk[0, krows, g], gold["dk"])
    assert maxerr(dv[0, krows, g], gold["dv"]) <= 2e-2, maxerr(dv[0, krows, g], gold["dv"])
    grp = w.H // w.Hkv
    bound = 4e-3 * np.sqrt(w.S)
    sdo = dod.double().sum(dim=1)[0].view(w.Hkv, grp, w.D).sum(1)
    assert (dv.double().sum(dim=1)[0] - sdo).abs().max().item() <= bound
    assert dk.double().sum(dim=1).abs().max().item() <= bound
