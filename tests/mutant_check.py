"""Small GPU parity checks of one build of libcpattn against the CPU oracle.

    python tests/mutant_check.py <path of libcpattn.so>

Prints one JSON line {check: passed}.  tests/test_gpu_mutations.py runs it
on the regular library (every check must pass) and on builds with a planted
mistake (some check must fail), each in a process of its own.  The bars are
those of the parity tests: bf16 O and gradients 2e-2, LSE 1e-3, float32
merge 1e-5, tile census bit-exact.
"""
import json
import os
import sys

import numpy as np
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from context_causal_attention_zigzag_gb300 import _binding  # noqa: E402

_binding.LIB_PATH = os.path.abspath(sys.argv[1])

import oracle  # noqa: E402
import context_causal_attention_zigzag_gb300 as cpa  # noqa: E402
from context_causal_attention_zigzag_gb300 import inputs  # noqa: E402

DEV = "cuda"
B, H, Hkv, S, D, CP = 1, 4, 2, 2048, 128, 4


def f32(x):
    return inputs.to_f32_numpy(x)


def err(gpu, ref):
    g = gpu.detach().to("cpu", torch.float64).numpy()
    return float(np.max(np.abs(g - ref)))


def draw(layout, seed):
    w = inputs.Workload("mut", B, H, Hkv, S, D, CP, layout, True, torch.bfloat16, seed=seed)
    return inputs.generate(w, with_dout=True)


def check_forward():
    q, k, v, _ = draw(cpa.ZIGZAG, 9101)
    out, lse = cpa.attention(q.to(DEV), k.to(DEV), v.to(DEV), CP, cpa.ZIGZAG, True)
    ro, rl = oracle.attn_fwd(f32(q), f32(k), f32(v), causal=True)
    return err(out, ro) <= 2e-2 and err(lse, rl) <= 1e-3


def check_step_partials():
    ok = True
    for layout in (cpa.ZIGZAG, cpa.CONTIGUOUS):
        q, k, v, _ = draw(layout, 9102 + layout)
        qs, ks, vs = (cpa.zigzag_permute(x.to(DEV), CP, layout) for x in (q, k, v))
        for t in range(CP):
            po, pl = cpa.ring_fwd_step(qs, ks, vs, CP, t, layout, True)
            ro, rl = oracle.ring_step(f32(q), f32(k), f32(v), CP, layout, t, causal=True)
            go = cpa.zigzag_unpermute(po, CP, layout).double().cpu().numpy()
            gl = cpa.zigzag_unpermute(pl, CP, layout, seq_dim=2).double().cpu().numpy()
            if not np.array_equal(np.isneginf(gl), np.isneginf(rl)):
                return False
            fin = ~np.isneginf(rl)
            ok &= bool(np.max(np.abs(go - ro)) <= 2e-2)
            ok &= bool(np.max(np.abs(gl[fin] - rl[fin])) <= 1e-3)
    return ok


def check_merge():
    g = torch.Generator().manual_seed(9103)
    o_a, o_b = (torch.randn((B, 256, H, D), generator=g) for _ in range(2))
    l_a, l_b = (torch.randn((B, H, 256), generator=g) for _ in range(2))
    mo, ml = cpa.lse_merge(*(x.to(DEV) for x in (o_a, l_a, o_b, l_b)))
    ro, rl = oracle.lse_merge(o_a.double().numpy(), l_a.double().numpy(),
                              o_b.double().numpy(), l_b.double().numpy())
    return err(mo, ro) <= 1e-5 and err(ml, rl) <= 1e-5


def check_census():
    q, k, v, _ = draw(cpa.CONTIGUOUS, 9104)
    qs, ks, vs = (cpa.zigzag_permute(x.to(DEV), CP, cpa.CONTIGUOUS) for x in (q, k, v))
    _, _, counts = cpa.ring_fwd_census(qs, ks, vs, CP, cpa.CONTIGUOUS, True)
    _, tile = cpa.plan(B, H, Hkv, S, D, CP, cpa.CONTIGUOUS, True, torch.bfloat16)
    closed, _ = cpa.tile_counts(S, CP, cpa.CONTIGUOUS, True, tile)
    return bool(np.array_equal(counts.cpu().numpy().astype(np.uint64), closed * (B * H)))


def check_backward():
    q, k, v, do = draw(cpa.ZIGZAG, 9105)
    _, _, dq, dk, dv = cpa.attention_fwd_bwd(q.to(DEV), k.to(DEV), v.to(DEV), do.to(DEV), CP,
                                             cpa.ZIGZAG, True, grad_dtype=torch.float32)
    rq, rk, rv = oracle.attn_bwd(f32(q), f32(k), f32(v), f32(do), causal=True)
    return all(err(g, r) <= 2e-2 for g, r in ((dq, rq), (dk, rk), (dv, rv)))


CHECKS = {"forward": check_forward, "step_partials": check_step_partials,
          "merge": check_merge, "census": check_census, "backward": check_backward}


def main():
    res = {}
    for name, fn in CHECKS.items():
        try:
            res[name] = bool(fn())
        except cpa.CpattnError as e:
            res[name] = False
            res[name + "_error"] = str(e)
    res["device_status"] = cpa.device_status()
    print(json.dumps(res), flush=True)


if __name__ == "__main__":
    main()
