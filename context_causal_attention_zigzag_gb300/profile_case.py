"""Runs one workload's forward (and backward) a few times: the program that
profiler captures (ncu) wrap.

    python -m context_causal_attention_zigzag_gb300.profile_case fwd_s32768
    python -m context_causal_attention_zigzag_gb300.profile_case bwd_s16384 [--onepass]
    python -m context_causal_attention_zigzag_gb300.profile_case bwd_s131072_g1
    python -m context_causal_attention_zigzag_gb300.profile_case docs_s16384 [--onepass]
    python -m context_causal_attention_zigzag_gb300.profile_case permute_s32768
    python -m context_causal_attention_zigzag_gb300.profile_case merge_s32768

Cases are reduced versions of the named workloads (same heads, head dim and
layout; fewer tokens or batches) so that a full counter capture of one launch
stays small: a few hundred MB on the device and a few ms per launch.
"""
import argparse

import torch

from . import _binding as cpa
from . import inputs

CASES = {
    # half of the S=32768 forward workload (one batch of two)
    "fwd_s32768": inputs.Workload("fwd_s32768", 1, 32, 8, 32768, 128, 8, cpa.ZIGZAG, True,
                                  torch.bfloat16, backward=False, seed=5),
    # the S=131072 forward+backward workload at S=16384 (1/64 of its tile pairs)
    "bwd_s16384": inputs.Workload("bwd_s16384", 1, 32, 8, 16384, 128, 4, cpa.ZIGZAG, True,
                                  torch.bfloat16, backward=True, seed=5),
    # one kv group of the S=131072 workload (4 query heads on 1 kv head): the
    # same per-head Q / dO working set as the full workload, 1/8 of its heads
    "bwd_s131072_g1": inputs.Workload("bwd_s131072_g1", 1, 4, 1, 131072, 128, 16, cpa.ZIGZAG,
                                      True, torch.bfloat16, backward=True, seed=5),
    # the packed-document workload reduced the same way (documents of mean
    # length 1024 instead of 8192)
    "docs_s16384": inputs.Workload("docs_s16384", 1, 32, 8, 16384, 128, 4, cpa.ZIGZAG, True,
                                   torch.bfloat16, backward=True, seed=5, doc_mean=1024,
                                   doc_seed=2006),
}


# The HBM-bound kernels on a query-sized tensor of the S=32768 shape (larger
# than L2): zigzag permute of a bf16 [1, 32768, 32, 128] tensor (256 MiB),
# LSE merge of two float32 partials of that shape (512 MiB each).
HBM_CASES = {"permute_s32768": (1, 32768, 32, 128, 8), "merge_s32768": (1, 32768, 32, 128, 8)}


def run_hbm(case: str, repeats: int) -> int:
    B, S, H, D, cp = HBM_CASES[case]
    dev = torch.device("cuda", torch.cuda.current_device())
    g = torch.Generator(device="cpu").manual_seed(6)
    if case.startswith("permute"):
        x = torch.randn((B, S, H, D), generator=g).to(torch.bfloat16).to(dev)
        y = torch.empty_like(x)
        for _ in range(repeats):
            cpa.zigzag_permute(x, cp, cpa.ZIGZAG, out=y)
    else:
        o_a = torch.randn((B, S, H, D), generator=g).to(dev)
        o_b = torch.randn((B, S, H, D), generator=g).to(dev)
        l_a = torch.randn((B, H, S), generator=g).to(dev)
        l_b = torch.randn((B, H, S), generator=g).to(dev)
        o_out, l_out = torch.empty_like(o_a), torch.empty_like(l_a)
        for _ in range(repeats):
            cpa.lse_merge(o_a, l_a, o_b, l_b, o_out, l_out)
    torch.cuda.synchronize()
    return cpa.device_status()


def run(case: str, repeats: int = 3, onepass: bool = False) -> int:
    if case in HBM_CASES:
        return run_hbm(case, repeats)
    w = CASES[case]
    dev = torch.device("cuda", torch.cuda.current_device())
    q, k, v, do = (x.to(dev) if x is not None else None for x in inputs.generate(w))
    qs, ks, vs = (cpa.zigzag_permute(x, w.cp, w.layout) for x in (q, k, v))
    dos = cpa.zigzag_permute(do, w.cp, w.layout) if do is not None else None
    cu = w.doc_offsets()
    bounds = cpa.doc_bounds(cu, w.S) if cu is not None else None
    for _ in range(repeats):
        if bounds is None:
            o, lse = cpa.ring_fwd(qs, ks, vs, w.cp, w.layout, w.causal)
        else:
            o, lse = cpa.ring_fwd_docs(qs, ks, vs, w.cp, bounds, w.layout, w.causal)
        if dos is not None and bounds is None:
            cpa.ring_bwd(qs, ks, vs, o, dos, lse, w.cp, w.layout, w.causal,
                         grad_dtype=torch.float32, onepass=onepass)
        elif dos is not None:
            cpa.ring_bwd_docs(qs, ks, vs, o, dos, lse, w.cp, bounds, w.layout, w.causal,
                              grad_dtype=torch.float32, onepass=onepass)
    torch.cuda.synchronize()
    return cpa.device_status()


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("case", choices=sorted(CASES) + sorted(HBM_CASES))
    ap.add_argument("--repeats", type=int, default=3)
    ap.add_argument("--onepass", action="store_true",
                    help="the one-pass backward (CPATTN_BWD_ONEPASS) instead of the two kernels")
    a = ap.parse_args()
    status = run(a.case, a.repeats, a.onepass)
    print(f"{a.case}: status {status}")
    raise SystemExit(0 if status == 0 else 1)


if __name__ == "__main__":
    main()
