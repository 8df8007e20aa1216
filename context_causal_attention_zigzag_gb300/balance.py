"""Per-iteration balance of the ring: useful tiles per (virtual rank, ring step).

"Sequence Parallelism IV: Megatron Context Parallel and Load-Balanced Rings",
TL;DR and section 3: ranks of a ring move in lockstep, so what matters is the
busiest rank of every ring iteration, not the average; the zigzag placement
pairs an early and a late chunk per rank so that every rank has the same
useful causal work at every step.

The report puts side by side, for the zigzag and the contiguous placement:
  * the kernel's own census (``cpattn_ring_fwd_census``: tile pairs the
    forward actually processed per rank and step, summed over batch and heads),
  * the library's closed form (``cpattn_tile_counts``), which it must equal
    exactly,
  * per step: max / mean over ranks (1.0 = perfectly balanced) and the
    lockstep efficiency  sum(work) / (cp * sum_t max_r work[r, t]).

    python -m context_causal_attention_zigzag_gb300.balance --S 32768 --cp 8
"""
import argparse
import json

import numpy as np
import torch

from . import _binding as cpa
from . import inputs


def closed_form(S, cp, layout, causal, tile):
    tiles, pairs = cpa.tile_counts(S, cp, layout, causal, tile)
    return tiles.astype(np.int64), pairs.astype(np.int64)


def summarize(counts):
    """counts[r, t] -> per-step max/mean and lockstep efficiency."""
    c = np.asarray(counts, dtype=np.float64)
    mean = c.mean(axis=0)
    mx = c.max(axis=0)
    ratio = np.where(mean > 0, mx / np.maximum(mean, 1e-30), 1.0)
    eff = float(c.sum() / (c.shape[0] * mx.sum())) if mx.sum() > 0 else 1.0
    return {"max_over_mean_per_step": ratio.tolist(), "worst_step_max_over_mean": float(ratio.max()),
            "lockstep_efficiency": eff}


def report(B=1, H=4, Hkv=4, S=8192, D=128, cp=4, causal=True, device="cuda", seed=7,
           run_kernel=True):
    """Balance report for both placements; the kernel census is included when
    a GPU is available and run_kernel is set."""
    out = {"S": S, "cp": cp, "B": B, "H": H, "Hkv": Hkv, "D": D, "causal": causal}
    for name, layout in (("zigzag", cpa.ZIGZAG), ("contiguous", cpa.CONTIGUOUS)):
        path, tile = cpa.plan(B, H, Hkv, S, D, cp, layout, causal, cpa.BF16)
        tiles, pairs = closed_form(S, cp, layout, causal, tile)
        entry = {"tile": tile, "path": "tcgen05" if path == cpa.PATH_TCGEN05 else "simt",
                 "closed_form_tiles_per_head": tiles.tolist(),
                 "closed_form_pairs_per_head": pairs.tolist(),
                 "closed_form": summarize(tiles)}
        if run_kernel and torch.cuda.is_available():
            w = inputs.Workload("balance", B, H, Hkv, S, D, cp, layout, causal, torch.bfloat16,
                                seed=seed)
            q, k, v, _ = inputs.generate(w)
            qs, ks, vs = (cpa.zigzag_permute(x.to(device), cp, layout) for x in (q, k, v))
            _, _, counts = cpa.ring_fwd_census(qs, ks, vs, cp, layout, causal)
            got = counts.cpu().numpy().astype(np.int64)
            entry["kernel_tiles"] = got.tolist()
            entry["kernel_equals_closed_form"] = bool(np.array_equal(got, tiles * B * H))
            entry["kernel"] = summarize(got)
        out[name] = entry
    return out


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    ap.add_argument("--B", type=int, default=1)
    ap.add_argument("--H", type=int, default=4)
    ap.add_argument("--Hkv", type=int, default=4)
    ap.add_argument("--S", type=int, default=8192)
    ap.add_argument("--D", type=int, default=128)
    ap.add_argument("--cp", type=int, default=4)
    ap.add_argument("--non-causal", action="store_true")
    ap.add_argument("--no-kernel", action="store_true")
    a = ap.parse_args()
    r = report(a.B, a.H, a.Hkv, a.S, a.D, a.cp, not a.non_causal, run_kernel=not a.no_kernel)
    print(json.dumps(r))


if __name__ == "__main__":
    main()
