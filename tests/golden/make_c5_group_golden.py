"""Writes the fp64 expected values of one kv group of the S=131072 workload.

Run once on any machine (about half an hour on 8 cores):

    python tests/golden/make_c5_group_golden.py

It calls only the CPU oracle.  The workload is B=1, H=32 query heads on
Hkv=8 kv heads, S=131072, D=128, causal, bf16 inputs with a dense dO
(N(0,1) everywhere).  Kv group 5 (query heads 20-23, kv head 5) takes its
values from the counter-based generator of ``inputs.group_inputs`` (seed
1005), which every machine reproduces bit for bit, so that values computed
here can be checked on another machine; the file stores the sha256 of those
inputs and the GPU test refuses to compare if its own draw differs.

Stored (``c5_kvgroup5_s131072.npz``), all from the attention definition of
"Context Parallelism for Long-Context Training", section "Prove attention
equivalence" (the sharded result must equal the unsharded one, outputs and
gradients):

* ``lse`` [4, S]: the LSE of every query row of the four heads (float32;
  rounding 6e-7 at most, far under the 1e-3 bar);
* ``o_rows`` [n] natural rows and ``o`` [4, n, D]: O on the first and last
  8 rows of every one of the 32 zigzag chunks and 64 more rows (float32);
* ``dq_rows`` / ``dq`` [4, m, D]: dQ of the definition on a subset of those
  rows (float64);
* ``k_rows`` / ``dk``, ``dv`` [nk, D]: dK and dV of kv head 5 at key rows
  0-31 (the longest sums over queries), the two keys on either side of every
  chunk border and the last key, summed over all four query heads and every
  query row (float64);
* ``meta``: the recipe and the input digest.

The whole forward of the four heads (17.6 TFLOP in float64) is what costs the
time; dK / dV at the listed keys reuse its O and LSE.
"""
import json
import os
import sys
import time

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(os.path.dirname(HERE))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import oracle  # noqa: E402
from context_causal_attention_zigzag_gb300 import inputs  # noqa: E402

WORKLOAD = "c5_bf16_s131072_fwdbwd"
GROUP = 5
OUT = os.path.join(HERE, "c5_kvgroup5_s131072.npz")


def key_rows(S: int, nchunk: int):
    c = S // nchunk
    keys = set(range(32))
    for b in range(1, nchunk):
        keys |= {b * c - 1, b * c}
    keys.add(S - 1)
    return np.array(sorted(keys), dtype=np.int64)


def o_rows(S: int, nchunk: int):
    c = S // nchunk
    rows = set()
    for b in range(nchunk):
        rows |= set(range(b * c, b * c + 8)) | set(range((b + 1) * c - 8, (b + 1) * c))
    rng = np.random.default_rng(20051)
    rows |= set(rng.integers(0, S, 64).tolist())
    return np.array(sorted(rows), dtype=np.int64)


def main():
    w = inputs.WORKLOADS[WORKLOAD]
    grp = w.H // w.Hkv
    nchunk = 2 * w.cp
    t0 = time.time()
    gq, gk, gv, gdo = inputs.group_inputs(w, GROUP)
    digest = inputs.digest(gq, gk, gv, gdo)
    q, k, v, do = (inputs.to_f32_numpy(x) for x in (gq, gk, gv, gdo))
    print(f"inputs {time.time() - t0:.1f} s, digest {digest}", flush=True)

    t0 = time.time()
    out, lse = oracle.attn_fwd(q, k, v, causal=w.causal)
    print(f"forward of {grp} heads: {time.time() - t0:.1f} s", flush=True)

    kr = key_rows(w.S, nchunk)
    t0 = time.time()
    dk, dv = oracle.attn_bwd_dkdv_rows(q, k, v, do, out, lse,
                                       np.stack([np.zeros_like(kr), np.zeros_like(kr), kr], 1),
                                       causal=w.causal)
    print(f"dK/dV at {len(kr)} keys: {time.time() - t0:.1f} s", flush=True)

    orows = o_rows(w.S, nchunk)
    o = np.stack([out[0, orows, h] for h in range(grp)]).astype(np.float32)
    dqr = orows[np.random.default_rng(20052).choice(len(orows), 128, replace=False)]
    dqr.sort()
    t0 = time.time()
    dq = oracle.attn_bwd_dq_rows(q, k, v, do,
                                 np.array([(0, h, i) for h in range(grp) for i in dqr]),
                                 causal=w.causal).reshape(grp, len(dqr), w.D)
    print(f"dQ at {len(dqr)} rows per head: {time.time() - t0:.1f} s", flush=True)

    meta = {
        "workload": WORKLOAD, "B": w.B, "H": w.H, "Hkv": w.Hkv, "S": w.S, "D": w.D,
        "cp": w.cp, "causal": w.causal, "dtype": "bf16", "group": GROUP,
        "query_heads": list(range(GROUP * grp, (GROUP + 1) * grp)), "seed": w.seed,
        "generator": "inputs.group_inputs (SplitMix64 counters, Box-Muller, float32, bf16)",
        "input_sha256": digest, "scale": 1.0 / float(np.sqrt(w.D)),
    }
    np.savez_compressed(OUT, meta=np.array(json.dumps(meta)), lse=lse[0].astype(np.float32),
                        o_rows=orows, o=o, dq_rows=dqr, dq=dq, k_rows=kr, dk=dk, dv=dv)
    print(f"wrote {OUT} ({os.path.getsize(OUT) / 1e6:.1f} MB)", flush=True)


if __name__ == "__main__":
    main()
