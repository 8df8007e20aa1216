"""Seeded synthetic inputs and the named workloads.

This module holds no attention arithmetic: it only draws random numbers and
names shapes.  Both the CUDA path's tests/benchmarks and the CPU oracle take
their inputs from here, so the two sides see identical values.

Recipe: a CPU ``torch.Generator`` seeded with ``seed``; ``randn`` in float32,
drawn in the order Q, K, V, dO (dO only when asked for), each then rounded to
the workload's dtype (round to nearest even for bf16).  Tensors are
[B, S, H, D] (K, V, dO: [B, S, Hkv, D] / [B, S, H, D]) in natural token order.
The pages publish no data set; these standard-normal draws are the
distribution every workload below names.

Expected values stored in tests/golden/ for a kv group of the S=131072
workload use the counter-based draws at the end of this module instead,
which every machine reproduces bit for bit.

Packed documents: the pages test document masks but give no length
distribution.  ``packed_doc_offsets`` draws document lengths from an
exponential distribution with a stated mean (many short documents, a few
long ones), from its own generator seeded with ``doc_seed``; the last
document is cut at S.
"""
import math
import os
from dataclasses import dataclass, field, replace
from typing import Optional, Tuple

import numpy as np
import torch

CONTIGUOUS = 0
ZIGZAG = 1


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    H: int
    Hkv: int
    S: int
    D: int
    cp: int
    layout: int
    causal: bool
    dtype: torch.dtype
    backward: bool = False
    seed: int = 0
    cp_sweep: Tuple[int, ...] = field(default_factory=tuple)
    doc_mean: int = 0   # > 0: packed documents of this mean length
    doc_seed: int = 0

    def with_(self, **kw) -> "Workload":
        return replace(self, **kw)

    @property
    def dtype_name(self) -> str:
        return {torch.float32: "f32", torch.bfloat16: "bf16"}[self.dtype]

    def doc_offsets(self):
        """Document offsets [0, ..., S], or None for one document."""
        if self.doc_mean <= 0:
            return None
        return packed_doc_offsets(self.S, self.doc_mean, self.doc_seed)

    def valid_pairs_per_head(self) -> int:
        cu = self.doc_offsets()
        lens = [self.S] if cu is None else [b - a for a, b in zip(cu[:-1], cu[1:])]
        return sum(n * (n + 1) // 2 if self.causal else n * n for n in lens)

    def useful_flops(self, backward: bool = False) -> float:
        """4*D flops per valid (q, k) pair forward, 10*D backward."""
        per = (10 if backward else 4) * self.D
        return float(per) * self.valid_pairs_per_head() * self.B * self.H


# The five workloads: shapes, ring size, layout, mask and dtype.  Seeds are
# 1000 + the workload's number.
WORKLOADS = {
    "c1_fp32_s256": Workload("c1_fp32_s256", 1, 2, 2, 256, 64, 2, ZIGZAG, True,
                             torch.float32, seed=1001),
    "c2_bf16_s8192": Workload("c2_bf16_s8192", 1, 32, 32, 8192, 128, 4, ZIGZAG, True,
                              torch.bfloat16, seed=1002),
    "c3_bf16_s32768_gqa": Workload("c3_bf16_s32768_gqa", 2, 32, 8, 32768, 128, 8, ZIGZAG, True,
                                   torch.bfloat16, seed=1003),
    "c4_bf16_s16384_bidir": Workload("c4_bf16_s16384_bidir", 1, 16, 16, 16384, 128, 4,
                                     CONTIGUOUS, False, torch.bfloat16, seed=1004,
                                     cp_sweep=(1, 2, 4, 8)),
    "c5_bf16_s131072_fwdbwd": Workload("c5_bf16_s131072_fwdbwd", 1, 32, 8, 131072, 128, 16,
                                       ZIGZAG, True, torch.bfloat16, backward=True, seed=1005),
}

# The S=131072 shape with packed documents (mean length 8192 tokens): the
# document-mask workload.
DOC_WORKLOADS = {
    "docs_bf16_s131072_fwdbwd": Workload("docs_bf16_s131072_fwdbwd", 1, 32, 8, 131072, 128, 16,
                                         ZIGZAG, True, torch.bfloat16, backward=True, seed=1006,
                                         doc_mean=8192, doc_seed=2006),
}


def packed_doc_offsets(S: int, mean_len: float, seed: int, min_len: int = 1):
    """Offsets [0, c1, ..., S] of documents packed into S tokens: lengths
    exponential with mean ``mean_len`` (at least ``min_len``), the last
    document cut at S."""
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    cu = [0]
    while cu[-1] < S:
        u = float(torch.rand((), generator=g, dtype=torch.float64))
        n = max(min_len, int(round(-mean_len * math.log1p(-u))))
        cu.append(min(S, cu[-1] + n))
    return cu


def generate(w: Workload, with_dout: Optional[bool] = None, pin: bool = False):
    """Returns (q, k, v, dout-or-None) as CPU tensors of w.dtype."""
    if with_dout is None:
        with_dout = w.backward
    g = torch.Generator(device="cpu")
    g.manual_seed(w.seed)

    def draw(shape):
        x = torch.randn(shape, generator=g, dtype=torch.float32).to(w.dtype)
        return x.pin_memory() if pin else x

    q = draw((w.B, w.S, w.H, w.D))
    k = draw((w.B, w.S, w.Hkv, w.D))
    v = draw((w.B, w.S, w.Hkv, w.D))
    do = draw((w.B, w.S, w.H, w.D)) if with_dout else None
    return q, k, v, do


def to_f32_numpy(x: torch.Tensor):
    """Exact float32 copy (bf16 and fp32 values are representable) as numpy."""
    return x.detach().to("cpu", torch.float32).contiguous().numpy()


# ---------------------------------------------------------------------------
# Counter-based draws that every machine reproduces bit for bit
# ---------------------------------------------------------------------------
#
# ``torch.randn`` on the CPU is not reproducible across machines: the same
# seeded workload drawn on an x86_64 host and on an aarch64 host gives
# tensors with different digests (its float32 normal sampler is vectorised
# differently per architecture).  Expected values computed on one machine
# and checked on another need draws that do not depend on the machine.  Here
# element n of a tensor gets two 64-bit words from SplitMix64 (Steele, Lea
# and Flood, "Fast splittable pseudorandom number generators", 2014: the
# state advances by the odd constant 0x9E3779B97F4A7C15 and each output is
# the state passed through two xor-shift-multiply rounds and a final
# xor-shift) used as a counter-based generator: the state for counter c is
# key + (c + 1) * 0x9E3779B97F4A7C15, so any element can be drawn on its own.
# The two words become uniforms u1 in (0, 1] and u2 in [0, 1) from their top
# 53 bits, and the Box-Muller transform sqrt(-2 ln u1) cos(2 pi u2) gives a
# standard normal in float64 (integer steps are exact everywhere; the
# float64 log / cos differ between math libraries by an ulp at most, which
# moves a bf16 rounding once in about 2^43 draws).  The value is then rounded
# to float32 and to the workload dtype (round to nearest even).

_GAMMA = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)


def _splitmix_out(z):
    z = (z ^ (z >> np.uint64(30))) * _M1
    z = (z ^ (z >> np.uint64(27))) * _M2
    return z ^ (z >> np.uint64(31))


def counter_key(seed: int, stream: int) -> int:
    """The generator key of one tensor (``stream``) of a seeded draw."""
    with np.errstate(over="ignore"):
        z = np.array([(int(seed) * 16 + int(stream)) & (2**64 - 1)], np.uint64) * _GAMMA
        return int(_splitmix_out(z)[0])


def counter_normal(key: int, index: np.ndarray) -> np.ndarray:
    """Standard normals (float64) for the counters ``index`` (natural flat
    element indices) of the tensor with generator key ``key``."""
    c = np.asarray(index, dtype=np.uint64) * np.uint64(2)
    k = np.uint64(key)
    with np.errstate(over="ignore"):
        w1 = _splitmix_out(k + (c + np.uint64(1)) * _GAMMA)
        w2 = _splitmix_out(k + (c + np.uint64(2)) * _GAMMA)
    u1 = ((w1 >> np.uint64(11)) + np.uint64(1)).astype(np.float64) * (2.0 ** -53)
    u2 = (w2 >> np.uint64(11)).astype(np.float64) * (2.0 ** -53)
    return np.sqrt(-2.0 * np.log(u1)) * np.cos(2.0 * np.pi * u2)


def counter_slice(key: int, full_shape, x0: int, nx: int, threads: int = 0) -> np.ndarray:
    """float32 draws of the heads [x0, x0 + nx) of a [B, S, X, D] tensor:
    element (b, s, x, d) takes counter ((b*S + s)*X + x)*D + d of the full
    tensor, so a slice holds the same values as the whole tensor would."""
    import concurrent.futures as cf
    B, S, X, D = (int(a) for a in full_shape)
    out = np.empty((B * S, nx, D), np.float32)
    rows = B * S
    step = 4096
    hx = np.arange(x0, x0 + nx, dtype=np.uint64)[:, None] * np.uint64(D)
    dd = np.arange(D, dtype=np.uint64)[None, :]
    inner = (hx + dd)[None]                       # [1, nx, D]

    def fill(r0):
        r1 = min(rows, r0 + step)
        base = np.arange(r0, r1, dtype=np.uint64)[:, None, None] * np.uint64(X * D)
        out[r0:r1] = counter_normal(key, base + inner).astype(np.float32)

    n = threads or min(16, os.cpu_count() or 1)
    with cf.ThreadPoolExecutor(max_workers=n) as ex:
        list(ex.map(fill, range(0, rows, step)))
    return out.reshape(B, S, nx, D)


def group_inputs(w: Workload, g: int):
    """Counter-based inputs of kv group ``g`` of workload ``w``: Q and dO of
    its query heads [g*H/Hkv, (g+1)*H/Hkv), K and V of kv head g, each value
    drawn for its natural index in the full tensor and rounded to w.dtype.
    Returns CPU tensors q [B,S,H/Hkv,D], k, v [B,S,1,D], dout [B,S,H/Hkv,D]."""
    grp = w.H // w.Hkv
    full_q = (w.B, w.S, w.H, w.D)
    full_k = (w.B, w.S, w.Hkv, w.D)
    parts = []
    for stream, (shape, x0, nx) in enumerate(((full_q, g * grp, grp), (full_k, g, 1),
                                              (full_k, g, 1), (full_q, g * grp, grp))):
        a = counter_slice(counter_key(w.seed, stream), shape, x0, nx)
        parts.append(torch.from_numpy(a).to(w.dtype))
    return tuple(parts)


def embed_group(w: Workload, g: int, full, group):
    """Writes the kv-group tensors ``group`` (from ``group_inputs``) into the
    full tensors ``full`` = (q, k, v, dout) in place."""
    grp = w.H // w.Hkv
    q, k, v, do = full
    gq, gk, gv, gdo = group
    q[:, :, g * grp:(g + 1) * grp] = gq
    k[:, :, g:g + 1] = gk
    v[:, :, g:g + 1] = gv
    do[:, :, g * grp:(g + 1) * grp] = gdo


def digest(*tensors) -> str:
    """sha256 over the raw bytes of the tensors, in order."""
    import hashlib
    h = hashlib.sha256()
    for t in tensors:
        t = t.detach().contiguous().cpu()
        if t.dtype == torch.bfloat16:
            t = t.view(torch.int16)
        h.update(t.numpy().tobytes())
    return h.hexdigest()
