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

Packed documents: the pages test document masks but give no length
distribution.  ``packed_doc_offsets`` draws document lengths from an
exponential distribution with a stated mean (many short documents, a few
long ones), from its own generator seeded with ``doc_seed``; the last
document is cut at S.
"""
import math
from dataclasses import dataclass, field, replace
from typing import Optional, Tuple

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
