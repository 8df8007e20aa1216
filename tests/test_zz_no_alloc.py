"""The allocation-free ring backward (cpattn_ring_bwd_noalloc).

Callers that cannot allocate device memory (a memory manager owns the whole
device, or cudaMalloc would stall a latency-critical loop) use this entry
point: its scratch is a fixed 64 MiB array inside the library.  These checks
call it through the C ABI and compare it with cpattn_ring_bwd (caller-owned
workspace) on the same inputs, twice in a row, so that contents the first
call leaves in the shared scratch cannot leak into the second.  This file is
collected last on purpose: a run that stops at its first failure has already
run every other test.
"""
import ctypes

import pytest
import torch

import context_causal_attention_zigzag_gb300 as cpa
from context_causal_attention_zigzag_gb300 import _binding, inputs

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.mark.parametrize("case", [
    # B, H, Hkv, S, D, cp, layout, causal, dtype, tol
    (1, 4, 2, 1024, 128, 4, cpa.ZIGZAG, True, torch.bfloat16, 2e-2),
    (1, 2, 2, 256, 64, 2, cpa.ZIGZAG, True, torch.float32, 1e-4),
    (2, 2, 1, 512, 128, 2, cpa.CONTIGUOUS, False, torch.bfloat16, 2e-2),
    (1, 4, 2, 1024, 128, 2, cpa.ZIGZAG, True, torch.float32, 1e-4),
])
def test_noalloc_backward_matches_workspace_backward(case):
    B, H, Hkv, S, D, cp, layout, causal, dtype, tol = case
    w = inputs.Workload("noalloc", B, H, Hkv, S, D, cp, layout, causal, dtype, seed=8100 + S)
    q, k, v, do = (x.to(DEV) for x in inputs.generate(w, with_dout=True))
    qs, ks, vs, dos = (cpa.zigzag_permute(x, cp, layout) for x in (q, k, v, do))
    o, lse = cpa.ring_fwd(qs, ks, vs, cp, layout, causal)
    ref = cpa.ring_bwd(qs, ks, vs, o, dos, lse, cp, layout, causal)
    for _ in range(2):
        got = cpa.ring_bwd_noalloc(qs, ks, vs, o, dos, lse, cp, layout, causal)
        torch.cuda.synchronize()
        for a, b in zip(got, ref):
            assert torch.isfinite(a.float()).all()
            assert (a.float() - b.float()).abs().max().item() <= tol
    assert cpa.device_status() == 0


def test_noalloc_rejects_problems_beyond_its_scratch():
    lib = cpa.lib()
    fake = ctypes.c_void_p(0x1000)
    null = ctypes.c_void_p(0)
    # B=1, H=32, S=8192, D=128: a 128 MiB float32 dQ accumulator > 64 MiB.
    rc = lib.cpattn_ring_bwd_noalloc(*([fake] * 9), 1, 32, 32, 8192, 128, 4, 1, 1, 1, 0.0, null)
    assert rc == _binding.ERR_WORKSPACE
    # A smaller problem of the same kind fits.
    need = lib.cpattn_ring_bwd_workspace_bytes(1, 32, 8, 1024, 128, 1)
    assert need <= 64 << 20
