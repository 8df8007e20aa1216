"""The allocation-free ring backward (cpattn_ring_bwd_noalloc).

Callers that cannot allocate device memory (a memory manager owns the whole
device, or cudaMalloc would stall a latency-critical loop) use this entry
point: its scratch is a fixed 64 MiB array inside the library.  These checks
call it through the C ABI and require the same bits as cpattn_ring_bwd
(caller-owned workspace) on the same inputs, twice in a row, so that contents
the first call leaves in the shared scratch cannot leak into the second, and
compare it with the fp64 oracle once.  This file is
collected last on purpose: a run that stops at its first failure has already
run every other test.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import context_causal_attention_zigzag_gb300 as cpa
from context_causal_attention_zigzag_gb300 import _binding, inputs

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.mark.parametrize("case", [
    # B, H, Hkv, S, D, cp, layout, causal, dtype, tol (against the oracle)
    (1, 4, 2, 1024, 128, 4, cpa.ZIGZAG, True, torch.bfloat16, 2e-2),
    (1, 2, 2, 256, 64, 2, cpa.ZIGZAG, True, torch.float32, 1e-4),
    (2, 2, 1, 512, 128, 2, cpa.CONTIGUOUS, False, torch.bfloat16, 2e-2),
    (1, 4, 2, 1024, 128, 2, cpa.ZIGZAG, True, torch.float32, 1e-4),
])
def test_noalloc_backward_matches_workspace_backward(case):
    B, H, Hkv, S, D, cp, layout, causal, dtype, tol = case
    w = inputs.Workload("noalloc", B, H, Hkv, S, D, cp, layout, causal, dtype, seed=8100 + S)
    qh, kh, vh, doh = inputs.generate(w, with_dout=True)
    q, k, v, do = (x.to(DEV) for x in (qh, kh, vh, doh))
    qs, ks, vs, dos = (cpa.zigzag_permute(x, cp, layout) for x in (q, k, v, do))
    o, lse = cpa.ring_fwd(qs, ks, vs, cp, layout, causal)
    ref = cpa.ring_bwd(qs, ks, vs, o, dos, lse, cp, layout, causal)
    # Both entry points run the same deterministic kernels on the same
    # inputs, so their gradients must agree bit for bit; anything an earlier
    # call left in the shared scratch would show up as a difference.
    for _ in range(2):
        got = cpa.ring_bwd_noalloc(qs, ks, vs, o, dos, lse, cp, layout, causal)
        torch.cuda.synchronize()
        for a, b in zip(got, ref):
            assert torch.equal(a, b)
    # And against the oracle (float32 gradients of bf16 inputs, as the other
    # parity tests compare them).
    g = cpa.ring_bwd_noalloc(qs, ks, vs, o, dos, lse, cp, layout, causal,
                             grad_dtype=torch.float32)
    f = inputs.to_f32_numpy
    rq, rk, rv = oracle.attn_bwd(f(qh), f(kh), f(vh), f(doh), causal=causal)
    for got, want in zip(g, (rq, rk, rv)):
        nat = cpa.zigzag_unpermute(got, cp, layout)
        err = float(np.max(np.abs(nat.double().cpu().numpy() - want)))
        assert err <= tol, err
    assert cpa.device_status() == 0


def test_noalloc_rejects_problems_beyond_its_scratch():
    lib = cpa.lib()
    fake = ctypes.c_void_p(0x1000)
    null = ctypes.c_void_p(0)
    # B=1, H=32, S=8192, D=128: a 272 MiB workspace (two float32 regions of
    # the query tensor's size, two of the kv tensors' size, Delta) > 64 MiB.
    rc = lib.cpattn_ring_bwd_noalloc(*([fake] * 9), 1, 32, 32, 8192, 128, 4, 1, 1, 1, 0.0, null)
    assert rc == _binding.ERR_WORKSPACE
    # A smaller problem of the same kind fits.
    need = lib.cpattn_ring_bwd_workspace_bytes(1, 32, 8, 1024, 128, 1)
    assert need <= 64 << 20
