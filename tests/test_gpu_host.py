"""The host-buffer entry point (cpattn_attention_host): natural-order host
tensors in and out, with the permutation done by the chunked copies and the
heads in pipelined parts (uploads and downloads on two side streams,
overlapping the neighbouring parts' kernels).  It runs the same
kernels as the device path, so its results must equal, bit for bit, the
device path's (cpattn_zigzag_permute -> ring forward -> ring backward ->
cpattn_zigzag_unpermute); the device path itself is checked against the
oracle in the other test files.
"""
import pytest
import torch

import context_causal_attention_zigzag_gb300 as cpa
from context_causal_attention_zigzag_gb300 import inputs

pytestmark = pytest.mark.gpu

CASES = [
    # B, H, Hkv, S, D, cp, layout, causal, dtype, grad_dtype
    (1, 4, 2, 2048, 128, 4, cpa.ZIGZAG, True, torch.bfloat16, torch.float32),
    (2, 4, 1, 1536, 128, 3, cpa.ZIGZAG, True, torch.bfloat16, None),
    (1, 2, 2, 2048, 128, 2, cpa.CONTIGUOUS, False, torch.bfloat16, torch.float32),
    (2, 2, 2, 256, 64, 2, cpa.ZIGZAG, True, torch.float32, None),
    (1, 8, 4, 2048, 128, 4, cpa.ZIGZAG, True, torch.bfloat16, torch.float32),
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "B{}H{}K{}S{}D{}cp{}L{}c{}".format(*c[:8]))
@pytest.mark.parametrize("backward", [True, False])
@pytest.mark.parametrize("split", ["one", "most"])
def test_host_path_equals_device_path(case, backward, split):
    # "most": as many head parts as the kv heads allow (each part one kv
    # head), so the pipelined per-part copies and launches are exercised.
    B, H, Hkv, S, D, cp, layout, causal, dtype, gdt = case
    parts = 1 if split == "one" else Hkv
    w = inputs.Workload("host", B, H, Hkv, S, D, cp, layout, causal, dtype, seed=9000 + S)
    q, k, v, do = inputs.generate(w, with_dout=True, pin=True)
    res = cpa.attention_host(q, k, v, do if backward else None, cp, layout, causal,
                             grad_dtype=gdt, parts=parts)
    torch.cuda.synchronize()
    dev = [x.cuda() for x in (q, k, v, do)]
    if backward:
        ref = cpa.attention_fwd_bwd(*dev, cp, layout, causal, grad_dtype=gdt)
    else:
        ref = cpa.attention(*dev[:3], cp, layout, causal)
    assert len(res) == len(ref)
    for name, a, b in zip(("out", "lse", "dq", "dk", "dv"), res, ref):
        assert not a.is_cuda and a.dtype == b.dtype and a.shape == b.shape, name
        assert torch.equal(a, b.cpu()), name
    assert cpa.device_status() == 0


def test_host_path_repeated_calls_reuse_workspace():
    # Two calls in a row with one workspace and the same output buffers: the
    # second call's results equal the first's (nothing left over matters).
    B, H, Hkv, S, D, cp = 1, 4, 2, 2048, 128, 4
    w = inputs.Workload("host2", B, H, Hkv, S, D, cp, cpa.ZIGZAG, True, torch.bfloat16, seed=91)
    q, k, v, do = inputs.generate(w, with_dout=True, pin=True)
    need = cpa.attention_host_workspace_bytes(B, H, Hkv, S, D, cp, cpa.ZIGZAG,
                                              cpa.BF16 | cpa.GRAD_F32, True)
    ws = torch.empty(need, device="cuda", dtype=torch.uint8)
    outs = cpa.attention_host(q, k, v, do, cp, grad_dtype=torch.float32, workspace=ws)
    torch.cuda.synchronize()
    first = [x.clone() for x in outs]
    outs = cpa.attention_host(q, k, v, do, cp, grad_dtype=torch.float32, workspace=ws)
    torch.cuda.synchronize()
    for a, b in zip(outs, first):
        assert torch.equal(a, b)
    assert cpa.device_status() == 0


def test_host_parts_choice_and_rejects():
    # The automatic choice: 8 parts for the S=131072 problem (8 kv heads),
    # one for small tensors; a parts value that does not divide Hkv is an
    # argument error.
    assert cpa.attention_host_parts(1, 32, 8, 131072, 128) == 8
    assert cpa.attention_host_parts(1, 4, 2, 2048, 128) == 1
    q = torch.zeros((1, 512, 4, 64), dtype=torch.bfloat16).pin_memory()
    k = torch.zeros((1, 512, 2, 64), dtype=torch.bfloat16).pin_memory()
    for bad in (3, 9, -1):
        with pytest.raises(cpa.CpattnError):
            cpa.attention_host(q, k, k, None, 2, parts=bad)
    assert cpa.device_status() == 0


def test_host_path_full_size_equals_device_path():
    # The S=131072 step that the end-to-end bench line times, through the
    # host path with the automatic number of head parts (8): bit for bit the
    # device path's results.
    w = inputs.WORKLOADS["c5_bf16_s131072_fwdbwd"]
    q, k, v, do = inputs.generate(w, pin=True)
    B, S, H, D = q.shape
    assert cpa.attention_host_parts(B, H, k.shape[2], S, D) == 8
    res = cpa.attention_host(q, k, v, do, w.cp, w.layout, w.causal, grad_dtype=torch.float32)
    torch.cuda.synchronize()
    ref = cpa.attention_fwd_bwd(*(x.cuda() for x in (q, k, v, do)), w.cp, w.layout, w.causal,
                                grad_dtype=torch.float32)
    for name, a, b in zip(("out", "lse", "dq", "dk", "dv"), res, ref):
        assert torch.equal(a, b.cpu()), name
    assert cpa.device_status() == 0


DOC_CASES = [
    # B, H, Hkv, S (real), D, cp, layout, causal, dtype, grad_dtype, cu_seqlens
    (1, 4, 2, 1000, 128, 2, cpa.ZIGZAG, True, torch.bfloat16, torch.float32, [0, 300, 1000]),
    (2, 4, 2, 777, 128, 3, cpa.CONTIGUOUS, True, torch.bfloat16, None, None),
    (1, 2, 2, 333, 64, 3, cpa.ZIGZAG, False, torch.float32, None, [0, 1, 200, 333]),
]


@pytest.mark.parametrize("case", DOC_CASES, ids=lambda c: "B{}H{}K{}S{}D{}cp{}L{}c{}".format(*c[:8]))
@pytest.mark.parametrize("backward", [True, False])
@pytest.mark.parametrize("split", ["one", "most"])
def test_host_docs_path_equals_device_docs_path(case, backward, split):
    # Any length and packed documents from host buffers: the padded device
    # sequence, the document rule, the real tokens back; the same results as
    # the device path (attention_docs / attention_docs_fwd_bwd), bit for bit.
    B, H, Hkv, S, D, cp, layout, causal, dtype, gdt, cu = case
    parts = 1 if split == "one" else Hkv
    w = inputs.Workload("hostdocs", B, H, Hkv, S, D, cp, layout, causal, dtype, seed=9500 + S)
    q, k, v, do = inputs.generate(w, with_dout=True, pin=True)
    res = cpa.attention_host_docs(q, k, v, do if backward else None, cp, cu, layout, causal,
                                  grad_dtype=gdt, parts=parts)
    torch.cuda.synchronize()
    dev = [x.cuda() for x in (q, k, v, do)]
    if backward:
        ref = cpa.attention_docs_fwd_bwd(*dev, cp, cu, layout, causal, grad_dtype=gdt)
    else:
        ref = cpa.attention_docs(*dev[:3], cp, cu, layout, causal)
    assert len(res) == len(ref)
    for name, a, b in zip(("out", "lse", "dq", "dk", "dv"), res, ref):
        assert not a.is_cuda and a.dtype == b.dtype and a.shape == b.shape, name
        assert torch.equal(a, b.cpu()), name
    assert cpa.device_status() == 0
