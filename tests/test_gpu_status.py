"""The device-side failure path, exercised without a GPU fault: a bounded
wait that nothing completes gives up, raises the device error word, the next
status read reports the timeout and clears it, and the context keeps working
(a forward after it still matches the oracle)."""
import pytest
import torch

import oracle
import context_causal_attention_zigzag_gb300 as cpa
from context_causal_attention_zigzag_gb300 import _binding, inputs

pytestmark = pytest.mark.gpu


def test_bounded_wait_gives_up_and_context_stays_usable():
    assert cpa.device_status() == _binding.OK
    cpa.wait_probe(50_000_000)  # 50 ms
    assert cpa.device_status() == _binding.ERR_DEVICE_TIMEOUT
    assert cpa.device_status() == _binding.OK  # read and cleared
    w = inputs.Workload("after", 1, 2, 1, 1024, 128, 2, cpa.ZIGZAG, True, torch.bfloat16,
                        seed=99)
    q, k, v, _ = inputs.generate(w, with_dout=False)
    out, lse = cpa.attention(q.cuda(), k.cuda(), v.cuda(), w.cp, w.layout, w.causal)
    ro, rl = oracle.attn_fwd(inputs.to_f32_numpy(q), inputs.to_f32_numpy(k),
                             inputs.to_f32_numpy(v))
    assert (out.double().cpu().numpy() - ro).__abs__().max() <= 2e-2
    assert (lse.double().cpu().numpy() - rl).__abs__().max() <= 1e-3
    assert cpa.device_status() == _binding.OK


def test_wait_probe_rejects_limits_out_of_range():
    for bad in (0, -1, 3_000_000_000):
        with pytest.raises(cpa.CpattnError):
            cpa.wait_probe(bad)
    assert cpa.device_status() == _binding.OK
