"""GPU parity of the shared-expert NVFP4 SwiGLU FFN (one group, no routing)
against the oracle, and bit-identity with the routed layer's one-expert,
top-1 case (every routing weight is then exactly 1)."""
import numpy as np
import pytest

from oracle import nvfp4_oracle as O
from nvfp4_mixture_experts_expert_gb300 import workloads as W
from helpers import OracleMoE, bf16_dev, bf16_host, cosine, dev, host, rel_frob

pytestmark = pytest.mark.gpu


def _layer(T, H=512, I=256, seed=81):
    wl = W.moe_workload(T, H, I, 1, 1, seed, zero_block_frac=0.03, tiny_block_frac=0.03)
    return wl, OracleMoE(wl)


@pytest.mark.parametrize("T", [300, 128, 1])
def test_shared_expert_matches_oracle(T):
    import torch
    from nvfp4_mixture_experts_expert_gb300 import api
    wl, orc = _layer(T)
    w = api.quantize_moe_weights(bf16_dev(wl.w13), bf16_dev(wl.w2))
    se = api.SharedExpertForward(wl.T, wl.H, wl.I)
    se.workspace[:4].fill_(0xFF)  # the call's first kernel clears the workspace status word
    buf = torch.full((wl.T + 3, wl.H), float("nan"), dtype=torch.bfloat16, device="cuda")
    se(bf16_dev(wl.hidden), w, dev(orc.a1_gs), dev(orc.a2_gs), wl.gate_limit, wl.up_limit, out=buf[:wl.T])
    torch.cuda.synchronize()
    assert se.status() == 0
    got = bf16_host(buf)
    assert np.all(np.isnan(got[wl.T:]))  # only the T rows of out are written
    ref = O.shared_expert_forward(W.bf16_bits_to_f32(wl.hidden), orc.w13q, orc.w2q, orc.a1_gs[0], orc.a2_gs[0],
                                  wl.gate_limit, wl.up_limit)
    got = got[:wl.T]
    assert np.all(np.isfinite(got))
    rf, cs = rel_frob(got, ref), cosine(got, ref)
    assert rf <= 2e-2 and cs >= 0.999, (rf, cs)


def test_shared_expert_equals_one_expert_top1_moe_bit_for_bit():
    import torch
    from nvfp4_mixture_experts_expert_gb300 import api
    wl, orc = _layer(257, seed=83)
    w = api.quantize_moe_weights(bf16_dev(wl.w13), bf16_dev(wl.w2))
    a1, a2 = dev(orc.a1_gs), dev(orc.a2_gs)
    moe = api.MoEForward(wl.T, wl.H, wl.I, 1, 1)
    ref = moe(bf16_dev(wl.hidden), dev(wl.logits), w, a1, a2, wl.gate_limit, wl.up_limit)
    se = api.SharedExpertForward(wl.T, wl.H, wl.I)
    out = se(bf16_dev(wl.hidden), w, a1, a2, wl.gate_limit, wl.up_limit)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(host(out.view(torch.int16)), host(ref.view(torch.int16)))


def test_shared_expert_zero_tokens_is_a_no_op():
    import torch
    from nvfp4_mixture_experts_expert_gb300 import binding as B
    assert B.nvfp4_shared_expert_workspace_size(0, 256, 128) > 0
    B.nvfp4_shared_expert_forward(None, 0, 256, 128, None, None, None, None, None, None, None, None, 10.0, 10.0,
                                  None, 0, None)
    torch.cuda.synchronize()
