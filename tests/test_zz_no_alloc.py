"""nvfp4_quantize_no_alloc: the quantizer for callers that cannot allocate
device memory (hosts that own the whole memory pool, or plugin interfaces
with no workspace argument).  Its reduction scratch lives in a fixed array
inside the library, so each call must still reproduce, byte for byte, what
nvfp4_quantize computes with a caller-provided workspace -- and a second call
must not be affected by what the first one left in that shared array.

This file is collected last on purpose: if it fails, a run that stops at the
first failure has already run every other test."""
import numpy as np
import pytest

from nvfp4_mixture_experts_expert_gb300 import workloads as W
from helpers import bf16_dev, host

pytestmark = pytest.mark.gpu


def quantize_both_ways(bits, rows, K, ld_x, group_stride_x, groups, rows_padded):
    import torch
    from nvfp4_mixture_experts_expert_gb300 import binding as B
    x = bf16_dev(bits)

    def outputs():
        return (torch.full((groups * rows_padded, K // 2), 0xAB, dtype=torch.uint8, device="cuda"),
                torch.full((groups * rows_padded * K // 16,), 0xCD, dtype=torch.uint8, device="cuda"),
                torch.full((groups,), float("nan"), dtype=torch.float32, device="cuda"))

    fp4_ref, sf_ref, gs_ref = outputs()
    wsb = B.nvfp4_quantize_workspace_size(groups)
    ws = torch.empty(wsb, dtype=torch.uint8, device="cuda")
    B.nvfp4_quantize(x, rows, K, ld_x, group_stride_x, groups, None, gs_ref, ws, wsb, fp4_ref, sf_ref, rows_padded)
    fp4, sf, gs = outputs()
    B.nvfp4_quantize_no_alloc(x, rows, K, ld_x, group_stride_x, groups, gs, fp4, sf, rows_padded)
    torch.cuda.synchronize()
    return (host(fp4), host(sf), host(gs)), (host(fp4_ref), host(sf_ref), host(gs_ref))


def test_two_calls_in_a_row_match_the_workspace_entry_point():
    # call 1: three strided groups of a (T, G, D) tensor
    wl = W.grouped_linear(seed=11, T=300, G=3, D=256, R=256)
    got, ref = quantize_both_ways(wl.x, wl.T, wl.D, wl.G * wl.D, wl.D, wl.G, 384)
    for a, b in zip(got, ref):
        np.testing.assert_array_equal(a, b)
    assert np.all(np.isfinite(got[2]))
    # call 2: more groups, other sizes and other data (a larger amax than call 1)
    rng = np.random.default_rng(12)
    x = W.f32_to_bf16_bits(rng.standard_normal((5, 200, 512)).astype(np.float32) * np.float32(40.0))
    got2, ref2 = quantize_both_ways(x, 200, 512, 512, 200 * 512, 5, 256)
    for a, b in zip(got2, ref2):
        np.testing.assert_array_equal(a, b)
    assert not np.array_equal(got2[2][:3], got[2])


def test_rejects_more_groups_than_the_fixed_scratch_holds():
    from nvfp4_mixture_experts_expert_gb300 import binding as B
    with pytest.raises(B.Nvfp4Error) as ei:
        B.nvfp4_quantize_no_alloc(16, 1, 64, 64, 64, 65, 16, 16, 16, 128)
    assert ei.value.status == B.NVFP4_ERR_UNSUPPORTED
    assert "64" in B.nvfp4_last_error()
