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


def quantize_both_ways(bits, rows, K, ld_x, group_stride_x, groups, rows_padded, x_offset_elems=0):
    import torch
    from nvfp4_mixture_experts_expert_gb300 import binding as B
    x = bf16_dev(bits)
    if x_offset_elems:  # a view that starts x_offset_elems into a copy: only 16-byte aligned
        buf = torch.zeros(x.numel() + x_offset_elems, dtype=torch.bfloat16, device="cuda")
        buf[x_offset_elems:] = x.reshape(-1)
        x = buf[x_offset_elems:]
        assert x.data_ptr() % 32 == 16

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


def test_no_rows_gives_unit_scales_and_zero_padding():
    """rows == 0: every group's amax reduction reads nothing (all partials 0),
    so gs must come out as 1 and every padded row as zero bytes -- exactly what
    the workspace entry point writes."""
    bits = np.zeros((2, 1, 128), np.uint16)
    got, ref = quantize_both_ways(bits, 0, 128, 128, 128, 2, 128)
    for a, b in zip(got, ref):
        np.testing.assert_array_equal(a, b)
    np.testing.assert_array_equal(got[2], np.ones(2, np.float32))
    assert not got[0].any() and not got[1].any()


def test_only_16_byte_aligned_input():
    """x starting 16 bytes past a 32-byte boundary takes the quantize kernel's
    two-load path; results still equal the workspace entry point's."""
    rng = np.random.default_rng(13)
    x = W.f32_to_bf16_bits(rng.standard_normal((2, 130, 256)).astype(np.float32))
    got, ref = quantize_both_ways(x, 130, 256, 256, 130 * 256, 2, 256, x_offset_elems=8)
    for a, b in zip(got, ref):
        np.testing.assert_array_equal(a, b)


def test_rejects_more_groups_than_the_fixed_scratch_holds():
    from nvfp4_mixture_experts_expert_gb300 import binding as B
    with pytest.raises(B.Nvfp4Error) as ei:
        B.nvfp4_quantize_no_alloc(16, 1, 64, 64, 64, 65, 16, 16, 16, 128)
    assert ei.value.status == B.NVFP4_ERR_UNSUPPORTED
    assert "64" in B.nvfp4_last_error()
