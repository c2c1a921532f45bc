"""GPU parity of NVFP4 quantization and scale assembly: nibbles, FP8 scales in
the tile layout and global scales must equal the oracle's bit for bit."""
import numpy as np
import pytest

from oracle import nvfp4_oracle as O
from nvfp4_mixture_experts_expert_gb300 import workloads as W
from helpers import bf16_dev, dev, host, oracle_packed_rows

pytestmark = pytest.mark.gpu


def api():
    from nvfp4_mixture_experts_expert_gb300 import api as A
    return A


def special_rows(R, K, seed):
    """Rows N(0,1) with a per-row lognormal gain, 5% zero blocks, 5% blocks below the
    underflow threshold after scaling, 2% channels x20."""
    wl = W.moe_workload(R, K, 128, 2, 1, seed, zero_block_frac=0.05, tiny_block_frac=0.05,
                        outlier_frac=0.02)
    x = W.bf16_bits_to_f32(wl.hidden) * np.exp(np.random.default_rng(seed).standard_normal((R, 1))).astype(np.float32)
    return W.f32_to_bf16_bits(x)


@pytest.mark.parametrize("R,K", [(1, 64), (130, 256), (300, 512), (257, 3584)])
def test_quantize_with_computed_global_scale(R, K):
    bits = special_rows(R, K, R + K)
    x = W.bf16_bits_to_f32(bits)
    gs = O.global_scale(np.abs(x).max())
    Rp = (R + 127) // 128 * 128
    packed, swz, _, _ = oracle_packed_rows(x, gs, Rp)
    fp4, sf, gs_dev = api().quantize(bf16_dev(bits))
    assert host(gs_dev)[0] == gs
    np.testing.assert_array_equal(host(fp4), packed)
    np.testing.assert_array_equal(host(sf), swz)


@pytest.mark.parametrize("gs", [1.0, 1234.5, 3e-3])
def test_quantize_with_given_global_scale(gs):
    R, K = 200, 320
    bits = special_rows(R, K, 7)
    x = W.bf16_bits_to_f32(bits)
    packed, swz, _, _ = oracle_packed_rows(x, np.float32(gs), 256)
    fp4, sf, gs_out = api().quantize(bf16_dev(bits), gs=dev(np.float32([gs])))
    np.testing.assert_array_equal(host(fp4), packed)
    np.testing.assert_array_equal(host(sf), swz)
    assert host(gs_out)[0] == np.float32(gs)


def test_quantize_all_zero_tensor_gives_unit_scale():
    bits = np.zeros((128, 64), np.uint16)
    fp4, sf, gs = api().quantize(bf16_dev(bits))
    assert host(gs)[0] == 1.0
    assert not host(fp4).any() and not host(sf).any()


def test_quantize_strided_groups_like_grouped_linear():
    """(T, G, D) input read as G groups of T rows (group stride D, row stride G*D)."""
    wl = W.grouped_linear(seed=3, T=200, G=3, D=256, R=256)
    x = W.bf16_bits_to_f32(wl.x)
    Rp = 256
    fp4, sf, gs = api().quantize_groups(bf16_dev(wl.x), wl.T, wl.D, wl.G * wl.D, wl.D, wl.G, rows_padded=Rp)
    fp4, sf, gs = host(fp4), host(sf), host(gs)
    for g in range(wl.G):
        xg = x[:, g, :]
        gsg = O.global_scale(np.abs(xg).max())
        assert gs[g] == gsg
        packed, swz, _, _ = oracle_packed_rows(xg, gsg, Rp)
        np.testing.assert_array_equal(fp4[g * Rp:(g + 1) * Rp], packed)
        n = Rp * wl.D // 16
        np.testing.assert_array_equal(sf[g * n:(g + 1) * n], swz)


def test_expert_weight_quantization():
    rng = np.random.default_rng(5)
    w = W.f32_to_bf16_bits(rng.standard_normal((3, 256, 192)).astype(np.float32) * np.float32(0.02))
    fp4, sf, gs = api().quantize_expert_weights(bf16_dev(w))
    nibs, scs, gss = O.quantize_expert_weights(W.bf16_bits_to_f32(w))
    np.testing.assert_array_equal(host(gs), gss)
    for e in range(3):
        np.testing.assert_array_equal(host(fp4)[e], O.pack_nibbles(nibs[e]))
        np.testing.assert_array_equal(host(sf)[e], O.assemble_scales(scs[e], np.array([0, 256]), np.array([0, 256])))


def test_assemble_scales_matches_oracle():
    import torch
    from nvfp4_mixture_experts_expert_gb300 import binding as B
    rng = np.random.default_rng(9)
    counts = [5, 0, 130, 128, 1]
    offsets = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    padded = np.concatenate([[0], np.cumsum([(c + 127) // 128 * 128 for c in counts])]).astype(np.int32)
    cap = int(padded[-1]) + 128
    for C in (6, 8, 256):
        lin = rng.integers(1, 0x7E, (offsets[-1], C), dtype=np.uint8)
        ref = O.assemble_scales(lin, offsets, padded)
        C4 = (C + 3) // 4 * 4
        out = torch.full((cap * C4,), 0xAB, dtype=torch.uint8, device="cuda")
        B.nvfp4_assemble_scales(dev(lin), C, dev(offsets), dev(padded), len(counts), cap, out)
        got = host(out)
        np.testing.assert_array_equal(got[:ref.size], ref)
        assert not got[ref.size:].any()  # capacity rows beyond the last slot are zero


def test_quantize_ties_saturation_and_thresholds():
    """Hand-picked blocks: exact E2M1 midpoints (ties to even), saturation, the
    underflow threshold on both sides, negative values rounding to zero."""
    rows = [
        [6, 0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5, -0.25, -0.75, -1.25, -1.75, -2.5, -3.5, -5, -6],
        [7, 6.5, -7, 0.1, -0.1, 3, 4, 2, 1, 0.5, 0, -0.0, 5.5, 4.5, 2.25, 0.125],
        [0.01171875, 0.001953125] + [0] * 14,
        [0.0117187, 0.005] + [0] * 14,
        [448 * 6 * 1.5] + [1] * 15,
    ]
    x = np.zeros((len(rows), 64), np.float32)  # K must be a multiple of 64: one hand block per row
    x[:, :16] = np.float32(rows)
    bits = W.f32_to_bf16_bits(x)
    xb = W.bf16_bits_to_f32(bits)
    packed, swz, _, _ = oracle_packed_rows(xb, np.float32(1.0), 128)
    fp4, sf, _ = api().quantize(bf16_dev(bits), gs=dev(np.float32([1.0])))
    np.testing.assert_array_equal(host(fp4), packed)
    np.testing.assert_array_equal(host(sf), swz)


@pytest.mark.parametrize("rows,K,ld_x,groups", [(2048, 3584, 3584, 1), (301, 192, 256, 1), (77, 320, 3 * 320, 3),
                                               (5, 64, 64, 300)])
def test_global_scale_sees_every_element_and_no_padding(rows, K, ld_x, groups):
    """gs = 2688 / amax must see each element of each group exactly where the
    strides put it: a single peak at the first, the last and random places of
    one group (a larger value sits in every padding column, which must not
    count) moves that group's scale and no other."""
    import torch
    rng = np.random.default_rng(rows + K + groups)
    gstride = K if ld_x == groups * K else rows * ld_x  # interleaved (T, G, D) or stacked groups
    n = gstride * (groups - 1) + (rows - 1) * ld_x + K if gstride == K else groups * rows * ld_x
    base = np.zeros(n, np.float32)
    valid = np.zeros(n, bool)
    for g in range(groups):
        for r in range(rows):
            at = g * gstride + r * ld_x
            base[at:at + K] = rng.uniform(-1, 1, K)
            valid[at:at + K] = True
    base[~valid] = 1e6
    places = [(0, 0, 0), (groups - 1, rows - 1, K - 1)] + [
        (int(rng.integers(groups)), int(rng.integers(rows)), int(rng.integers(K))) for _ in range(4)]
    for g0, r0, c0 in places:
        x = base.copy()
        x[g0 * gstride + r0 * ld_x + c0] = -37.0
        bits = W.f32_to_bf16_bits(x)
        _, _, gs = api().quantize_groups(bf16_dev(bits), rows, K, ld_x, gstride, groups)
        gs = host(gs)
        xb = W.bf16_bits_to_f32(bits)
        for g in range(groups):
            xs = np.concatenate([xb[g * gstride + r * ld_x:g * gstride + r * ld_x + K] for r in range(rows)])
            assert gs[g] == O.global_scale(np.abs(xs).max()), (g0, r0, c0, g)
        assert gs[g0] == O.global_scale(np.float32(37.0))
    torch.cuda.synchronize()


def test_many_small_groups_bytes_and_scales():
    """300 groups of 5 rows (the amax grid gives each group very few blocks)."""
    G, T, D = 300, 5, 64
    rng = np.random.default_rng(11)
    x = (rng.standard_normal((G, T, D)) * np.exp(rng.standard_normal((G, 1, 1)) * 3)).astype(np.float32)
    bits = W.f32_to_bf16_bits(x)
    xb = W.bf16_bits_to_f32(bits)
    fp4, sf, gs = api().quantize_groups(bf16_dev(bits), T, D, D, T * D, G, rows_padded=128)
    fp4, sf, gs = host(fp4), host(sf), host(gs)
    for g in range(G):
        gsg = O.global_scale(np.abs(xb[g]).max())
        assert gs[g] == gsg
        packed, swz, _, _ = oracle_packed_rows(xb[g], gsg, 128)
        np.testing.assert_array_equal(fp4[g * 128:(g + 1) * 128], packed)
        np.testing.assert_array_equal(sf[g * 128 * D // 16:(g + 1) * 128 * D // 16], swz)


def test_scales_only_when_nothing_to_quantize():
    """rows = rows_padded = 0: no bytes to write, every group's gs is 1."""
    import torch
    from nvfp4_mixture_experts_expert_gb300 import binding as B
    G = 5
    gs_out = torch.full((G,), -1.0, dtype=torch.float32, device="cuda")
    wsb = B.nvfp4_quantize_workspace_size(G)
    ws = torch.empty(wsb, dtype=torch.uint8, device="cuda")
    B.nvfp4_quantize(None, 0, 128, 128, 0, G, None, gs_out, ws, wsb, None, None, 0)
    assert (host(gs_out) == 1.0).all()
