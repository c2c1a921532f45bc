"""Pins of the oracle's FP8 L1 output (reading R20): OCP E4M3 values in
blocks of 16 features with a power-of-two scale 2^k per block, k the least
integer with max|h| <= 448 * 2^k.  Checked against exact float64 arithmetic,
hand-worked codes and the E4M3 error bound, and the forward against the bf16
L1 output it approximates."""
import numpy as np
import pytest

from oracle import nvfp4_oracle as O
from nvfp4_mixture_experts_expert_gb300 import workloads as W


def test_block_exponent_is_the_least_power_of_two_covering_the_block():
    rng = np.random.default_rng(1)
    edges = np.ldexp(448.0, np.arange(-60, 60))
    vals = np.concatenate([edges, np.nextafter(edges, 0), np.nextafter(edges, np.inf),
                           np.exp(rng.uniform(-80, 80, 4000))])
    k = O.fp8_block_exponent(vals)
    assert np.all(vals <= np.ldexp(448.0, k))
    assert np.all(vals > np.ldexp(448.0, k - 1))  # k - 1 would not cover it
    assert O.fp8_block_exponent(0.0) == 0
    assert O.fp8_block_exponent(1e-300) == -126 and O.fp8_block_exponent(1e300) == 126  # clamped


def test_hand_worked_codes():
    # 300 <= 448: k = 0; 300 = 1.171875 * 2^8 -> mantissa 1.375/8 rounds to 1/8: 288, code (15 << 3) | 1
    # -0.1 = -1.6 * 2^-4 -> 1.625 * 2^-4, code 0x80 | (3 << 3) | 5; 2^-10 -> subnormal step 2^-9 rounds to 0 (tie to even)
    h = np.zeros((1, 16), np.float32)
    h[0, :4] = [300.0, -0.1, 2.0 ** -10, 3 * 2.0 ** -10]
    codes, k = O.fp8_block_encode(h)
    assert k.tolist() == [[0]]
    assert codes[0, :4].tolist() == [0x79, 0x9D, 0x00, 0x02]  # 3 * 2^-10 = 1.5 steps -> 2 steps (even)
    np.testing.assert_array_equal(O.fp8_block_decode(codes, k)[0, :4],
                                  np.float32([288.0, -0.1015625, 0.0, 2.0 ** -8]))
    # the same block times 2^10: 448 * 2^9 < 307200 <= 448 * 2^10, so k = 10 and the codes repeat
    codes2, k2 = O.fp8_block_encode(h * np.float32(1024.0))
    assert k2.tolist() == [[10]]
    np.testing.assert_array_equal(codes2, codes)


def test_round_trip_error_bound_and_signs():
    rng = np.random.default_rng(2)
    h = W.bf16_bits_to_f32(W.f32_to_bf16_bits(
        (rng.standard_normal((64, 256)) * np.exp(rng.uniform(-20, 20, (64, 1)))).astype(np.float32)))
    h[3, 16:32] = 0.0
    h[5, 0] = -0.0
    codes, k = O.fp8_block_encode(h)
    back = O.fp8_block_decode(codes, k).astype(np.float64)
    scale = np.repeat(np.exp2(k.astype(np.float64)), 16, axis=1)
    blk = h.astype(np.float64).reshape(64, 16, 16)
    scaled_max = np.max(np.abs(blk), axis=2) / np.exp2(k)
    nz = scaled_max > 0
    assert np.all((scaled_max[nz] > 224) & (scaled_max[nz] <= 448))  # the block max lands in the top binade
    err = np.abs(back - h)
    normal = np.abs(h) >= scale * 2.0 ** -6
    assert np.all(err[normal] <= np.abs(h[normal]) * 2.0 ** -4)   # half a step of 3 mantissa bits
    assert np.all(err[~normal] <= scale[~normal] * 2.0 ** -10)    # half the subnormal step 2^-9
    assert k[3, 1] == 0 and not codes[3, 16:32].any()             # zero block: k = 0, codes 0
    assert codes[5, 0] == 0                                      # -0 stores as +0
    assert np.all((codes == 0) | (np.signbit(back) == np.signbit(h)))
    # values on the scaled E4M3 grid come back exactly
    grid = O.e4m3_decode(np.arange(0, 0x7F, dtype=np.uint8))
    g = np.zeros((1, 128), np.float32)
    g[0, :127] = grid * 2.0 ** 5
    c, kk = O.fp8_block_encode(g)
    np.testing.assert_array_equal(O.fp8_block_decode(c, kk), g)


def test_forward_with_fp8_l1_output_tracks_the_bf16_one():
    wl = W.moe_workload(96, 256, 128, 6, 2, 5)
    hidden = W.bf16_bits_to_f32(wl.hidden)
    w13q = O.quantize_expert_weights(W.bf16_bits_to_f32(wl.w13))
    w2q = O.quantize_expert_weights(W.bf16_bits_to_f32(wl.w2))
    a1 = np.full(wl.E, O.global_scale(np.abs(hidden).max()), np.float32)
    ref, ri = O.moe_forward(hidden, wl.logits, wl.top_k, w13q, w2q, a1, None, return_intermediates=True)
    got, gi = O.moe_forward(hidden, wl.logits, wl.top_k, w13q, w2q, a1, None, return_intermediates=True,
                            l1_fp8=True)
    # both against the layer with the exact bf16 h fed to the L2 weights (no L2 activation
    # quantization): the FP8 step costs little next to the NVFP4 requantization both paths do
    meta = ri["meta"]
    exact = np.zeros(ref.shape)
    for e, d in ri["experts"].items():
        lo, n = int(meta["offsets"][e]), int(meta["counts"][e])
        B = O.dequant_blocks(w2q[0][e], w2q[1][e]) / np.float64(w2q[2][e])
        np.add.at(exact, d["toks"], meta["row_weight"][lo:lo + n, None] * (d["h"].astype(np.float64) @ B.T))
    err = lambda a: np.linalg.norm(a - exact) / np.linalg.norm(exact)
    assert 0 < err(got) <= 1.2 * err(ref) and err(got) <= 0.15, (err(got), err(ref))
    for e, d in gi["experts"].items():
        h = ri["experts"][e]["h"]
        codes, k = O.fp8_block_encode(h)
        np.testing.assert_array_equal(d["h"], O.fp8_block_decode(codes, k))  # the L2 input is h8
        assert np.linalg.norm(d["h"] - h) <= 0.04 * np.linalg.norm(h)
        assert d["a2_gs"] == O.global_scale(np.max(np.abs(d["h"])))          # its scale from h8
    with pytest.raises(ValueError):
        O.moe_forward(hidden, wl.logits, wl.top_k, w13q, w2q, a1, a1, l1_fp8=True)
