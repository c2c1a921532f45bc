"""Pins of the oracle's NVFP4 block quantizer: hand-worked golden blocks,
the dequantization error bound, the forced (zero / underflow) block rule,
the global-scale convention and the 128x4 scale-tile layout (no GPU)."""
import json
import os

import numpy as np
import pytest

from oracle import nvfp4_oracle as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "quant_blocks.json")


def load_cases():
    with open(GOLDEN) as f:
        return json.load(f)["cases"]


@pytest.mark.parametrize("case", load_cases(), ids=lambda c: c["name"])
def test_golden_blocks(case):
    x = np.float32(case["x"])[None, :]
    nib, s = O.quantize_blocks(x, np.float32(case["gs"]))
    assert int(s[0, 0]) == case["scale"]
    assert nib[0].tolist() == case["nibbles"]
    deq = O.dequant_blocks(nib, s)[0]
    np.testing.assert_array_equal(deq, np.float64(case["dequant"]))
    assert np.all(np.isfinite(deq))


def test_global_scale_convention():
    assert O.global_scale(0.0) == np.float32(1.0)
    assert O.global_scale(448.0 * 6) == np.float32(1.0)
    assert O.global_scale(2.0) == np.float32(1344.0)
    # vllm page (checkpoint input_scale paragraph): the decode form of this
    # scale for a unit amax is 1/2688 = 0.000372
    assert round(1.0 / float(O.global_scale(1.0)), 6) == 0.000372
    # the tensor amax lands exactly on the largest code pair (scale 448, nibble 6)
    x = np.zeros((1, 16), np.float32)
    x[0, 3] = 3.25
    gs = O.global_scale(3.25)
    nib, s = O.quantize_blocks(x, gs)
    assert int(s[0, 0]) == 0x7E and int(nib[0, 3]) == 7


def random_blocks(n, rng):
    x = rng.standard_normal((n, 16)).astype(np.float32)
    x *= np.exp(rng.uniform(-12, 8, (n, 1))).astype(np.float32)
    return x


def test_dequant_error_bound():
    rng = np.random.default_rng(4)
    x = random_blocks(20000, rng)
    gs = np.float32(3.0)
    nib, s = O.quantize_blocks(x, gs)
    xs = (x * gs).astype(np.float32).astype(np.float64)
    deq = O.dequant_blocks(nib, s)
    b = np.abs(xs).max(axis=1)
    forced = b < 6 * 2.0 ** -9
    sc = O.e4m3_decode(s[:, 0])
    bound = np.maximum(sc, b - 6 * sc)[:, None] * (1 + 1e-6)
    err = np.abs(xs - deq)
    assert np.all(err[~forced] <= bound[~forced])
    assert np.all(deq[forced] == 0) and np.all(s[forced] == 0) and np.all(nib[forced] == 0)
    assert np.all(np.abs(xs[forced]) < 6 * 2.0 ** -9)
    assert forced.any() and (~forced).any()


def test_forced_range_includes_values_plain_rounding_keeps():
    # b/6 in [2^-10, 2^-9): plain round-to-nearest of the scale would give code 0x01,
    # the explicit rule forces 0.
    b = np.float32(6 * 2.0 ** -10 * 1.5)
    assert O.e4m3_encode(np.float32([b / np.float32(6)]))[0] == 1
    x = np.zeros((1, 16), np.float32)
    x[0, 0] = b
    nib, s = O.quantize_blocks(x, np.float32(1))
    assert int(s[0, 0]) == 0 and int(nib[0, 0]) == 0


def test_block_exactly_at_the_underflow_threshold_is_kept():
    # amax = 6 * 2^-9: b/6 = 2^-9 is the smallest E4M3 subnormal (code 0x01), the
    # block survives and its maximum maps to E2M1 6.0 (code 7); the next FP32
    # value below the threshold is forced to zero.
    t = np.float32(6 * 2.0 ** -9)
    x = np.zeros((2, 16), np.float32)
    x[0, 0], x[0, 1] = t, -t / np.float32(2)
    x[1, 0] = np.nextafter(t, np.float32(0))
    nib, s = O.quantize_blocks(x, np.float32(1))
    assert int(s[0, 0]) == 0x01
    assert int(nib[0, 0]) == 0x7 and int(nib[0, 1]) == 0xD  # -3.0 = sign bit | code 5
    assert int(s[1, 0]) == 0 and not nib[1].any()


def test_scale_applies_per_row():
    rng = np.random.default_rng(5)
    x = rng.standard_normal((3, 32)).astype(np.float32)
    gs = np.float32([1.0, 2.0, 0.5])
    nib, s = O.quantize_blocks(x, gs)
    for r in range(3):
        n1, s1 = O.quantize_blocks(x[r:r + 1], gs[r])
        np.testing.assert_array_equal(nib[r], n1[0])
        np.testing.assert_array_equal(s[r], s1[0])


# ----------------------------------------------------------------- scale tile layout

def test_sf_layout_is_a_bijection_with_512_byte_tiles():
    rows, cols = 384, 12
    rr, cc = np.meshgrid(np.arange(rows), np.arange(cols), indexing="ij")
    off = O.sf_tile_offset(rr, cc, cols)
    assert sorted(off.ravel().tolist()) == list(range(rows * cols))
    # every 128-row x 4-column tile occupies 512 consecutive bytes
    for rt in range(rows // 128):
        for ct in range(cols // 4):
            t = off[rt * 128:(rt + 1) * 128, ct * 4:(ct + 1) * 4]
            assert t.max() - t.min() == 511
    # within a tile the 4 scales of one row are adjacent bytes and rows r, r+32,
    # r+64, r+96 share one 16-byte line
    assert (off[5, 1] - off[5, 0]) == 1
    assert (off[37, 0] - off[5, 0]) == 4 and (off[6, 0] - off[5, 0]) == 16


def test_assemble_and_unswizzle_roundtrip_with_padding():
    rng = np.random.default_rng(6)
    counts = [5, 0, 130, 128]
    offsets = np.concatenate([[0], np.cumsum(counts)])
    padded = np.concatenate([[0], np.cumsum([(c + 127) // 128 * 128 for c in counts])])
    C = 6  # pads to 8 columns
    lin = rng.integers(1, 255, (offsets[-1], C), dtype=np.uint8)
    swz = O.assemble_scales(lin, offsets, padded)
    assert swz.size == padded[-1] * 8
    full = O.unswizzle_scales(swz, padded[-1], 8)
    for g, c in enumerate(counts):
        np.testing.assert_array_equal(full[padded[g]:padded[g] + c, :C], lin[offsets[g]:offsets[g] + c])
        assert np.all(full[padded[g] + c:padded[g + 1]] == 0)
    assert np.all(full[:, C:] == 0)
