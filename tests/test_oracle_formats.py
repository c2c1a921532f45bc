"""Pins of the oracle's FP4 (E2M1) and FP8 (E4M3) encoders against brute force
and, for E4M3, against torch's float8_e4m3fn conversion (no GPU)."""
import numpy as np
import pytest
import torch

from oracle import nvfp4_oracle as O

GRID = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])


def brute_e2m1(q):
    """Nearest of the 8 magnitudes by explicit distance; exact ties take the even code."""
    q = np.asarray(q, np.float32)
    # beyond 1e6 every distance is dominated by |q|; the clip keeps f64 differences exact
    a = np.minimum(np.abs(q).astype(np.float64), 1e6)
    d = np.abs(a[:, None] - GRID[None, :])
    best = d.min(axis=1, keepdims=True)
    cand = d == best
    # among tied candidates prefer an even code index
    even = cand & (np.arange(8)[None, :] % 2 == 0)
    pick = np.where(even.any(axis=1), even.argmax(axis=1), cand.argmax(axis=1))
    neg = np.signbit(q) & (pick != 0)
    return (pick | (neg << 3)).astype(np.uint8)


def around(values, n_ulps):
    vals = np.asarray(values, np.float32)
    bits = vals.view(np.int32)[:, None] + np.arange(-n_ulps, n_ulps + 1, dtype=np.int32)[None, :]
    bits = bits[bits >= 0]
    return bits.astype(np.int32).view(np.float32)


def test_e2m1_brute_force_lattice_and_midpoints():
    mids = [0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0]
    pts = [around(mids, 2000), around(GRID[1:], 2000), around([6.0, 7.0, 8.0], 500)]
    # a prime-stride lattice over every fp32 bit pattern in [0, 8]
    lat = (np.arange(0, 0x41000000, 1021, dtype=np.int64)).astype(np.int32).view(np.float32)
    rng = np.random.default_rng(1)
    rnd = rng.uniform(0, 9, 200000).astype(np.float32)
    q = np.concatenate(pts + [lat, rnd, np.float32([0.0, 1e-30, 1e30, 6.0000005])])
    q = np.concatenate([q, -q])
    np.testing.assert_array_equal(O.e2m1_encode(q), brute_e2m1(q))


@pytest.mark.parametrize("q,nib", [(-0.75, 0xA), (0.25, 0x0), (2.5, 0x4), (5.0, 0x6),
                                   (7.0, 0x7), (-0.1, 0x0), (0.75, 0x2), (1.75, 0x4),
                                   (3.5, 0x6), (1.25, 0x2), (-6.0, 0xF), (-0.0, 0x0)])
def test_e2m1_hand_values(q, nib):
    assert int(O.e2m1_encode(np.float32([q]))[0]) == nib


def e4m3_table():
    codes = np.arange(0, 0x7F)
    return codes, O.e4m3_decode(codes)


def test_e4m3_decode_known_points():
    # 0x38 = 1.0, 0x7E = 448 (largest finite), 0x01 = 2^-9 (smallest subnormal), 0x08 = 2^-6
    assert O.e4m3_decode(0x38) == 1.0
    assert O.e4m3_decode(0x7E) == 448.0
    assert O.e4m3_decode(0x01) == 2.0 ** -9
    assert O.e4m3_decode(0x08) == 2.0 ** -6
    assert np.isnan(O.e4m3_decode(0x7F))
    vals = O.e4m3_decode(np.arange(0x7F))
    assert np.all(np.diff(vals) > 0)  # monotone over the positive codes


def brute_e4m3(v):
    codes, vals = e4m3_table()
    v = np.asarray(v, np.float64)
    d = np.abs(v[:, None] - vals[None, :])
    best = d.min(axis=1, keepdims=True)
    cand = d == best
    even = cand & (codes[None, :] % 2 == 0)
    return np.where(even.any(axis=1), even.argmax(axis=1), cand.argmax(axis=1)).astype(np.uint8)


def test_e4m3_brute_force():
    codes, vals = e4m3_table()
    mids = (vals[:-1] + vals[1:]) / 2
    pts = [around(vals[1:].astype(np.float32), 64), around(mids.astype(np.float32), 64),
           around([448.0, 464.0, 480.0, 1e4], 64)]
    rng = np.random.default_rng(2)
    rnd = np.exp(rng.uniform(np.log(1e-4), np.log(500), 200000)).astype(np.float32)
    v = np.concatenate(pts + [rnd, np.float32([0.0, 1e-30, 2.0 ** -10, 2.0 ** -10 * 1.0001])])
    v = v[v >= 0]
    np.testing.assert_array_equal(O.e4m3_encode(v), brute_e4m3(v))


def test_e4m3_matches_torch_in_range():
    rng = np.random.default_rng(3)
    v = np.concatenate([np.exp(rng.uniform(np.log(1e-4), np.log(448), 100000)),
                        O.e4m3_decode(np.arange(0x7F))]).astype(np.float32)
    v = v[v <= 448]
    t = torch.from_numpy(v).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    np.testing.assert_array_equal(O.e4m3_encode(v), t)


def test_e4m3_exhaustive_against_torch_and_brute_force():
    """Every fp32 bit pattern in [0, 448] against torch's float8_e4m3fn cast
    (1.14e9 values, about 30 s), and every one in (448, 464] against the
    brute-force encoder (saturation, where torch gives NaN above 464)."""
    top = int(np.float32(448.0).view(np.int32))
    step = 1 << 22  # 4 M values per chunk keeps the peak memory near 200 MB
    for lo in range(0, top + 1, step):
        v = np.arange(lo, min(lo + step, top + 1), dtype=np.int64).astype(np.int32).view(np.float32)
        ref = torch.from_numpy(v).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
        np.testing.assert_array_equal(O.e4m3_encode(v), ref)
    hi = int(np.float32(464.0).view(np.int32))
    v = np.arange(top + 1, hi + 1, dtype=np.int64).astype(np.int32).view(np.float32)
    np.testing.assert_array_equal(O.e4m3_encode(v), brute_e4m3(v))


@pytest.mark.parametrize("v,code", [(7.0 / 6.0, 0x39), (1.0, 0x38), (2.0 ** -9, 0x01),
                                    (2.0 ** -10, 0x00), (2.0 ** -10 * 1.0001, 0x01),
                                    (448.0, 0x7E), (500.0, 0x7E), (1e9, 0x7E)])
def test_e4m3_hand_values(v, code):
    assert int(O.e4m3_encode(np.float32([v]))[0]) == code


def test_e4m3_saturates_where_torch_gives_nan():
    t = torch.tensor([500.0]).to(torch.float8_e4m3fn).view(torch.uint8).item()
    assert t & 0x7F == 0x7F  # torch: NaN
    assert int(O.e4m3_encode(np.float32([500.0]))[0]) == 0x7E  # satfinite


def test_pack_unpack_roundtrip_and_order():
    nib = np.array([[1, 2, 3, 4]], np.uint8)
    packed = O.pack_nibbles(nib)
    assert packed.tolist() == [[0x21, 0x43]]  # low nibble = even K index
    np.testing.assert_array_equal(O.unpack_nibbles(packed), nib)


def test_bf16_round_matches_torch():
    """The oracle's FP32 -> bf16 rounding (nearest, ties to even) against
    torch's conversion: random magnitudes over the whole exponent range, exact
    ties in both directions, values next to ties, signed zeros and the largest
    finite values."""
    rng = np.random.default_rng(4)
    r = (rng.standard_normal(200000) * np.exp(rng.uniform(-80, 80, 200000))).astype(np.float32)
    base = rng.integers(0, 1 << 16, 5000).astype(np.uint32) << 16
    ties = (base | 0x8000).view(np.float32)          # exactly halfway between two bf16 values
    near = np.concatenate([(base | 0x7FFF).view(np.float32), (base | 0x8001).view(np.float32)])
    edge = np.float32([0.0, -0.0, 3.3895314e38, -3.3895314e38, 1e-40, -1e-40, 1.0, 1.00390625])
    x = np.concatenate([r, ties, near, edge])
    x = x[np.isfinite(x) & (np.abs(x) < 3.389e38)]
    want = torch.from_numpy(x).to(torch.bfloat16).float().numpy()
    got = O.bf16_round(x)
    np.testing.assert_array_equal(got.view(np.uint32), want.view(np.uint32))
