"""Pins for oracle.formats: the e4m3fn codec and bf16 rounding.

The encoder is checked against an independent nearest-code search over the
decoded table (brute force), at every midpoint of the grid and one fp32 ulp on
either side, on every finite bf16 bit pattern times several powers of two, and
on random fp32 bit patterns; the decoder against the format's fixed points.
torch's own float8_e4m3fn cast serves as a third opinion after clamping (it
does not saturate by itself).
"""

import numpy as np
import pytest

pytestmark = pytest.mark.filterwarnings("ignore:invalid value encountered in cast")
import torch

from oracle.formats import decode_e4m3, encode_e4m3, round_bf16, round_e4m3_sat

ALL = np.arange(256, dtype=np.uint8)


def finite_table():
    vals = decode_e4m3(ALL)
    ok = ~np.isnan(vals)
    return ALL[ok], vals[ok]


def brute_force_encode(v):
    """Nearest finite e4m3 code by exhaustive search; ties -> even mantissa;
    magnitudes above 448 saturate; zero keeps its sign."""
    codes, vals = finite_table()
    v = np.asarray(v, dtype=np.float64)
    a = np.minimum(np.abs(v), 448.0)
    pos = vals >= 0
    pc, pv = codes[pos & ((codes & 0x80) == 0)], vals[pos & ((codes & 0x80) == 0)]
    d = np.abs(a[:, None] - pv[None, :])
    dmin = d.min(axis=1, keepdims=True)
    tie = d == dmin
    even = (pc & 1) == 0
    # prefer an even-mantissa code among the nearest ones
    pick = np.where(tie & even[None, :], 1, 0) * 2 + np.where(tie, 1, 0)
    best = pc[np.argmax(pick, axis=1)]
    return np.where(np.signbit(v), best | 0x80, best).astype(np.uint8)


def test_decode_fixed_points():
    v = decode_e4m3(ALL)
    assert v[0x00] == 0.0 and not np.signbit(v[0x00])
    assert v[0x80] == 0.0 and np.signbit(v[0x80])
    assert v[0x01] == 2.0 ** -9            # smallest subnormal
    assert v[0x07] == 7 * 2.0 ** -9        # largest subnormal
    assert v[0x08] == 2.0 ** -6            # smallest normal
    assert v[0x38] == 1.0                  # exponent field 7 = bias
    assert v[0x7E] == 448.0                # largest finite
    assert np.isnan(v[0x7F]) and np.isnan(v[0xFF])
    assert np.sum(np.isnan(v)) == 2
    pos = v[:0x7F]
    assert np.all(np.diff(pos) > 0)        # positive codes strictly increasing
    assert np.array_equal(v[0x80:0xFF], -v[0x00:0x7F])


def test_decode_matches_torch_view():
    t = torch.from_numpy(ALL.copy()).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    v = decode_e4m3(ALL)
    same = (t == v) | (np.isnan(t) & np.isnan(v))
    assert same.all()


def test_encode_roundtrips_every_code():
    codes, vals = finite_table()
    assert np.array_equal(encode_e4m3(vals), codes)


def test_encode_midpoints_and_neighbours():
    codes, vals = finite_table()
    pos = np.sort(vals[vals > 0])
    grid = np.concatenate([[0.0], pos])
    mids = (grid[:-1] + grid[1:]) / 2
    f32 = mids.astype(np.float32)
    assert np.array_equal(f32.astype(np.float64), mids)   # midpoints are fp32-exact
    up = np.nextafter(f32, np.float32(np.inf)).astype(np.float64)
    dn = np.nextafter(f32, np.float32(0)).astype(np.float64)
    probe = np.concatenate([mids, up, dn, grid, [448.0, 450.0, 464.0, 464.1, 480.0, 1e30]])
    probe = np.concatenate([probe, -probe])
    assert np.array_equal(encode_e4m3(probe), brute_force_encode(probe))


def test_encode_all_bf16_times_powers_of_two():
    bits = np.arange(65536, dtype=np.uint32) << 16
    v = bits.view(np.float32).astype(np.float64)
    v = v[np.isfinite(v)]
    for k in (-20, -9, -3, 0, 4, 9):
        p = v * 2.0 ** k
        p = p[np.isfinite(p)]
        # clamp the enormous ones for the brute-force distance arithmetic
        p = np.clip(p, -1e6, 1e6)
        for chunk in np.array_split(p, 8):
            assert np.array_equal(encode_e4m3(chunk), brute_force_encode(chunk))


def test_encode_random_fp32_patterns():
    rng = np.random.default_rng(1234)
    bits = rng.integers(0, 2 ** 32, size=200_000, dtype=np.uint64).astype(np.uint32)
    v = bits.view(np.float32).astype(np.float64)
    v = np.clip(v[np.isfinite(v)], -1e6, 1e6)
    for chunk in np.array_split(v, 20):
        assert np.array_equal(encode_e4m3(chunk), brute_force_encode(chunk))


def test_encode_matches_torch_cast_after_clamp():
    rng = np.random.default_rng(7)
    v = np.concatenate([rng.standard_normal(100_000) * s for s in (1e-3, 1.0, 50.0, 300.0)])
    v = np.clip(v.astype(np.float32), -448, 448)
    t = torch.from_numpy(v).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(encode_e4m3(v.astype(np.float64)), t)


def test_saturation_and_nan():
    assert encode_e4m3(np.array([1e9]))[0] == 0x7E
    assert encode_e4m3(np.array([-1e9]))[0] == 0xFE
    assert encode_e4m3(np.array([np.nan]))[0] == 0x7F
    assert round_e4m3_sat(np.array([465.0]))[0] == 448.0


def test_round_bf16_matches_torch_on_fp32_inputs():
    rng = np.random.default_rng(3)
    bits = rng.integers(0, 2 ** 32, size=300_000, dtype=np.uint64).astype(np.uint32)
    v = bits.view(np.float32)
    v = v[np.isfinite(v)]
    t = torch.from_numpy(v).to(torch.bfloat16).to(torch.float64).numpy()
    r = round_bf16(v.astype(np.float64))
    assert np.array_equal(np.isinf(t), np.isinf(r))
    fin = np.isfinite(t)
    assert np.array_equal(t[fin], r[fin])


@pytest.mark.parametrize("x,expect", [(1.0, 1.0), (1.00390625, 1.0), (1.01171875, 1.015625),
                                      (257.0, 256.0), (259.0, 260.0), (-3.0, -3.0)])
def test_round_bf16_ties_to_even(x, expect):
    assert round_bf16(np.array([x]))[0] == expect
