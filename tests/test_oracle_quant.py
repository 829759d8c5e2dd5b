"""Pins for oracle.quant: the power-of-two scale rule and the rowwise /
per-group colwise quantizers, checked against hand-computed codes, the
invariants the scale rule implies, and group isolation."""

import numpy as np
import pytest

from oracle.formats import decode_e4m3
from oracle.quant import pow2_scale, quant_colwise_grouped, quant_colwise_grouped_dual, quant_rowwise


def is_pow2(s):
    m, _ = np.frexp(s)
    return np.all(m == 0.5)


@pytest.mark.parametrize("amax,expect", [
    (448.0, 1.0),          # 448/448 = 1
    (1.0, 256.0),          # 448 -> 256
    (0.5, 512.0),          # 896 -> 512
    (3.5, 128.0),          # exactly 128
    (3.515625, 64.0),      # 127.44... -> 64
    (0.0, 2.0 ** 48),      # EPS clamp: 4.48e14 -> 2^48
    (1e-30, 2.0 ** 48),
    (1000.0, 0.25),        # 0.448 -> 0.25
])
def test_pow2_scale_values(amax, expect):
    assert pow2_scale(np.array([amax]))[0] == expect


def test_pow2_scale_invariants():
    rng = np.random.default_rng(0)
    amax = np.abs(rng.standard_normal(100_000)) * np.exp2(rng.integers(-30, 30, 100_000))
    s = pow2_scale(amax)
    assert is_pow2(s)
    r = (448.0 / np.maximum(amax, 1e-12)).astype(np.float32).astype(np.float64)
    assert np.all(s <= r) and np.all(2 * s > r)


def test_scale_uses_fp32_rounding_before_floor():
    # 448 / amax just below 2^k in float64 but rounding up to 2^k in fp32
    amax = 448.0 / (2.0 ** 7 * (1 - 2.0 ** -30))
    assert 448.0 / amax < 128.0
    assert pow2_scale(np.array([amax]))[0] == 128.0


def test_rowwise_hand_example():
    x = np.array([[1.0, -2.0, 0.5, 0.0, 3.5],
                  [0.0, 0.0, 0.0, 0.0, 0.0]])
    q, s = quant_rowwise(x)
    assert s[0] == 128.0 and s[1] == 2.0 ** 48
    # 128 = 2^7 -> e=14 m=0; -256 -> 0xF8; 64 -> 0x68; 0 -> 0; 448 -> 0x7E
    assert q[0].tolist() == [0x70, 0xF8, 0x68, 0x00, 0x7E]
    assert q[1].tolist() == [0] * 5


def test_rowwise_invariants():
    rng = np.random.default_rng(1)
    x = rng.standard_normal((64, 96)) * np.exp2(rng.integers(-12, 12, (64, 1)))
    x = x.astype(np.float32).astype(np.float64)
    q, s = quant_rowwise(x)
    d = decode_e4m3(q)
    assert np.all(np.abs(d) <= 448)
    dq = np.max(np.abs(d), axis=1)
    assert np.all((dq >= 224) & (dq <= 448))
    # each dequantized value is within half an e4m3 spacing of x (relative 2^-4)
    err = np.abs(d / s[:, None] - x)
    assert np.all(err <= np.abs(x) * 2.0 ** -4 + 2.0 ** -10 / s[:, None])


def test_colwise_single_group_is_rowwise_of_transpose():
    rng = np.random.default_rng(2)
    x = rng.standard_normal((40, 24))
    qt, sc = quant_colwise_grouped(x, [0, 40])
    q2, s2 = quant_rowwise(x.T)
    assert np.array_equal(qt, q2) and np.array_equal(sc, s2)


def test_colwise_groups_are_isolated_and_indexed():
    rng = np.random.default_rng(3)
    x = rng.standard_normal((30, 8))
    offs = [0, 10, 10, 30]                  # middle group empty
    qt, sc = quant_colwise_grouped(x, offs)
    x2 = x.copy()
    x2[10:] *= 1000.0                        # only group 2 changes
    qt2, sc2 = quant_colwise_grouped(x2, offs)
    assert np.array_equal(sc[:8], sc2[:8]) and np.array_equal(qt[:, :10], qt2[:, :10])
    assert np.all(sc[8:16] == 2.0 ** 48)     # empty group: amax 0 -> 2^48
    for g, (r0, r1) in enumerate([(0, 10), (10, 10), (10, 30)]):
        for c in range(8):
            col = x[r0:r1, c]
            if r1 > r0:
                s = pow2_scale(np.array([np.max(np.abs(col))]))[0]
                assert sc[c + 8 * g] == s
                assert np.array_equal(qt[c, r0:r1], quant_rowwise(col[None, :])[0][0])


def test_dual_equals_two_singles():
    rng = np.random.default_rng(4)
    a, b = rng.standard_normal((20, 6)), rng.standard_normal((20, 10))
    offs = [0, 7, 20]
    (q1, s1), (q2, s2) = quant_colwise_grouped_dual(a, b, offs)
    assert np.array_equal(q1, quant_colwise_grouped(a, offs)[0])
    assert np.array_equal(s2, quant_colwise_grouped(b, offs)[1])
