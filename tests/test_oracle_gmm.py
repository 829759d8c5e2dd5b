"""Pins for oracle.gmm: brute-force loops on tiny inputs, the adjoint identity
that ties forward, dgrad and wgrad together (it catches a transposed operand or
a wrong group index in any of the three), closed forms (all-ones input gives
column sums), the trans_b identity, empty groups, and the FP8 scale rule."""

import numpy as np
import pytest

from oracle.formats import decode_e4m3, encode_e4m3
from oracle.gmm import (expert_of_rows, gmm_dgrad, gmm_dgrad_fp8, gmm_fwd, gmm_fwd_fp8,
                        gmm_wgrad, gmm_wgrad_fp8)


def brute_fwd(x, w, sizes):
    M, K = len(x), len(x[0])
    N = len(w[0][0])
    out = [[0.0] * N for _ in range(M)]
    r = 0
    for e, m in enumerate(sizes):
        for i in range(r, r + m):
            for n in range(N):
                acc = 0.0
                for k in range(K):
                    acc += x[i][k] * w[e][k][n]
                out[i][n] = acc
        r += m
    return np.array(out)


def int_inputs(rng, sizes, K, N):
    M = sum(sizes)
    x = rng.integers(-2, 3, (M, K)).astype(np.float64)
    w = rng.integers(-2, 3, (len(sizes), K, N)).astype(np.float64)
    return x, w


@pytest.mark.parametrize("sizes", [[2, 0, 3], [1], [0, 0, 4], [3, 1, 0, 2]])
def test_fwd_brute_force(sizes):
    rng = np.random.default_rng(sum(sizes))
    x, w = int_inputs(rng, sizes, 5, 3)
    ref = brute_fwd(x.tolist(), w.tolist(), sizes)
    assert np.array_equal(gmm_fwd(x, w, sizes), ref.reshape(sum(sizes), 3))


def test_single_expert_is_plain_matmul_brute_force():
    rng = np.random.default_rng(9)
    x, w = int_inputs(rng, [6], 4, 5)
    ref = np.array([[sum(x[i, k] * w[0, k, n] for k in range(4)) for n in range(5)] for i in range(6)])
    assert np.array_equal(gmm_fwd(x, w, [6]), ref)


@pytest.mark.parametrize("sizes", [[5, 0, 7, 1], [16], [0, 9, 0], [130, 0, 37, 200]])
def test_adjoint_identity(sizes):
    # <fwd(x, w), G> = <x, dgrad(G, w)> = <w, wgrad(x, G)>, exactly for integers
    rng = np.random.default_rng(len(sizes))
    K, N = 6, 4
    x, w = int_inputs(rng, sizes, K, N)
    G = rng.integers(-3, 4, (sum(sizes), N)).astype(np.float64)
    a = np.sum(gmm_fwd(x, w, sizes) * G)
    b = np.sum(x * gmm_dgrad(G, w, sizes))
    c = np.sum(w * gmm_wgrad(x, G, sizes))
    assert a == b == c


def test_wgrad_brute_force_and_empty_group_zero():
    sizes = [2, 0, 3]
    rng = np.random.default_rng(5)
    x, _ = int_inputs(rng, sizes, 3, 2)
    G = rng.integers(-3, 4, (5, 2)).astype(np.float64)
    gw = gmm_wgrad(x, G, sizes)
    assert np.all(gw[1] == 0)
    for e, (r0, r1) in enumerate([(0, 2), (2, 2), (2, 5)]):
        for k in range(3):
            for n in range(2):
                assert gw[e, k, n] == sum(x[r, k] * G[r, n] for r in range(r0, r1))


def test_ones_input_gives_column_sums():
    sizes = [3, 4]
    rng = np.random.default_rng(6)
    w = rng.standard_normal((2, 5, 7))
    out = gmm_fwd(np.ones((7, 5)), w, sizes)
    assert np.allclose(out[:3], w[0].sum(axis=0)[None, :], rtol=0, atol=1e-12)
    assert np.allclose(out[3:], w[1].sum(axis=0)[None, :], rtol=0, atol=1e-12)


def test_trans_b_identity():
    sizes = [2, 3]
    rng = np.random.default_rng(7)
    x, w = int_inputs(rng, sizes, 4, 6)
    assert np.array_equal(gmm_fwd(x, w, sizes), gmm_fwd(x, w.transpose(0, 2, 1).copy(), sizes, trans_b=True))


def test_dgrad_is_fwd_with_transposed_weights():
    sizes = [3, 0, 2]
    rng = np.random.default_rng(8)
    _, w = int_inputs(rng, sizes, 4, 6)
    G = rng.integers(-3, 4, (5, 6)).astype(np.float64)
    assert np.array_equal(gmm_dgrad(G, w, sizes), gmm_fwd(G, w.transpose(0, 2, 1), sizes))


def test_expert_of_rows():
    assert expert_of_rows([2, 0, 3], [0, 1, 2, 4]).tolist() == [0, 0, 2, 2]


def fp8_int_operands(rng, shape):
    # small integers are exact e4m3 values (|v| <= 16)
    v = rng.integers(-16, 17, shape).astype(np.float64)
    q = encode_e4m3(v)
    assert np.array_equal(decode_e4m3(q), v)
    return v, q


def test_fp8_fwd_scales_divide():
    sizes = [3, 0, 2]
    rng = np.random.default_rng(10)
    xv, xq = fp8_int_operands(rng, (5, 4))
    wv, wq = fp8_int_operands(rng, (3, 6, 4))          # [E, N, K]
    sx = np.exp2(rng.integers(-3, 4, 5)).astype(np.float64)
    sw = np.exp2(rng.integers(-3, 4, (3, 6))).astype(np.float64)
    out = gmm_fwd_fp8(xq, sx, wq, sw, sizes)
    plain = gmm_fwd(xv, wv, sizes, trans_b=True)
    e_of = expert_of_rows(sizes, np.arange(5))
    assert np.array_equal(out, plain / (sx[:, None] * sw[e_of]))


def test_fp8_dgrad_and_wgrad_scales_divide():
    sizes = [2, 3, 0]
    rng = np.random.default_rng(11)
    gv, gq = fp8_int_operands(rng, (5, 6))             # grad_out [M, N]
    wv, wq = fp8_int_operands(rng, (3, 4, 6))          # [E, K, N]
    sgo = np.exp2(rng.integers(-3, 4, 5)).astype(np.float64)
    sw = np.exp2(rng.integers(-3, 4, (3, 4))).astype(np.float64)
    gx = gmm_dgrad_fp8(gq, sgo, wq, sw, sizes)
    e_of = expert_of_rows(sizes, np.arange(5))
    assert np.array_equal(gx, gmm_dgrad(gv, wv, sizes) / (sgo[:, None] * sw[e_of]))

    xv, xq = fp8_int_operands(rng, (5, 4))             # x [M, K]
    sx = np.exp2(rng.integers(-3, 4, 3 * 4)).astype(np.float64)
    sg = np.exp2(rng.integers(-3, 4, 3 * 6)).astype(np.float64)
    gw = gmm_wgrad_fp8(xq.T.copy(), sx, gq.T.copy(), sg, sizes)
    ref = gmm_wgrad(xv, gv, sizes) / (sx.reshape(3, 4)[:, :, None] * sg.reshape(3, 6)[:, None, :])
    assert np.array_equal(gw, ref)
    assert np.all(gw[2] == 0)
