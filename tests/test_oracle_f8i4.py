"""Pins for oracle.f8i4: the INT4 block quantizer, the nibble packing and the
FP8 x INT4 grouped GEMM, checked against hand-computed values and bytes, every
byte of the packing, the quantizer's invariants and exact round trips, a
brute-force loop over the definition, and the reduction to the (separately
pinned) MXFP8 GEMM of oracle.mx when the integers are written as e4m3 codes."""

import numpy as np

from oracle.f8i4 import decode_int4, gmm_fwd_f8i4, int4_block_scale, pack_int4, quant_int4_rows, unpack_int4
from oracle.formats import decode_e4m3, encode_e4m3
from oracle.mx import gmm_fwd_mx
from oracle.quant import quant_rowwise


def test_hand_example_three_blocks():
    w = np.zeros((1, 96))
    w[0, :5] = [3.5, -1.0, 0.3, -0.25, 0.75]      # amax 3.5: 7 / 3.5 = 2 -> s = 2
    w[0, 64:68] = [1.0, -0.875, 0.625, 0.1]        # amax 1: 7 -> s = 4; block 1 is all zero
    q, b = quant_int4_rows(w)
    # s = 2: 7, -2, 0.6 -> 1, -0.5 -> 0 (half to even), 1.5 -> 2
    assert q[0, :5].tolist() == [7, -2, 1, 0, 2]
    # s = 4: 4, -3.5 -> -4 (half to even), 2.5 -> 2 (half to even), 0.4 -> 0
    assert q[0, 64:68].tolist() == [4, -4, 2, 0]
    assert not q[0, 5:64].any() and not q[0, 68:].any()
    # bytes of the decode factors 1/2, 2^-42 (amax 0: 7e12 -> 2^42), 1/4
    assert b.tolist() == [[126, 85, 125]]


def test_scale_rule_values():
    s, b = int4_block_scale(np.array([7.0, 7.0001, 6.9999, 1e-12, 0.0, 3.0e38, 1.0]))
    assert s.tolist() == [1.0, 0.5, 1.0, 2.0 ** 42, 2.0 ** 42, 2.0 ** -126, 4.0]
    assert b.tolist() == [127, 128, 127, 85, 85, 253, 125]


def test_packing_every_byte():
    allb = np.arange(256, dtype=np.uint8).reshape(1, 256)
    q = unpack_int4(allb)
    lo, hi = q[0, 0::2].astype(int), q[0, 1::2].astype(int)
    for v in range(256):
        nl, nh = v & 15, v >> 4
        assert lo[v] == (nl - 16 if nl >= 8 else nl) and hi[v] == (nh - 16 if nh >= 8 else nh)
    assert np.array_equal(pack_int4(q), allb)
    # element 2j is the low nibble of byte j
    assert pack_int4(np.array([[-1, 0, 0, -1, 7, -8, -8, 7]], dtype=np.int8)).tolist() == [[0x0F, 0xF0, 0x87, 0x78]]


def test_quantizer_invariants():
    rng = np.random.default_rng(0)
    w = (rng.standard_normal((40, 256)) * np.exp2(rng.integers(-30, 30, (40, 8))).repeat(32, axis=1))
    w = w.astype(np.float32).astype(np.float64)
    w[5, 32:64] = 0.0
    q, b = quant_int4_rows(w)
    assert q.min() >= -7 and q.max() <= 7                         # s <= 7 / amax
    amax = np.abs(w).reshape(40, 8, 32).max(axis=2)
    qmax = np.abs(q.astype(int)).reshape(40, 8, 32).max(axis=2)
    live = amax > 0
    assert np.all((qmax[live] >= 4) & (qmax[live] <= 7))           # amax * s in (3.5, 7]
    assert np.all(qmax[~live] == 0) and b[5, 1] == 85
    # error of the decoded value: at most half a step of its block
    step = np.exp2(b.astype(np.float64) - 127).repeat(32, axis=1)
    assert np.all(np.abs(decode_int4(q, b) - w) <= 0.5 * step)


def test_exact_round_trip_for_representable_blocks():
    rng = np.random.default_rng(1)
    R, K = 6, 128
    q0 = rng.integers(-7, 8, (R, K))
    q0[:, ::32] = rng.choice([-7, 7], (R, K // 32))             # every block reaches magnitude 7
    j = rng.integers(-40, 40, (R, K // 32))
    w = q0 * np.exp2(j).repeat(32, axis=1)
    q, b = quant_int4_rows(w)
    assert np.array_equal(q.astype(int), q0)
    assert np.array_equal(b.astype(int), 127 + j)
    assert np.array_equal(decode_int4(q, b), w)


def _problem(sizes, K, N, seed):
    rng = np.random.default_rng(seed)
    M, E = int(np.sum(sizes)), len(sizes)
    x = rng.standard_normal((M, K)).astype(np.float32).astype(np.float64)
    w = (rng.standard_normal((E * N, K)) * 0.02).astype(np.float32).astype(np.float64)
    xq, sx = quant_rowwise(x)
    q, b = quant_int4_rows(w)
    return xq, sx, q.reshape(E, N, K), b.reshape(E, N, K // 32)


def test_gemm_brute_force_tiny():
    sizes, K, N = [2, 0, 3], 64, 5
    xq, sx, q, b = _problem(sizes, K, N, 2)
    out = gmm_fwd_f8i4(xq, sx, pack_int4(q.reshape(-1, K)).reshape(3, N, K // 2), b, sizes)
    xv = decode_e4m3(xq)
    e_of = [0, 0, 2, 2, 2]
    for r in range(5):
        for n in range(N):
            acc = 0.0
            for k in range(K):
                acc += xv[r, k] / sx[r] * float(q[e_of[r], n, k]) * 2.0 ** (int(b[e_of[r], n, k // 32]) - 127)
            assert abs(out[r, n] - acc) <= 1e-12 * max(1.0, abs(acc))


def test_gemm_equals_mx_gemm_of_the_same_values():
    sizes, K, N = [7, 0, 30, 1, 12], 256, 48
    xq, sx, q, b = _problem(sizes, K, N, 3)
    E = len(sizes)
    out = gmm_fwd_f8i4(xq, sx, pack_int4(q.reshape(-1, K)).reshape(E, N, K // 2), b, sizes)
    # integers -8..7 are exact e4m3 values; the row scale of x is a block byte on every block
    wcodes = encode_e4m3(q.astype(np.float64))
    assert np.array_equal(decode_e4m3(wcodes), q.astype(np.float64))
    _, ex = np.frexp(sx)
    xbytes = np.repeat((127 - (ex - 1))[:, None], K // 32, axis=1).astype(np.uint8)
    ref = gmm_fwd_mx(xq, xbytes, wcodes, b, sizes)
    assert np.array_equal(out, ref)


def test_empty_groups_and_single_group():
    sizes, K, N = [0, 9, 0], 64, 16
    xq, sx, q, b = _problem(sizes, K, N, 4)
    wp = pack_int4(q.reshape(-1, K)).reshape(3, N, K // 2)
    out = gmm_fwd_f8i4(xq, sx, wp, b, sizes)
    # E = 1 of the same expert is a plain matmul of the decoded values
    one = gmm_fwd_f8i4(xq, sx, wp[1:2], b[1:2], [9])
    plain = (decode_e4m3(xq) / sx[:, None]) @ decode_int4(q[1], b[1]).T
    assert np.array_equal(out, one) and np.allclose(one, plain, rtol=1e-13, atol=0)
