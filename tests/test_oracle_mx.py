"""Pins for oracle.mx: the MXFP8 block quantizer and the block-scaled grouped
GEMM, checked against hand-computed codes and bytes, the reduction to the
(separately pinned) rowwise quantizer when a row is one block, exact
round trips, and a brute-force loop over the definition."""

import numpy as np

from oracle.formats import decode_e4m3
from oracle.mx import decode_mx, gmm_fwd_mx, quant_mx_rows
from oracle.quant import quant_rowwise


def test_hand_example_two_blocks():
    x = np.zeros((1, 64))
    x[0, :4] = [1.0, -2.0, 0.5, 0.0]     # block 0: amax 2 -> 448/2 = 224 -> s = 128
    q, e = quant_mx_rows(x)               # block 1: all zero -> s = 2^48
    assert e.tolist() == [[127 - 7, 127 - 48]]
    # 128 = 2^7 -> 0x70; -256 -> 0xF8; 64 -> 0x68; 0 -> 0x00
    assert q[0, :4].tolist() == [0x70, 0xF8, 0x68, 0x00]
    assert not q[0, 4:].any()


def test_one_block_rows_reduce_to_rowwise():
    rng = np.random.default_rng(0)
    x = (rng.standard_normal((50, 32)) * np.exp2(rng.integers(-20, 20, (50, 1)))).astype(np.float32).astype(np.float64)
    x[3] = 0.0
    q, e = quant_mx_rows(x)
    qr, sr = quant_rowwise(x)
    assert np.array_equal(q, qr)
    assert np.array_equal(np.exp2(127.0 - e[:, 0].astype(np.float64)), sr)


def test_blocks_are_independent_rows_of_32():
    rng = np.random.default_rng(1)
    x = (rng.standard_normal((7, 256)) * np.exp2(rng.integers(-6, 6, (7, 8)).repeat(32, axis=1))).astype(np.float32)
    x = x.astype(np.float64)
    q, e = quant_mx_rows(x)
    qb, sb = quant_rowwise(x.reshape(-1, 32))
    assert np.array_equal(q, qb.reshape(7, 256))
    assert np.array_equal(np.exp2(127.0 - e.reshape(-1).astype(np.float64)), sb)
    # changing one block leaves every other block's codes and byte alone
    y = x.copy()
    y[2, 64:96] *= 1000.0
    q2, e2 = quant_mx_rows(y)
    mask = np.ones_like(q, dtype=bool)
    mask[2, 64:96] = False
    assert np.array_equal(q[mask], q2[mask])
    emask = np.ones_like(e, dtype=bool)
    emask[2, 2] = False
    assert np.array_equal(e[emask], e2[emask])
    # 1000x is about 2^10: the decode factor of that block grows by 2^9 or 2^10
    assert int(e2[2, 2]) - int(e[2, 2]) in (9, 10)


def test_exact_round_trip_for_representable_blocks():
    # every block holds e4m3 values times 2^j with one element at 448 * 2^j:
    # the scale is exactly 2^-j and decoding gives the input back
    rng = np.random.default_rng(2)
    R, K = 9, 128
    codes = rng.integers(0, 0x7E, (R, K), dtype=np.uint8) | (rng.integers(0, 2, (R, K), dtype=np.uint8) << 7)
    codes[:, ::32] = 0x7E
    j = rng.integers(-20, 20, (R, K // 32))
    x = decode_e4m3(codes) * np.exp2(j).repeat(32, axis=1)
    q, e = quant_mx_rows(x)
    assert np.array_equal(decode_mx(q, e), x)
    assert np.array_equal(e.astype(np.int64), 127 + j)


def test_relative_error_bound():
    rng = np.random.default_rng(3)
    x = (rng.standard_normal((32, 512)) * 3.0).astype(np.float32).astype(np.float64)
    q, e = quant_mx_rows(x)
    d = decode_mx(q, e)
    blk = np.abs(x).reshape(32, 16, 32).max(axis=2).repeat(32, axis=1)
    # e4m3 keeps 3 mantissa bits: error <= 2^-4 of the value, or half the
    # subnormal step (2^-10 of the scaled unit) for tiny elements
    assert np.all(np.abs(d - x) <= np.maximum(np.abs(x) * 2.0 ** -4, blk / 448.0 * 2.0 ** -9 * 2))


def test_gemm_hand_example():
    xq = np.full((1, 32), 0x38, dtype=np.uint8)       # 1.0
    xs = np.array([[127]], dtype=np.uint8)            # x 1
    wq = np.full((1, 1, 32), 0x40, dtype=np.uint8)    # 2.0
    ws = np.array([[[128]]], dtype=np.uint8)          # x 2
    out = gmm_fwd_mx(xq, xs, wq, ws, [1])
    assert out.tolist() == [[32 * 1.0 * 2.0 * 2.0]]


def test_gemm_brute_force():
    rng = np.random.default_rng(4)
    E, N, K = 3, 5, 64
    sizes = [2, 0, 3]
    M = sum(sizes)
    xq = rng.integers(0, 0x7F, (M, K), dtype=np.uint8) ^ (rng.integers(0, 2, (M, K), dtype=np.uint8) << 7)
    wq = rng.integers(0, 0x7F, (E, N, K), dtype=np.uint8) ^ (rng.integers(0, 2, (E, N, K), dtype=np.uint8) << 7)
    xs = rng.integers(110, 140, (M, K // 32), dtype=np.uint8)
    ws = rng.integers(110, 140, (E, N, K // 32), dtype=np.uint8)
    out = gmm_fwd_mx(xq, xs, wq, ws, sizes)
    dv = {c: float(decode_e4m3(np.array([c], dtype=np.uint8))[0]) for c in range(256)}
    starts = [0, 2, 2]
    for e in range(E):
        for r in range(starts[e], starts[e] + sizes[e]):
            for n in range(N):
                acc = 0.0
                for k in range(K):
                    a = dv[int(xq[r, k])] * 2.0 ** (int(xs[r, k // 32]) - 127)
                    b = dv[int(wq[e, n, k])] * 2.0 ** (int(ws[e, n, k // 32]) - 127)
                    acc += a * b
                assert abs(out[r, n] - acc) <= 1e-12 * max(1.0, abs(acc)), (e, r, n)


def test_colwise_one_block_groups_reduce_to_fp8_colwise():
    # groups of at most 32 rows hold one block per column: the MX colwise codes
    # equal the per-group colwise FP8 codes, and 2^(127 - byte) its scales
    from oracle.mx import quant_mx_colwise_grouped
    from oracle.quant import quant_colwise_grouped

    rng = np.random.default_rng(5)
    sizes = [32, 0, 7, 19]
    off = np.concatenate([[0], np.cumsum(sizes)])
    x = (rng.standard_normal((off[-1], 24)) * np.exp2(rng.integers(-9, 9, (1, 24)))).astype(np.float32)
    x = x.astype(np.float64)
    q, e = quant_mx_colwise_grouped(x, off)
    qf, sf = quant_colwise_grouped(x, off)
    assert np.array_equal(q, qf)
    for g, m in enumerate(sizes):
        if m:
            assert np.array_equal(np.exp2(127.0 - e[g][:, 0].astype(np.float64)), sf[g * 24:(g + 1) * 24])
        else:
            assert e[g].shape == (24, 0)


def test_colwise_blocks_start_at_each_group():
    from oracle.mx import quant_mx_colwise_grouped

    x = np.zeros((70, 2))
    x[:40, 0] = 1.0           # group 0: rows 0..39 -> blocks [0, 32), [32, 40)
    x[39, 0] = 100.0          # only the second block of group 0 sees 100
    x[40:70, 0] = 2.0         # group 1: rows 40..69 -> one block
    q, e = quant_mx_colwise_grouped(x, [0, 40, 70])
    # amax 1 -> s 256 (byte 119); amax 100 -> 448/100 -> s 4 (byte 125); amax 2 -> s 128 (byte 120)
    assert e[0][0].tolist() == [119, 125] and e[1][0].tolist() == [120]
    assert e[0][1].tolist() == [127 - 48, 127 - 48] and e[1][1].tolist() == [127 - 48]


def test_wgrad_brute_force():
    from oracle.mx import gmm_wgrad_mx, quant_mx_colwise_grouped

    rng = np.random.default_rng(6)
    sizes = [5, 0, 40]
    off = np.concatenate([[0], np.cumsum(sizes)])
    M, K, N = off[-1], 3, 4
    x = rng.standard_normal((M, K)).astype(np.float32).astype(np.float64)
    go = rng.standard_normal((M, N)).astype(np.float32).astype(np.float64)
    xq, xs = quant_mx_colwise_grouped(x, off)
    gq, gs = quant_mx_colwise_grouped(go, off)
    out = gmm_wgrad_mx(xq, xs, gq, gs, sizes)
    dv = {c: float(decode_e4m3(np.array([c], dtype=np.uint8))[0]) for c in range(256)}
    for e in range(3):
        for k in range(K):
            for n in range(N):
                acc = 0.0
                for r in range(off[e], off[e + 1]):
                    b = (r - off[e]) // 32
                    acc += dv[int(xq[k, r])] * 2.0 ** (int(xs[e][k, b]) - 127) * \
                        dv[int(gq[n, r])] * 2.0 ** (int(gs[e][n, b]) - 127)
                assert abs(out[e, k, n] - acc) <= 1e-12 * max(1.0, abs(acc))
    assert not out[1].any()


def test_fwd_equals_rowwise_fp8_when_a_row_shares_one_scale():
    # every block of a row (and of a weight row) with the same e8m0 byte: the MX
    # product is the rowwise-scaled FP8 product with scale 2^(127 - byte)
    from oracle.gmm import gmm_fwd_fp8

    rng = np.random.default_rng(7)
    sizes, K, N = [3, 0, 5], 96, 7
    E, M = len(sizes), sum(sizes)
    xq = rng.integers(0, 0x7F, (M, K), dtype=np.uint8) ^ (rng.integers(0, 2, (M, K), dtype=np.uint8) << 7)
    wq = rng.integers(0, 0x7F, (E, N, K), dtype=np.uint8) ^ (rng.integers(0, 2, (E, N, K), dtype=np.uint8) << 7)
    bx = rng.integers(100, 150, M).astype(np.uint8)
    bw = rng.integers(100, 150, (E, N)).astype(np.uint8)
    xs = np.repeat(bx[:, None], K // 32, axis=1)
    ws = np.repeat(bw[:, :, None], K // 32, axis=2)
    mx = gmm_fwd_mx(xq, xs, wq, ws, sizes)
    fp8 = gmm_fwd_fp8(xq, np.exp2(127.0 - bx), wq, np.exp2(127.0 - bw.astype(np.float64)).ravel(), sizes)
    assert np.allclose(mx, fp8, rtol=1e-12, atol=0)


def test_wgrad_equals_fp8_colwise_when_groups_hold_one_block():
    # groups of at most 32 rows: one MX block per column and group, whose scale is
    # the FP8 per-group colwise scale, so the two wgrads agree
    from oracle.gmm import gmm_wgrad_fp8
    from oracle.mx import gmm_wgrad_mx, quant_mx_colwise_grouped
    from oracle.quant import quant_colwise_grouped

    rng = np.random.default_rng(8)
    sizes = [17, 0, 32, 5]
    off = np.concatenate([[0], np.cumsum(sizes)])
    M, K, N = off[-1], 6, 5
    x = (rng.standard_normal((M, K)) * 3).astype(np.float32).astype(np.float64)
    go = rng.standard_normal((M, N)).astype(np.float32).astype(np.float64)
    qx, ex = quant_mx_colwise_grouped(x, off)
    qg, eg = quant_mx_colwise_grouped(go, off)
    mx = gmm_wgrad_mx(qx, ex, qg, eg, sizes)
    fx, sx = quant_colwise_grouped(x, off)
    fg, sg = quant_colwise_grouped(go, off)
    fp8 = gmm_wgrad_fp8(fx, sx, fg, sg, sizes)
    assert np.allclose(mx, fp8, rtol=1e-12, atol=0)
