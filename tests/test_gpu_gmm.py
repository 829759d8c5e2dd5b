"""GPU parity of mgemm_fwd / mgemm_dgrad / mgemm_wgrad against oracle.gmm.

Sizes are small enough for the float64 oracle to finish in seconds but span
several 128 x 256 tiles and ragged tails in every dimension (group edges inside
a tile, K and N not multiples of the tile, empty groups, a one-row group).
Tolerances: max|err| <= 1e-2 * max|ref| (bf16 operands) and 3e-2 * max|ref|
(FP8 operands); integer-valued inputs are exact in fp32, so there the bf16
result must equal the oracle rounded to bf16 bit for bit.  Guard rows beyond
the outputs and a poisoned status word check that nothing else is written."""

import numpy as np
import pytest
import torch

from oracle import formats, gmm as og, quant as oq
from tests.helpers import (BF16_TOL, FP8_TOL, assert_close, colwise_padding, is_sentinel, new_args, sentinel_bf16,
                           to_np, unpad_colwise)

pytestmark = pytest.mark.gpu
DEV = "cuda"
BF = torch.bfloat16


def B():
    from mixture_experts_grouped_gmm_gb300 import binding

    return binding


def fill(sizes):
    E = len(sizes)
    args = new_args(E, DEV)
    B().mgemm_fill_args(torch.tensor(sizes, dtype=torch.int64, device=DEV), E, int(np.sum(sizes)), args)
    return args


def rand_bf16(shape, seed, kind="uniform"):
    g = torch.Generator(device=DEV).manual_seed(seed)
    if kind == "uniform":
        t = torch.rand(shape, generator=g, device=DEV)
    elif kind == "normal":
        t = torch.randn(shape, generator=g, device=DEV)
    else:  # small integers: products and sums exact in fp32
        t = torch.randint(-2, 3, shape, generator=g, device=DEV).float()
    return t.to(BF)


CASES = [
    # sizes, K, N
    ([15, 16, 19, 14], 128, 256),                 # tiny config
    ([0, 20, 20, 24], 128, 256),                  # tiny, empty group
    ([0, 300, 1, 129, 250], 320, 520),            # ragged: K, N not tile multiples
    ([700], 192, 264),                            # E = 1 (a plain matmul)
    ([5, 0, 0, 0, 0, 0, 3, 0], 64, 64),           # sparse rows among many groups
]


def bf16_fwd(sizes, K, N, x, w, trans_b):
    M, E = int(np.sum(sizes)), len(sizes)
    out = sentinel_bf16((M + 8, N), DEV)
    B().mgemm_fwd(fill(sizes), B().MGEMM_BF16, trans_b, x, None, w, None, out, M, K, N, E)
    torch.cuda.synchronize()
    assert is_sentinel(out[M:]), "fwd wrote past M rows"
    return out[:M]


@pytest.mark.parametrize("sizes,K,N", CASES)
@pytest.mark.parametrize("trans_b", [0, 1])
def test_fwd_bf16(sizes, K, N, trans_b):
    M, E = int(np.sum(sizes)), len(sizes)
    x = rand_bf16((M, K), 1)
    w = rand_bf16((E, N, K) if trans_b else (E, K, N), 2)
    out = bf16_fwd(sizes, K, N, x, w, trans_b)
    ref = og.gmm_fwd(to_np(x), to_np(w), sizes, trans_b=bool(trans_b))
    assert_close(to_np(out), ref, BF16_TOL, "fwd")


@pytest.mark.parametrize("sizes,K,N,kind", [
    ([128] * 8, 256, 3072, "uniform"),
    ([128, 0, 300, 7, 128, 256, 64, 141], 192, 3008, "normal"),  # last tile 128 of 192 columns
    ([128, 0, 300, 7, 128, 256, 64, 141], 192, 3008, "int"),
])
def test_fwd_bf16_weight_streaming_192_wide(sizes, K, N, kind):
    # 8 row tiles at most 256 rows per expert and w [E, K, N]: 192-wide tiles
    # take one wave (16 x 8 tiles) where 128-wide ones take two, so these
    # launches run the 192-wide, 5-stage form
    M, E = int(np.sum(sizes)), len(sizes)
    x = rand_bf16((M, K), 21, kind)
    w = rand_bf16((E, K, N), 22, kind)
    out = bf16_fwd(sizes, K, N, x, w, 0)
    ref = og.gmm_fwd(to_np(x), to_np(w), sizes, trans_b=False)
    if kind == "int":
        assert np.array_equal(to_np(out), formats.round_bf16(ref)), "integer inputs: exact"
    else:
        assert_close(to_np(out), ref, BF16_TOL, "fwd 192-wide")


@pytest.mark.parametrize("sizes,K,N", [([128] * 8, 256, 3072), ([128, 0, 300, 7, 128, 256, 64, 141], 192, 3008)])
def test_fwd_bf16_kmajor_weight_streaming_192_wide(sizes, K, N):
    # w [E, N, K] with the shapes of the 192-wide weight-streaming case: the
    # K-major 192-wide form
    M, E = int(np.sum(sizes)), len(sizes)
    x = rand_bf16((M, K), 33, "normal")
    w = rand_bf16((E, N, K), 34, "normal")
    out = bf16_fwd(sizes, K, N, x, w, 1)
    ref = og.gmm_fwd(to_np(x), to_np(w), sizes, trans_b=True)
    assert_close(to_np(out), ref, BF16_TOL, "fwd 192-wide, K-major weights")


@pytest.mark.parametrize("sizes,K,N", CASES)
def test_dgrad_bf16(sizes, K, N):
    M, E = int(np.sum(sizes)), len(sizes)
    go = rand_bf16((M, N), 3, "normal")
    w = rand_bf16((E, K, N), 4, "normal")
    gx = sentinel_bf16((M + 8, K), DEV)
    B().mgemm_dgrad(fill(sizes), B().MGEMM_BF16, go, None, w, None, gx, M, K, N, E)
    torch.cuda.synchronize()
    assert is_sentinel(gx[M:])
    assert_close(to_np(gx[:M]), og.gmm_dgrad(to_np(go), to_np(w), sizes), BF16_TOL, "dgrad")


@pytest.mark.parametrize("sizes,K,N", CASES + [([130, 0, 1, 64, 63, 200], 128, 256)])
def test_wgrad_bf16(sizes, K, N):
    M, E = int(np.sum(sizes)), len(sizes)
    x = rand_bf16((M, K), 5, "normal")
    go = rand_bf16((M, N), 6, "normal")
    gw = sentinel_bf16((E + 1, K, N), DEV)
    B().mgemm_wgrad(fill(sizes), B().MGEMM_BF16, x, None, go, None, gw, M, K, N, E)
    torch.cuda.synchronize()
    assert is_sentinel(gw[E:]), "wgrad wrote past E experts"
    ref = og.gmm_wgrad(to_np(x), to_np(go), sizes)
    got = to_np(gw[:E])
    for e in range(E):
        if sizes[e] == 0:
            assert np.all(got[e] == 0), "empty expert must get an exact zero gradient"
    assert_close(got, ref, BF16_TOL, "wgrad")


def test_integer_inputs_are_bit_exact():
    sizes, K, N = [0, 300, 1, 129, 250], 320, 520
    M, E = int(np.sum(sizes)), len(sizes)
    x = rand_bf16((M, K), 7, "int")
    w = rand_bf16((E, K, N), 8, "int")
    go = rand_bf16((M, N), 9, "int")
    args = fill(sizes)
    out = torch.empty(M, N, dtype=BF, device=DEV)
    gx = torch.empty(M, K, dtype=BF, device=DEV)
    gw = torch.empty(E, K, N, dtype=BF, device=DEV)
    B().mgemm_fwd(args, 0, 0, x, None, w, None, out, M, K, N, E)
    B().mgemm_dgrad(args, 0, go, None, w, None, gx, M, K, N, E)
    B().mgemm_wgrad(args, 0, x, None, go, None, gw, M, K, N, E)
    torch.cuda.synchronize()
    xs, ws, gs = to_np(x), to_np(w), to_np(go)
    assert np.array_equal(to_np(out), formats.round_bf16(og.gmm_fwd(xs, ws, sizes)))
    assert np.array_equal(to_np(gx), formats.round_bf16(og.gmm_dgrad(gs, ws, sizes)))
    assert np.array_equal(to_np(gw), formats.round_bf16(og.gmm_wgrad(xs, gs, sizes)))


def test_repeat_calls_identical():
    sizes, K, N = [0, 300, 1, 129, 250], 320, 520
    M, E = int(np.sum(sizes)), len(sizes)
    x, w = rand_bf16((M, K), 1), rand_bf16((E, K, N), 2)
    a = bf16_fwd(sizes, K, N, x, w, 0).clone()
    b = bf16_fwd(sizes, K, N, x, w, 0)
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))


def test_bad_status_blocks_every_gemm():
    sizes, K, N = [3, 5], 64, 64
    E, M = 2, 8
    args = new_args(E, DEV)
    B().mgemm_fill_args(torch.tensor([3, 4], dtype=torch.int64, device=DEV), E, M, args)   # sum 7 != 8
    x, w, go = rand_bf16((M, K), 1), rand_bf16((E, K, N), 2), rand_bf16((M, N), 3)
    out = sentinel_bf16((M, N), DEV)
    gx = sentinel_bf16((M, K), DEV)
    gw = sentinel_bf16((E, K, N), DEV)
    B().mgemm_fwd(args, 0, 0, x, None, w, None, out, M, K, N, E)
    B().mgemm_dgrad(args, 0, go, None, w, None, gx, M, K, N, E)
    B().mgemm_wgrad(args, 0, x, None, go, None, gw, M, K, N, E)
    torch.cuda.synchronize()
    assert B().args_status(args) == 2
    assert is_sentinel(out) and is_sentinel(gx) and is_sentinel(gw)


def test_wgrad_all_groups_empty_writes_zeros():
    E, K, N = 3, 64, 256
    args = new_args(E, DEV)
    B().mgemm_fill_args(torch.zeros(E, dtype=torch.int64, device=DEV), E, 0, args)
    gw = sentinel_bf16((E, K, N), DEV)
    dummy = torch.empty(16, K, dtype=BF, device=DEV)
    B().mgemm_wgrad(args, 0, dummy, None, dummy, None, gw, 0, K, N, E)
    torch.cuda.synchronize()
    assert (to_np(gw) == 0).all()


# ----------------------------------------------------------------- FP8 path
def quant_rows_gpu(t):
    R, C = t.shape
    q = torch.empty(R, C, dtype=torch.uint8, device=DEV)
    s = torch.empty(R, dtype=torch.float32, device=DEV)
    B().mgemm_quant_rowwise(t, q, s)
    return q, s


FP8_CASES = [
    ([15, 16, 19, 14], 128, 256),
    ([5, 0, 37, 100, 2], 256, 272),           # M = 144; group starts off 16-row boundaries
    ([0, 300, 1, 129, 250, 0, 0, 24], 320, 528),
    ([48], 512, 256),
    ([7, 0, 93, 33], 128, 144),               # M = 133: wgrad reads the padded layout, any M
]


@pytest.mark.parametrize("sizes,K,N", FP8_CASES)
def test_fp8_fwd_dgrad_wgrad(sizes, K, N):
    M, E = int(np.sum(sizes)), len(sizes)
    args = fill(sizes)
    x = rand_bf16((M, K), 21, "normal")
    go = rand_bf16((M, N), 22, "normal")
    w_nk = (rand_bf16((E, N, K), 23, "normal").float() * 0.02).to(BF)
    w_kn = w_nk.transpose(1, 2).contiguous()
    # quantize (bit-exact against the oracle)
    xq, sx = quant_rows_gpu(x)
    goq, sgo = quant_rows_gpu(go)
    wq, sw = quant_rows_gpu(w_nk.view(E * N, K))
    wdq, swd = quant_rows_gpu(w_kn.view(E * K, N))
    ld = B().mgemm_colwise_ld(M, E)
    xqt = torch.empty(K * ld, dtype=torch.uint8, device=DEV)
    goqt = torch.empty(N * ld, dtype=torch.uint8, device=DEV)
    sxc = torch.empty(E * K, dtype=torch.float32, device=DEV)
    sgoc = torch.empty(E * N, dtype=torch.float32, device=DEV)
    B().mgemm_quant_colwise_grouped(args, E, M, go, goqt, sgoc, x, xqt, sxc, ld=ld)
    torch.cuda.synchronize()
    xqt_u, goqt_u = unpad_colwise(to_np(xqt), K, ld, sizes), unpad_colwise(to_np(goqt), N, ld, sizes)
    assert (colwise_padding(to_np(xqt), K, ld, sizes) == 0).all()
    xs, gos = to_np(x), to_np(go)
    q_ref, s_ref = oq.quant_rowwise(xs)
    assert np.array_equal(to_np(xq), q_ref) and np.array_equal(to_np(sx), s_ref)
    offs = np.concatenate([[0], np.cumsum(sizes)])
    (gqt_ref, sgc_ref), (xqt_ref, sxc_ref) = oq.quant_colwise_grouped_dual(gos, xs, offs)
    assert np.array_equal(goqt_u, gqt_ref) and np.array_equal(to_np(sgoc), sgc_ref)
    assert np.array_equal(xqt_u, xqt_ref) and np.array_equal(to_np(sxc), sxc_ref)

    out = sentinel_bf16((M + 8, N), DEV)
    gx = sentinel_bf16((M + 8, K), DEV)
    gw = sentinel_bf16((E + 1, K, N), DEV)
    B().mgemm_fwd(args, B().MGEMM_FP8_E4M3, 1, xq, sx, wq, sw, out, M, K, N, E)
    B().mgemm_dgrad(args, B().MGEMM_FP8_E4M3, goq, sgo, wdq, swd, gx, M, K, N, E)
    B().mgemm_wgrad(args, B().MGEMM_FP8_E4M3, xqt, sxc, goqt, sgoc, gw, M, K, N, E, ld=ld)
    torch.cuda.synchronize()
    assert is_sentinel(out[M:]) and is_sentinel(gx[M:]) and is_sentinel(gw[E:])
    ref_f = og.gmm_fwd_fp8(to_np(xq), to_np(sx), to_np(wq).reshape(E, N, K), to_np(sw), sizes)
    ref_d = og.gmm_dgrad_fp8(to_np(goq), to_np(sgo), to_np(wdq).reshape(E, K, N), to_np(swd), sizes)
    ref_w = og.gmm_wgrad_fp8(xqt_u, to_np(sxc), goqt_u, to_np(sgoc), sizes)
    assert_close(to_np(out[:M]), ref_f, FP8_TOL, "fp8 fwd")
    assert_close(to_np(gx[:M]), ref_d, FP8_TOL, "fp8 dgrad")
    got_w = to_np(gw[:E])
    for e in range(E):
        if sizes[e] == 0:
            assert np.all(got_w[e] == 0)
    assert_close(got_w, ref_w, FP8_TOL, "fp8 wgrad")
    # the FP8 result also tracks the unquantized bf16 product (quantization error only)
    assert_close(to_np(out[:M]), og.gmm_fwd(xs, to_np(w_nk), sizes, trans_b=True), 0.1, "fp8 vs bf16 fwd")

