"""GPU parity of the MXFP8 path against oracle.mx: the block quantizer bit for
bit (codes and e8m0 bytes), and the block-scaled grouped GEMM (forward, and
dgrad through the same call) element by element, over ragged and empty groups,
contractions that are not a multiple of the four-block scale rows, partial
output tiles, the DeepSeek-sized step on sampled rows, and CUDA-graph replay
with new group sizes.

GEMM tolerance: the oracle contracts the same decoded values in float64; the
kernel accumulates exact e4m3 x e4m3 products scaled by powers of two in fp32
and rounds once to bf16.  Per element |out - ref| <= 2^-8 |ref| (bf16 RNE,
8 significant bits) + 2^-9 max|ref| (fp32 accumulation order over K <= 2048)."""

import numpy as np
import pytest
import torch

from oracle.mx import decode_mx, gmm_fwd_mx, gmm_wgrad_mx, quant_mx_colwise_grouped, quant_mx_rows
from tests.helpers import colwise_padding, new_args, padded_offsets, to_np, unpad_colwise

pytestmark = pytest.mark.gpu
DEV = "cuda"


def B():
    from mixture_experts_grouped_gmm_gb300 import binding

    return binding


def blocky(R, K, seed, lo=-12, hi=12):
    """bf16 [R, K] on the device whose 32-element blocks span 2^lo .. 2^hi."""
    g = torch.Generator(device=DEV).manual_seed(seed)
    base = torch.randn(R, K, generator=g, device=DEV)
    sc = torch.exp2(torch.randint(lo, hi, (R, K // 32), generator=g, device=DEV).float())
    return (base * sc.repeat_interleave(32, dim=1)).to(torch.bfloat16)


def quant_gpu(x):
    R, C = x.shape
    ld = B().mx_ld_sf(C)
    q = torch.full((R, C), 0xAB, dtype=torch.uint8, device=DEV)
    sf = torch.full((R, ld), 0xCD, dtype=torch.uint8, device=DEV)
    B().mgemm_quant_mx(x, q, sf)
    return q, sf


def check_quant(x):
    q, sf = quant_gpu(x)
    torch.cuda.synchronize()
    C = x.shape[1]
    qo, so = quant_mx_rows(to_np(x))
    assert np.array_equal(to_np(q), qo)
    assert np.array_equal(to_np(sf)[:, :C // 32], so)
    assert (to_np(sf)[:, C // 32:] == 0xCD).all()        # nothing written past C / 32


@pytest.mark.parametrize("R,C", [(1, 32), (37, 128), (64, 1408), (257, 2048), (3, 5120), (9, 96)])
def test_quant_mx_shapes(R, C):
    x = blocky(R, C, seed=R * 7 + C)
    x[0, :32] = 0                                        # an all-zero block: byte 79, codes 0
    check_quant(x)


def test_quant_mx_extremes_and_strided_rows():
    g = torch.Generator(device=DEV).manual_seed(3)
    big = torch.randn(16, 800, generator=g, device=DEV)
    big[0, :32] = 3.0e38                                # near the bf16 maximum
    big[1, 32:64] = 1e-38                               # subnormal-range magnitudes
    big[2, :] = 0.0
    big[3, 64:96] = -448.0
    x = big.to(torch.bfloat16)[:, :640]                 # row stride 800 elements
    check_quant(x)


def gemm_case(sizes, K, N, seed):
    # GPU: quantize + GEMM on the device; reference: the oracle's quantize of
    # the same bf16 inputs, then its GEMM (the codes agree bit for bit)
    E, M = len(sizes), sum(sizes)
    x = blocky(M, K, seed)
    w = blocky(E * N, K, seed + 1)
    xq, sx = quant_gpu(x)
    wq, sw = quant_gpu(w)
    gs = torch.tensor(sizes, dtype=torch.int64, device=DEV)
    args = new_args(E, DEV)
    B().mgemm_fill_args(gs, E, M, args)
    out = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device=DEV)
    B().mgemm_fwd_mx(args, xq, sx, wq.view(E, N, K), sw, out, M, K, N, E)
    torch.cuda.synchronize()
    qx, ex = quant_mx_rows(to_np(x))
    qw, ew = quant_mx_rows(to_np(w))
    assert np.array_equal(to_np(xq), qx) and np.array_equal(to_np(wq), qw)
    ref = gmm_fwd_mx(qx, ex, qw.reshape(E, N, K), ew.reshape(E, N, K // 32), sizes)
    return to_np(out), ref


def assert_mx_close(got, ref, what=""):
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    m = np.max(np.abs(ref)) if ref.size else 0.0
    bad = np.abs(got - ref) > np.abs(ref) * 2.0 ** -8 + m * 2.0 ** -9
    assert not bad.any(), f"{what}: {int(bad.sum())} elements off, first at {np.argwhere(bad)[0]}"


@pytest.mark.parametrize("sizes,K,N", [
    ([128], 128, 128),
    ([100, 0, 300, 57], 512, 384),
    ([1, 2, 3, 250, 0, 129], 1408, 200),       # K % 512 != 0; a partial last column tile
    ([0, 0, 70], 2048, 1408),
    ([33] * 12, 640, 136),
    ([300, 0, 700, 260], 512, 400),            # groups averaging >= 256 rows: CTA pairs, partial pair tiles
    ([1024], 384, 192),                        # E = 1 on CTA pairs, one column tile
    ([2500, 0, 2400, 4828], 256, 384),         # large groups, two 192-wide column tiles
])
def test_fwd_mx_parity(sizes, K, N):
    got, ref = gemm_case(sizes, K, N, seed=len(sizes) * 100 + K + N)
    assert_mx_close(got, ref, f"sizes={sizes} K={K} N={N}")


def test_dgrad_mx_through_fwd():
    # grad_x = grad_out . w[e]^T: grad_out [M, N] quantized along N, w stored
    # [E, K, N] quantized along N, i.e. the forward call with the roles of K, N swapped
    sizes, K, N = [90, 0, 200], 256, 384
    E, M = len(sizes), sum(sizes)
    go = blocky(M, N, 11)
    w_kn = blocky(E * K, N, 12)
    goq, sgo = quant_gpu(go)
    wq, sw = quant_gpu(w_kn)
    args = new_args(E, DEV)
    B().mgemm_fill_args(torch.tensor(sizes, dtype=torch.int64, device=DEV), E, M, args)
    gx = torch.empty(M, K, dtype=torch.bfloat16, device=DEV)
    B().mgemm_fwd_mx(args, goq, sgo, wq.view(E, K, N), sw, gx, M, N, K, E)
    torch.cuda.synchronize()
    qg, eg = quant_mx_rows(to_np(go))
    qw, ew = quant_mx_rows(to_np(w_kn))
    ref = gmm_fwd_mx(qg, eg, qw.reshape(E, K, N), ew.reshape(E, K, N // 32), sizes)
    assert_mx_close(to_np(gx), ref, "dgrad")


def test_fwd_mx_deepseek_size_sampled_rows():
    from mixture_experts_grouped_gmm_gb300 import workloads

    d = workloads.deepseek(device=DEV, T=16384, with_weights=False)
    M, K, N, E = d["M"], d["K"], d["N"], d["E"]
    x = d["x"]
    w = blocky(E * N, K, 5, lo=-4, hi=4)
    xq, sx = quant_gpu(x)
    wq, sw = quant_gpu(w)
    args = new_args(E, DEV)
    B().mgemm_fill_args(d["group_sizes"], E, M, args)
    out = torch.empty(M, N, dtype=torch.bfloat16, device=DEV)
    B().mgemm_fwd_mx(args, xq, sx, wq.view(E, N, K), sw, out, M, K, N, E)
    torch.cuda.synchronize()
    sizes = d["group_sizes"].cpu().numpy()
    off = np.concatenate([[0], np.cumsum(sizes)])
    rng = np.random.default_rng(0)
    rows = np.unique(np.concatenate([rng.integers(0, M, 48), off[1:-1][sizes[1:] > 0], [M - 1]]))
    xs = decode_mx(*quant_mx_rows(to_np(x[rows])))
    got = to_np(out[rows])
    experts = np.searchsorted(off, rows, side="right") - 1
    for e in np.unique(experts):
        we = decode_mx(*quant_mx_rows(to_np(w[e * N:(e + 1) * N])))
        sel = experts == e
        assert_mx_close(got[sel], xs[sel] @ we.T, f"rows {rows[sel][:4]} (expert {e})")


def test_fwd_mx_graph_replays_with_new_sizes():
    E, M, K, N = 5, 600, 384, 256
    gs = torch.zeros(E, dtype=torch.int64, device=DEV)
    x = blocky(M, K, 21)
    w = blocky(E * N, K, 22)
    xq = torch.empty(M, K, dtype=torch.uint8, device=DEV)
    sx = torch.empty(M, B().mx_ld_sf(K), dtype=torch.uint8, device=DEV)
    wq, sw = quant_gpu(w)
    args = new_args(E, DEV)
    out = torch.empty(M, N, dtype=torch.bfloat16, device=DEV)

    def step():
        B().mgemm_fill_args(gs, E, M, args)
        B().mgemm_quant_mx(x, xq, sx)
        B().mgemm_fwd_mx(args, xq, sx, wq.view(E, N, K), sw, out, M, K, N, E)

    gs.copy_(torch.tensor([600, 0, 0, 0, 0]))
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        step()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step()
    for sizes in ([100, 200, 0, 250, 50], [0, 0, 0, 0, 600], [1, 1, 1, 1, 596]):
        gs.copy_(torch.tensor(sizes))
        graph.replay()
        torch.cuda.synchronize()
        qx, ex = quant_mx_rows(to_np(x))
        qw, ew = quant_mx_rows(to_np(w))
        ref = gmm_fwd_mx(qx, ex, qw.reshape(E, N, K), ew.reshape(E, N, K // 32), sizes)
        assert_mx_close(to_np(out), ref, f"replay {sizes}")


def rowblocky(M, C, seed, lo=-10, hi=10):
    """bf16 [M, C] on the device whose 32-row runs of each column span 2^lo .. 2^hi."""
    g = torch.Generator(device=DEV).manual_seed(seed)
    base = torch.randn(M, C, generator=g, device=DEV)
    sc = torch.exp2(torch.randint(lo, hi, (M // 32 + 1, C), generator=g, device=DEV).float())
    return (base * sc.repeat_interleave(32, dim=0)[:M]).to(torch.bfloat16)


def colwise_mx_gpu(xs, sizes):
    E, M = len(sizes), sum(sizes)
    args = new_args(E, DEV)
    B().mgemm_fill_args(torch.tensor(sizes, dtype=torch.int64, device=DEV), E, M, args)
    ld = B().mgemm_colwise_ld(M, E)
    outs = [torch.full((x.shape[1] * ld,), 0xAB, dtype=torch.uint8, device=DEV) for x in xs]
    sfs = [torch.full((ld // 128 * x.shape[1] * 4,), 0xCD, dtype=torch.uint8, device=DEV) for x in xs]
    if len(xs) == 2:
        B().mgemm_quant_colwise_mx(args, E, M, xs[0], outs[0], sfs[0], xs[1], outs[1], sfs[1], ld)
    else:
        B().mgemm_quant_colwise_mx(args, E, M, xs[0], outs[0], sfs[0], ld=ld)
    torch.cuda.synchronize()
    return args, ld, outs, sfs


def check_colwise_mx(x, sizes, out, sf, ld):
    C = x.shape[1]
    off = np.concatenate([[0], np.cumsum(sizes)])
    qo, so = quant_mx_colwise_grouped(to_np(x), off)
    assert np.array_equal(unpad_colwise(to_np(out), C, ld, sizes), qo)
    assert not colwise_padding(to_np(out), C, ld, sizes).any()          # padding holds zero codes
    sfv = to_np(sf).reshape(ld // 128, C, 4)
    po = padded_offsets(sizes)
    for g, m in enumerate(sizes):
        for b in range(so[g].shape[1]):
            r = po[g] + 32 * b
            assert np.array_equal(sfv[r // 128, :, (r % 128) // 32], so[g][:, b]), (g, b)


@pytest.mark.parametrize("sizes,C1,C2", [
    ([100, 0, 300, 57], 64, 0),
    ([1, 2, 3, 250, 0, 129], 136, 200),
    ([0, 0, 70], 2048, 1408),
    ([32] * 9, 8, 24),
])
def test_quant_colwise_mx(sizes, C1, C2):
    M = sum(sizes)
    xs = [rowblocky(M, C1, C1 + M)] + ([rowblocky(M, C2, C2 + M + 1)] if C2 else [])
    _, ld, outs, sfs = colwise_mx_gpu(xs, sizes)
    for x, o, f in zip(xs, outs, sfs):
        check_colwise_mx(x, sizes, o, f, ld)


@pytest.mark.parametrize("sizes,K,N", [
    ([100, 0, 300, 57], 128, 192),
    ([1, 2, 3, 250, 0, 129], 256, 400),
    ([0, 0, 700], 384, 64),
    ([33] * 12, 144, 208),
])
def test_wgrad_mx_parity(sizes, K, N):
    E, M = len(sizes), sum(sizes)
    x = rowblocky(M, K, 31 + K)
    go = rowblocky(M, N, 32 + N)
    args, ld, (xq, gq), (sx, sg) = colwise_mx_gpu([x, go], sizes)
    gw = torch.full((E, K, N), float("nan"), dtype=torch.bfloat16, device=DEV)
    B().mgemm_wgrad_mx(args, xq, sx, gq, sg, gw, M, K, N, E, ld)
    torch.cuda.synchronize()
    off = np.concatenate([[0], np.cumsum(sizes)])
    qx, ex = quant_mx_colwise_grouped(to_np(x), off)
    qg, eg = quant_mx_colwise_grouped(to_np(go), off)
    ref = gmm_wgrad_mx(qx, ex, qg, eg, sizes)
    got = to_np(gw)
    for e in range(E):
        assert_mx_close(got[e], ref[e], f"expert {e} (m = {sizes[e]})")


def test_mx_step_deepseek_size_sampled():
    # the MXFP8 backward on the DeepSeek routing: dual colwise MX of (grad_out,
    # x) and the wgrad; checked on sampled columns of every group
    from mixture_experts_grouped_gmm_gb300 import workloads

    d = workloads.deepseek(device=DEV, T=16384, with_weights=False)
    M, K, N, E = d["M"], d["K"], d["N"], d["E"]
    sizes = d["group_sizes"].cpu().numpy().tolist()
    x, go = d["x"], d["grad_out"]
    args, ld, (gq, xq), (sg, sx) = colwise_mx_gpu([go, x], sizes)
    gw = torch.empty(E, K, N, dtype=torch.bfloat16, device=DEV)
    B().mgemm_wgrad_mx(args, xq, sx, gq, sg, gw, M, K, N, E, ld)
    torch.cuda.synchronize()
    off = np.concatenate([[0], np.cumsum(sizes)])
    rng = np.random.default_rng(1)
    kc = np.sort(rng.choice(K, 12, replace=False))
    nc = np.sort(rng.choice(N, 12, replace=False))
    qx, ex = quant_mx_colwise_grouped(to_np(x[:, kc]), off)
    qg, eg = quant_mx_colwise_grouped(to_np(go[:, nc]), off)
    # the GPU's codes of the sampled columns, bit for bit
    assert np.array_equal(unpad_colwise(to_np(xq), K, ld, sizes)[kc], qx)
    assert np.array_equal(unpad_colwise(to_np(gq), N, ld, sizes)[nc], qg)
    ref = gmm_wgrad_mx(qx, ex, qg, eg, sizes)
    got = to_np(gw[:, torch.as_tensor(kc, device=DEV)][:, :, torch.as_tensor(nc, device=DEV)])
    for e in range(E):
        assert_mx_close(got[e], ref[e], f"expert {e}")


@pytest.mark.parametrize("sizes,K,N", [
    ([5], 128, 8),                               # one tile, N = 8 (one 128-wide tile, mostly outside N)
    ([3, 0, 1, 2] * 64, 256, 136),               # 256 experts with one to three rows or none
    ([0, 0, 0, 513], 640, 64),
])
def test_fwd_mx_edges(sizes, K, N):
    got, ref = gemm_case(sizes, K, N, seed=len(sizes) + K + N)
    assert_mx_close(got, ref, f"sizes={sizes[:6]}.. K={K} N={N}")


@pytest.mark.parametrize("sizes,K,N", [
    ([7, 0, 33], 16, 16),                        # the smallest K and N
    ([1, 2, 3, 0] * 64, 32, 48),                 # 256 experts, tiny groups
    ([0, 0, 0, 0, 97], 128, 192),                # a single non-empty expert
])
def test_wgrad_mx_edges(sizes, K, N):
    E, M = len(sizes), sum(sizes)
    x = rowblocky(M, K, 41 + K)
    go = rowblocky(M, N, 42 + N)
    args, ld, (xq, gq), (sx, sg) = colwise_mx_gpu([x, go], sizes)
    gw = torch.full((E, K, N), float("nan"), dtype=torch.bfloat16, device=DEV)
    B().mgemm_wgrad_mx(args, xq, sx, gq, sg, gw, M, K, N, E, ld)
    torch.cuda.synchronize()
    off = np.concatenate([[0], np.cumsum(sizes)])
    qx, ex = quant_mx_colwise_grouped(to_np(x), off)
    qg, eg = quant_mx_colwise_grouped(to_np(go), off)
    ref = gmm_wgrad_mx(qx, ex, qg, eg, sizes)
    got = to_np(gw)
    for e in range(E):
        if sizes[e] == 0:
            assert not got[e].any(), f"expert {e}: empty group must give zeros"
        else:
            assert_mx_close(got[e], ref[e], f"expert {e}")


def test_wgrad_mx_no_rows_writes_zeros():
    E, K, N = 3, 128, 192
    args = new_args(E, DEV)
    B().mgemm_fill_args(torch.zeros(E, dtype=torch.int64, device=DEV), E, 0, args)
    gw = torch.full((E, K, N), float("nan"), dtype=torch.bfloat16, device=DEV)
    B().mgemm_wgrad_mx(args, None, None, None, None, gw, 0, K, N, E, 0)
    torch.cuda.synchronize()
    assert not gw.float().any()
