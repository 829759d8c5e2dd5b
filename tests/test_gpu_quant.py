"""GPU parity of the FP8 quantize kernels against oracle.quant: bytes and
scales must match bit for bit.  Includes every finite bf16 magnitude up to 448
through the cast at several power-of-two scales, ragged and empty groups, the
dual form with different widths, and strided rows."""

import numpy as np
import pytest
import torch

from oracle.quant import quant_colwise_grouped, quant_rowwise
from tests.helpers import colwise_padding, new_args, padded_offsets, to_np, unpad_colwise

pytestmark = pytest.mark.gpu
DEV = "cuda"


def B():
    from mixture_experts_grouped_gmm_gb300 import binding

    return binding


def rowwise_gpu(x, ld_out=None):
    R, C = x.shape
    ld_out = ld_out or ((C + 15) // 16) * 16
    out = torch.full((R, ld_out), 0xAB, dtype=torch.uint8, device=DEV)
    sc = torch.empty(R, dtype=torch.float32, device=DEV)
    B().mgemm_quant_rowwise(x, out, sc)
    torch.cuda.synchronize()
    return out, sc


def check_rowwise(x):
    out, sc = rowwise_gpu(x)
    C = x.shape[1]
    q, s = quant_rowwise(to_np(x))
    assert np.array_equal(to_np(out)[:, :C], q)
    assert np.array_equal(to_np(sc), s)
    if out.shape[1] > C:
        assert (to_np(out)[:, C:] == 0xAB).all()      # nothing written past C


@pytest.mark.parametrize("R,C", [(1, 8), (64, 128), (33, 1408), (7, 2048), (5, 5120), (9, 6152), (3, 8200),
                                 (300, 256), (2, 4096)])
def test_rowwise_shapes(R, C):
    g = torch.Generator(device=DEV).manual_seed(R * 1000 + C)
    x = torch.randn(R, C, generator=g, device=DEV) * torch.exp2(torch.randint(-20, 20, (R, 1), generator=g,
                                                                               device=DEV).float())
    x = x.to(torch.bfloat16)
    x[0] = 0                                            # all-zero row: scale 2^48, codes 0
    check_rowwise(x)


def test_rowwise_strided_rows():
    g = torch.Generator(device=DEV).manual_seed(1)
    big = torch.randn(40, 1000, generator=g, device=DEV).to(torch.bfloat16)
    x = big[:, :768]                                    # row stride 1000 elements
    out = torch.full((40, 800), 0xAB, dtype=torch.uint8, device=DEV)
    sc = torch.empty(40, dtype=torch.float32, device=DEV)
    B().mgemm_quant_rowwise(x, out[:, :768], sc)
    torch.cuda.synchronize()
    q, s = quant_rowwise(to_np(x))
    assert np.array_equal(to_np(out)[:, :768], q) and (to_np(out)[:, 768:] == 0xAB).all()
    assert np.array_equal(to_np(sc), s)


@pytest.mark.parametrize("anchor", [448.0, 1.0, 2.0 ** -7, 2.0 ** 20])
def test_cast_every_bf16_magnitude(anchor):
    # every finite bf16 value v with |v| <= anchor, one row per 255 values plus
    # the anchor, so the row scale is pow2floor(448 / anchor) and the cast sees v * s
    bits = torch.from_numpy(np.arange(65536, dtype=np.uint16).view(np.int16))
    v = bits.view(torch.bfloat16).float()
    v = v[torch.isfinite(v) & (v.abs() <= anchor)]
    n = (v.numel() + 254) // 255
    rows = torch.full((n * 255,), 0.0)
    rows[: v.numel()] = v
    x = torch.cat([rows.view(n, 255), torch.full((n, 1), anchor)], dim=1)
    x = torch.cat([x, torch.zeros(n, 256)], dim=1).to(torch.bfloat16).to(DEV)   # C = 512
    check_rowwise(x)


def colwise_case(sizes, C1, C2=None, seed=0):
    E = len(sizes)
    M = int(np.sum(sizes))
    g = torch.Generator(device=DEV).manual_seed(seed)
    a1 = (torch.randn(M, C1, generator=g, device=DEV) * 3).to(torch.bfloat16)
    gs = torch.tensor(sizes, dtype=torch.int64, device=DEV)
    args = new_args(E, DEV)
    B().mgemm_fill_args(gs, E, M, args)
    ld = B().mgemm_colwise_ld(M, E)
    o1 = torch.full((C1 * ld,), 0xAB, dtype=torch.uint8, device=DEV)
    s1 = torch.full((E * C1,), -1.0, dtype=torch.float32, device=DEV)
    a2 = o2 = s2 = None
    if C2:
        a2 = (torch.randn(M, C2, generator=g, device=DEV) * 1e-3).to(torch.bfloat16)
        o2 = torch.full((C2 * ld,), 0xAB, dtype=torch.uint8, device=DEV)
        s2 = torch.full((E * C2,), -1.0, dtype=torch.float32, device=DEV)
    B().mgemm_quant_colwise_grouped(args, E, M, a1, o1, s1, a2, o2, s2, ld=ld)
    torch.cuda.synchronize()
    offs = np.concatenate([[0], np.cumsum(sizes)])
    used = padded_offsets(sizes)[-1]
    q1, r1 = quant_colwise_grouped(to_np(a1), offs)
    assert np.array_equal(to_np(s1), r1)
    assert np.array_equal(unpad_colwise(to_np(o1), C1, ld, sizes), q1)
    assert (colwise_padding(to_np(o1), C1, ld, sizes) == 0).all(), "padding must hold zero codes"
    assert (to_np(o1).reshape(C1, ld)[:, used:] == 0xAB).all(), "bytes past the last group are not written"
    if C2:
        q2, r2 = quant_colwise_grouped(to_np(a2), offs)
        assert np.array_equal(to_np(s2), r2)
        assert np.array_equal(unpad_colwise(to_np(o2), C2, ld, sizes), q2)
        assert (colwise_padding(to_np(o2), C2, ld, sizes) == 0).all()


@pytest.mark.parametrize("sizes,C1,C2", [
    ([64], 64, None),
    ([10, 0, 30, 24], 128, None),          # M = 64, empty group
    ([7, 0, 93], 72, None),                # M = 100: not a multiple of 16
    ([1, 200, 0, 55, 0, 0, 4], 200, 136),  # dual, different widths
    ([300, 301, 3, 0, 420], 64, 64),       # dual, same widths, groups across 128-row chunks
    ([0, 0, 0, 16], 8, 8),
])
def test_colwise(sizes, C1, C2):
    colwise_case(sizes, C1, C2, seed=len(sizes) * 7 + C1)


def test_colwise_large_groups_deepseek_like():
    rng = np.random.default_rng(3)
    sizes = rng.integers(0, 2000, 16)
    sizes[[2, 9]] = 0
    sizes[-1] += (16 - sizes.sum() % 16) % 16
    colwise_case(sizes.tolist(), 256, 96, seed=11)


def test_colwise_group_over_many_segments():
    # one group of 20000 rows (79 boxes of 256 rows) over 24 column blocks of
    # two tensors, next to tiny and empty groups
    colwise_case([20000, 3, 0, 4997], 1024, 512, seed=5)


def test_colwise_split_groups_every_chunk_shape():
    # Groups of more than 5 boxes (1280 rows) are split across the CTAs of a
    # cluster: 6 boxes over 8 CTAs (some CTAs read none), 9, 12 (every chunk
    # stays in the ring), 47 (chunks of 5 and 6 boxes: some are read twice),
    # next to small and empty groups, over two tensors of different widths.
    colwise_case([1281, 12000, 0, 2100, 1300, 3000, 17, 250], 200, 136, seed=21)


def test_colwise_status_blocks_writes():
    E, M, C = 3, 48, 64
    gs = torch.tensor([16, -1, 33], dtype=torch.int64, device=DEV)
    args = new_args(E, DEV)
    B().mgemm_fill_args(gs, E, M, args)
    a = torch.randn(M, C, device=DEV).to(torch.bfloat16)
    ld = B().mgemm_colwise_ld(M, E)
    o = torch.full((C * ld,), 0xAB, dtype=torch.uint8, device=DEV)
    s = torch.full((E * C,), -1.0, device=DEV)
    B().mgemm_quant_colwise_grouped(args, E, M, a, o, s)
    torch.cuda.synchronize()
    assert (to_np(o) == 0xAB).all() and (to_np(s) == -1.0).all()


@pytest.mark.parametrize("sizes", [[300, 0, 77, 1000, 5, 130], [300, 0, 77, 3000, 5, 1500]])
def test_colwise_repeated_on_one_args_block(sizes):
    # the work counter in the args header is handed back at 0, so a second call
    # with the same args block sees every item again (with and without groups
    # split across CTAs)
    E, M = len(sizes), int(np.sum(sizes))
    gs = torch.tensor(sizes, dtype=torch.int64, device=DEV)
    args = new_args(E, DEV)
    B().mgemm_fill_args(gs, E, M, args)
    offs = np.concatenate([[0], np.cumsum(sizes)])
    for rep in range(3):
        a = (torch.randn(M, 136, generator=torch.Generator(device=DEV).manual_seed(rep), device=DEV)).to(torch.bfloat16)
        ld = B().mgemm_colwise_ld(M, E)
        o = torch.full((136 * ld,), 0xAB, dtype=torch.uint8, device=DEV)
        s = torch.full((E * 136,), -1.0, dtype=torch.float32, device=DEV)
        B().mgemm_quant_colwise_grouped(args, E, M, a, o, s)
        torch.cuda.synchronize()
        q, r = quant_colwise_grouped(to_np(a), offs)
        assert np.array_equal(unpad_colwise(to_np(o), 136, ld, sizes), q) and np.array_equal(to_np(s), r)
        assert int(args[12:16].view(torch.int32).item()) == 0


@pytest.mark.parametrize("sizes,K", [([0, 1, 0, 0], 5120), ([3, 0, 2] + [0] * 125, 5120), ([40, 0, 88], 2048),
                                     ([7] * 300, 272), ([0, 0], 128)])
def test_fill_args_quant_rowwise_fused_equals_the_two_calls(sizes, K):
    # one launch: the args block equals mgemm_fill_args' byte for byte, the codes
    # and scales equal mgemm_quant_rowwise's and the oracle's
    from oracle import quant as oq

    E, M = len(sizes), int(np.sum(sizes))
    gs = torch.tensor(sizes, dtype=torch.int64, device=DEV)
    x = (torch.randn(max(M, 1), K, device=DEV) * 3.0).to(torch.bfloat16)[:M]
    a1 = torch.zeros(B().mgemm_args_bytes(E), dtype=torch.uint8, device=DEV)
    a2 = torch.full_like(a1, 0xA5)
    q1 = torch.empty(M, K, dtype=torch.uint8, device=DEV)
    s1 = torch.empty(M, dtype=torch.float32, device=DEV)
    q2, s2 = torch.empty_like(q1), torch.empty_like(s1)
    B().mgemm_fill_args(gs, E, M, a1)
    if M:
        B().mgemm_quant_rowwise(x, q1, s1)
    B().mgemm_fill_args_quant_rowwise(gs, E, M, a2, x, q2, s2)
    torch.cuda.synchronize()
    from tests.helpers import parse_args

    p1, p2 = parse_args(a1, E), parse_args(a2, E)
    na = p1["n_active"]
    for k in ("active",):                      # defined for the n_active non-empty groups
        p1[k], p2[k] = p1[k][:na], p2[k][:na]
    for k in ("mtile_start", "ptile_start"):   # and their prefix ends
        p1[k], p2[k] = p1[k][:na + 1], p2[k][:na + 1]
    assert p1 == p2
    assert torch.equal(q1, q2) and torch.equal(s1, s2)
    if M:
        qr, sr = oq.quant_rowwise(to_np(x))
        assert np.array_equal(to_np(q2), qr) and np.array_equal(to_np(s2), sr)
