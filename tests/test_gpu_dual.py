"""GPU checks of mgemm_dgrad_wgrad: both gradients of the bf16 grouped GEMM in
one call.

Its outputs must equal those of mgemm_dgrad and mgemm_wgrad bit for bit
(the one-launch form runs the same tiles with the same contraction order on
other CTAs), whether the sizes take the one-launch form or the two calls in
turn; and they are compared with the oracle at the bf16 tolerance.  Guard rows
past both outputs must stay untouched."""

import numpy as np
import pytest
import torch

from oracle import gmm as og
from tests.helpers import BF16_TOL, assert_close, is_sentinel, new_args, sentinel_bf16, to_np

pytestmark = pytest.mark.gpu
DEV = "cuda"
BF = torch.bfloat16


def B():
    from mixture_experts_grouped_gmm_gb300 import binding

    return binding


def rand_bf16(shape, seed):
    g = torch.Generator(device=DEV).manual_seed(seed)
    return torch.randn(shape, generator=g, device=DEV).to(BF)


def fill(sizes, E, M):
    args = new_args(E, DEV)
    B().mgemm_fill_args(torch.as_tensor(sizes, dtype=torch.int64, device=DEV), E, M, args)
    return args


def run_both(sizes, K, N, seed=0):
    M, E = int(np.sum(sizes)), len(sizes)
    x = rand_bf16((M, K), seed)
    w = rand_bf16((E, K, N), seed + 1)
    go = rand_bf16((M, N), seed + 2)
    args = fill(sizes, E, M)
    gx = sentinel_bf16((M + 8, K), DEV)
    gw = sentinel_bf16((E + 1, K, N), DEV)
    B().mgemm_dgrad_wgrad(args, go, w, x, gx, gw, M, K, N, E)
    gx_ref = torch.empty(M, K, dtype=BF, device=DEV)
    gw_ref = torch.empty(E, K, N, dtype=BF, device=DEV)
    B().mgemm_dgrad(args, B().MGEMM_BF16, go, None, w, None, gx_ref, M, K, N, E)
    B().mgemm_wgrad(args, B().MGEMM_BF16, x, None, go, None, gw_ref, M, K, N, E)
    torch.cuda.synchronize()
    assert B().args_status(args) == 0
    assert is_sentinel(gx[M:]), "grad_x written past M rows"
    assert is_sentinel(gw[E:]), "grad_w written past E experts"
    assert torch.equal(gx[:M].view(torch.int16), gx_ref.view(torch.int16)), "grad_x differs from mgemm_dgrad"
    assert torch.equal(gw[:E].view(torch.int16), gw_ref.view(torch.int16)), "grad_w differs from mgemm_wgrad"
    return x, w, go, gx[:M], gw[:E]


# sizes, K, N; every case here is in the memory-bound regime (groups of at
# most 256 rows on average) and the size model takes the one-launch form (the
# test asserts that as well); dgrad tiles 64, 128 and 256 wide
DUAL_CASES = [
    ([15, 16, 19, 14], 512, 256),                     # tiny: few tiles, most CTAs idle
    ([0, 300, 1, 129, 250], 2048, 520),               # ragged groups, an empty and a one-row group, N % 256 != 0
    ([128] * 8, 2048, 1536),                          # GRIN-like, smaller
    ([5, 0, 0, 0, 0, 0, 3, 0], 768, 256),             # sparse rows among many groups
    ([200, 0, 57, 311, 64, 90, 0, 170], 1280, 776),   # K % 256 != 0, N % 8 == 0 only
]


@pytest.mark.parametrize("sizes,K,N", DUAL_CASES)
def test_dgrad_wgrad_one_launch(sizes, K, N):
    M, E = int(np.sum(sizes)), len(sizes)
    split = B().mgemm_dgrad_wgrad_split(M, K, N, E)
    assert 0 < split < B().mgemm_num_sms(), f"expected the one-launch form, split {split}"
    x, w, go, gx, gw = run_both(sizes, K, N)
    ref_x = og.gmm_dgrad(to_np(go), to_np(w), sizes)
    assert_close(to_np(gx), ref_x, BF16_TOL, "dgrad")
    ref_w = og.gmm_wgrad(to_np(x), to_np(go), sizes)
    for e in range(E):
        if sizes[e] == 0:
            assert np.all(to_np(gw[e]) == 0), "empty expert must get an exact zero gradient"
    assert_close(to_np(gw), ref_w, BF16_TOL, "wgrad")


def test_dgrad_wgrad_two_calls_when_groups_are_large():
    # 1024 rows per group: compute-bound GEMMs, the two calls run in turn
    sizes, K, N = [1024, 1024], 256, 256
    M, E = 2048, 2
    assert B().mgemm_dgrad_wgrad_split(M, K, N, E) == 0
    x, w, go, gx, gw = run_both(sizes, K, N, seed=5)
    assert_close(to_np(gx), og.gmm_dgrad(to_np(go), to_np(w), sizes), BF16_TOL, "dgrad")
    assert_close(to_np(gw), og.gmm_wgrad(to_np(x), to_np(go), sizes), BF16_TOL, "wgrad")


def test_dgrad_wgrad_no_rows():
    E, K, N = 3, 128, 256
    args = fill([0, 0, 0], E, 0)
    gw = sentinel_bf16((E, K, N), DEV)
    B().mgemm_dgrad_wgrad(args, None, sentinel_bf16((E, K, N), DEV), None, None, gw, 0, K, N, E)
    torch.cuda.synchronize()
    assert (to_np(gw) == 0).all()


def test_dgrad_wgrad_split_at_grin_size():
    # GRIN-MoE gmm (M = 1024, K = 4096, N = 6400, E = 8): 128 dgrad tiles, two per dgrad CTA
    split = B().mgemm_dgrad_wgrad_split(1024, 4096, 6400, 8)
    assert split == 64, split
    # predicted gains below 6% take the two calls (measured there: the one launch 6% / 1% slower)
    assert B().mgemm_dgrad_wgrad_split(1024, 1024, 6400, 8) == 0
    assert B().mgemm_dgrad_wgrad_split(4096, 2048, 1536, 16) == 0


def test_dgrad_wgrad_bad_status_writes_nothing():
    sizes, K, N = [3, 5], 256, 256
    E, M = 2, 8
    args = new_args(E, DEV)
    B().mgemm_fill_args(torch.tensor(sizes[:1] + [4], dtype=torch.int64, device=DEV), E, M, args)  # sum 7 != 8
    x, w, go = rand_bf16((M, K), 1), rand_bf16((E, K, N), 2), rand_bf16((M, N), 3)
    assert B().mgemm_dgrad_wgrad_split(M, K, N, E) > 0
    gx = sentinel_bf16((M, K), DEV)
    gw = sentinel_bf16((E, K, N), DEV)
    B().mgemm_dgrad_wgrad(args, go, w, x, gx, gw, M, K, N, E)
    torch.cuda.synchronize()
    assert B().args_status(args) == 2
    assert is_sentinel(gx) and is_sentinel(gw)
