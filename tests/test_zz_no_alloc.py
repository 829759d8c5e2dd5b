"""The forward entry point for callers that cannot allocate device memory.

mgemm_fwd_noalloc keeps the args block (the tile schedule derived from the
group sizes) in a static device array inside the library, so a caller that may
not call cudaMalloc -- code running inside another framework's launch callback,
a loop where an allocation could stall the device, a runtime with a fixed
workspace -- only passes inputs and the output.  These tests call it through
the C ABI twice in a row with different problems (the second with fewer
experts, so stale contents of the shared array would show) and compare each
result with the regular path: a caller-allocated args block filled by
mgemm_fill_args and passed to mgemm_fwd.  This file is collected last."""

import ctypes

import numpy as np
import pytest
import torch

from tests.helpers import BF16_TOL, assert_close, new_args, to_np

DEV = "cuda"
BF = torch.bfloat16


@pytest.fixture(scope="module", autouse=True)
def built_library():
    from mixture_experts_grouped_gmm_gb300 import build

    build.build()


def B():
    from mixture_experts_grouped_gmm_gb300 import binding

    return binding


def rand_bf16(shape, seed):
    g = torch.Generator(device=DEV).manual_seed(seed)
    return torch.randn(shape, generator=g, device=DEV).to(BF)


def regular_fwd(gs, x, w, trans_b, M, K, N, E):
    args = new_args(E, DEV)
    B().mgemm_fill_args(gs, E, M, args)
    out = torch.empty(M, N, dtype=BF, device=DEV)
    B().mgemm_fwd(args, B().MGEMM_BF16, trans_b, x, None, w, None, out, M, K, N, E)
    return out


@pytest.mark.gpu
def test_noalloc_forward_matches_regular_path_twice():
    cases = [
        ([0, 300, 1, 129, 250, 64, 0, 40], 320, 520, 0),   # E = 8, w [E, K, N]
        ([5, 0, 77, 130, 2], 192, 264, 1),                 # E = 5, w [E, N, K]
    ]
    for i, (sizes, K, N, trans_b) in enumerate(cases):
        E, M = len(sizes), int(np.sum(sizes))
        gs = torch.tensor(sizes, dtype=torch.int64, device=DEV)
        x = rand_bf16((M, K), 10 + i)
        w = rand_bf16((E, N, K) if trans_b else (E, K, N), 20 + i)
        out = torch.full((M, N), float("nan"), dtype=BF, device=DEV)
        B().mgemm_fwd_noalloc(gs, B().MGEMM_BF16, trans_b, x, None, w, None, out, M, K, N, E)
        ref = regular_fwd(gs, x, w, trans_b, M, K, N, E)
        torch.cuda.synchronize()
        assert_close(to_np(out), to_np(ref), BF16_TOL, f"no-alloc forward, call {i + 1}")


def test_noalloc_rejects_too_many_experts():
    # checked on the host before any CUDA call, so this runs without a GPU
    lib = B().lib()
    p = ctypes.c_void_p(0x10000)
    too_many = 1025
    assert lib.mgemm_fwd_noalloc(p, too_many, 0, 0, p, None, p, None, p, 64, 128, 256, None) == -3
    assert lib.mgemm_fwd_noalloc(None, 8, 0, 0, p, None, p, None, p, 64, 128, 256, None) == -1
    # the stated maximum fits the library's array: E = 1024 passes the size check (and then,
    # without a GPU here, fails at the first CUDA call rather than as too many experts)
    assert lib.mgemm_fwd_noalloc(p, 1024, 0, 0, p, None, p, None, p, 64, 128, 256, None) not in (-1, -3)
