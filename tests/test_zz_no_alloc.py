"""The forward entry point for callers that cannot allocate device memory.

mgemm_fwd_noalloc keeps the args block (the tile schedule derived from the
group sizes) in a static device array inside the library, so a caller that may
not call cudaMalloc -- code running inside another framework's launch callback,
a loop where an allocation could stall the device, a runtime with a fixed
workspace -- only passes inputs and the output.  The GPU tests call it through
the C ABI twice in a row with different problems (the second with fewer
experts, so stale contents of the shared array would show).  Each result must
equal, bit for bit, the regular path on the same inputs (a caller-allocated
args block filled by mgemm_fill_args and passed to mgemm_fwd: the same kernel
on the same schedule), and match the oracle within the GEMM tolerance.  The
FP8 cases reach the few-rows kernels (sparse groups) and the CTA-pair kernels
(groups of 256 rows and more).  This file is collected last."""

import ctypes

import numpy as np
import pytest
import torch

from oracle import gmm as og
from tests.helpers import BF16_TOL, FP8_TOL, assert_close, new_args, to_np

DEV = "cuda"
BF = torch.bfloat16


@pytest.fixture(scope="module", autouse=True)
def built_library():
    from mixture_experts_grouped_gmm_gb300 import build

    build.build()


def B():
    from mixture_experts_grouped_gmm_gb300 import binding

    return binding


def rand_bf16(shape, seed, scale=1.0):
    g = torch.Generator(device=DEV).manual_seed(seed)
    return (torch.randn(shape, generator=g, device=DEV) * scale).to(BF)


def regular_fwd(gs, dtype, x, sx, w, sw, trans_b, M, K, N, E):
    args = new_args(E, DEV)
    B().mgemm_fill_args(gs, E, M, args)
    out = torch.empty(M, N, dtype=BF, device=DEV)
    B().mgemm_fwd(args, dtype, trans_b, x, sx, w, sw, out, M, K, N, E)
    return out


def quant_rows_gpu(t):
    R, C = t.shape
    q = torch.empty(R, C, dtype=torch.uint8, device=DEV)
    s = torch.empty(R, dtype=torch.float32, device=DEV)
    B().mgemm_quant_rowwise(t, q, s)
    return q, s


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
        ref = regular_fwd(gs, B().MGEMM_BF16, x, None, w, None, trans_b, M, K, N, E)
        torch.cuda.synchronize()
        assert torch.equal(out.view(torch.int16), ref.view(torch.int16)), f"no-alloc bf16 call {i + 1} != mgemm_fwd"
        want = og.gmm_fwd(to_np(x), to_np(w), sizes, trans_b=bool(trans_b))
        assert_close(to_np(out), want, BF16_TOL, f"no-alloc bf16 call {i + 1} vs oracle")


@pytest.mark.gpu
def test_noalloc_fp8_forward_matches_regular_path_twice():
    cases = [
        ([0, 700, 400, 0], 256, 272),            # E = 4, M / E >= 256 rows: CTA pairs
        ([1, 0, 0, 2, 0, 1, 0, 0, 0, 3], 512, 256),  # E = 10, 7 rows: the few-rows kernels
    ]
    for i, (sizes, K, N) in enumerate(cases):
        E, M = len(sizes), int(np.sum(sizes))
        gs = torch.tensor(sizes, dtype=torch.int64, device=DEV)
        xq, sx = quant_rows_gpu(rand_bf16((M, K), 30 + i))
        wq, sw = quant_rows_gpu(rand_bf16((E * N, K), 40 + i, 0.02))
        out = torch.full((M, N), float("nan"), dtype=BF, device=DEV)
        B().mgemm_fwd_noalloc(gs, B().MGEMM_FP8_E4M3, 1, xq, sx, wq, sw, out, M, K, N, E)
        ref = regular_fwd(gs, B().MGEMM_FP8_E4M3, xq, sx, wq, sw, 1, M, K, N, E)
        torch.cuda.synchronize()
        assert torch.equal(out.view(torch.int16), ref.view(torch.int16)), f"no-alloc fp8 call {i + 1} != mgemm_fwd"
        want = og.gmm_fwd_fp8(to_np(xq), to_np(sx), to_np(wq).reshape(E, N, K), to_np(sw), sizes)
        assert_close(to_np(out), want, FP8_TOL, f"no-alloc fp8 call {i + 1} vs oracle")


def test_noalloc_host_checks_reject_before_any_launch():
    # Each of these is rejected on the host before any CUDA call (the pointers
    # are never dereferenced), so this runs with or without a GPU.
    lib = B().lib()
    p = ctypes.c_void_p(0x10000)
    odd = ctypes.c_void_p(0x10008)
    f = lib.mgemm_fwd_noalloc
    assert f(p, 1025, 0, 0, p, None, p, None, p, 64, 128, 256, None) == -3   # E over the array's maximum
    assert f(None, 8, 0, 0, p, None, p, None, p, 64, 128, 256, None) == -1   # no group sizes
    assert f(p, 0, 0, 0, p, None, p, None, p, 64, 128, 256, None) == -1      # E < 1
    assert f(p, 8, 0, 0, p, None, p, None, p, -1, 128, 256, None) == -1      # M < 0
    assert f(p, 8, 7, 0, p, None, p, None, p, 64, 128, 256, None) == -1      # unknown dtype
    assert f(p, 8, 0, 0, None, None, p, None, p, 64, 128, 256, None) == -1   # no x
    assert f(p, 8, 0, 0, odd, None, p, None, p, 64, 128, 256, None) == -2    # x not 16-byte aligned
    assert f(p, 8, 0, 0, p, None, p, None, p, 64, 120, 260, None) == -2     # N % 8 != 0
    assert f(p, 8, 1, 0, p, p, p, p, p, 64, 128, 256, None) == -5           # FP8 needs w [E, N, K]
    assert f(p, 8, 1, 1, p, None, p, p, p, 64, 128, 256, None) == -1        # FP8 without sx
