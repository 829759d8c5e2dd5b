"""The bounded pipeline waits of the GEMM kernels, made to run out.

Every mbarrier wait in the library's kernels gives up after a limit: the
kernel then records status 4 (MGEMM_STATUS_TIMEOUT) in the args block, lets its
other roles leave their loops, waits for the copies and MMAs it already issued,
frees tensor memory and returns, so the context stays usable and later calls
skip their work (the status word's failure handling is planned around the
argument kernels of "Support GPU-resident batch sizes", review of the k = 0
workaround kernels).

To make a wait run out without a faulty producer, this test builds and loads a
separate copy of the library, compiled with MGEMM_WAIT_LIMIT_NS=0: there a
pipeline wait whose phase is not already complete gives up at once, so every
CTA's first wait for data still in flight times out (the drain keeps its own
1 s limit).  The product library and its binding never load that copy.  After
the timed-out call the product library runs an ordinary GEMM on the same
device, which must match the oracle: nothing (tensor memory, a barrier) was
left held."""

import ctypes

import numpy as np
import pytest
import torch

from oracle import gmm as og
from tests.helpers import BF16_TOL, assert_close, is_sentinel, new_args, parse_args, sentinel_bf16, to_np

pytestmark = pytest.mark.gpu
DEV = "cuda"
BF = torch.bfloat16


def _probe_library():
    from mixture_experts_grouped_gmm_gb300 import binding, build

    L = ctypes.CDLL(build.build_variant("mgemm_waitprobe", {"MGEMM_WAIT_LIMIT_NS": 0}))
    for name in ("mgemm_fill_args", "mgemm_fwd", "mgemm_last_error"):
        res, argt = binding._SIGS[name]
        getattr(L, name).restype = res
        getattr(L, name).argtypes = argt
    return L


def test_gemm_wait_timeout_sets_status_and_leaves_the_device_usable():
    from mixture_experts_grouped_gmm_gb300 import binding as B

    L = _probe_library()
    sizes = [300, 200, 12, 0, 500]
    E, M, K, N = len(sizes), int(np.sum(sizes)), 512, 384
    g = torch.Generator(device=DEV).manual_seed(3)
    x = torch.randn(M, K, generator=g, device=DEV).to(BF)
    w = torch.randn(E, K, N, generator=g, device=DEV).to(BF)
    gs = torch.tensor(sizes, dtype=torch.int64, device=DEV)
    p = lambda t: ctypes.c_void_p(t.data_ptr())  # noqa: E731
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)

    args = new_args(E, DEV)
    out = sentinel_bf16((M, N), DEV)
    assert L.mgemm_fill_args(p(gs), E, M, p(args), stream) == 0
    rc = L.mgemm_fwd(p(args), B.MGEMM_BF16, 0, p(x), None, p(w), None, p(out), M, K, N, E, stream)
    assert rc == 0, f"mgemm_fwd of the wait-probe build: {rc} ({L.mgemm_last_error().decode()})"
    torch.cuda.synchronize()  # the kernel returned
    assert parse_args(args, E)["status"] == 4, "the timed-out waits record MGEMM_STATUS_TIMEOUT"
    assert is_sentinel(out), "no tile is stored after a timeout"

    # the product library, same device, right after
    args2 = new_args(E, DEV)
    out2 = sentinel_bf16((M, N), DEV)
    B.mgemm_fill_args(gs, E, M, args2)
    B.mgemm_fwd(args2, B.MGEMM_BF16, 0, x, None, w, None, out2, M, K, N, E)
    torch.cuda.synchronize()
    assert parse_args(args2, E)["status"] == 0
    assert_close(to_np(out2), og.gmm_fwd(to_np(x), to_np(w), sizes), BF16_TOL, "GEMM after a timed-out one")
