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


def _probe_library_full():
    from mixture_experts_grouped_gmm_gb300 import binding, build

    L = ctypes.CDLL(build.build_variant("mgemm_waitprobe", {"MGEMM_WAIT_LIMIT_NS": 0}))
    for name in ("mgemm_fwd_fp8_sparse", "mgemm_fill_args_quant_rowwise", "mgemm_fwd_f8i4", "mgemm_last_error"):
        res, argt = binding._SIGS[name]
        getattr(L, name).restype = res
        getattr(L, name).argtypes = argt
    return L


def _fp8_weights(E, N, K, seed):
    from mixture_experts_grouped_gmm_gb300 import binding as B

    g = torch.Generator(device=DEV).manual_seed(seed)
    w = (torch.randn(E * N, K, generator=g, device=DEV) * 0.02).to(BF)
    wq = torch.empty(E * N, K, dtype=torch.uint8, device=DEV)
    sw = torch.empty(E * N, dtype=torch.float32, device=DEV)
    B.mgemm_quant_rowwise(w, wq, sw)
    return wq, sw


# one token on one expert (CTA pairs split the contraction); 16 rows in four groups on 64 tiles
# of 128 weight rows each (unpaired, more tiles than half the SMs)
@pytest.mark.parametrize("sizes,K,N", [([1], 1024, 1024), ([3, 4, 5, 4], 2048, 8192)])
def test_sparse_fwd_wait_timeout_sets_status_and_leaves_the_device_usable(sizes, K, N):
    from mixture_experts_grouped_gmm_gb300 import binding as B
    from oracle import quant as oq

    L = _probe_library_full()
    E, M = len(sizes), int(np.sum(sizes))
    wq, sw = _fp8_weights(E, N, K, 4)
    x = torch.randn(M, K, generator=torch.Generator(device=DEV).manual_seed(5), device=DEV).to(BF)
    gs = torch.tensor(sizes, dtype=torch.int64, device=DEV)
    p = lambda t: ctypes.c_void_p(t.data_ptr())  # noqa: E731
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    out = torch.empty(M, N, dtype=BF, device=DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    rc = L.mgemm_fwd_fp8_sparse(p(gs), E, p(x), K, p(wq), p(sw), p(out), p(st), M, K, N, stream)
    assert rc == 0, f"the wait-probe build: {rc} ({L.mgemm_last_error().decode()})"
    torch.cuda.synchronize()  # the kernel returned
    assert int(st.item()) == 4, "the timed-out waits raise the status to MGEMM_STATUS_TIMEOUT"

    # the product library, same device, right after
    st2 = torch.zeros(1, dtype=torch.int32, device=DEV)
    out2 = torch.empty(M, N, dtype=BF, device=DEV)
    B.mgemm_fwd_fp8_sparse(gs, E, x, wq, sw, out2, st2)
    torch.cuda.synchronize()
    assert int(st2.item()) == 0
    xq, sx = oq.quant_rowwise(to_np(x))
    want = og.gmm_fwd_fp8(xq, sx, to_np(wq).reshape(E, N, K), to_np(sw), sizes)
    assert_close(to_np(out2), want, 3e-2, "sparse fwd after a timed-out one")


def test_f8i4_pairs_wait_timeout_sets_status_and_leaves_the_device_usable():
    from mixture_experts_grouped_gmm_gb300 import binding as B
    from oracle import f8i4 as of

    L = _probe_library_full()
    sizes, K, N = [0, 2, 5], 1024, 512          # 7 rows: CTA pairs split each tile's contraction
    E, M = len(sizes), int(np.sum(sizes))
    g = torch.Generator(device=DEV).manual_seed(6)
    w = (0.02 * torch.randn(E, N, K, generator=g, device=DEV)).to(BF)
    wp = torch.empty(E, N, K // 2, dtype=torch.uint8, device=DEV)
    sf = torch.empty(B.int4_scale_bytes(E, N, K), dtype=torch.uint8, device=DEV)
    B.mgemm_quant_int4(w, wp, sf)
    x = torch.randn(M, K, generator=g, device=DEV).to(BF)
    gs = torch.tensor(sizes, dtype=torch.int64, device=DEV)
    p = lambda t: ctypes.c_void_p(t.data_ptr())  # noqa: E731
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)

    args = new_args(E, DEV)
    xq = torch.empty(M, K, dtype=torch.uint8, device=DEV)
    sx = torch.empty(M, dtype=torch.float32, device=DEV)
    out = torch.empty(M, N, dtype=BF, device=DEV)
    assert L.mgemm_fill_args_quant_rowwise(p(gs), E, M, p(args), p(x), K, K, p(xq), K, p(sx), stream) == 0
    rc = L.mgemm_fwd_f8i4(p(args), p(xq), p(sx), p(wp), p(sf), p(out), M, K, N, E, stream)
    assert rc == 0, f"the wait-probe build: {rc} ({L.mgemm_last_error().decode()})"
    torch.cuda.synchronize()  # the kernel returned
    assert parse_args(args, E)["status"] == 4, "the timed-out waits record MGEMM_STATUS_TIMEOUT"

    # the product library, same device, right after
    args2 = new_args(E, DEV)
    out2 = torch.empty(M, N, dtype=BF, device=DEV)
    B.mgemm_fill_args_quant_rowwise(gs, E, M, args2, x, xq, sx)
    B.mgemm_fwd_f8i4(args2, xq, sx, wp, sf, out2, M, K, N, E)
    torch.cuda.synchronize()
    assert parse_args(args2, E)["status"] == 0
    q, b = of.quant_int4_rows(w.double().cpu().numpy().reshape(E * N, K))
    want = of.gmm_fwd_f8i4(to_np(xq), to_np(sx), of.pack_int4(q).reshape(E, N, K // 2), b.reshape(E, N, K // 32), sizes)
    assert_close(to_np(out2), want, 3e-2, "F8I4 after a timed-out one")
