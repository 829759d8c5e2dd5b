"""GPU parity of mgemm_fwd_fp8_sparse, the sparse-M FP8 forward in one launch
(the group-size scan, the rowwise cast of the token rows and the grouped GEMM
of "F8I4 Grouped Gemm Optimization for Sparse M": tiles only for the
non-empty groups).  Its output must equal, bit for bit, the three calls it
replaces (mgemm_fill_args, mgemm_quant_rowwise, mgemm_fwd with FP8 operands),
and match the oracle within the FP8 tolerance; rows past M are untouched and
invalid group sizes are reported in the status word with nothing written."""

import numpy as np
import pytest
import torch

from oracle import gmm as og
from oracle import quant as oq
from tests.helpers import FP8_TOL, assert_close, is_sentinel, new_args, sentinel_bf16, to_np

pytestmark = pytest.mark.gpu
DEV = "cuda"
BF = torch.bfloat16


def B():
    from mixture_experts_grouped_gmm_gb300 import binding

    return binding


def weights(E, N, K, seed):
    g = torch.Generator(device=DEV).manual_seed(seed)
    w = (torch.randn(E * N, K, generator=g, device=DEV) * 0.02).to(BF)
    wq = torch.empty(E * N, K, dtype=torch.uint8, device=DEV)
    sw = torch.empty(E * N, dtype=torch.float32, device=DEV)
    B().mgemm_quant_rowwise(w, wq, sw)
    return wq, sw


def three_calls(gs, E, x, wq, sw, N):
    M, K = x.shape
    args = new_args(E, DEV)
    xq = torch.empty(M, K, dtype=torch.uint8, device=DEV)
    sx = torch.empty(M, dtype=torch.float32, device=DEV)
    B().mgemm_fill_args(gs, E, M, args)
    B().mgemm_quant_rowwise(x, xq, sx)
    out = torch.empty(M, N, dtype=BF, device=DEV)
    B().mgemm_fwd(args, B().MGEMM_FP8_E4M3, 1, xq, sx, wq, sw, out, M, K, N, E)
    return out


@pytest.mark.parametrize("sizes,K,N", [
    ([1, 0, 3, 0, 2], 256, 208),        # N not a multiple of the 64-wide tile
    ([3, 1], 128, 200),                 # N % 16 == 8: accepted here, not by mgemm_fwd (oracle only)
    ([0, 0, 5], 384, 128),              # K = 3 blocks of 128 (the last stage holds one)
    ([16], 512, 256),                   # E = 1, the most rows
    ([2] * 8, 1024, 64),                # eight groups of two
    ([5, 11], 2048, 128),               # more units than one register batch of the cast
    ([16], 4096, 64),                   # four batches
    ([3, 0, 4], 384, 136),              # rows of 48 units: a warp's units straddle two rows
])
@pytest.mark.parametrize("ld_pad", [0, 40])
def test_sparse_fwd_equals_the_three_calls(sizes, K, N, ld_pad):
    E, M = len(sizes), int(np.sum(sizes))
    g = torch.Generator(device=DEV).manual_seed(M + K)
    x = (torch.randn(M, K + ld_pad, generator=g, device=DEV) * 3).to(BF)[:, :K]   # row stride K + ld_pad
    x[M // 2, 7] = 0.0
    if M > 3:
        x[3].zero_()                                                             # an all-zero row
    gs = torch.tensor(sizes, dtype=torch.int64, device=DEV)
    wq, sw = weights(E, N, K, 7)
    out = sentinel_bf16((M + 4, N), DEV)
    st = torch.full((1,), -7, dtype=torch.int32, device=DEV)
    B().mgemm_fwd_fp8_sparse(gs, E, x, wq, sw, out[:M], st)
    ref = three_calls(gs, E, x.contiguous(), wq, sw, N) if N % 16 == 0 else None
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    assert is_sentinel(out[M:]), "wrote past M rows"
    if ref is not None:
        assert torch.equal(out[:M].view(torch.int16), ref.view(torch.int16)), "differs from the three calls"
    xq, sx = oq.quant_rowwise(to_np(x))
    want = og.gmm_fwd_fp8(xq, sx, to_np(wq).reshape(E, N, K), to_np(sw), sizes)
    assert_close(to_np(out[:M]), want, FP8_TOL, "sparse fwd vs oracle")


@pytest.mark.parametrize("total_m", [1, 2, 4, 16])
def test_sparse_fwd_at_the_sparse_m_shape(total_m):
    # E = 128, K = 5120, N = 8192, tokens routed to random experts: the bench's workload
    from mixture_experts_grouped_gmm_gb300 import workloads

    E, K, N = 128, 5120, 8192
    d = workloads.sparse_m(total_m, E=E, K=K, N=N, device=DEV, with_weights=False)
    wq, sw = weights(E, N, K, total_m)
    out = torch.empty(total_m, N, dtype=BF, device=DEV)
    st = torch.full((1,), -7, dtype=torch.int32, device=DEV)
    B().mgemm_fwd_fp8_sparse(d["group_sizes"], E, d["x"], wq, sw, out, st)
    ref = three_calls(d["group_sizes"], E, d["x"], wq, sw, N)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    assert torch.equal(out.view(torch.int16), ref.view(torch.int16))


def test_sparse_fwd_reports_bad_sizes():
    E, K, N = 4, 256, 64
    wq, sw = weights(E, N, K, 3)
    x = torch.randn(5, K, device=DEV).to(BF)
    for sizes, code in (([2, -1, 4, 0], 1), ([2, 1, 1, 0], 2)):   # negative; sum 4 != M = 5
        out = sentinel_bf16((5, N), DEV)
        st = torch.full((1,), -7, dtype=torch.int32, device=DEV)
        B().mgemm_fwd_fp8_sparse(torch.tensor(sizes, dtype=torch.int64, device=DEV), E, x, wq, sw, out, st)
        torch.cuda.synchronize()
        assert int(st.item()) == code and is_sentinel(out)
