"""GPU parity of mgemm_fwd_fp8_sparse, the sparse-M FP8 forward in one launch
(the group-size scan, the rowwise cast of the token rows and the grouped GEMM
of "F8I4 Grouped Gemm Optimization for Sparse M": work only for the non-empty
groups).  Its output must match the oracle within the FP8 tolerance and the
three calls it replaces (mgemm_fill_args, mgemm_quant_rowwise, mgemm_fwd with
FP8 operands): bit for bit when no CTA pairs split the contraction (more
tiles of 128 output columns than half the SMs), else within one bf16 rounding
step (the two halves' fp32 sums are added once more).  Rows past M are
untouched and invalid group sizes are reported in the status word with
nothing written."""

import numpy as np
import pytest
import torch

from oracle import gmm as og
from oracle import quant as oq
from oracle.formats import decode_e4m3 as decode
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


def paired(M, E, N):
    """Whether the call splits each tile's contraction over a CTA pair (the library's rule)."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    return 2 * min(M, E) * ((N + 127) // 128) <= sms


def status():
    return torch.full((1,), -7, dtype=torch.int32, device=DEV)


def assert_within_one_step(got, ref, what):
    """|got - ref| <= one bf16 step (2^-7 relative) of ref, elementwise, plus the fp32 rounding slack."""
    g, r = got.float(), ref.float()
    bound = r.abs() * 2.0 ** -7 + r.abs().max() * 2.0 ** -20
    bad = (g - r).abs() > bound
    assert not bool(bad.any()), f"{what}: {int(bad.sum())} outputs differ by more than one bf16 step"


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
    ([3, 4, 5, 4], 2048, 8192),         # more tiles than SMs: CTAs whose tiles span two groups
    ([1] * 16, 256, 1040),              # tiles of 120 weight rows (on 148+ SMs), the last of 80
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
    st = status()
    B().mgemm_fwd_fp8_sparse(gs, E, x, wq, sw, out[:M], st)
    ref = three_calls(gs, E, x.contiguous(), wq, sw, N) if N % 16 == 0 else None
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    assert is_sentinel(out[M:]), "wrote past M rows"
    if ref is not None:
        if paired(M, E, N):
            assert_within_one_step(out[:M], ref, "vs the three calls")
        else:
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
    st = status()
    B().mgemm_fwd_fp8_sparse(d["group_sizes"], E, d["x"], wq, sw, out, st)
    ref = three_calls(d["group_sizes"], E, d["x"], wq, sw, N)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    if paired(total_m, E, N):
        assert_within_one_step(out, ref, "vs the three calls")
    else:
        assert torch.equal(out.view(torch.int16), ref.view(torch.int16)), "differs from the three calls"
    # sampled outputs against the oracle (rows computed one by one in float64)
    sizes = d["group_sizes"].cpu().tolist()
    xq, sx = oq.quant_rowwise(to_np(d["x"]))
    cols = np.random.default_rng(total_m).choice(N, 64, replace=False)
    e_of = og.expert_of_rows(sizes, np.arange(total_m))
    wv = to_np(wq.view(E, N, K)[:, torch.as_tensor(cols, device=DEV)])
    want = np.stack([(decode(xq[r]) / sx[r]) @ (decode(wv[e_of[r]]) / to_np(sw).reshape(E, N)[e_of[r], cols][:, None]).T
                     for r in range(total_m)])
    assert_close(to_np(out)[:, cols], want, FP8_TOL, "sampled columns vs oracle")


def test_sparse_fwd_reports_bad_sizes():
    E, K, N = 4, 256, 64
    wq, sw = weights(E, N, K, 3)
    x = torch.randn(5, K, device=DEV).to(BF)
    for sizes, code in (([2, -1, 4, 0], 1), ([2, 1, 1, 0], 2)):   # negative; sum 4 != M = 5
        out = sentinel_bf16((5, N), DEV)
        st = status()
        B().mgemm_fwd_fp8_sparse(torch.tensor(sizes, dtype=torch.int64, device=DEV), E, x, wq, sw, out, st)
        torch.cuda.synchronize()
        assert int(st.item()) == code and is_sentinel(out)


@pytest.mark.parametrize("K", [256, 384, 1024, 5120])
def test_sparse_fwd_pairs_split_the_contraction(K):
    # one token on one expert: 8 tiles, so CTA pairs take one half of K each (K = 256 with 64 KB
    # stages has a single stage per tile and runs unpaired); repeated calls reuse the handoff
    E, N = 1, 1024
    wq, sw = weights(E, N, K, 5)
    gs = torch.tensor([1], dtype=torch.int64, device=DEV)
    for seed in (1, 2):
        x = torch.randn(1, K, generator=torch.Generator(device=DEV).manual_seed(seed), device=DEV).to(BF)
        out = sentinel_bf16((1, N), DEV)
        st = status()
        B().mgemm_fwd_fp8_sparse(gs, E, x, wq, sw, out, st)
        ref = three_calls(gs, E, x, wq, sw, N)
        torch.cuda.synchronize()
        assert int(st.item()) == 0
        assert_within_one_step(out, ref, "vs the three calls")
        xq, sx = oq.quant_rowwise(to_np(x))
        want = og.gmm_fwd_fp8(xq, sx, to_np(wq).reshape(E, N, K), to_np(sw), [1])
        assert_close(to_np(out), want, FP8_TOL, "pairs vs oracle")


@pytest.mark.parametrize("total_m", [1, 4])
def test_sparse_fwd_graph_replay_follows_device_sizes(total_m):
    # the launch reads the group sizes on the device: captured once in a CUDA graph, it follows
    # new sizes written into the same tensor between replays (no host round trip)
    E, K, N = 8, 1024, 512
    wq, sw = weights(E, N, K, 9)
    x = (torch.randn(total_m, K, generator=torch.Generator(device=DEV).manual_seed(2), device=DEV) * 2).to(BF)
    gs = torch.zeros(E, dtype=torch.int64, device=DEV)
    gs[0] = total_m
    out = torch.empty(total_m, N, dtype=BF, device=DEV)
    st = status()
    B().mgemm_fwd_fp8_sparse(gs, E, x, wq, sw, out, st)  # warm-up outside the capture
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        B().mgemm_fwd_fp8_sparse(gs, E, x, wq, sw, out, st)
    for sizes in ([0] * 5 + [total_m, 0, 0], [total_m - total_m // 2, 0, 0, total_m // 2, 0, 0, 0, 0]):
        gs.copy_(torch.tensor(sizes, dtype=torch.int64))
        st.fill_(0)
        graph.replay()
        ref = three_calls(gs, E, x, wq, sw, N)
        torch.cuda.synchronize()
        assert int(st.item()) == 0
        if paired(total_m, E, N):
            assert_within_one_step(out, ref, f"replay with sizes {sizes}")
        else:
            assert torch.equal(out.view(torch.int16), ref.view(torch.int16)), f"replay with sizes {sizes}"
