"""GPU parity of the routed layer's calls (mgemm_topk_softmax,
mgemm_gather_rows, mgemm_fwd_scatter, mgemm_silu_and_mul, mgemm_topk_sum,
mgemm_fill_args with M = -1) and of moe.fused_experts / moe.fused_moe, against
oracle.routing.  Expert ids are compared exactly.

Integer outputs (gather) are compared bit for bit; GEMM outputs, and the
whole layer, within 1e-2 * max|ref|.  The layer rounds to bf16 three times
where the float64 oracle does not (the gated rows, the scattered entries and
the final sum), each a relative error of at most 2^-9 of the value rounded;
the gated rows' errors enter the second GEMM's sums with both signs, so the
layer's max|err| stays a small multiple of 2^-9 * max|ref| (< 1e-2).
Rows the kernels must not touch are pre-filled with a sentinel and checked."""

import numpy as np
import pytest
import torch

from oracle import routing as R
from tests.helpers import BF16_TOL, assert_close, is_sentinel, new_args, parse_args, sentinel_bf16, to_np

pytestmark = pytest.mark.gpu
DEV = "cuda"
BF = torch.bfloat16


def B():
    from mixture_experts_grouped_gmm_gb300 import binding

    return binding


def routing_ids(T, k, E, seed):
    """Top-k distinct experts per token (uniform), int32 [T, k]."""
    g = torch.Generator().manual_seed(seed)
    return torch.stack([torch.randperm(E, generator=g)[:k] for _ in range(T)]).to(torch.int32)


def aligned(ids, E):
    from mixture_experts_grouped_gmm_gb300 import moe

    sid, eid, npp, gs = moe.align(ids.to(DEV), E)
    torch.cuda.synchronize()
    return sid, eid, npp, gs


def test_fill_args_sum_mode_matches_explicit_M():
    gs = torch.tensor([256, 0, 128, 384, 0, 128], dtype=torch.int64, device=DEV)
    a1, a2 = new_args(6, DEV), new_args(6, DEV)
    B().mgemm_fill_args(gs, 6, 896, a1)
    B().mgemm_fill_args(gs, 6, -1, a2)
    torch.cuda.synchronize()
    assert torch.equal(a1, a2)
    assert parse_args(a2, 6)["status"] == 0


def test_gather_rows_bit_exact():
    T, k, E, K = 300, 2, 8, 136
    ids = routing_ids(T, k, E, 1)
    sid, eid, npp, gs = aligned(ids, E)
    x = torch.randn(T, K, device=DEV).to(BF)
    cap = sid.numel()
    dst = sentinel_bf16((cap, K), DEV)
    B().mgemm_gather_rows(x, sid, npp, T * k, k, dst)
    torch.cuda.synchronize()
    tot = int(npp)
    ref = R.gather_rows(to_np(x), sid.cpu().numpy(), tot, T * k, k)
    assert np.array_equal(to_np(dst[:tot]), ref.astype(np.float32))
    assert is_sentinel(dst[tot:]), "rows past the padded total must stay untouched"


@pytest.mark.parametrize("with_weights", [False, True])
@pytest.mark.parametrize("T,k,E,K,N", [(300, 2, 8, 256, 384), (5, 2, 16, 128, 256), (1000, 6, 64, 192, 136)])
def test_fwd_scatter_against_oracle(T, k, E, K, N, with_weights):
    ids = routing_ids(T, k, E, T + E)
    sid, eid, npp, gs = aligned(ids, E)
    n, cap = T * k, sid.numel()
    args = new_args(E, DEV)
    B().mgemm_fill_args(gs, E, -1, args)
    x = torch.randn(T, K, device=DEV).to(BF)
    w = (0.05 * torch.randn(E, N, K, device=DEV)).to(BF)
    a = torch.empty(cap, K, dtype=BF, device=DEV)
    B().mgemm_gather_rows(x, sid, npp, n, k, a)
    wts = torch.rand(n, device=DEV) if with_weights else None
    out = sentinel_bf16((n + 4, N), DEV)
    B().mgemm_fwd_scatter(args, B().MGEMM_BF16, 1, a, w, out, sid, n, wts, cap, K, N, E)
    torch.cuda.synchronize()
    assert parse_args(args, E)["status"] == 0
    assert is_sentinel(out[n:]), "wrote past the entry rows"
    ref = R.fused_moe_gemm(to_np(x), to_np(w), sid.cpu().numpy(), eid.cpu().numpy(), int(npp), n, k, 128,
                           None if wts is None else wts.cpu().numpy())
    assert not np.isnan(ref).any()  # every entry is placed
    assert_close(to_np(out[:n]), ref, BF16_TOL, "fwd_scatter")


def test_silu_and_mul():
    x = (3 * torch.randn(257, 2 * 136, device=DEV)).to(BF)
    out = torch.empty(257, 136, dtype=BF, device=DEV)
    B().mgemm_silu_and_mul(x, out)
    torch.cuda.synchronize()
    ref = R.silu_and_mul(to_np(x))
    got = to_np(out).astype(np.float64)
    # one bf16 rounding of an fp32 result: within 2^-8 relative, plus fp32 exp error
    assert np.all(np.abs(got - ref) <= 2.0 ** -8 * np.abs(ref) + 1e-6)


def test_topk_sum():
    T, k, H = 129, 3, 264
    c = torch.randn(T * k, H, device=DEV).to(BF)
    out = torch.empty(T, H, dtype=BF, device=DEV)
    B().mgemm_topk_sum(c, T, k, out)
    torch.cuda.synchronize()
    ref = to_np(c).astype(np.float64).reshape(T, k, H).sum(axis=1)
    got = to_np(out).astype(np.float64)
    assert np.all(np.abs(got - ref) <= 2.0 ** -8 * np.abs(ref) + 1e-5)


@pytest.mark.parametrize("T,k,E,H,F", [(200, 2, 8, 256, 384), (3, 2, 8, 128, 128),
                                       (2100, 2, 8, 128, 128)])  # 4200 entries: the three-kernel alignment
def test_fused_moe_layer(T, k, E, H, F):
    from mixture_experts_grouped_gmm_gb300 import moe

    torch.manual_seed(T)
    x = torch.randn(T, H, device=DEV).to(BF)
    w1 = (0.05 * torch.randn(E, 2 * F, H, device=DEV)).to(BF)
    w2 = (0.05 * torch.randn(E, H, F, device=DEV)).to(BF)
    logits = torch.randn(T, E, device=DEV)
    probs = torch.softmax(logits, dim=-1)
    tw, tid = torch.topk(probs, k, dim=-1)
    tw = tw / tw.sum(dim=-1, keepdim=True)
    out = moe.fused_experts(x, w1, w2, tw, tid)
    torch.cuda.synchronize()
    # oracle: the same steps in float64 (no bf16 caches in between)
    sid, eid, tot, _ = R.moe_align_block_size(tid.cpu().numpy(), 128, E)
    n = T * k
    c1 = R.fused_moe_gemm(to_np(x), to_np(w1), sid, eid, tot, n, k, 128)
    c2 = R.silu_and_mul(c1)
    c3 = R.fused_moe_gemm(c2, to_np(w2), sid, eid, tot, n, 1, 128, topk_weights=tw.cpu().numpy().ravel())
    ref = c3.reshape(T, k, H).sum(axis=1)
    assert_close(to_np(out), ref, BF16_TOL, "fused_moe")


@pytest.mark.parametrize("T,E,k,renorm,kind", [
    (1000, 8, 2, True, "normal"), (333, 64, 6, False, "normal"), (64, 128, 40, True, "normal"),
    (40, 1024, 1024, False, "normal"), (200, 64, 6, True, "ties"), (17, 3, 3, True, "ties"),
])
def test_topk_softmax(T, E, k, renorm, kind):
    g = torch.Generator(device=DEV).manual_seed(T + E)
    if kind == "normal":
        logits = torch.randn(T, E, generator=g, device=DEV)
    else:  # few distinct values: many equal logits, ties go to the lower id
        logits = torch.randint(-2, 3, (T, E), generator=g, device=DEV).float()
    w = torch.empty(T, k, device=DEV)
    i = torch.empty(T, k, dtype=torch.int32, device=DEV)
    B().mgemm_topk_softmax(logits, k, renorm, w, i)
    torch.cuda.synchronize()
    rw, ri = R.topk_softmax(logits.cpu().numpy(), k, renorm)
    assert np.array_equal(i.cpu().numpy(), ri), "expert ids must match exactly"
    # fp32 exp and an fp32 sum over E terms
    assert np.allclose(w.cpu().numpy(), rw, rtol=1e-4, atol=1e-7)


def test_fused_moe_from_gating_logits():
    from mixture_experts_grouped_gmm_gb300 import moe

    T, k, E, H, F = 150, 2, 8, 256, 256
    torch.manual_seed(5)
    x = torch.randn(T, H, device=DEV).to(BF)
    w1 = (0.05 * torch.randn(E, 2 * F, H, device=DEV)).to(BF)
    w2 = (0.05 * torch.randn(E, H, F, device=DEV)).to(BF)
    gating = torch.randn(T, E, device=DEV)
    out = moe.fused_moe(x, w1, w2, gating, k, True)
    torch.cuda.synchronize()
    tw, tid = R.topk_softmax(gating.cpu().numpy(), k, True)
    sid, eid, tot, _ = R.moe_align_block_size(tid, 128, E)
    n = T * k
    c1 = R.fused_moe_gemm(to_np(x), to_np(w1), sid, eid, tot, n, k, 128)
    c3 = R.fused_moe_gemm(R.silu_and_mul(c1), to_np(w2), sid, eid, tot, n, 1, 128, topk_weights=tw.ravel())
    ref = c3.reshape(T, k, H).sum(axis=1)
    assert_close(to_np(out), ref, BF16_TOL, "fused_moe from gating logits")


@pytest.mark.parametrize("sizes,K,F", [([130, 0, 257, 64, 1], 192, 200), ([128] * 4, 256, 384), ([700], 64, 1000)])
def test_fwd_gated_against_oracle(sizes, K, F):
    # silu_and_mul fused into the GEMM epilogue: out = silu(x . w_gate^T) * (x . w_up^T)
    from oracle import gmm as og

    M, E = int(np.sum(sizes)), len(sizes)
    args = new_args(E, DEV)
    B().mgemm_fill_args(torch.tensor(sizes, dtype=torch.int64, device=DEV), E, M, args)
    x = torch.randn(M, K, device=DEV).to(BF)
    w = (0.1 * torch.randn(E, 2 * F, K, device=DEV)).to(BF)
    out = sentinel_bf16((M + 8, F), DEV)
    B().mgemm_fwd_gated(args, x, w, out, M, K, F, E)
    torch.cuda.synchronize()
    assert is_sentinel(out[M:]), "wrote past M rows"
    ref = R.silu_and_mul(og.gmm_fwd(to_np(x), to_np(w), sizes, trans_b=True))
    assert_close(to_np(out[:M]), ref, BF16_TOL, "fwd_gated")


@pytest.mark.parametrize("T,k,E,H,F,renorm", [
    (1, 2, 8, 128, 128, True),     # one token
    (37, 4, 4, 128, 256, True),    # top_k = E: every token in every expert
    (50, 1, 1, 256, 128, False),   # one expert, top-1, no renormalization
    (9, 3, 16, 136, 200, True),    # H, F not multiples of the 64-element k-block
    (2, 2, 8, 1024, 2048, True),   # decode: k-chunk boxes (gate and up rows of a stage in one copy)
])
def test_fused_moe_edges(T, k, E, H, F, renorm):
    from mixture_experts_grouped_gmm_gb300 import moe

    torch.manual_seed(T * 7 + E)
    x = torch.randn(T, H, device=DEV).to(BF)
    w1 = (0.05 * torch.randn(E, 2 * F, H, device=DEV)).to(BF)
    w2 = (0.05 * torch.randn(E, H, F, device=DEV)).to(BF)
    gating = torch.randn(T, E, device=DEV)
    out = moe.fused_moe(x, w1, w2, gating, k, renorm)
    torch.cuda.synchronize()
    tw, tid = R.topk_softmax(gating.cpu().numpy(), k, renorm)
    ref = np.stack([R.fused_moe_token(to_np(x)[t], to_np(w1), to_np(w2), tid[t], tw[t]) for t in range(T)])
    assert_close(to_np(out), ref, BF16_TOL, "fused_moe edge case")


@pytest.mark.parametrize("T,k,E,H,F", [
    (1, 2, 8, 1024, 2048),     # one token: 8-row A slots, four blocks per stage
    (4, 2, 8, 512, 384),       # a partial last column tile
    (9, 3, 16, 256, 520),      # 27 entries: 32-row A slots, padding rows inside them
    (12, 2, 2, 320, 256),      # 24 entries over 2 experts; K = 320: chunks past K are zeros
    (16, 2, 64, 4096, 128),    # 32 entries over 64 experts (the largest group_rows_max, 32)
    (5, 1, 3, 192, 1040),      # top-1, K = 192 (three of a stage's four chunks inside K)
])
def test_fwd_gated_gather_matches_gather_then_gated(T, k, E, H, F):
    from mixture_experts_grouped_gmm_gb300 import moe

    torch.manual_seed(T * 31 + H)
    x = torch.randn(T, H, device=DEV).to(BF)
    w1 = (0.05 * torch.randn(E, 2 * F, H, device=DEV)).to(BF)
    tid = torch.stack([torch.randperm(E, device=DEV)[:k] for _ in range(T)]).to(torch.int32)
    n = T * k
    sid, _, npp, _, args = moe.align_args(tid, E)
    cap = sid.numel()
    rows = min(cap, n + min(E, n) * 127)
    a1 = torch.empty(cap, H, dtype=BF, device=DEV)
    B().mgemm_gather_rows(x, sid, npp, n, k, a1)
    ref = sentinel_bf16((cap, F), DEV)
    got = sentinel_bf16((cap, F), DEV)
    B().mgemm_fwd_gated(args, a1, w1, ref, rows, H, F, E, n)
    B().mgemm_fwd_gated_gather(args, x, sid, n, k, w1, got, rows, H, F, E, n)
    torch.cuda.synchronize()
    # the same rows in the same order (padding rows zero in both), the same MMAs: equal bits
    assert torch.equal(got.view(torch.int16), ref.view(torch.int16))
    # and the routed rows against the oracle
    s = sid.cpu().numpy()
    real = np.nonzero(s[:rows] < n)[0]
    e_of = np.searchsorted(np.asarray(parse_args(args, E)["offsets"]), real, side="right") - 1
    xr = to_np(x)[s[real] // k]
    w = to_np(w1)
    want = np.stack([R.silu_and_mul(xr[i:i + 1] @ w[e_of[i]].T)[0] for i in range(len(real))])
    assert_close(to_np(got[torch.as_tensor(real, device=DEV)]), want, BF16_TOL, "gathered gated rows")


def test_fwd_gated_gather_rejects_other_shapes():
    E, F = 4, 64
    sid = torch.zeros(512, dtype=torch.int32, device=DEV)
    args = new_args(E, DEV)
    out = torch.empty(512, F, dtype=BF, device=DEV)
    x = torch.zeros(2, 136, dtype=BF, device=DEV)
    w1 = torch.zeros(E, 2 * F, 136, dtype=BF, device=DEV)
    with pytest.raises(B().MgemmError):   # K % 64 != 0
        B().mgemm_fwd_gated_gather(args, x, sid, 3, 2, w1, out, 512, 136, F, E, 3)
    x = torch.zeros(40, 256, dtype=BF, device=DEV)
    w1 = torch.zeros(E, 2 * F, 256, dtype=BF, device=DEV)
    with pytest.raises(B().MgemmError):   # group_rows_max > 32
        B().mgemm_fwd_gated_gather(args, x, sid, 80, 2, w1, out, 512, 256, F, E, 33)
