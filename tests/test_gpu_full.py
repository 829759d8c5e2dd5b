"""Full-size parity on the benchmark workloads, in the launch configuration the
benchmark times (same entry points, same persistent grid).  The oracle
recomputes sampled outputs one by one: sampled rows (and columns) for forward
and dgrad, sampled K-rows of every expert for wgrad, sampled rows for the
rowwise quantize and sampled columns of every group for the colwise quantize.
Quantized bytes and scales must match bit for bit; GEMM outputs within the
tolerance of their operand type."""

import numpy as np
import pytest
import torch

from mixture_experts_grouped_gmm_gb300 import workloads
from oracle import gmm as og, quant as oq
from tests.helpers import BF16_TOL, FP8_TOL, assert_close, new_args, padded_offsets, rows_by_expert, to_np

pytestmark = pytest.mark.gpu
DEV = "cuda"
BF = torch.bfloat16


def B():
    from mixture_experts_grouped_gmm_gb300 import binding

    return binding


def fill(gs, E, M):
    args = new_args(E, DEV)
    B().mgemm_fill_args(gs, E, M, args)
    return args


def sample_rows(sizes, per_group=3, seed=0):
    """First, last and a random row of every non-empty group, sorted."""
    rng = np.random.default_rng(seed)
    off = np.concatenate([[0], np.cumsum(sizes)])
    rows = []
    for e in range(len(sizes)):
        if sizes[e] > 0:
            rows += [off[e], off[e + 1] - 1] + list(rng.integers(off[e], off[e + 1], per_group - 2))
    return np.unique(np.asarray(rows, dtype=np.int64))


def test_grin_fwd_bwd_full_size():
    d = workloads.grin(device=DEV)
    M, K, N, E = d["M"], d["K"], d["N"], d["E"]
    sizes = d["group_sizes"].cpu().numpy()
    args = fill(d["group_sizes"], E, M)
    out = torch.empty(M, N, dtype=BF, device=DEV)
    gx = torch.empty(M, K, dtype=BF, device=DEV)
    gw = torch.empty(E, K, N, dtype=BF, device=DEV)
    go = torch.ones(M, N, dtype=BF, device=DEV)          # loss = out.sum()
    # the bench's launches: fill, fwd, and the backward in one launch
    assert B().mgemm_dgrad_wgrad_split(M, K, N, E) > 0
    B().mgemm_fwd(args, 0, 0, d["x"], None, d["w"], None, out, M, K, N, E)
    B().mgemm_dgrad_wgrad(args, go, d["w"], d["x"], gx, gw, M, K, N, E)
    torch.cuda.synchronize()
    # bit for bit the two separate calls
    gx2, gw2 = torch.empty_like(gx), torch.empty_like(gw)
    B().mgemm_dgrad(args, 0, go, None, d["w"], None, gx2, M, K, N, E)
    B().mgemm_wgrad(args, 0, d["x"], None, go, None, gw2, M, K, N, E)
    torch.cuda.synchronize()
    assert torch.equal(gx, gx2) and torch.equal(gw, gw2)
    del gx2, gw2
    rows = sample_rows(sizes, 4)
    rt = torch.as_tensor(rows, device=DEV)
    sub = rows_by_expert(sizes, rows)
    rng = np.random.default_rng(1)
    ns = torch.as_tensor(np.sort(rng.choice(N, 384, replace=False)), device=DEV)
    kk = torch.as_tensor(np.sort(rng.choice(K, 256, replace=False)), device=DEV)
    xs = to_np(d["x"][rt])
    assert_close(to_np(out[rt][:, ns]), og.gmm_fwd(xs, to_np(d["w"][:, :, ns]), sub), BF16_TOL, "grin fwd")
    assert_close(to_np(gx[rt][:, kk]), og.gmm_dgrad(np.ones((len(rows), N)), to_np(d["w"][:, kk, :]), sub),
                 BF16_TOL, "grin dgrad")
    ks = torch.as_tensor(np.sort(rng.choice(K, 12, replace=False)), device=DEV)
    ref = og.gmm_wgrad(to_np(d["x"][:, ks]), np.ones((M, len(ns))), sizes)       # [E, 12, 384]
    assert_close(to_np(gw[:, ks][:, :, ns]), ref, BF16_TOL, "grin wgrad")


def quant_rows(t):
    R, C = t.shape
    q = torch.empty(R, C, dtype=torch.uint8, device=DEV)
    s = torch.empty(R, dtype=torch.float32, device=DEV)
    B().mgemm_quant_rowwise(t, q, s)
    return q, s


@pytest.fixture(scope="module")
def sparse_weights():
    d = workloads.sparse_m(1, device=DEV)            # w_nk [128, 8192, 5120] bf16 (seeded)
    E, N, K = d["w_nk"].shape
    wq, sw = quant_rows(d["w_nk"].view(E * N, K))
    torch.cuda.synchronize()
    ns = np.sort(np.random.default_rng(2).choice(N, 96, replace=False))
    # the rowwise quantize of the weights is bit-exact on sampled rows (e, n)
    for e in (0, 77, 127):
        q_ref, s_ref = oq.quant_rowwise(to_np(d["w_nk"][e, torch.as_tensor(ns[:8], device=DEV)]))
        assert np.array_equal(to_np(wq.view(E, N, K)[e, torch.as_tensor(ns[:8], device=DEV)]), q_ref)
        assert np.array_equal(to_np(sw.view(E, N)[e, torch.as_tensor(ns[:8], device=DEV)]), s_ref)
    yield dict(wq=wq, sw=sw, E=E, N=N, K=K, ns=ns)
    del d


@pytest.mark.parametrize("total_m", [1, 2, 4, 16, 64, 256])
def test_sparse_m_fp8_full_size(sparse_weights, total_m):
    W = sparse_weights
    E, N, K = W["E"], W["N"], W["K"]
    d = workloads.sparse_m(total_m, device=DEV, with_weights=False)
    sizes = d["group_sizes"].cpu().numpy()
    args = fill(d["group_sizes"], E, total_m)
    xq, sx = quant_rows(d["x"])
    out = torch.empty(total_m, N, dtype=BF, device=DEV)
    B().mgemm_fwd(args, 1, 1, xq, sx, W["wq"], W["sw"], out, total_m, K, N, E)
    torch.cuda.synchronize()
    q_ref, s_ref = oq.quant_rowwise(to_np(d["x"]))
    assert np.array_equal(to_np(xq), q_ref) and np.array_equal(to_np(sx), s_ref)
    rows = np.arange(total_m) if total_m <= 16 else sample_rows(sizes, 3)[:24]
    ns = W["ns"]
    sub = rows_by_expert(sizes, rows)
    experts = [e for e in range(E) if sub[e] > 0]
    # oracle on the touched experts and sampled columns only
    wq_s = to_np(W["wq"].view(E, N, K)[torch.as_tensor(experts, device=DEV)][:, torch.as_tensor(ns, device=DEV)])
    sw_s = to_np(W["sw"].view(E, N)[torch.as_tensor(experts, device=DEV)][:, torch.as_tensor(ns, device=DEV)])
    ref = og.gmm_fwd_fp8(to_np(xq)[rows], to_np(sx)[rows], wq_s, sw_s, [sub[e] for e in experts])
    got = to_np(out)[rows][:, ns]
    assert_close(got, ref, FP8_TOL, f"sparse-M fwd total_M={total_m}")


@pytest.mark.parametrize("proj", ["up", "down"])
def test_deepseek_fp8_step_full_size(proj):
    # the up projection (K = 2048 -> N = 1408) and the down projection (K = 1408 -> N = 2048)
    d = workloads.deepseek(device=DEV, **({} if proj == "up" else {"H": 1408, "F": 2048}))
    M, K, N, E = d["M"], d["K"], d["N"], d["E"]
    sizes = d["group_sizes"].cpu().numpy()
    assert (sizes == 0).sum() >= 1
    w_kn = d["w"]                                    # [E, K, N] master
    w_nk = w_kn.transpose(1, 2).contiguous()
    args = fill(d["group_sizes"], E, M)
    xq, sx = quant_rows(d["x"])
    goq, sgo = quant_rows(d["grad_out"])
    wq, sw = quant_rows(w_nk.view(E * N, K))
    wdq, swd = quant_rows(w_kn.view(E * K, N))
    ld = B().mgemm_colwise_ld(M, E)
    xqt = torch.empty(K * ld, dtype=torch.uint8, device=DEV)
    goqt = torch.empty(N * ld, dtype=torch.uint8, device=DEV)
    sxc = torch.empty(E * K, dtype=torch.float32, device=DEV)
    sgoc = torch.empty(E * N, dtype=torch.float32, device=DEV)
    B().mgemm_quant_colwise_grouped(args, E, M, d["grad_out"], goqt, sgoc, d["x"], xqt, sxc, ld=ld)
    out = torch.empty(M, N, dtype=BF, device=DEV)
    gx = torch.empty(M, K, dtype=BF, device=DEV)
    gw = torch.empty(E, K, N, dtype=BF, device=DEV)
    B().mgemm_fwd(args, 1, 1, xq, sx, wq, sw, out, M, K, N, E)
    B().mgemm_dgrad(args, 1, goq, sgo, wdq, swd, gx, M, K, N, E)
    B().mgemm_wgrad(args, 1, xqt, sxc, goqt, sgoc, gw, M, K, N, E, ld=ld)
    torch.cuda.synchronize()

    rows = sample_rows(sizes, 3, seed=4)
    rt = torch.as_tensor(rows, device=DEV)
    # rowwise quantize: bit-exact on sampled rows
    q_ref, s_ref = oq.quant_rowwise(to_np(d["x"][rt]))
    assert np.array_equal(to_np(xq[rt]), q_ref) and np.array_equal(to_np(sx[rt]), s_ref)
    # colwise dual: bit-exact on sampled columns, every group (gathered from the padded layout)
    offs = np.concatenate([[0], np.cumsum(sizes)])
    po = padded_offsets(sizes)
    keep = torch.as_tensor(np.concatenate([np.arange(po[g], po[g] + int(m)) for g, m in enumerate(sizes)]),
                           device=DEV)
    for tens, qt, sc, C, cs in ((d["x"], xqt, sxc, K, [0, 1, 777, K - 1]), (d["grad_out"], goqt, sgoc, N, [0, 5, N - 1])):
        ct = torch.as_tensor(cs, device=DEV)
        qr, sr = oq.quant_colwise_grouped(to_np(tens[:, ct]), offs)
        assert np.array_equal(to_np(qt.view(C, ld)[ct][:, keep]), qr)
        assert np.array_equal(to_np(sc.view(E, C)[:, ct]), sr.reshape(E, len(cs)))
    # GEMMs on sampled rows and output columns
    sub = rows_by_expert(sizes, rows)
    rng = np.random.default_rng(5)
    ns = torch.as_tensor(np.sort(rng.choice(N, 64, replace=False)), device=DEV)
    ks = torch.as_tensor(np.sort(rng.choice(K, 64, replace=False)), device=DEV)
    ref_f = og.gmm_fwd_fp8(to_np(xq[rt]), to_np(sx[rt]), to_np(wq.view(E, N, K)[:, ns]),
                           to_np(sw.view(E, N)[:, ns]), sub)
    assert_close(to_np(out[rt][:, ns]), ref_f, FP8_TOL, "deepseek fwd")
    ref_d = og.gmm_dgrad_fp8(to_np(goq[rt]), to_np(sgo[rt]), to_np(wdq.view(E, K, N)[:, ks]),
                             to_np(swd.view(E, K)[:, ks]), sub)
    assert_close(to_np(gx[rt][:, ks]), ref_d, FP8_TOL, "deepseek dgrad")
    k6 = ks[:6]
    ref_w = og.gmm_wgrad_fp8(to_np(xqt.view(K, ld)[k6][:, keep]), to_np(sxc.view(E, K)[:, k6]).reshape(-1),
                             to_np(goqt.view(N, ld)[ns][:, keep]), to_np(sgoc.view(E, N)[:, ns]).reshape(-1), sizes)
    assert_close(to_np(gw[:, k6][:, :, ns]), ref_w, FP8_TOL, "deepseek wgrad")
    for e in np.nonzero(sizes == 0)[0]:
        assert bool((gw[int(e)] == 0).all())


def test_mixtral_up_down_full_size():
    d = workloads.mixtral(device=DEV)
    M, H, F, E = d["M"], d["H"], d["F"], d["E"]
    sizes = d["group_sizes"].cpu().numpy()
    args = fill(d["group_sizes"], E, M)
    up = torch.empty(M, 2 * F, dtype=BF, device=DEV)
    B().mgemm_fwd(args, 0, 0, d["x"], None, d["w1"], None, up, M, H, 2 * F, E)
    h = (torch.nn.functional.silu(up[:, :F].float()) * up[:, F:].float()).to(BF)
    down = torch.empty(M, H, dtype=BF, device=DEV)
    B().mgemm_fwd(args, 0, 0, h, None, d["w2"], None, down, M, F, H, E)
    torch.cuda.synchronize()
    rows = sample_rows(sizes, 3, seed=6)
    rt = torch.as_tensor(rows, device=DEV)
    sub = rows_by_expert(sizes, rows)
    cols = np.sort(np.random.default_rng(7).choice(2 * F, 512, replace=False))
    ct = torch.as_tensor(cols, device=DEV)
    experts = [e for e in range(E) if sub[e] > 0]
    w1s = to_np(d["w1"][:, :, ct])
    assert_close(to_np(up[rt][:, ct]), og.gmm_fwd(to_np(d["x"][rt]), w1s, sub), BF16_TOL, "mixtral up")
    c2 = torch.as_tensor(np.sort(np.random.default_rng(8).choice(H, 256, replace=False)), device=DEV)
    assert_close(to_np(down[rt][:, c2]), og.gmm_fwd(to_np(h[rt]), to_np(d["w2"][:, :, c2]), sub), BF16_TOL,
                 "mixtral down")
    assert len(experts) == E


def test_mixtral_routed_layer_full_size():
    # moe.fused_experts at the benchmark's Mixtral shape and launch configuration
    # (same routing, weights viewed as [E, 2F, H] / [E, H, F]); sampled tokens
    # recomputed one by one in float64 by the oracle, one expert at a time
    from mixture_experts_grouped_gmm_gb300 import moe
    from oracle.routing import fused_moe_token

    d = workloads.mixtral(device=DEV)
    T, H, F, E = d["T"], d["H"], d["F"], d["E"]
    w1 = d["w1"].view(E, 2 * F, H)
    w2 = d["w2"].view(E, H, F)
    g = torch.Generator(device=DEV).manual_seed(1)
    x = torch.randn(T, H, generator=g, device=DEV).to(BF)
    tw = d["topk_weights"].to(DEV)
    tid = d["topk_ids"].to(DEV).to(torch.int32)
    out = moe.fused_experts(x, w1, w2, tw, tid)
    torch.cuda.synchronize()
    toks = np.unique(np.concatenate([[0, T - 1], np.random.default_rng(9).integers(0, T, 10)]))
    ids, wts, xs = tid.cpu().numpy(), tw.cpu().numpy(), to_np(x)
    ref = np.zeros((len(toks), H))
    for e in range(E):
        users = [(i, t, j) for i, t in enumerate(toks) for j in range(ids.shape[1]) if ids[t, j] == e]
        if not users:
            continue
        w1e, w2e = {e: to_np(w1[e]).astype(np.float64)}, {e: to_np(w2[e]).astype(np.float64)}
        for i, t, j in users:
            ref[i] += fused_moe_token(xs[t], w1e, w2e, [e], [wts[t, j]])
        del w1e, w2e
    assert_close(to_np(out[torch.as_tensor(toks, device=DEV)]), ref, BF16_TOL, "mixtral routed layer")
