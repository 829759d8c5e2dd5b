"""Every call is CUDA-graph capturable and never reads the group sizes on the
host: each pipeline is captured once, then replayed after new inputs --
including new group sizes and new routing -- are written into the captured
buffers, and each replay must equal (bit for bit) the same calls run eagerly
on those inputs.  Covers the bf16 training step (fill, fwd, dgrad, wgrad; and
with the one-launch backward mgemm_dgrad_wgrad), the
FP8 step (rowwise and dual colwise quantize, fwd, dgrad, wgrad; the colwise
work counter must come back to 0 between replays) and the routed layer from
gating logits (routing, alignment, gather, gated GEMM, scattered GEMM, top-k
sum)."""

import pytest
import torch

from tests.helpers import new_args

pytestmark = pytest.mark.gpu
DEV = "cuda"
BF = torch.bfloat16
U8 = torch.uint8


def B():
    from mixture_experts_grouped_gmm_gb300 import binding

    return binding


def capture(fn):
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        fn()  # warm-up outside the graph (one-time attribute setup)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fn()
    return g


def test_bf16_step_graph_replays_with_new_sizes():
    E, M, K, N = 6, 700, 192, 264
    gs = torch.zeros(E, dtype=torch.int64, device=DEV)
    x = torch.empty(M, K, dtype=BF, device=DEV)
    w = torch.empty(E, K, N, dtype=BF, device=DEV)
    go = torch.empty(M, N, dtype=BF, device=DEV)
    args = new_args(E, DEV)
    out = torch.empty(M, N, dtype=BF, device=DEV)
    gx = torch.empty(M, K, dtype=BF, device=DEV)
    gw = torch.empty(E, K, N, dtype=BF, device=DEV)

    def step(a=args, o=out, g_x=gx, g_w=gw):
        B().mgemm_fill_args(gs, E, M, a)
        B().mgemm_fwd(a, 0, 0, x, None, w, None, o, M, K, N, E)
        B().mgemm_dgrad(a, 0, go, None, w, None, g_x, M, K, N, E)
        B().mgemm_wgrad(a, 0, x, None, go, None, g_w, M, K, N, E)

    graph = capture(step)
    for rep, sizes in enumerate(([100, 0, 250, 50, 300, 0], [0, 700, 0, 0, 0, 0], [117, 117, 117, 117, 116, 116])):
        gs.copy_(torch.tensor(sizes, dtype=torch.int64))
        x.copy_(torch.randn(M, K, device=DEV).to(BF))
        w.copy_(torch.randn(E, K, N, device=DEV).to(BF))
        go.copy_(torch.randn(M, N, device=DEV).to(BF))
        graph.replay()
        torch.cuda.synchronize()
        a2 = new_args(E, DEV)
        o2, gx2, gw2 = torch.empty_like(out), torch.empty_like(gx), torch.empty_like(gw)
        step(a2, o2, gx2, gw2)
        torch.cuda.synchronize()
        assert torch.equal(out, o2) and torch.equal(gx, gx2) and torch.equal(gw, gw2), f"replay {rep}"


def test_bf16_step_one_launch_backward_graph_replays_with_new_sizes():
    # the same step with mgemm_dgrad_wgrad (its one-launch form at these sizes):
    # each replay equals the separate calls run eagerly, bit for bit
    E, M, K, N = 6, 700, 192, 264
    assert B().mgemm_dgrad_wgrad_split(M, K, N, E) > 0
    gs = torch.zeros(E, dtype=torch.int64, device=DEV)
    x = torch.empty(M, K, dtype=BF, device=DEV)
    w = torch.empty(E, K, N, dtype=BF, device=DEV)
    go = torch.empty(M, N, dtype=BF, device=DEV)
    args = new_args(E, DEV)
    out = torch.empty(M, N, dtype=BF, device=DEV)
    gx = torch.empty(M, K, dtype=BF, device=DEV)
    gw = torch.empty(E, K, N, dtype=BF, device=DEV)

    def step():
        B().mgemm_fill_args(gs, E, M, args)
        B().mgemm_fwd(args, 0, 0, x, None, w, None, out, M, K, N, E)
        B().mgemm_dgrad_wgrad(args, go, w, x, gx, gw, M, K, N, E)

    graph = capture(step)
    for rep, sizes in enumerate(([100, 0, 250, 50, 300, 0], [0, 700, 0, 0, 0, 0], [117, 117, 117, 117, 116, 116])):
        gs.copy_(torch.tensor(sizes, dtype=torch.int64))
        x.copy_(torch.randn(M, K, device=DEV).to(BF))
        w.copy_(torch.randn(E, K, N, device=DEV).to(BF))
        go.copy_(torch.randn(M, N, device=DEV).to(BF))
        graph.replay()
        torch.cuda.synchronize()
        a2 = new_args(E, DEV)
        o2, gx2, gw2 = torch.empty_like(out), torch.empty_like(gx), torch.empty_like(gw)
        B().mgemm_fill_args(gs, E, M, a2)
        B().mgemm_fwd(a2, 0, 0, x, None, w, None, o2, M, K, N, E)
        B().mgemm_dgrad(a2, 0, go, None, w, None, gx2, M, K, N, E)
        B().mgemm_wgrad(a2, 0, x, None, go, None, gw2, M, K, N, E)
        torch.cuda.synchronize()
        assert torch.equal(out, o2) and torch.equal(gx, gx2) and torch.equal(gw, gw2), f"replay {rep}"


def test_fp8_step_graph_replays():
    E, M, K, N = 5, 640, 256, 144
    ld = B().mgemm_colwise_ld(M, E)
    gs = torch.zeros(E, dtype=torch.int64, device=DEV)
    x = torch.empty(M, K, dtype=BF, device=DEV)
    go = torch.empty(M, N, dtype=BF, device=DEV)
    wq = torch.empty(E * N, K, dtype=U8, device=DEV)   # [E, N, K] e4m3
    sw = torch.empty(E * N, device=DEV)
    args = new_args(E, DEV)

    def alloc():
        return dict(xq=torch.empty(M, K, dtype=U8, device=DEV), sx=torch.empty(M, device=DEV),
                    gq=torch.empty(M, N, dtype=U8, device=DEV), sg=torch.empty(M, device=DEV),
                    xc=torch.zeros(K * ld, dtype=U8, device=DEV), sxc=torch.empty(E * K, device=DEV),
                    gc=torch.zeros(N * ld, dtype=U8, device=DEV), sgc=torch.empty(E * N, device=DEV),
                    out=torch.empty(M, N, dtype=BF, device=DEV), gw=torch.empty(E, K, N, dtype=BF, device=DEV))

    def step(a, b):
        B().mgemm_fill_args(gs, E, M, a)
        B().mgemm_quant_rowwise(x, b["xq"], b["sx"])
        B().mgemm_fwd(a, 1, 1, b["xq"], b["sx"], wq, sw, b["out"], M, K, N, E)
        B().mgemm_quant_colwise_grouped(a, E, M, go, b["gc"], b["sgc"], x, b["xc"], b["sxc"], ld=ld)
        B().mgemm_wgrad(a, 1, b["xc"], b["sxc"], b["gc"], b["sgc"], b["gw"], M, K, N, E, ld=ld)

    bufs = alloc()
    graph = capture(lambda: step(args, bufs))
    for rep, sizes in enumerate(([128, 0, 300, 12, 200], [640, 0, 0, 0, 0], [1, 2, 3, 4, 630])):
        gs.copy_(torch.tensor(sizes, dtype=torch.int64))
        x.copy_(torch.randn(M, K, device=DEV).to(BF))
        go.copy_(torch.randn(M, N, device=DEV).to(BF))
        wq.copy_(torch.randint(0, 0x70, (E * N, K), dtype=U8, device=DEV))
        sw.copy_(torch.rand(E * N, device=DEV) + 0.5)
        graph.replay()
        torch.cuda.synchronize()
        assert int(args[12:16].view(torch.int32).item()) == 0, "colwise work counter handed back at 0"
        a2, b2 = new_args(E, DEV), alloc()
        step(a2, b2)
        torch.cuda.synchronize()
        for k in ("xq", "sx", "out", "sxc", "sgc", "gw"):
            assert torch.equal(bufs[k], b2[k]), f"replay {rep}: {k}"
        # column-major codes: each column's groups and their zero padding (the
        # bytes past the padded total are not part of the output)
        P = sum((m + 127) // 128 * 128 for m in sizes)
        for k, C in (("xc", K), ("gc", N)):
            assert torch.equal(bufs[k].view(C, ld)[:, :P], b2[k].view(C, ld)[:, :P]), f"replay {rep}: {k}"


@pytest.mark.parametrize("T,H", [
    (40, 128),   # routing kernel, then the one-CTA alignment of the given ids
    (1, 256),    # decode: routing + alignment + args in one launch, the first GEMM gathering its rows
    (4, 256),
    (16, 128),   # the largest batch of the one-launch routing and of the gathering GEMM (32 entries)
])
def test_routed_layer_graph_replays_with_new_routing(T, H):
    from mixture_experts_grouped_gmm_gb300 import moe

    E, F, k = 8, 256, 2
    x = torch.empty(T, H, dtype=BF, device=DEV)
    gating = torch.empty(T, E, device=DEV)
    w1 = (0.05 * torch.randn(E, 2 * F, H, device=DEV)).to(BF)
    w2 = (0.05 * torch.randn(E, H, F, device=DEV)).to(BF)
    res = {}

    def layer():
        res["y"] = moe.fused_moe(x, w1, w2, gating, k, True)

    x.copy_(torch.randn(T, H, device=DEV).to(BF))
    gating.copy_(torch.randn(T, E, device=DEV))
    graph = capture(layer)
    for rep in range(3):
        x.copy_(torch.randn(T, H, device=DEV).to(BF))
        gating.copy_(torch.randn(T, E, device=DEV) * (rep + 1))
        graph.replay()
        torch.cuda.synchronize()
        y_graph = res["y"].clone()
        y_eager = moe.fused_moe(x, w1, w2, gating, k, True)
        torch.cuda.synchronize()
        assert torch.equal(y_graph, y_eager), f"replay {rep}"
