"""GPU checks of the public Python surface: the autograd ``gmm`` op (forward
and backward through the C ABI, both weight layouts) against the oracle, and
calls into the library from a thread other than the one that loaded it (the
autograd engine runs backward on its own threads)."""

import numpy as np
import pytest
import torch

from oracle import gmm as og
from tests.helpers import BF16_TOL, assert_close, to_np
from tests.test_gpu_gmm import BF, DEV, B, fill, rand_bf16

pytestmark = pytest.mark.gpu


def test_autograd_gmm_matches_oracle():
    from mixture_experts_grouped_gmm_gb300 import gmm

    sizes, K, N = [0, 300, 1, 129, 250], 320, 520
    M, E = int(np.sum(sizes)), len(sizes)
    gs = torch.tensor(sizes, dtype=torch.int64, device=DEV)
    for trans_b in (False, True):
        x = rand_bf16((M, K), 11, "normal").requires_grad_(True)
        w = rand_bf16((E, N, K) if trans_b else (E, K, N), 12, "normal").requires_grad_(True)
        out = gmm(x, w, gs, trans_b=trans_b)
        G = rand_bf16((M, N), 13, "normal")
        out.backward(G)
        torch.cuda.synchronize()
        xs, ws, Gs = to_np(x), to_np(w), to_np(G)
        wk = ws.transpose(0, 2, 1) if trans_b else ws            # [E, K, N]
        assert_close(to_np(out), og.gmm_fwd(xs, wk, sizes), BF16_TOL, "autograd fwd")
        assert_close(to_np(x.grad), og.gmm_dgrad(Gs, wk, sizes), BF16_TOL, "autograd dgrad")
        gw = og.gmm_wgrad(xs, Gs, sizes)
        if trans_b:
            gw = gw.transpose(0, 2, 1)
        assert_close(to_np(w.grad), gw, BF16_TOL, "autograd wgrad")


def test_calls_from_another_thread():
    # autograd runs backward on its own thread; the library must work there too
    import threading

    sizes, K, N = [0, 300, 1, 129, 250], 320, 520
    M, E = int(np.sum(sizes)), len(sizes)
    args = fill(sizes)
    go, w = rand_bf16((M, N), 3, "normal"), rand_bf16((E, K, N), 4, "normal")
    gx = torch.empty(M, K, dtype=BF, device=DEV)
    err = []

    def work():
        try:
            B().mgemm_dgrad(args, 0, go, None, w, None, gx, M, K, N, E)
            torch.cuda.synchronize()
        except Exception as e:  # surfaced below
            err.append(e)

    th = threading.Thread(target=work)
    th.start()
    th.join()
    assert not err, err
    assert_close(to_np(gx), og.gmm_dgrad(to_np(go), to_np(w), sizes), BF16_TOL, "dgrad from a thread")


@pytest.mark.parametrize("sizes,K,N", [([0, 300, 1, 129, 250], 320, 272), ([5, 0, 2], 128, 64), ([700], 256, 128)])
def test_fwd_fp8_strided_equals_contiguous(sizes, K, N):
    # the same codes laid out as the padded column-major output of the colwise
    # cast (w[e, n, k] at n ld + e Kp + k) give the contiguous [E, N, K] result bit for bit
    M, E = int(np.sum(sizes)), len(sizes)
    args = fill(sizes)
    g = torch.Generator(device=DEV).manual_seed(3)
    xq = torch.randint(0, 0x7E, (M, K), generator=g, device=DEV).to(torch.uint8)
    wq = torch.randint(0, 0x7E, (E, N, K), generator=g, device=DEV).to(torch.uint8)
    sx = torch.exp2(torch.randint(-4, 4, (M,), generator=g, device=DEV).float())
    sw = torch.exp2(torch.randint(-4, 4, (E * N,), generator=g, device=DEV).float())
    Kp = -(-K // 128) * 128
    ld = E * Kp + 128
    ws = torch.zeros(N, ld, dtype=torch.uint8, device=DEV)
    for e in range(E):
        ws[:, e * Kp:e * Kp + K] = wq[e]
    a = torch.empty(M, N, dtype=BF, device=DEV)
    b = torch.empty(M, N, dtype=BF, device=DEV)
    B().mgemm_fwd(args, B().MGEMM_FP8_E4M3, 1, xq, sx, wq, sw, a, M, K, N, E)
    B().mgemm_fwd_fp8_strided(args, xq, sx, ws, ld, Kp, sw, b, M, K, N, E)
    torch.cuda.synchronize()
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))


def test_autograd_gmm_fp8_matches_oracle():
    # the FP8 training op on bf16 master tensors: forward, dgrad and wgrad against
    # the oracle's own quantization of the same inputs (FP8 tolerance)
    from mixture_experts_grouped_gmm_gb300 import gmm_fp8
    from oracle import quant as oq

    from tests.helpers import FP8_TOL

    sizes, K, N = [0, 300, 1, 129, 250], 320, 272
    M, E = int(np.sum(sizes)), len(sizes)
    gs = torch.tensor(sizes, dtype=torch.int64, device=DEV)
    x = rand_bf16((M, K), 21, "normal").requires_grad_(True)
    w = (rand_bf16((E, K, N), 22, "normal").float() * 0.05).to(BF).requires_grad_(True)
    G = rand_bf16((M, N), 23, "normal")
    out = gmm_fp8(x, w, gs)
    out.backward(G)
    torch.cuda.synchronize()
    xs, ws, Gs = to_np(x), to_np(w), to_np(G)
    offs = np.concatenate([[0], np.cumsum(sizes)])
    xq, sx = oq.quant_rowwise(xs)
    wt, sw = oq.quant_colwise_grouped(ws.reshape(E * K, N), np.arange(E + 1) * K)   # per (e, n) over K
    wq = wt.reshape(N, E, K).transpose(1, 0, 2)                                       # [E, N, K]
    assert_close(to_np(out), og.gmm_fwd_fp8(xq, sx, wq, sw, sizes), FP8_TOL, "fp8 op fwd")
    goq, sgo = oq.quant_rowwise(Gs)
    wdq, swd = oq.quant_rowwise(ws.reshape(E * K, N))
    assert_close(to_np(x.grad), og.gmm_dgrad_fp8(goq, sgo, wdq.reshape(E, K, N), swd, sizes), FP8_TOL, "fp8 op dgrad")
    (gqt, sgc), (xqt, sxc) = oq.quant_colwise_grouped_dual(Gs, xs, offs)
    assert_close(to_np(w.grad), og.gmm_wgrad_fp8(xqt, sxc, gqt, sgc, sizes), FP8_TOL, "fp8 op wgrad")
    # and the FP8 result tracks the bf16 one (quantization error only)
    assert_close(to_np(out), og.gmm_fwd(xs, ws, sizes), 0.1, "fp8 op vs bf16")
