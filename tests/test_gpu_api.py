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
