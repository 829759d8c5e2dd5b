"""Host logic of the gmm autograd op (CPU, no kernels run): which library calls
its forward and backward make.  The binding's calls are replaced by recorders,
so only the Python dispatch is exercised."""

import pytest
import torch

from mixture_experts_grouped_gmm_gb300 import binding as B
from mixture_experts_grouped_gmm_gb300.gmm import gmm

CALLS = ["mgemm_fill_args", "mgemm_fwd", "mgemm_dgrad", "mgemm_wgrad", "mgemm_dgrad_wgrad"]


@pytest.fixture
def recorded(monkeypatch):
    log = []
    for name in CALLS:
        monkeypatch.setattr(B, name, (lambda n: lambda *a, **k: log.append(n))(name))
    monkeypatch.setattr(B, "mgemm_args_bytes", lambda E: 64 + 32 * E)
    return log


def run(trans_b, grad_x, grad_w):
    M, K, N, E = 16, 32, 48, 2
    x = torch.zeros(M, K, dtype=torch.bfloat16, requires_grad=grad_x)
    w = torch.zeros((E, N, K) if trans_b else (E, K, N), dtype=torch.bfloat16, requires_grad=grad_w)
    out = gmm(x, w, torch.tensor([8, 8]), trans_b=trans_b)
    out.float().sum().backward()


@pytest.mark.parametrize("trans_b,grad_x,grad_w,expect", [
    (False, True, True, ["mgemm_dgrad_wgrad"]),                      # both gradients: one call
    (False, True, False, ["mgemm_dgrad"]),
    (False, False, True, ["mgemm_wgrad"]),
    (True, True, True, ["mgemm_fwd", "mgemm_wgrad"]),                 # w [E, N, K]: grad_x is a forward GEMM
])
def test_gmm_calls(recorded, trans_b, grad_x, grad_w, expect):
    run(trans_b, grad_x, grad_w)
    assert recorded[:2] == ["mgemm_fill_args", "mgemm_fwd"]
    assert recorded[2:] == expect
