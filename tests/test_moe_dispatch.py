"""Host logic of moe.fused_moe / moe.fused_experts (CPU, no kernels run): which
library calls each batch size takes.  The binding's calls are replaced by
recorders, so only the Python dispatch is exercised."""

import pytest
import torch

from mixture_experts_grouped_gmm_gb300 import binding as B
from mixture_experts_grouped_gmm_gb300 import moe

CALLS = ["mgemm_topk_softmax", "mgemm_moe_align", "mgemm_moe_route_align", "mgemm_fill_args", "mgemm_gather_rows",
         "mgemm_fwd_gated", "mgemm_fwd_gated_gather", "mgemm_fwd_scatter", "mgemm_topk_sum"]


@pytest.fixture
def recorded(monkeypatch):
    log = []
    for name in CALLS:
        monkeypatch.setattr(B, name, (lambda n: lambda *a, **k: log.append(n))(name))
    monkeypatch.setattr(B, "mgemm_args_bytes", lambda E: 64 + 32 * E)
    monkeypatch.setattr(B, "mgemm_moe_align_workspace_bytes", lambda n, E: 16)
    return log


def layer(T, E, H, F, k):
    x = torch.zeros(T, H, dtype=torch.bfloat16)
    w1 = torch.zeros(E, 2 * F, H, dtype=torch.bfloat16)
    w2 = torch.zeros(E, H, F, dtype=torch.bfloat16)
    return x, w1, w2


@pytest.mark.parametrize("T,H,expect", [
    (1, 256, ["mgemm_moe_route_align", "mgemm_fwd_gated_gather", "mgemm_fwd_scatter", "mgemm_topk_sum"]),
    (16, 128, ["mgemm_moe_route_align", "mgemm_fwd_gated_gather", "mgemm_fwd_scatter", "mgemm_topk_sum"]),
    (16, 136, ["mgemm_moe_route_align", "mgemm_gather_rows", "mgemm_fwd_gated", "mgemm_fwd_scatter",
               "mgemm_topk_sum"]),                                   # H % 64 != 0: the gather copy
    (17, 256, ["mgemm_topk_softmax", "mgemm_moe_route_align", "mgemm_gather_rows", "mgemm_fwd_gated",
               "mgemm_fwd_scatter", "mgemm_topk_sum"]),              # routed over many CTAs, ids aligned in one
    (2049, 128, ["mgemm_topk_softmax", "mgemm_moe_align", "mgemm_fill_args", "mgemm_gather_rows",
                 "mgemm_fwd_gated", "mgemm_fwd_scatter", "mgemm_topk_sum"]),  # 4098 entries: three-kernel align
])
def test_fused_moe_calls(recorded, T, H, expect):
    x, w1, w2 = layer(T, 8, H, 64, 2)
    moe.fused_moe(x, w1, w2, torch.zeros(T, 8), 2, True)
    assert recorded == expect


def test_fused_experts_aligns_given_ids_in_one_launch_up_to_the_limit(recorded):
    x, w1, w2 = layer(2048, 8, 128, 64, 2)
    moe.fused_experts(x, w1, w2, torch.zeros(2048, 2), torch.zeros(2048, 2, dtype=torch.int32))
    assert recorded[0] == "mgemm_moe_route_align"        # 4096 entries: the limit
    recorded.clear()
    x, w1, w2 = layer(2049, 8, 128, 64, 2)
    moe.fused_experts(x, w1, w2, torch.zeros(2049, 2), torch.zeros(2049, 2, dtype=torch.int32))
    assert recorded[:2] == ["mgemm_moe_align", "mgemm_fill_args"]


def test_fused_moe_rejects_non_bf16(recorded):
    x, w1, w2 = layer(1, 8, 128, 64, 2)
    with pytest.raises(B.MgemmError):
        moe.fused_moe(x.float(), w1, w2, torch.zeros(1, 8), 2, True)
    assert recorded == []
