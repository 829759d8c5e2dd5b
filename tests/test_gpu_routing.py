"""GPU parity of mgemm_moe_align against oracle.routing.moe_align_block_size.

The result is unique (stable order inside each expert), so every output is
compared bit for bit: sorted_ids over its whole buffer, expert_ids, the padded
total and the padded group sizes.  Cases: the worked example of the
docstring, the workload shapes (DeepSeek-MoE 16384 tokens x top-6 over 64
experts, Mixtral 4096 x top-2 over 8, sparse decode rows over 128 experts),
ragged chunk tails, out-of-range ids, empty experts, no entries, block sizes 1
and 4096, and 1024 experts."""

import json
import os

import numpy as np
import pytest
import torch

from oracle.routing import moe_align_block_size

pytestmark = pytest.mark.gpu
DEV = "cuda"
GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "moe_align_example.json")


def B():
    from mixture_experts_grouped_gmm_gb300 import binding

    return binding


def run_gpu(ids, E, block, with_sizes=True):
    t = torch.as_tensor(np.asarray(ids, dtype=np.int32)).to(DEV)
    n = t.numel()
    cap, max_blocks = B().moe_align_buffer_sizes(n, E, block)
    sid = torch.full((cap + 64,), -7, dtype=torch.int32, device=DEV)        # guard entries past the buffer
    eid = torch.full((max_blocks + 64,), -7, dtype=torch.int32, device=DEV)
    npp = torch.full((2,), -7, dtype=torch.int32, device=DEV)
    gs = torch.full((E + 1,), -7, dtype=torch.int64, device=DEV) if with_sizes else None
    ws = torch.empty(B().mgemm_moe_align_workspace_bytes(n, E), dtype=torch.uint8, device=DEV)
    B().mgemm_moe_align(t, E, block, sid, eid, npp, ws, gs)
    torch.cuda.synchronize()
    assert (sid[cap:] == -7).all() and (eid[max_blocks:] == -7).all() and int(npp[1]) == -7
    if with_sizes:
        assert int(gs[E]) == -7
    return (sid[:cap].cpu().tolist(), eid[:max_blocks].cpu().tolist(), int(npp[0]),
            gs[:E].cpu().tolist() if with_sizes else None)


def compare(ids, E, block, with_sizes=True):
    sid, eid, total, gs = run_gpu(ids, E, block, with_sizes)
    r_sid, r_eid, r_total, r_gs = moe_align_block_size(ids, block, E)
    assert total == r_total
    assert sid == r_sid
    assert eid == r_eid
    if with_sizes:
        assert gs == r_gs


def test_worked_example():
    g = json.load(open(GOLDEN))
    compare(g["topk_ids"], g["num_experts"], g["block_size"])
    sid, _, total, _ = run_gpu(g["topk_ids"], g["num_experts"], g["block_size"])
    assert sid[:total] == g["sorted_token_ids_prefix"]


def zipf_ids(T, k, E, s, seed, empty=4):
    """Top-k experts per token, drawn without replacement from a Zipf(s) popularity
    over a seeded permutation, with `empty` experts never chosen."""
    rng = np.random.default_rng(seed)
    perm = rng.permutation(E)
    pop = 1.0 / np.arange(1, E + 1) ** s
    pop[-empty:] = 0 if empty else pop[-empty:]
    pop = pop / pop.sum()
    out = np.empty((T, k), dtype=np.int32)
    for t in range(T):
        out[t] = perm[rng.choice(E, size=k, replace=False, p=pop)]
    return out


@pytest.mark.parametrize("T,k,E,block,seed", [
    (4096, 2, 8, 128, 1),     # Mixtral routing shape
    (1000, 6, 64, 128, 2),    # ragged chunk tail (6000 entries)
    (3, 1, 128, 128, 3),      # sparse decode rows
    (300, 4, 1024, 16, 4),    # 1024 experts, most empty
    (513, 3, 5, 1, 5),        # block size 1: no padding
    (70, 2, 3, 4096, 6),      # block size 4096
])
def test_uniform_routing(T, k, E, block, seed):
    ids = np.random.default_rng(seed).integers(0, E, size=(T, k)).astype(np.int32)
    compare(ids, E, block)


def test_deepseek_shape_zipf():
    # 16384 tokens x top-6 over 64 experts, Zipf(1.2) popularity, 4 experts never chosen
    ids = zipf_ids(16384, 6, 64, 1.2, seed=0)
    compare(ids, 64, 128)


def test_out_of_range_ids_and_no_group_sizes():
    rng = np.random.default_rng(9)
    ids = rng.integers(-3, 12, size=(2500, 2)).astype(np.int32)
    compare(ids, 10, 8, with_sizes=False)


def test_no_entries():
    compare(np.zeros((0, 2), dtype=np.int32), 4, 16)


def test_repeat_is_identical():
    ids = np.random.default_rng(11).integers(0, 16, size=(5000, 2)).astype(np.int32)
    a = run_gpu(ids, 16, 64)
    b = run_gpu(ids, 16, 64)
    assert a == b
