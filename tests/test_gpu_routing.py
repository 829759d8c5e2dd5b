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


# ---------------------------------------------------------------- mgemm_moe_route_align
# One launch for routing + alignment + args block: every output must equal,
# bit for bit, what mgemm_topk_softmax, mgemm_moe_align and mgemm_fill_args
# (M = -1) write, and the alignment and ids must equal the oracle's.

def _guarded(n, fill, dtype):
    return torch.full((n + 64,), fill, dtype=dtype, device=DEV)


def _fused(gating, ids, T, E, k, renorm, block):
    n = T * k
    cap, mb = B().moe_align_buffer_sizes(n, E, block)
    nb = B().mgemm_args_bytes(E)
    sid, eid = _guarded(cap, -7, torch.int32), _guarded(mb, -7, torch.int32)
    npp, gs = _guarded(1, -7, torch.int32), _guarded(E, -7, torch.int64)
    args = _guarded(nb, 0xA5, torch.uint8)
    if gating is not None:
        w = torch.full((T, k), float("nan"), device=DEV)
        i = torch.full((T, k), -7, dtype=torch.int32, device=DEV)
    else:
        w, i = None, ids.clone()
    B().mgemm_moe_route_align(gating, T, E, k, renorm, block, w, i, sid, eid, npp, args, gs)
    torch.cuda.synchronize()
    assert (sid[cap:] == -7).all() and (eid[mb:] == -7).all() and (npp[1:] == -7).all() and (gs[E:] == -7).all()
    assert (args[nb:] == 0xA5).all()
    return w, i, sid[:cap], eid[:mb], npp[:1], gs[:E], args[:nb]


def _separate(gating, ids, T, E, k, renorm, block):
    n = T * k
    cap, mb = B().moe_align_buffer_sizes(n, E, block)
    nb = B().mgemm_args_bytes(E)
    if gating is not None:
        w = torch.full((T, k), float("nan"), device=DEV)
        i = torch.full((T, k), -7, dtype=torch.int32, device=DEV)
        B().mgemm_topk_softmax(gating, k, renorm, w, i)
    else:
        w, i = None, ids.clone()
    sid = torch.full((cap,), -7, dtype=torch.int32, device=DEV)
    eid = torch.full((mb,), -7, dtype=torch.int32, device=DEV)
    npp = torch.full((1,), -7, dtype=torch.int32, device=DEV)
    gs = torch.full((E,), -7, dtype=torch.int64, device=DEV)
    ws = torch.empty(B().mgemm_moe_align_workspace_bytes(n, E), dtype=torch.uint8, device=DEV)
    B().mgemm_moe_align(i, E, block, sid, eid, npp, ws, gs)
    args = torch.full((nb,), 0xA5, dtype=torch.uint8, device=DEV)
    B().mgemm_fill_args(gs, E, -1, args)
    torch.cuda.synchronize()
    return w, i, sid, eid, npp, gs, args


def _check_route_align(gating, ids, T, E, k, renorm, block):
    from oracle import args as OA
    from oracle import routing as OR

    f = _fused(gating, ids, T, E, k, renorm, block)
    s = _separate(gating, ids, T, E, k, renorm, block)
    names = ("topk_weights", "topk_ids", "sorted_ids", "expert_ids", "num_post_padded", "group_sizes", "args")
    for name, a, b in zip(names, f, s):
        if a is None:
            assert b is None
            continue
        if a.dtype == torch.float32:  # same bits, NaN sentinels included
            a, b = a.view(torch.int32), b.view(torch.int32)
        assert torch.equal(a, b), name
    # the oracle: the alignment of the ids, and the args block of its padded sizes
    ids_np = f[1].cpu().numpy()
    if gating is not None:
        _, r_ids = OR.topk_softmax(gating.cpu().numpy(), k, renorm)
        assert np.array_equal(ids_np, r_ids)
    r_sid, r_eid, r_total, r_gs = moe_align_block_size(ids_np, block, E)
    assert f[2].cpu().tolist() == r_sid and f[3].cpu().tolist() == r_eid
    assert int(f[4][0]) == r_total and f[5].cpu().tolist() == r_gs
    from tests.helpers import parse_args

    got = parse_args(f[6], E)
    ref = OA.fill_args(r_gs, r_total)
    assert got["status"] == ref["status"] and got["n_active"] == ref["n_active"]
    assert got["offsets"] == ref["offsets"] and got["M"] == r_total
    assert got["active"][:ref["n_active"]] == ref["active"]
    assert got["mtile_start"][:ref["n_active"] + 1] == ref["mtile_start"]
    assert got["wgrad_order"] == ref["wgrad_order"]


@pytest.mark.parametrize("T,E,k,renorm,block,kind", [
    (1, 8, 2, True, 128, "normal"),       # Mixtral decode, one token
    (8, 128, 8, True, 128, "normal"),     # the 128-thread form's limits (8 tokens, 128 experts)
    (6, 100, 3, False, 16, "normal"),     # 128 threads, E not a multiple of 32
    (9, 128, 8, True, 128, "normal"),     # one token past it: 1024 threads
    (8, 256, 8, True, 128, "normal"),     # the 256-thread form's limits (DeepSeek-V3-like routing)
    (1, 160, 6, False, 64, "ties"),       # 256 threads, E not a power of two
    (9, 256, 8, True, 128, "normal"),     # one token past it: 1024 threads
    (16, 64, 6, True, 128, "normal"),     # DeepSeek-MoE routing, decode batch
    (64, 128, 8, False, 128, "normal"),   # 512 entries over 128 experts
    (2048, 8, 2, True, 128, "normal"),    # 4096 entries: the largest batch (four placement rounds)
    (4096, 16, 1, False, 64, "normal"),   # 4096 tokens, top-1
    (37, 1024, 4, True, 16, "normal"),    # 1024 experts (NV = 32), most empty
    (300, 64, 6, True, 128, "ties"),      # equal logits go to the lower id
    (5, 3, 3, False, 1, "ties"),          # block size 1, top_k = E
    (9, 40, 2, True, 4096, "normal"),     # block size 4096
    (0, 4, 2, True, 128, "normal"),       # no tokens
])
def test_route_align_matches_separate_calls_and_oracle(T, E, k, renorm, block, kind):
    g = torch.Generator(device=DEV).manual_seed(T * 7 + E)
    if kind == "normal":
        logits = torch.randn(T, E, generator=g, device=DEV)
    else:
        logits = torch.randint(-2, 3, (T, E), generator=g, device=DEV).float()
    _check_route_align(logits, None, T, E, k, renorm, block)


@pytest.mark.parametrize("T,E,k,block,lo", [
    (1000, 10, 4, 8, -3),      # out-of-range ids are not placed
    (3, 128, 1, 128, 0),       # sparse decode rows
    (1024, 1024, 4, 16, 0),    # 4096 entries over 1024 experts
    (7, 2, 5, 128, 0),         # top_k above E (given ids may repeat)
])
def test_route_align_given_ids(T, E, k, block, lo):
    ids = torch.as_tensor(np.random.default_rng(T + E).integers(lo, E + (2 if lo < 0 else 0), size=(T, k))
                          .astype(np.int32)).to(DEV)
    _check_route_align(None, ids, T, E, k, False, block)


def test_route_align_worked_example():
    gd = json.load(open(GOLDEN))
    ids = torch.as_tensor(np.asarray(gd["topk_ids"], dtype=np.int32)).to(DEV)
    T, k = ids.shape
    _, _, sid, _, npp, _, _ = _fused(None, ids, T, gd["num_experts"], k, False, gd["block_size"])
    assert sid[:int(npp[0])].cpu().tolist() == gd["sorted_token_ids_prefix"]


def test_route_align_rejects_more_entries_than_the_limit():
    lim = B().MGEMM_ROUTE_ALIGN_MAX_ENTRIES
    with pytest.raises(B().MgemmError):
        _fused(torch.zeros(lim // 2 + 1, 8, device=DEV), None, lim // 2 + 1, 8, 2, False, 128)
