"""Pins for oracle.routing.moe_align_block_size.

* The worked example printed in the docstring of moe_align_block_size
  (pytorch-labs/applied-ai issue 24, column-major fused MoE script), stored in
  tests/golden/moe_align_example.json.
* An independent construction: numpy's stable argsort of the flat expert ids
  gives the same within-expert order, then padding by arithmetic; compared on
  random inputs and exhaustively on tiny ones.
* Invariants the docstring fixes: every entry placed once, blocks of one
  expert each, padded total divisible by block_size, pad id = numel."""

import itertools
import json
import os

import numpy as np
import pytest

from oracle.routing import buffer_sizes, moe_align_block_size

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "moe_align_example.json")


def test_worked_example():
    g = json.load(open(GOLDEN))
    flat = [v for row in g["topk_ids"] for v in row]
    assert flat == g["flattened"]
    sid, eid, total, gs = moe_align_block_size(g["topk_ids"], g["block_size"], g["num_experts"])
    n = len(flat)
    assert n == g["padding_id"]
    assert total == g["num_tokens_post_padded"]
    assert sid[:total] == g["sorted_token_ids_prefix"]
    cap, max_blocks = buffer_sizes(n, g["num_experts"], g["block_size"])
    assert len(sid) == cap and all(v == n for v in sid[total:])
    assert eid[: total // g["block_size"]] == [1, 2, 3, 4]
    assert len(eid) == max_blocks and all(v == -1 for v in eid[total // g["block_size"]:])
    assert gs == [0, 4, 4, 4, 4]


def by_argsort(flat, block, E):
    """Same result from numpy's stable argsort (invalid ids sort last and are dropped)."""
    flat = np.asarray(flat, dtype=np.int64).ravel()
    n = flat.size
    valid = (flat >= 0) & (flat < E)
    key = np.where(valid, flat, E)
    order = np.argsort(key, kind="stable")
    sid, eid, gs = [], [], []
    for e in range(E):
        ids = order[key[order] == e].tolist()
        p = (len(ids) + block - 1) // block * block
        sid += ids + [n] * (p - len(ids))
        eid += [e] * (p // block)
        gs.append(p)
    return sid, eid, gs


def check(flat, block, E):
    sid, eid, total, gs = moe_align_block_size(flat, block, E)
    s2, e2, g2 = by_argsort(flat, block, E)
    assert sid[:total] == s2 and eid[: total // block] == e2 and gs == g2
    n = len(np.asarray(flat).ravel())
    flat_l = np.asarray(flat).ravel().tolist()
    # invariants
    assert total % block == 0 and total == sum(gs)
    placed = [v for v in sid[:total] if v != n]
    assert sorted(placed) == [i for i, v in enumerate(flat_l) if 0 <= v < E]
    for b in range(total // block):
        blk = sid[b * block:(b + 1) * block]
        real = [v for v in blk if v != n]
        assert real == sorted(real)
        assert all(flat_l[v] == eid[b] for v in real)
        assert blk == real + [n] * (block - len(real))  # padding only at an expert's end
    assert eid[: total // block] == sorted(eid[: total // block])


@pytest.mark.parametrize("T,k,E,block,seed", [
    (64, 2, 8, 16, 0), (100, 6, 64, 128, 1), (7, 3, 5, 4, 2), (1, 1, 128, 128, 3), (333, 4, 16, 1, 4),
    (50, 2, 1024, 8, 5),
])
def test_random_against_argsort(T, k, E, block, seed):
    rng = np.random.default_rng(seed)
    ids = rng.integers(0, E, size=(T, k))
    check(ids, block, E)


def test_invalid_ids_are_not_placed():
    ids = [[0, 5, -1], [2, 2, 9], [4, 0, 1]]
    check(ids, 2, 5)
    sid, eid, total, gs = moe_align_block_size(ids, 2, 5)
    # entries 1, 2 and 5 carry the out-of-range ids 5, -1 and 9
    assert all(i not in sid[:total] for i in (1, 2, 5))
    assert gs == [2, 2, 2, 0, 2]


def test_no_entries():
    sid, eid, total, gs = moe_align_block_size([], 4, 3)
    assert total == 0 and sid == [0] * 9 and eid == [-1] * 2 and gs == [0, 0, 0]


def test_exhaustive_tiny():
    for E in (1, 2, 3):
        for n in range(0, 5):
            for flat in itertools.product(range(-1, E + 1), repeat=n):
                for block in (1, 2, 3):
                    check(list(flat), block, E)


def test_fused_moe_gemm_hand_example():
    # tokens 0..2 with top-2 experts [[0,1],[1,2],[0,2]], block 2: worked by hand
    from oracle.routing import fused_moe_gemm
    sid, eid, tot, _ = moe_align_block_size([[0, 1], [1, 2], [0, 2]], 2, 3)
    A = np.arange(6, dtype=float).reshape(3, 2)
    Bw = np.arange(24, dtype=float).reshape(3, 4, 2)
    out = fused_moe_gemm(A, Bw, sid, eid, tot, 6, 2, 2)
    assert out[0].tolist() == [1, 3, 5, 7]          # token 0 . expert 0
    assert out[4].tolist() == [5, 23, 41, 59]       # token 2 . expert 0
    assert out[5].tolist() == [149, 167, 185, 203]  # token 2 . expert 2
    w = np.array([0.5, 2, 1, 1, 1, 4])
    outw = fused_moe_gemm(A, Bw, sid, eid, tot, 6, 2, 2, topk_weights=w)
    assert np.array_equal(outw, out * w[:, None])


def test_fused_moe_gemm_against_einsum():
    # every entry against a dense per-entry matmul (numpy einsum), padding and
    # out-of-range ids leave NaN rows
    from oracle.routing import fused_moe_gemm
    rng = np.random.default_rng(7)
    T, k, E, K, N, block = 50, 3, 6, 16, 12, 8
    ids = rng.integers(-1, E, size=(T, k))
    sid, eid, tot, _ = moe_align_block_size(ids, block, E)
    A = rng.standard_normal((T, K))
    Bw = rng.standard_normal((E, N, K))
    wts = rng.random(T * k)
    out = fused_moe_gemm(A, Bw, sid, eid, tot, T * k, k, block, topk_weights=wts)
    flat = ids.ravel()
    for i in range(T * k):
        if 0 <= flat[i] < E:
            ref = np.einsum("k,nk->n", A[i // k], Bw[flat[i]]) * wts[i]
            assert np.allclose(out[i], ref, rtol=1e-13, atol=1e-12)
        else:
            assert np.isnan(out[i]).all()


def test_silu_and_mul_closed_forms():
    from scipy.special import expit

    from oracle.routing import silu_and_mul
    x = np.array([[0.0, 1.0, 3.0, -2.0], [50.0, -50.0, 1.0, 1.0]])
    h = silu_and_mul(x)
    assert h.shape == (2, 2)
    assert h[0, 0] == 0.0                                   # silu(0) = 0
    assert np.isclose(h[0, 1], 1.0 * expit(1.0) * -2.0)    # silu(v) = v * sigmoid(v)
    assert np.isclose(h[1, 0], 50.0, rtol=1e-15)            # silu(v) -> v for large v
    assert abs(h[1, 1]) < 1e-19                             # silu(v) -> 0 for very negative v


def test_gather_rows_pads_with_zeros():
    from oracle.routing import gather_rows
    sid, eid, tot, _ = moe_align_block_size([[1, 0], [0, 0]], 4, 2)
    src = np.array([[1.0, 2.0], [3.0, 4.0]])
    g = gather_rows(src, sid, tot, 4, 2)
    # expert 0: entries 1, 2, 3 (tokens 0, 1, 1) + 1 pad; expert 1: entry 0 (token 0) + 3 pads
    assert g.tolist() == [[1, 2], [3, 4], [3, 4], [0, 0], [1, 2], [0, 0], [0, 0], [0, 0]]


def test_topk_softmax_against_torch_and_by_hand():
    import torch

    from oracle.routing import topk_softmax
    rng = np.random.default_rng(3)
    g = rng.standard_normal((64, 16)).astype(np.float32)   # distinct logits: no ties
    w, i = topk_softmax(g, 4, False)
    p = torch.softmax(torch.from_numpy(g).double(), dim=-1)
    tw, ti = torch.topk(p, 4, dim=-1)
    assert np.array_equal(i, ti.numpy()) and np.allclose(w, tw.numpy(), rtol=1e-14)
    wr, ir = topk_softmax(g, 4, True)
    assert np.array_equal(ir, i) and np.allclose(wr.sum(axis=1), 1.0, rtol=1e-14)
    assert np.allclose(wr, w / w.sum(axis=1, keepdims=True), rtol=1e-14)
    # by hand: logits [0, ln 3, ln 3, 0]: probabilities [1/8, 3/8, 3/8, 1/8]; ties -> lower id
    h = np.array([[0.0, np.log(3.0), np.log(3.0), 0.0]])
    w2, i2 = topk_softmax(h, 3, False)
    assert i2.tolist() == [[1, 2, 0]]
    assert np.allclose(w2, [[3 / 8, 3 / 8, 1 / 8]], rtol=1e-14)


def test_fused_moe_token_matches_the_composed_layer():
    # the per-token form against align + fused_moe_gemm + silu_and_mul +
    # fused_moe_gemm (weighted) + sum over the top-k entries
    from oracle.routing import fused_moe_gemm, fused_moe_token, silu_and_mul
    rng = np.random.default_rng(11)
    T, k, E, H, F = 20, 2, 5, 12, 8
    x = rng.standard_normal((T, H))
    w1 = rng.standard_normal((E, 2 * F, H))
    w2 = rng.standard_normal((E, H, F))
    ids = np.stack([rng.permutation(E)[:k] for _ in range(T)])
    wts = rng.random((T, k))
    sid, eid, tot, _ = moe_align_block_size(ids, 4, E)
    c1 = fused_moe_gemm(x, w1, sid, eid, tot, T * k, k, 4)
    c3 = fused_moe_gemm(silu_and_mul(c1), w2, sid, eid, tot, T * k, 1, 4, topk_weights=wts.ravel())
    layer = c3.reshape(T, k, H).sum(axis=1)
    for t in range(T):
        assert np.allclose(fused_moe_token(x[t], w1, w2, ids[t], wts[t]), layer[t], rtol=1e-12, atol=1e-12)
