"""Pins for oracle.args.fill_args: exhaustive small cases checked against the
properties the pages fix (sizes sum to M, rows contiguous by expert, only
non-empty groups scheduled, at most min(M, E) of them, wgrad problems sorted by
contraction length descending), plus hand-worked examples."""

import itertools

import pytest

from oracle.args import fill_args


def check_valid(sizes, M, a, tile_m):
    E = len(sizes)
    assert a["status"] == 0
    off = a["offsets"]
    assert len(off) == E + 1 and off[0] == 0 and off[E] == M
    for e in range(E):
        assert off[e + 1] - off[e] == sizes[e]
    nz = [e for e in range(E) if sizes[e] > 0]
    assert a["active"] == nz
    assert a["n_active"] == len(nz) <= min(M, E)
    ms = a["mtile_start"]
    assert len(ms) == len(nz) + 1 and ms[0] == 0
    for i, e in enumerate(nz):
        t = ms[i + 1] - ms[i]
        assert (t - 1) * tile_m < sizes[e] <= t * tile_m     # t = ceil(m / tile_m) >= 1
    order = a["wgrad_order"]
    assert sorted(order) == list(range(E))
    for i in range(E - 1):
        p, q = order[i], order[i + 1]
        assert sizes[p] > sizes[q] or (sizes[p] == sizes[q] and p < q)


@pytest.mark.parametrize("E", [1, 2, 3, 4])
def test_exhaustive_small(E):
    for M in range(0, 9):
        for sizes in itertools.product(range(M + 1), repeat=E):
            if sum(sizes) != M:
                continue
            for tile_m in (1, 2, 3, 128):
                check_valid(list(sizes), M, fill_args(sizes, M, tile_m), tile_m)


def test_status_codes():
    assert fill_args([1, -1, 2], 2)["status"] == 1
    assert fill_args([-5, 10], 3)["status"] == 1          # negative checked first
    assert fill_args([1, 2, 3], 7)["status"] == 2
    assert fill_args([1, 2, 3], 6)["status"] == 0
    assert fill_args([0, 0], 0)["status"] == 0


def test_hand_worked_example():
    # sizes 0,3,0,130,5 (M = 138): offsets are running sums; groups 1, 3, 4 are
    # non-empty; row tiles of 128: 1, 2, 1; wgrad order 130 > 5 > 3 > 0 = 0.
    a = fill_args([0, 3, 0, 130, 5], 138, 128)
    assert a["offsets"] == [0, 0, 3, 3, 133, 138]
    assert a["active"] == [1, 3, 4]
    assert a["mtile_start"] == [0, 1, 3, 4]
    assert a["wgrad_order"] == [3, 4, 1, 0, 2]


def test_sparse_m_single_token_many_groups():
    # one routed token among 128 groups: one problem, one row tile
    sizes = [0] * 128
    sizes[77] = 1
    a = fill_args(sizes, 1, 128)
    assert a["active"] == [77] and a["mtile_start"] == [0, 1]
    assert a["wgrad_order"][0] == 77


def test_grin_sizes():
    a = fill_args([128] * 8, 1024, 128)
    assert a["offsets"] == [128 * i for i in range(9)]
    assert a["mtile_start"] == list(range(9))
    assert a["wgrad_order"] == list(range(8))      # all equal: ascending id
