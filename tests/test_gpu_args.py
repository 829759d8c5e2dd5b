"""GPU parity of mgemm_fill_args against oracle.args.fill_args: bit-exact
offsets, active list, tile prefix and wgrad order, and the status codes."""

import numpy as np
import pytest
import torch

from oracle.args import fill_args
from tests.helpers import new_args, padded_offsets, parse_args

pytestmark = pytest.mark.gpu
DEV = "cuda"


def run_fill(sizes, M=None):
    from mixture_experts_grouped_gmm_gb300 import binding as B

    E = len(sizes)
    M = int(np.sum(sizes)) if M is None else M
    gs = torch.tensor(np.asarray(sizes, dtype=np.int64), device=DEV)
    args = new_args(E, DEV)
    B.mgemm_fill_args(gs, E, M, args)
    torch.cuda.synchronize()
    return parse_args(args, E)


def compare(sizes):
    E = len(sizes)
    got = run_fill(sizes)
    ref = fill_args(sizes, int(np.sum(sizes)), 128)
    assert got["status"] == ref["status"] == 0
    assert got["E"] == E and got["M"] == int(np.sum(sizes))
    assert got["offsets"] == ref["offsets"]
    assert got["n_active"] == ref["n_active"]
    na = ref["n_active"]
    assert got["active"][:na] == ref["active"]
    assert got["mtile_start"][:na + 1] == ref["mtile_start"]
    assert got["wgrad_order"] == ref["wgrad_order"]
    assert got["poffsets"] == padded_offsets(sizes)
    # row-tile pairs (256 rows) of the active groups, prefix summed (header: ptile_start)
    pairs = [0]
    for m in sizes:
        if m > 0:
            pairs.append(pairs[-1] + (-(-int(m) // 128) + 1) // 2)
    assert got["ptile_start"][:na + 1] == pairs


@pytest.mark.parametrize("E", [1, 2, 4, 8, 31, 32, 33, 64, 128, 129, 500, 1000, 1024])
def test_fill_args_random(E):
    rng = np.random.default_rng(E)
    for trial in range(4):
        sizes = rng.integers(0, 400, E)
        sizes[rng.random(E) < 0.35] = 0
        if trial == 1:
            sizes = rng.integers(0, 4, E)            # many ties
        if trial == 2:
            sizes = np.zeros(E, dtype=np.int64)
            sizes[rng.integers(0, E)] = 1            # one token, one group (sparse M)
        if trial == 3:
            sizes = np.full(E, 128)                  # all equal
        compare(sizes.tolist())


def test_fill_args_all_empty():
    compare([0, 0, 0, 0])


def test_fill_args_status_codes():
    assert run_fill([3, -1, 4], M=6)["status"] == 1
    assert run_fill([3, 1, 4], M=9)["status"] == 2
    assert run_fill([3, 1, 4], M=8)["status"] == 0


def test_fill_args_is_deterministic():
    sizes = np.random.default_rng(5).integers(0, 50, 300).tolist()
    a = run_fill(sizes)
    b = run_fill(sizes)
    assert a == b
