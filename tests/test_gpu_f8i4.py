"""GPU parity of the FP8 x INT4 row ("F8I4 Grouped Gemm Optimization for Sparse
M", FBGEMM PR #3854): mgemm_quant_int4 bit for bit against oracle.f8i4 (packed
nibbles and e8m0 bytes, including every finite bf16 magnitude as a block
maximum), and mgemm_fwd_f8i4 against the oracle's GEMM element by element at
the FP8 tolerance (3e-2 * max|ref|) on ragged, empty and one-row groups, in
both tile forms (64-wide for few rows per group, 128-wide beyond), with K not a
multiple of the kernel's blocks per stage, guard rows untouched, a poisoned
status word, integer-valued inputs bit-exact after bf16 rounding, and the
sparse-M shape (E=128, K=5120, N=8192) on sampled columns."""

import numpy as np
import pytest
import torch

from oracle import f8i4 as of
from oracle import formats
from tests.helpers import FP8_TOL, assert_close, is_sentinel, new_args, sentinel_bf16, to_np

pytestmark = pytest.mark.gpu
DEV = "cuda"
BF = torch.bfloat16


def B():
    from mixture_experts_grouped_gmm_gb300 import binding

    return binding


def quant_int4_gpu(w):
    E, N, K = w.shape
    packed = torch.empty(E, N, K // 2, dtype=torch.uint8, device=DEV)
    sf = torch.empty(B().int4_scale_bytes(E, N, K), dtype=torch.uint8, device=DEV)
    B().mgemm_quant_int4(w, packed, sf)
    return packed, sf


def sf_rows(sf, E, N, K):
    """[E][K/128][N][4] (the kernel's layout) -> [E, N, K/32]."""
    return to_np(sf).reshape(E, K // 128, N, 4).transpose(0, 2, 1, 3).reshape(E, N, K // 32)


def quant_rows_gpu(t):
    R, C = t.shape
    q = torch.empty(R, C, dtype=torch.uint8, device=DEV)
    s = torch.empty(R, dtype=torch.float32, device=DEV)
    B().mgemm_quant_rowwise(t, q, s)
    return q, s


def test_quant_int4_bit_exact():
    g = torch.Generator(device=DEV).manual_seed(0)
    E, N, K = 3, 72, 384
    w = torch.randn(E, N, K, generator=g, device=DEV)
    w = w * torch.exp2(torch.randint(-40, 40, (E, N, K // 32, 1), generator=g, device=DEV).float()).repeat_interleave(
        32, dim=2).view(E, N, K)
    w[0, 3, 32:64] = 0.0                 # an all-zero block
    w[1, 5, :32] = 1e-30                 # tiny
    w = w.to(BF)
    packed, sf = quant_int4_gpu(w)
    torch.cuda.synchronize()
    q_ref, b_ref = of.quant_int4_rows(to_np(w).reshape(E * N, K))
    assert np.array_equal(to_np(packed).reshape(E * N, K // 2), of.pack_int4(q_ref))
    assert np.array_equal(sf_rows(sf, E, N, K).reshape(E * N, K // 32), b_ref)


def test_quant_int4_every_bf16_magnitude():
    # block maxima over every finite positive bf16 value: the scale byte is bit-exact
    mags = torch.arange(1, 0x7F80, dtype=torch.int32, device=DEV).to(torch.int16).view(BF)
    nb = mags.numel()
    K = 128
    rows = -(-nb // (K // 32))
    blocks = torch.zeros(rows * (K // 32), 32, dtype=BF, device=DEV)
    blocks[:nb, 0] = mags
    blocks[:nb, 1] = -(mags.float() * 0.37).to(BF)     # a second value below the maximum
    w = blocks.view(1, rows, K)
    packed, sf = quant_int4_gpu(w)
    torch.cuda.synchronize()
    q_ref, b_ref = of.quant_int4_rows(to_np(w)[0])
    assert np.array_equal(sf_rows(sf, 1, rows, K)[0], b_ref)
    assert np.array_equal(to_np(packed)[0], of.pack_int4(q_ref))


def f8i4_problem(sizes, K, N, seed, scale=0.02):
    M, E = int(np.sum(sizes)), len(sizes)
    g = torch.Generator(device=DEV).manual_seed(seed)
    x = torch.randn(M, K, generator=g, device=DEV).to(BF)
    w = (torch.randn(E, N, K, generator=g, device=DEV) * scale).to(BF)
    xq, sx = quant_rows_gpu(x)
    packed, sf = quant_int4_gpu(w)
    return M, E, x, w, xq, sx, packed, sf


def run_f8i4(sizes, K, N, xq, sx, packed, sf, guard=8):
    M, E = int(np.sum(sizes)), len(sizes)
    args = new_args(E, DEV)
    B().mgemm_fill_args(torch.tensor(sizes, dtype=torch.int64, device=DEV), E, M, args)
    out = sentinel_bf16((M + guard, N), DEV)
    B().mgemm_fwd_f8i4(args, xq, sx, packed, sf, out, M, K, N, E)
    torch.cuda.synchronize()
    return args, out


F8I4_CASES = [
    ([1, 0, 0, 2, 0, 1, 0, 0, 0, 3], 512, 256),      # 7 rows, sparse groups: CTA pairs, one slot each
    ([2, 0, 5], 5120, 1024),                         # 7 rows, the sparse-M contraction: pairs, 10 slots each
    ([5, 0, 37, 30, 2], 384, 200),                   # K = 3 blocks (not a multiple of 4), N % 64 != 0
    ([0, 300, 1, 129, 250, 0, 0, 24], 256, 136),     # 128-wide tiles, group edges inside tiles
    ([700], 640, 320),                               # E = 1
    ([130, 0, 257, 64, 1], 128, 64),                 # one block of K
]


@pytest.mark.parametrize("sizes,K,N", F8I4_CASES)
def test_fwd_f8i4_against_oracle(sizes, K, N):
    M, E, x, w, xq, sx, packed, sf = f8i4_problem(sizes, K, N, 11)
    _, out = run_f8i4(sizes, K, N, xq, sx, packed, sf)
    assert is_sentinel(out[M:]), "wrote past the M rows"
    ref = of.gmm_fwd_f8i4(to_np(xq), to_np(sx), to_np(packed), sf_rows(sf, E, N, K), sizes)
    assert_close(to_np(out[:M]), ref, FP8_TOL, "f8i4 fwd")
    # the quantized product also tracks the bf16 one (quantization error only)
    from oracle import gmm as og

    assert_close(to_np(out[:M]), og.gmm_fwd(to_np(x), to_np(w), sizes, trans_b=True), 0.25, "f8i4 vs bf16")


@pytest.mark.parametrize("sizes,K,N", [([3, 0, 4, 1], 384, 128), ([200, 140], 256, 256),
                                       ([3, 0, 4, 1], 1024, 128)])   # 8 rows, K = 1024: CTA pairs split K
def test_fwd_f8i4_integer_inputs_bit_exact(sizes, K, N):
    # x in {-3..3} (codes x * 128 exact), w integers in [-7, 7] with a 7 in every
    # block (scale 1): every product and partial sum is an integer below 2^24, so
    # the fp32 accumulation is exact and the bf16 output equals the oracle's rounding
    M, E = int(np.sum(sizes)), len(sizes)
    g = torch.Generator(device=DEV).manual_seed(5)
    x = torch.randint(-3, 4, (M, K), generator=g, device=DEV).float()
    x[:, 0] = 3.0
    w = torch.randint(-7, 8, (E, N, K), generator=g, device=DEV).float()
    w[:, :, ::32] = 7.0
    xq, sx = quant_rows_gpu(x.to(BF))
    packed, sf = quant_int4_gpu(w.to(BF))
    _, out = run_f8i4(sizes, K, N, xq, sx, packed, sf)
    ref = of.gmm_fwd_f8i4(to_np(xq), to_np(sx), to_np(packed), sf_rows(sf, E, N, K), sizes)
    assert np.array_equal(to_np(out[:M]), formats.round_bf16(ref))


def test_fwd_f8i4_poisoned_status_writes_nothing():
    sizes, K, N = [3, 0, 9], 256, 128
    M, E, x, w, xq, sx, packed, sf = f8i4_problem(sizes, K, N, 3)
    args = new_args(E, DEV)
    B().mgemm_fill_args(torch.tensor(sizes, dtype=torch.int64, device=DEV), E, M, args)
    args[0] = 1
    out = sentinel_bf16((M, N), DEV)
    B().mgemm_fwd_f8i4(args, xq, sx, packed, sf, out, M, K, N, E)
    torch.cuda.synchronize()
    assert is_sentinel(out)


@pytest.mark.parametrize("total_m", [1, 4, 16])
def test_fwd_f8i4_sparse_m_shape(total_m):
    # E = 128, K = 5120, N = 8192, tokens routed to random experts (the sparse-M
    # workload), checked on 256 sampled columns
    from mixture_experts_grouped_gmm_gb300 import workloads

    E, K, N = 128, 5120, 8192
    d = workloads.sparse_m(total_m, E=E, K=K, N=N, device=DEV, with_weights=False)
    sizes = d["group_sizes"].tolist()
    touched = [e for e in range(E) if sizes[e]]
    g = torch.Generator(device=DEV).manual_seed(total_m)
    w = torch.zeros(E, N, K, dtype=BF, device=DEV)
    for e in touched:
        w[e] = (torch.randn(N, K, generator=g, device=DEV) * 0.02).to(BF)
    xq, sx = quant_rows_gpu(d["x"])
    packed, sf = quant_int4_gpu(w)
    _, out = run_f8i4(sizes, K, N, xq, sx, packed, sf)
    cols = np.sort(np.random.default_rng(total_m).choice(N, 256, replace=False))
    ct = torch.as_tensor(cols, device=DEV)
    sfr = sf_rows(sf, E, N, K)[:, cols]
    ref = of.gmm_fwd_f8i4(to_np(xq), to_np(sx), to_np(packed[:, ct]), sfr, sizes)
    assert_close(to_np(out[:total_m][:, ct]), ref, FP8_TOL, "f8i4 sparse-M")
