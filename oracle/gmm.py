"""Grouped GEMM forward / dgrad / wgrad (oracle; test infrastructure only).

Sources:
* "Support GPU-resident batch sizes" (tgale96/grouped_gemm PR #21):
  the benchmark script calls ``gg.ops.gmm(x, w, batch_sizes)`` with
  x[M, K], w[E, K, N] and batch_sizes of E entries summing to M (rows of x are
  contiguous by expert), then ``out.sum().backward()``; the review of
  csrc/grouped_gemm.cu shows ``CutlassGroupedGemm<trans_a, trans_b>`` and
  ops_test.py loops over ``trans_b``.  Reading: forward out_e = x_e @ w[e]
  (w[e] transposed when trans_b, i.e. w stored [E, N, K]); dgrad
  grad_x_e = grad_out_e @ w[e]^T; wgrad grad_w[e] = x_e^T @ grad_out_e, a
  contraction over the m_e rows of group e ("dynamic k"), zero when m_e = 0
  (ZeroOutK0Outputs).
* "[moe training] Optimize FP8 MoE backward pass" (pytorch/ao commit 34322b5):
  operands are quantized as A_scaled = A * scale, so the FP8 product is
  divided by the scales.  Forward: x rowwise (one scale per row); backward
  grad_A: grad_output rowwise; backward grad_B: grad_output and A per group
  and column.

Readings for the FP8 weight scales (not printed): forward w is e4m3 stored
[E, N, K] with one scale per (e, n); dgrad w is e4m3 stored [E, K, N] with one
scale per (e, k); outputs are bf16.

Arithmetic: every product and sum in float64 over the values exactly as
stored (bf16 values, or decoded e4m3 codes); ``np.matmul`` is the contraction
primitive; rounding to bf16 is left to the caller (formats.round_bf16).
"""

import numpy as np

from .formats import decode_e4m3


def _bounds(group_sizes):
    off = np.concatenate([[0], np.cumsum(np.asarray(group_sizes, dtype=np.int64))])
    return [(int(off[e]), int(off[e + 1])) for e in range(len(group_sizes))]


def gmm_fwd(x, w, group_sizes, trans_b=False):
    """x [M, K]; w [E, K, N] (or [E, N, K] with trans_b) -> out [M, N] float64."""
    x = np.asarray(x, dtype=np.float64)
    w = np.asarray(w, dtype=np.float64)
    N = w.shape[1] if trans_b else w.shape[2]
    out = np.zeros((x.shape[0], N))
    for e, (r0, r1) in enumerate(_bounds(group_sizes)):
        if r1 > r0:
            we = w[e].T if trans_b else w[e]
            out[r0:r1] = x[r0:r1] @ we
    return out


def gmm_dgrad(grad_out, w, group_sizes):
    """grad_out [M, N]; w [E, K, N] -> grad_x [M, K] = grad_out_e @ w[e]^T."""
    go = np.asarray(grad_out, dtype=np.float64)
    w = np.asarray(w, dtype=np.float64)
    gx = np.zeros((go.shape[0], w.shape[1]))
    for e, (r0, r1) in enumerate(_bounds(group_sizes)):
        if r1 > r0:
            gx[r0:r1] = go[r0:r1] @ w[e].T
    return gx


def gmm_wgrad(x, grad_out, group_sizes):
    """x [M, K]; grad_out [M, N] -> grad_w [E, K, N] = x_e^T @ grad_out_e."""
    x = np.asarray(x, dtype=np.float64)
    go = np.asarray(grad_out, dtype=np.float64)
    E = len(group_sizes)
    gw = np.zeros((E, x.shape[1], go.shape[1]))
    for e, (r0, r1) in enumerate(_bounds(group_sizes)):
        if r1 > r0:
            gw[e] = x[r0:r1].T @ go[r0:r1]
    return gw


def gmm_fwd_fp8(xq, sx, wq, sw, group_sizes):
    """xq e4m3 [M, K] + sx [M]; wq e4m3 [E, N, K] + sw [E, N] -> out [M, N].

    out[r, n] = (sum_k xq[r, k] * wq[e, n, k]) / (sx[r] * sw[e, n]).
    """
    x = decode_e4m3(xq)
    w = decode_e4m3(wq)
    sx = np.asarray(sx, dtype=np.float64)
    sw = np.asarray(sw, dtype=np.float64).reshape(w.shape[0], w.shape[1])
    out = np.zeros((x.shape[0], w.shape[1]))
    for e, (r0, r1) in enumerate(_bounds(group_sizes)):
        if r1 > r0:
            out[r0:r1] = (x[r0:r1] @ w[e].T) / (sx[r0:r1, None] * sw[e][None, :])
    return out


def gmm_dgrad_fp8(goq, sgo, wq, sw, group_sizes):
    """goq e4m3 [M, N] + sgo [M]; wq e4m3 [E, K, N] + sw [E, K] -> grad_x [M, K]."""
    go = decode_e4m3(goq)
    w = decode_e4m3(wq)
    sgo = np.asarray(sgo, dtype=np.float64)
    sw = np.asarray(sw, dtype=np.float64).reshape(w.shape[0], w.shape[1])
    gx = np.zeros((go.shape[0], w.shape[1]))
    for e, (r0, r1) in enumerate(_bounds(group_sizes)):
        if r1 > r0:
            gx[r0:r1] = (go[r0:r1] @ w[e].T) / (sgo[r0:r1, None] * sw[e][None, :])
    return gx


def gmm_wgrad_fp8(xq_t, sx, goq_t, sgo, group_sizes):
    """Per-group colwise-quantized operands, stored column-major.

    xq_t e4m3 [K, M] (xq_t[k, r] codes x[r, k]) + sx [E * K] (index k + K * e);
    goq_t e4m3 [N, M] + sgo [E * N] (index n + N * e) -> grad_w [E, K, N].
    grad_w[e, k, n] = (sum over rows r of group e of x[r, k] * go[r, n])
                      / (sx[k + K e] * sgo[n + N e]).
    """
    xt = decode_e4m3(xq_t)
    gt = decode_e4m3(goq_t)
    K, N = xt.shape[0], gt.shape[0]
    E = len(group_sizes)
    sx = np.asarray(sx, dtype=np.float64).reshape(E, K)
    sgo = np.asarray(sgo, dtype=np.float64).reshape(E, N)
    gw = np.zeros((E, K, N))
    for e, (r0, r1) in enumerate(_bounds(group_sizes)):
        if r1 > r0:
            gw[e] = (xt[:, r0:r1] @ gt[:, r0:r1].T) / (sx[e][:, None] * sgo[e][None, :])
    return gw


def expert_of_rows(group_sizes, rows):
    """Expert id owning each row index (rows must lie in [0, M))."""
    off = np.cumsum(np.asarray(group_sizes, dtype=np.int64))
    return np.searchsorted(off, np.asarray(rows), side="right")
