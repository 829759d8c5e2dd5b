"""MXFP8 (block-scaled e4m3) quantize and grouped GEMM (oracle; test
infrastructure only).

Source: "[moe training] Optimize FP8 MoE backward pass: fused colwise kernel +
AMD tuning" (pytorch/ao commit 34322b5), commit message: the MXFP8 grouped MM
path exists beside the FP8 one and needs its token groups padded to a multiple
of 32 rows (the FP8 path 16); its tests run on SM100-class GPUs only.  The page
names the format and its block of 32 and prints nothing more.

Readings (the page is silent on the arithmetic):
* A block is 32 consecutive elements of one row along the contraction
  dimension; every block has one shared scale, stored as an e8m0 byte (a bare
  biased exponent: byte b means 2^(b - 127)).
* The block's scale follows the same power-of-two rule as the rowwise and
  colwise quantizers of this build (``quant.pow2_scale``: s = 2^floor(log2(
  fp32(448 / max(amax, 1e-12))))), applied to the block's magnitude maximum;
  codes are the saturating e4m3 cast of x * s.  The e8m0 byte stores the
  decode factor 1 / s = 2^-log2(s), i.e. byte = 127 - log2(s); for every
  finite bf16 input it lies in [79, 254] (amax = 0 gives s = 2^48, byte 79).
* The grouped GEMM multiplies decoded values: operand value = e4m3 value of
  the code times 2^(byte - 127) of its block; for group e,
  out[r, n] = sum_k xv[r, k] * wv[e, n, k] (forward, w stored [E, N, K]);
  dgrad is the same contraction with grad_out and w stored [E, K, N]
  quantized along N.
* wgrad contracts over the token rows of a group, so its blocks run down the
  columns: 32 consecutive rows of one column counted from the group's first
  row (the page's 32-row padding of the groups makes every block whole; here
  a group's last block may be short and its missing rows count as zeros).

Arithmetic: float64 numpy, ``np.matmul`` per group as the contraction.
"""

import numpy as np

from .formats import decode_e4m3, encode_e4m3
from .quant import pow2_scale

MX_BLOCK = 32
E8M0_BIAS = 127


def quant_mx_rows(x):
    """x: [R, K] float64 holding bf16 values, K % 32 == 0 ->
    (codes uint8 [R, K], e8m0 uint8 [R, K // 32])."""
    x = np.asarray(x, dtype=np.float64)
    R, K = x.shape
    assert K % MX_BLOCK == 0
    xb = x.reshape(R, K // MX_BLOCK, MX_BLOCK)
    amax = np.max(np.abs(xb), axis=2) if K else np.zeros((R, 0))
    s = pow2_scale(amax)                                    # [R, K/32], powers of two
    codes = encode_e4m3(xb * s[:, :, None]).reshape(R, K)   # x * s is exact
    _, ex = np.frexp(s)                                     # s = 0.5 * 2^ex
    log2s = ex - 1
    e8m0 = (E8M0_BIAS - log2s).astype(np.int64)
    assert np.all((e8m0 >= 0) & (e8m0 <= 254))
    return codes.astype(np.uint8), e8m0.astype(np.uint8)


def decode_mx(codes, e8m0):
    """codes uint8 [R, K], e8m0 uint8 [R, K // 32] -> float64 values [R, K]."""
    v = decode_e4m3(codes)
    R, K = v.shape
    f = np.ldexp(1.0, np.asarray(e8m0, dtype=np.int64) - E8M0_BIAS)  # [R, K/32]
    return (v.reshape(R, K // MX_BLOCK, MX_BLOCK) * f[:, :, None]).reshape(R, K)


def gmm_fwd_mx(xq, xs, wq, ws, group_sizes):
    """xq [M, K] + xs [M, K/32]; wq [E, N, K] + ws [E, N, K/32] -> out [M, N]."""
    x = decode_mx(xq, xs)
    E, N, K = wq.shape
    w = decode_mx(np.asarray(wq).reshape(E * N, K), np.asarray(ws).reshape(E * N, K // MX_BLOCK)).reshape(E, N, K)
    out = np.zeros((x.shape[0], N))
    off = np.concatenate([[0], np.cumsum(np.asarray(group_sizes, dtype=np.int64))])
    for e in range(E):
        r0, r1 = int(off[e]), int(off[e + 1])
        if r1 > r0:
            out[r0:r1] = x[r0:r1] @ w[e].T
    return out


def quant_mx_colwise_grouped(x, offsets):
    """Per-group colwise MX quantize (the wgrad operands): in each group g
    (rows offsets[g] .. offsets[g+1]) and column c, blocks of 32 consecutive
    rows counted from the group's first row; the last block of a group may be
    short (its missing rows count as zeros, which do not change the maximum).

    x: [M, C] float64 holding bf16 values; offsets: G + 1 exclusive offsets.
    Returns (codes_t uint8 [C, M], e8m0: list over groups of uint8
    [C, ceil(m_g / 32)]).
    """
    x = np.asarray(x, dtype=np.float64)
    M, C = x.shape
    codes_t = np.zeros((C, M), dtype=np.uint8)
    scales = []
    for g in range(len(offsets) - 1):
        r0, r1 = int(offsets[g]), int(offsets[g + 1])
        nb = -(-(r1 - r0) // MX_BLOCK)
        blk = np.zeros((nb * MX_BLOCK, C))
        blk[:r1 - r0] = x[r0:r1]
        q, e = quant_mx_rows(blk.T.copy())          # rows = columns of x, blocks along the group's rows
        codes_t[:, r0:r1] = q[:, :r1 - r0]
        scales.append(e)
    return codes_t, scales


def gmm_wgrad_mx(xq_t, xs, goq_t, gos, group_sizes):
    """grad_w[e] = sum over the rows of group e of x_r^T go_r on decoded MX
    values.  xq_t [K, M], goq_t [N, M] (column-major codes); xs, gos: per-group
    lists of [K or N, ceil(m_e / 32)] e8m0 bytes (blocks along the group's
    rows) -> [E, K, N]; zero for an empty group."""
    K, N = xq_t.shape[0], goq_t.shape[0]
    E = len(group_sizes)
    out = np.zeros((E, K, N))
    off = np.concatenate([[0], np.cumsum(np.asarray(group_sizes, dtype=np.int64))])
    for e in range(E):
        r0, r1 = int(off[e]), int(off[e + 1])
        if r1 == r0:
            continue
        nb = xs[e].shape[1]
        pad = nb * MX_BLOCK - (r1 - r0)
        xa = np.concatenate([xq_t[:, r0:r1], np.zeros((K, pad), dtype=np.uint8)], axis=1)
        ga = np.concatenate([goq_t[:, r0:r1], np.zeros((N, pad), dtype=np.uint8)], axis=1)
        out[e] = decode_mx(xa, xs[e]) @ decode_mx(ga, gos[e]).T
    return out
