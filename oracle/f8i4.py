"""FP8 x INT4 grouped GEMM for sparse M (oracle; test infrastructure only).

Source: "F8I4 Grouped Gemm Optimization for Sparse M" (pytorch/FBGEMM PR
#3854), title and Summary: a grouped GEMM of FP8 activations and INT4 weights,
whose problems are set up for min(total_M, groups) groups, so that at
total_M = 1 with 128 groups the latency is about 3x lower.  The page gives no
INT4 packing, no weight-scale format and no activation quantization.

Readings (the plainest ones the rest of this build supports):
* Activations: the rowwise FP8 quantize of this build (``quant.quant_rowwise``:
  e4m3 codes and one power-of-two fp32 scale per row, x_q = x * s).
* Weights: stored like the FP8 forward weights, w[E, N, K] (one row per output
  column n, contraction K contiguous).  Values are two's-complement 4-bit
  integers q in [-8, 7], packed two per byte along K: byte j of a row holds
  element 2j in its low nibble and element 2j + 1 in its high nibble.
* Weight scales: one per block of 32 consecutive K elements of a row (the MX
  block of this build), with the power-of-two rule of the FP8 quantizers moved
  to the INT4 range: s = 2^floor(log2(fp32(7 / max(amax, 1e-12)))), amax the
  block's magnitude maximum; q = clamp(round_half_even(w * s), -8, 7) (w * s is
  exact, s being a power of two; s <= 7 / amax keeps |q| <= 7, so -8 is never
  produced, though it decodes).  The scale is stored as the e8m0 byte of the
  decode factor 1 / s: byte = 127 - log2(s), in [85, 253] for every finite
  bf16 input (amax = 0 gives s = 2^42, byte 85).
* The GEMM multiplies decoded values and divides by the row scale of x:
  out[r, n] = (1 / sx[r]) * sum_k e4m3(xq[r, k]) * q[e, n, k] * 2^(byte - 127),
  e the group of row r; outputs are bf16 (the rounding is the caller's).

Every integer in [-8, 7] is an exact e4m3 value and the row scale of x is a
power of two, so the same product is an MXFP8 product (``mx.gmm_fwd_mx``) of
the e4m3 codes of q with the weight bytes and x's codes with the byte
127 - log2(sx[r]) on every block of row r; the tests pin this oracle to that.

Arithmetic: float64 numpy, one ``np.matmul`` per group as the contraction.
"""

import numpy as np

from .formats import decode_e4m3

I4_BLOCK = 32
I4_MAX = 7.0
E8M0_BIAS = 127
EPS = 1e-12


def int4_block_scale(amax):
    """amax (float64 >= 0, any shape) -> (s, byte): the power-of-two scale of
    each block and the e8m0 byte 127 - log2(s) of its decode factor."""
    amax = np.asarray(amax, dtype=np.float64)
    s64 = I4_MAX / np.maximum(amax, EPS)
    s32 = s64.astype(np.float32).astype(np.float64)   # rounded once to fp32 (nearest even)
    _, ex = np.frexp(s32)                              # s32 = f * 2^ex, f in [0.5, 1)
    log2s = ex - 1
    s = np.ldexp(1.0, log2s)
    byte = (E8M0_BIAS - log2s).astype(np.int64)
    return s, byte


def quant_int4_rows(w):
    """w: [R, K] float64 holding bf16 values, K % 32 == 0 ->
    (q int8 [R, K] in [-8, 7], e8m0 bytes uint8 [R, K // 32])."""
    w = np.asarray(w, dtype=np.float64)
    R, K = w.shape
    assert K % I4_BLOCK == 0
    wb = w.reshape(R, K // I4_BLOCK, I4_BLOCK)
    amax = np.max(np.abs(wb), axis=2) if K else np.zeros((R, 0))
    s, byte = int4_block_scale(amax)
    q = np.rint(wb * s[:, :, None])                   # np.rint rounds half to even
    q = np.clip(q, -8, 7).astype(np.int8).reshape(R, K)
    assert np.all((byte >= 0) & (byte <= 254))
    return q, byte.astype(np.uint8)


def pack_int4(q):
    """int8 [R, K] in [-8, 7], K even -> uint8 [R, K // 2]: element 2j in the
    low nibble of byte j, element 2j + 1 in the high nibble (two's complement)."""
    q = np.asarray(q, dtype=np.int64)
    assert q.shape[-1] % 2 == 0 and np.all((q >= -8) & (q <= 7))
    nib = q & 0xF
    return (nib[..., 0::2] | (nib[..., 1::2] << 4)).astype(np.uint8)


def unpack_int4(p):
    """uint8 [R, K // 2] -> int8 [R, K]: the inverse of ``pack_int4``."""
    p = np.asarray(p, dtype=np.int64)
    lo, hi = p & 0xF, (p >> 4) & 0xF
    out = np.empty(p.shape[:-1] + (2 * p.shape[-1],), dtype=np.int64)
    out[..., 0::2], out[..., 1::2] = lo, hi
    return np.where(out >= 8, out - 16, out).astype(np.int8)


def decode_int4(q, byte):
    """q int8 [R, K], bytes uint8 [R, K // 32] -> float64 values q * 2^(byte - 127)."""
    q = np.asarray(q, dtype=np.float64)
    R, K = q.shape
    f = np.ldexp(1.0, np.asarray(byte, dtype=np.int64) - E8M0_BIAS)
    return (q.reshape(R, K // I4_BLOCK, I4_BLOCK) * f[:, :, None]).reshape(R, K)


def gmm_fwd_f8i4(xq, sx, wp, wb, group_sizes):
    """xq uint8 [M, K] e4m3 codes + sx [M] row scales; wp uint8 [E, N, K // 2]
    packed INT4 + wb uint8 [E, N, K // 32] e8m0 bytes -> out [M, N] float64.
    Only the non-empty groups contribute rows (an empty group has none)."""
    x = decode_e4m3(xq) / np.asarray(sx, dtype=np.float64)[:, None]
    E, N, Kh = np.asarray(wp).shape
    K = 2 * Kh
    out = np.zeros((x.shape[0], N))
    off = np.concatenate([[0], np.cumsum(np.asarray(group_sizes, dtype=np.int64))])
    for e in range(E):
        r0, r1 = int(off[e]), int(off[e + 1])
        if r1 > r0:
            w = decode_int4(unpack_int4(wp[e]), np.asarray(wb[e]).reshape(N, K // I4_BLOCK))
            out[r0:r1] = x[r0:r1] @ w.T
    return out
