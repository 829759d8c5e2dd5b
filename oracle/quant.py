"""FP8 absmax scaling and saturating e4m3 cast (oracle; test infrastructure only).

Source: "[moe training] Optimize FP8 MoE backward pass: fused colwise kernel +
AMD tuning" (pytorch/ao commit 34322b5).
* Commit message: the forward pass of the FP8 grouped MM replaces the 3-op
  sequence  tensor_to_scale(A, axiswise_dim=-1);  A_scaled = A.to(float32) *
  A_scales;  A_fp8 = to_fp8_saturated(A_scaled)  by one fused rowwise kernel;
  the backward pass quantizes grad_output rowwise and (grad_output, A) per
  group and column with one dual kernel.
* bench_colwise_block_configs.py, ``_colwise_kernel``: per group (rows
  offs[g-1] (0 for g = 0) to offs[g]) and column, amax = max |x| over the
  group's rows; s = fp32(fp8_max / clamp(amax, min=EPS)) computed from a
  float64 amax, EPS = 1e-12; s = 2^floor(log2(s)); scale stored at
  ``col + N * g``; q = clamp(x * s, fp8_min, fp8_max) cast to e4m3.
* ``run_experiment``: the colwise output is column-major, i.e. the transpose
  stored row-major (``as_strided(size, (1, M))``).

Readings:
* The rowwise scale formula is not printed; it uses the same rule as the
  printed colwise kernel (power-of-two floor included), applied per row.
* ``floor(log2(s))`` is taken exactly from the binary exponent of the fp32
  value s (s > 0 and normal for every finite input).
* The printed scale-store mask ``arange(BLOCK_SIZE) < N`` is read as
  ``col < N``.
* An empty group has amax = 0, so its scale is pow2floor(fp32(448 / 1e-12))
  = 2^48 for every column; it has no rows to write.
* Offsets here are the exclusive-scan form (length G + 1, offsets[0] = 0):
  group g owns rows [offsets[g], offsets[g+1]), the same ranges as the page's
  end-offset form.
"""

import numpy as np

from .formats import E4M3_MAX, encode_e4m3

EPS = 1e-12


def pow2_scale(amax):
    """amax (float64, >= 0) -> power-of-two fp32 scale, as float64 values."""
    amax = np.asarray(amax, dtype=np.float64)
    s64 = E4M3_MAX / np.maximum(amax, EPS)
    s32 = s64.astype(np.float32).astype(np.float64)   # round to fp32, nearest even
    _, ex = np.frexp(s32)                              # s32 = f * 2^ex, f in [0.5, 1)
    return np.ldexp(1.0, ex - 1)


def quant_rowwise(x):
    """x: [R, C] float64 holding bf16 values -> (codes uint8 [R, C], scales [R])."""
    x = np.asarray(x, dtype=np.float64)
    amax = np.max(np.abs(x), axis=1) if x.shape[1] > 0 else np.zeros(x.shape[0])
    s = pow2_scale(amax)
    q = encode_e4m3(x * s[:, None])        # x * s is exact: s is a power of two
    return q, s


def quant_colwise_grouped(x, offsets):
    """Per-group, per-column quantize.

    x: [M, C] float64 holding bf16 values; offsets: G + 1 exclusive offsets.
    Returns (codes_t uint8 [C, M], scales [G * C]) where ``codes_t[c, r]`` is
    the e4m3 code of x[r, c] (column-major storage of the [M, C] result) and
    ``scales[c + C * g]`` is the scale of column c in group g.
    """
    x = np.asarray(x, dtype=np.float64)
    M, C = x.shape
    G = len(offsets) - 1
    codes_t = np.zeros((C, M), dtype=np.uint8)
    scales = np.zeros(G * C, dtype=np.float64)
    for g in range(G):
        r0, r1 = int(offsets[g]), int(offsets[g + 1])
        blk = x[r0:r1]
        amax = np.max(np.abs(blk), axis=0) if r1 > r0 else np.zeros(C)
        s = pow2_scale(amax)
        scales[g * C:(g + 1) * C] = s
        if r1 > r0:
            codes_t[:, r0:r1] = encode_e4m3(blk * s[None, :]).T
    return codes_t, scales


def quant_colwise_grouped_dual(x1, x2, offsets):
    """The dual form: the same per-group colwise quantize of two tensors that
    share the row groups (grad_output and A in the backward pass)."""
    return quant_colwise_grouped(x1, offsets), quant_colwise_grouped(x2, offsets)
