"""Number formats used by the path: FP8 e4m3fn and bf16, written from their
format definitions (oracle; test infrastructure only).

FP8 e4m3fn -- the NVIDIA variant named ``torch.float8_e4m3fn`` / ``tl.float8e4nv``
in the FP8_DTYPE_MAP of bench_colwise_block_configs.py ("[moe training]
Optimize FP8 MoE backward pass", pytorch/ao commit 34322b5).  The page also
names the AMD ``float8_e4m3fnuz`` (max 240); that variant is not used here.

  byte  = s eeee mmm,  bias 7
  e = 0        : subnormal, value = (-1)^s * m * 2^-9
  1 <= e <= 15 : normal,    value = (-1)^s * (1 + m/8) * 2^(e-7)
  e = 15, m = 7: NaN (no infinities)          -> largest finite = 448

The cast used by the quantize kernels (``_colwise_kernel``: clamp to
[fp8_min, fp8_max], then ``.to(out_dtype)``) is read as: clamp to [-448, 448],
then round to nearest, ties to even, on the e4m3 grid including subnormals,
keeping the sign of zero.

bf16: 1 sign, 8 exponent bits (bias 127), 7 stored mantissa bits.  GEMM outputs
are rounded to bf16 with round-to-nearest-even.
"""

import numpy as np

E4M3_MAX = 448.0
E4M3_MIN_NORMAL_EXP = -6      # smallest normal = 2^-6
E4M3_MANT_BITS = 3
E4M3_NAN_POS = 0x7F


def decode_e4m3(codes):
    """e4m3fn bytes (uint8 array) -> float64 values; S.1111.111 -> NaN."""
    c = np.asarray(codes).astype(np.int64)
    neg = (c & 0x80) != 0
    e = (c >> 3) & 0xF
    m = (c & 0x7).astype(np.float64)
    mag = np.where(e == 0, m * 2.0 ** -9, (1.0 + m / 8.0) * np.exp2(e.astype(np.float64) - 7.0))
    mag = np.where((e == 15) & ((c & 7) == 7), np.nan, mag)
    return np.where(neg, -mag, mag)


def round_e4m3_sat(v):
    """Saturating round-to-nearest-even of float values onto the e4m3 grid.

    Returns float64 values that lie on the grid (NaN stays NaN).  Steps: clamp
    |v| to 448; find the spacing of the grid in |v|'s binade (2^(E-3) for a
    normal binade 2^E, 2^-9 for the subnormal range below 2^-6); round
    |v| / spacing to the nearest integer with ties to even; multiply back.
    Division and multiplication by a power of two are exact in float64.
    """
    v = np.asarray(v, dtype=np.float64)
    neg = np.signbit(v)
    nan = np.isnan(v)
    a = np.minimum(np.abs(np.where(nan, 0.0, v)), E4M3_MAX)
    _, ex = np.frexp(a)                # a = f * 2^ex, f in [0.5, 1)  (a > 0)
    binade = np.maximum(ex - 1, E4M3_MIN_NORMAL_EXP)
    spacing = np.ldexp(1.0, binade - E4M3_MANT_BITS)
    r = np.rint(a / spacing) * spacing  # np.rint rounds half to even
    r = np.where(neg, -r, r)
    return np.where(nan, np.nan, r)


def encode_e4m3(v):
    """float values -> e4m3fn bytes (uint8), via :func:`round_e4m3_sat`.

    Zero keeps its sign (0x00 / 0x80); NaN maps to 0x7F with its sign bit.
    """
    v = np.asarray(v, dtype=np.float64)
    r = round_e4m3_sat(v)
    nan = np.isnan(r)
    a = np.abs(np.where(nan, 0.0, r))
    sign = np.where(np.signbit(v), 0x80, 0x00).astype(np.int64)
    _, ex = np.frexp(a)
    binade = ex - 1
    normal = a >= 2.0 ** E4M3_MIN_NORMAL_EXP
    # normal: field = binade + 7, mantissa = (a / 2^binade - 1) * 8
    e_field = np.where(normal, binade + 7, 0)
    mant_n = (np.ldexp(a, -binade) - 1.0) * 8.0
    mant_s = a / 2.0 ** -9
    mant = np.where(normal, mant_n, mant_s)
    mant = np.where(a == 0.0, 0.0, mant)
    code = sign | (e_field.astype(np.int64) << 3) | np.rint(mant).astype(np.int64)
    code = np.where(nan, sign | E4M3_NAN_POS, code)
    return code.astype(np.uint8)


def round_bf16(v):
    """Round float64 values to the nearest bf16 value (ties to even).

    bf16 keeps 8 significant bits: spacing 2^(E-7) in binade 2^E, and 2^-133
    below the smallest normal 2^-126.  Magnitudes that round past the largest
    finite bf16 become infinities.
    """
    v = np.asarray(v, dtype=np.float64)
    a = np.abs(v)
    _, ex = np.frexp(a)
    binade = np.maximum(ex - 1, -126)
    spacing = np.ldexp(1.0, binade - 7)
    r = np.rint(a / spacing) * spacing
    bf16_max = (2.0 - 2.0 ** -7) * 2.0 ** 127
    r = np.where(r > bf16_max, np.inf, r)
    r = np.where(np.isnan(v), np.nan, r)
    return np.where(np.signbit(v), -r, r)
