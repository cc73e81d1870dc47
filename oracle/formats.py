"""Number formats used by the layer, written out in fp64 (oracle; test use only).

* bfloat16: 8 significant bits, round to nearest, ties to even.
* FP8 E4M3 ("e4m3fn" in the OCP 8-bit float spec): 1 sign, 4 exponent (bias 7),
  3 mantissa bits; largest finite 448, smallest normal 2^-6, subnormal step
  2^-9; no infinities.  Encoding is round-to-nearest-even with saturation to
  +-448 ("satfinite").
* UE8M0: an unsigned 8-bit power-of-two scale 2^(byte-127).

The per-token 1x128 activation quantisation follows "Support DeepGEMM for
standard MoE dispatch" (sglang PR #33128 report), section "实现拆解" step 3:
the FP8 activations are quantised *directly* with a power-of-two (UE8M0)
scale instead of quantising with a real scale and rounding that scale
afterwards (which the report says costs up to a factor-2 representation
error).  Reading adopted where the report is silent: for each 128-column
group the exponent is the smallest integer s with amax <= 448 * 2^s, clamped
to [-127, 127] (s = -127 when amax == 0), and every element is divided by
that final scale before rounding to E4M3.

MXFP8 (the 1x32 variant, which the standard-dispatch report lists as not yet
covered, section "风险与影响" item 5) is read as the same element format and
the same exponent rule over 32-column blocks (the OCP microscaling block
size), for activations, the GEMM1 output and each weight row.  The FP4
variant of the same item is read as FP4 (E2M1) expert weights with one UE8M0
scale per row and 32-column block (OCP MXFP4), the activations and h staying
MXFP8.
"""

import math

import numpy as np

E4M3_MAX = 448.0
BF16_MAX = (2.0 - 2.0 ** -7) * 2.0 ** 127
_BF16_MIN_NORMAL_EXP = -126
_E4M3_MIN_NORMAL_EXP = -6


def bf16_round(x):
    """Round finite fp64 values to the nearest bfloat16 value (ties to even).

    Returns fp64 holding bf16-representable values.  Values whose rounding
    exceeds the bf16 range become +-inf, as IEEE round-to-nearest does.
    """
    x = np.asarray(x, dtype=np.float64)
    _, e = np.frexp(x)                     # |x| = m * 2^e with m in [0.5, 1)
    lead = np.maximum(e - 1, _BF16_MIN_NORMAL_EXP)   # exponent of the leading bit
    step = np.ldexp(1.0, lead - 7)         # spacing of bf16 values in that binade
    q = np.rint(x / step) * step           # x / step is exact (power of two)
    return np.where(np.abs(q) > BF16_MAX, np.copysign(np.inf, x), q)


def bf16_bits(x):
    """uint16 bit patterns of bf16-representable fp64 values."""
    f = np.asarray(x, dtype=np.float64).astype(np.float32)   # exact for bf16 values
    return (f.view(np.uint32) >> 16).astype(np.uint16)


def e4m3_round(v):
    """Round finite fp64 values to the E4M3 grid: nearest, ties to even, then
    saturate to +-448.  The sign of zero is kept."""
    v = np.asarray(v, dtype=np.float64)
    a = np.abs(v)
    _, e = np.frexp(a)
    lead = np.maximum(e - 1, _E4M3_MIN_NORMAL_EXP)   # subnormals share the 2^-6 binade step
    step = np.ldexp(1.0, lead - 3)
    q = np.minimum(np.rint(a / step) * step, E4M3_MAX)
    return np.copysign(q, v)


def e4m3_bits(q):
    """uint8 E4M3 encodings of values already on the E4M3 grid (|q| <= 448)."""
    q = np.asarray(q, dtype=np.float64)
    sign = np.signbit(q).astype(np.uint16) << 7
    a = np.abs(q)
    _, e = np.frexp(a)
    normal = a >= 2.0 ** _E4M3_MIN_NORMAL_EXP
    exp_field = np.where(normal, e - 1 + 7, 0)
    frac = np.where(normal, a / np.ldexp(1.0, e - 1) - 1.0, a / 2.0 ** -6)
    mant = np.rint(frac * 8.0)
    return (sign | (exp_field.astype(np.uint16) << 3) | mant.astype(np.uint16)).astype(np.uint8)


def e4m3_from_bits(b):
    """Decode E4M3 bytes to fp64 (0x7f / 0xff are NaN)."""
    b = np.asarray(b, dtype=np.uint8).astype(np.int64)
    sign = np.where(b & 0x80, -1.0, 1.0)
    ef = (b >> 3) & 0xF
    mf = b & 0x7
    val = np.where(ef == 0, mf / 8.0 * 2.0 ** -6, (1.0 + mf / 8.0) * np.ldexp(1.0, ef - 7))
    val = np.where((b & 0x7F) == 0x7F, np.nan, val)
    return sign * val


def ue8m0_exponent(amax):
    """Smallest integer s with amax <= 448 * 2^s, clamped to [-127, 127].

    Written from frexp: amax = m * 2^e (m in [0.5, 1)) and 448 * 2^s =
    0.875 * 2^(s+9), so s = e - 9 when m <= 0.875 and e - 8 otherwise.
    amax == 0 gives -127.  The scale byte stored on the wire is s + 127.
    """
    a = np.asarray(amax, dtype=np.float64)
    m, e = np.frexp(a)
    s = np.where(m > 0.875, e - 8, e - 9)
    s = np.where(a == 0.0, -127, s)
    return np.clip(s, -127, 127).astype(np.int64)


def quant_fp8_groups(x, group):
    """Per-row FP8 quantisation with one UE8M0 scale per ``group`` consecutive
    columns (128: the layer's 1x128 format; 32: the MXFP8 1x32 format).

    x: [R, C] fp64 (C % group == 0).  Returns (q, s): q [R, C] fp64 on the
    E4M3 grid (the stored FP8 values) and s [R, C/group] int64 exponents; the
    value the GEMM consumes is q * 2^s.
    """
    x = np.asarray(x, dtype=np.float64)
    R, C = x.shape
    if C % group:
        raise ValueError(f"quantisation groups are {group} columns wide")
    g = x.reshape(R, C // group, group)
    s = ue8m0_exponent(np.abs(g).max(axis=2) if C else np.zeros((R, 0)))
    scaled = g * np.ldexp(1.0, -s)[..., None]   # exact: power-of-two factor
    q = e4m3_round(scaled)
    return q.reshape(R, C), s


def dequant_groups(q, s, group):
    """q [R, C] on the E4M3 grid and s [R, C/group] -> fp64 values q * 2^s."""
    R, C = q.shape
    return (q.reshape(R, C // group, group) * np.ldexp(1.0, s)[..., None]).reshape(R, C)


def quant_fp8_1x128(x):
    """The layer's activation format: ``quant_fp8_groups(x, 128)``."""
    return quant_fp8_groups(x, 128)


def dequant_1x128(q, s):
    """q [R, C] on the E4M3 grid and s [R, C/128] -> fp64 values q * 2^s."""
    return dequant_groups(q, s, 128)


def quant_mxfp8_1x32(x):
    """MXFP8 activation format: E4M3 elements sharing one UE8M0 scale per 32
    consecutive columns, the block size of the OCP microscaling formats.  The
    exponent follows the layer's rule (smallest s with amax <= 448 * 2^s),
    applied per 32-column block: ``quant_fp8_groups(x, 32)``."""
    return quant_fp8_groups(x, 32)


def e2m1_from_codes(codes):
    """FP4 E2M1 (the OCP microscaling FP4 element: 1 sign, 2 exponent bits with
    bias 1, 1 mantissa bit, subnormals, no inf / NaN) codes 0..15 -> fp64.
    Magnitudes 0, 0.5, 1, 1.5, 2, 3, 4, 6."""
    c = np.asarray(codes, dtype=np.int64)
    sign = np.where(c & 8, -1.0, 1.0)
    ef = (c >> 1) & 3
    mf = c & 1
    mag = np.where(ef == 0, 0.5 * mf, np.ldexp(1.0 + 0.5 * mf, ef - 1))
    return sign * mag


def unpack_fp4(packed):
    """uint8 [..., C/2] -> codes [..., C]: element 2j in the low nibble of byte
    j, element 2j + 1 in the high nibble."""
    p = np.asarray(packed, dtype=np.uint8)
    out = np.empty(p.shape[:-1] + (2 * p.shape[-1],), dtype=np.int64)
    out[..., 0::2] = p & 0xF
    out[..., 1::2] = p >> 4
    return out


def exp2i(s):
    """2^s for integer s as fp64 (exact)."""
    return math.ldexp(1.0, int(s))
