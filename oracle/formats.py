"""Bit-level decode and round-to-nearest-even encode of every format on the path.

TEST INFRASTRUCTURE ONLY (see the package docstring): never imported by the
product path.

Formats (sign, exponent bits e, mantissa bits m, bias B):

* E4M3 "fn"  (1,4,3, B=7)  finite only; the single NaN pattern S.1111.111;
  max (1+6/8)*2**(15-7) = 448.  "Numerics: FP32 to INT4, and why bf16 won",
  the paragraph on the two formats that break the IEEE rules, and the
  scalar_types listing (float8_e4m3fn, NanRepr.EXTD_RANGE_MAX_MIN).
* E5M2        (1,5,2, B=15) IEEE: all-ones exponent is inf/NaN; max 57344.
* E2M1        (1,2,1)      no inf, no NaN; magnitudes {0,.5,1,1.5,2,3,4,6}.
  Same page, "MXFP4 and the block-scaled family" (E2M1_values literal).
* E8M0 "fnu"  (0,8,0, B=127) a bare power of two 2**(c-127); code 255 is NaN
  (OCP MX; scalar_types float8_e8m0fnu with EXTD_RANGE_MAX_MIN).
* bf16 = float16_e8m7, fp16 = float16_e5m10 (IEEE), same listing.
* INT4: two's-complement nibble in [-8, 7] (scalar_types int4, max 7 min -8).

Encoders round the exact input value once, to nearest, ties to the even code
(even mantissa), and -- for the "satfinite" FP8/FP4 casts -- clamp magnitudes
above the format maximum to that maximum (FreeToken PR #805:
``cvt.rn.satfinite.e4m3x2.f32``; vLLM ``scaled_fp8_conversion`` clamps with
fmaxf/fminf before the convert, quoted on the "Numerics" page).  Signed zero is
kept (a negative input that rounds to zero gets the negative-zero code).

Two independent formulations are provided so each can pin the other:
``round_to_grid`` (nearest value among the enumerated finite grid) and
``round_binade`` (scale into the binade, round the significand half-to-even).

Parity: pinned by the page values (448, 57344, 65504, 3.3895313892515355e38,
int4 [-8,7], 200.04 -> 208, 2**-10 -> 0, the E2M1 lists), by brute force over
all 16 E2M1 and 256 E4M3 codes, by the Marlin bit-trick identity, and by
agreement with torch's CPU casts (tests/test_oracle_pins.py).
"""

import numpy as np

# ----------------------------------------------------------------------------
# raw bit views
# ----------------------------------------------------------------------------

def f32_from_bits(u):
    return np.asarray(u, dtype=np.uint32).view(np.float32)


def bits_from_f32(x):
    return np.asarray(x, dtype=np.float32).view(np.uint32)


# ----------------------------------------------------------------------------
# decoders: code -> exact value (float64)
# ----------------------------------------------------------------------------

def decode_minifloat(codes, e_bits, m_bits, bias, ieee_specials):
    """Value of sign.exponent.mantissa codes, written out from the definition.

    normal   (E != 0): (-1)**s * 2**(E - bias) * (1 + M / 2**m)
    subnormal (E == 0): (-1)**s * 2**(1 - bias) * (M / 2**m)
    ``ieee_specials``: the all-ones exponent is inf (M == 0) or NaN.
    """
    c = np.asarray(codes).astype(np.int64)
    s = (c >> (e_bits + m_bits)) & 1
    E = (c >> m_bits) & ((1 << e_bits) - 1)
    M = c & ((1 << m_bits) - 1)
    sign = np.where(s == 1, -1.0, 1.0)
    normal = np.ldexp(1.0 + M / float(1 << m_bits), (E - bias).astype(np.int64))
    sub = np.ldexp(M / float(1 << m_bits), np.int64(1 - bias))
    v = sign * np.where(E == 0, sub, normal)
    if ieee_specials:
        top = E == (1 << e_bits) - 1
        v = np.where(top & (M == 0), sign * np.inf, v)
        v = np.where(top & (M != 0), np.nan, v)
    return v


def e4m3_decode(codes):
    """E4M3 'fn': IEEE layout, no infinities, only S.1111.111 is NaN."""
    c = np.asarray(codes).astype(np.int64)
    v = decode_minifloat(c, 4, 3, 7, ieee_specials=False)
    return np.where((c & 0x7F) == 0x7F, np.nan, v)


def e5m2_decode(codes):
    return decode_minifloat(codes, 5, 2, 15, ieee_specials=True)


E2M1_MAGNITUDES = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])


def e2m1_decode(codes):
    """E2M1 nibble: bit 3 is the sign, bits 2..0 index the eight magnitudes."""
    c = np.asarray(codes).astype(np.int64) & 0xF
    mag = E2M1_MAGNITUDES[c & 7]
    return np.where(c & 8, -mag, mag)


def e8m0_decode(codes):
    """E8M0: 2**(c - 127); code 255 is NaN."""
    c = np.asarray(codes).astype(np.int64)
    return np.where(c == 255, np.nan, np.ldexp(1.0, c - 127))


def bf16_decode(bits):
    """bf16 is the upper half of an fp32 bit pattern."""
    u = np.asarray(bits).astype(np.uint32) << 16
    with np.errstate(invalid="ignore"):
        return f32_from_bits(u).astype(np.float64)


def fp16_decode(bits):
    return np.asarray(bits).astype(np.uint16).view(np.float16).astype(np.float64)


def int4_decode(nibbles):
    """Two's-complement 4-bit integer."""
    n = (np.asarray(nibbles) & 0xF).astype(np.int8)
    return np.where(n >= 8, n - 16, n).astype(np.int8)


# ----------------------------------------------------------------------------
# rounding, formulation A: nearest point of the enumerated finite grid
# ----------------------------------------------------------------------------

def _nonneg_grid(decoder, n_codes):
    """(values, codes) of every non-negative finite code, in increasing order."""
    codes = np.arange(n_codes)
    vals = decoder(codes)
    keep = np.isfinite(vals) & (vals >= 0) & ~np.signbit(vals)
    return vals[keep], codes[keep]


E4M3_GRID, E4M3_GRID_CODES = _nonneg_grid(e4m3_decode, 0x80)
E2M1_GRID, E2M1_GRID_CODES = _nonneg_grid(e2m1_decode, 0x8)


def round_to_grid(x, grid, grid_codes, sign_bit):
    """Round |x| to the nearest grid value, ties to the even code; saturate.

    ``grid`` holds every non-negative finite value in increasing order with
    its code; values above the top of the grid saturate to it (satfinite).
    Returns the code with ``sign_bit`` set for negative inputs (incl. -0.0).
    """
    x = np.asarray(x, dtype=np.float64)
    mag = np.minimum(np.abs(x), grid[-1])
    hi = np.searchsorted(grid, mag, side="left")          # grid[hi-1] < mag <= grid[hi]
    hi = np.clip(hi, 0, len(grid) - 1)
    lo = np.clip(hi - 1, 0, len(grid) - 1)
    d_lo = mag - grid[lo]
    d_hi = grid[hi] - mag
    pick_hi = (d_hi < d_lo) | ((d_hi == d_lo) & (grid_codes[hi] % 2 == 0))
    idx = np.where(pick_hi, hi, lo)
    code = grid_codes[idx].astype(np.int64)
    neg = np.signbit(x)
    return np.where(neg, code | sign_bit, code)


def e4m3_encode(x):
    """fp32 -> E4M3, round to nearest even once, saturate to +-448."""
    return round_to_grid(x, E4M3_GRID, E4M3_GRID_CODES, 0x80).astype(np.uint8)


def e2m1_encode(x):
    """fp32 -> E2M1 nibble, round to nearest even once, saturate to +-6."""
    return round_to_grid(x, E2M1_GRID, E2M1_GRID_CODES, 0x8).astype(np.uint8)


# ----------------------------------------------------------------------------
# rounding, formulation B: significand rounding inside the binade
# ----------------------------------------------------------------------------

def round_binade(x, p, emin):
    """Round x (exact in float64) to p significant bits, ties to even.

    The binade exponent is floor(log2|x|), clamped below at ``emin`` (the
    minimum normal exponent) so that subnormals keep a fixed spacing.  No upper
    clamp: callers decide about overflow.  Returns float64 (sign of zero kept).
    """
    x = np.asarray(x, dtype=np.float64)
    _, e = np.frexp(x)                       # |x| = f * 2**e with f in [0.5, 1)
    ex = np.maximum(e.astype(np.int64) - 1, emin)
    ulp = np.ldexp(1.0, ex - (p - 1))
    return np.round(x / ulp) * ulp           # numpy rounds half to even


BF16_MAX = float(np.ldexp(2.0 - 2.0 ** -7, 127))


def bf16_round(x):
    """Exact value -> nearest bf16 value (float64), ties to even, IEEE overflow."""
    r = round_binade(x, 8, -126)
    return np.where(np.abs(r) > BF16_MAX, np.copysign(np.inf, r), r)


def bf16_encode_f32(x):
    """float32 -> bf16 bit pattern, round to nearest even, on the bit pattern.

    Keep the upper 16 bits after adding 0x7FFF plus the lowest kept bit: a
    discarded half above 0x8000 carries, below does not, and exactly 0x8000
    carries only when the kept part is odd (ties to even).  A carry out of the
    mantissa bumps the exponent, and past the largest finite value it yields
    the infinity pattern, as IEEE overflow under round-to-nearest does.
    Finite inputs only.
    """
    u = bits_from_f32(np.asarray(x, dtype=np.float32)).astype(np.uint32)
    return ((u + np.uint32(0x7FFF) + ((u >> 16) & np.uint32(1))) >> 16).astype(np.uint16)


def bf16_encode(x):
    """Exact value -> bf16 bit pattern (uint16), round to nearest even once.

    float32 input uses the bit-pattern rounding above; any other input (the
    float64 products) is rounded once from its exact value by ``bf16_round``.
    """
    x = np.asarray(x)
    if x.dtype == np.float32:
        return bf16_encode_f32(x)
    r = bf16_round(x).astype(np.float32)      # exact: r is a bf16 value
    return (bits_from_f32(r) >> 16).astype(np.uint16)


def e4m3_round_binade(x):
    """Formulation B of the E4M3 satfinite cast, as a value (cross-check only)."""
    x = np.asarray(x, dtype=np.float64)
    return round_binade(np.clip(x, -448.0, 448.0), 4, -6)


def e2m1_round_binade(x):
    """Formulation B of the E2M1 satfinite cast, as a value (cross-check only)."""
    x = np.asarray(x, dtype=np.float64)
    return round_binade(np.clip(x, -6.0, 6.0), 2, 0)


# ----------------------------------------------------------------------------
# closed forms quoted on the "Numerics" page
# ----------------------------------------------------------------------------

def ieee_max_finite(e, m):
    """Largest finite IEEE value with e exponent and m mantissa bits:
    (2 - 2**-m) * 2**(2**e - 2 - B), B = 2**(e-1) - 1."""
    B = 2 ** (e - 1) - 1
    return (2.0 - 2.0 ** -m) * 2.0 ** (2 ** e - 2 - B)
