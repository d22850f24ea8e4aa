"""Quantizers, written step by step in the order the pages give them.

TEST INFRASTRUCTURE ONLY (see the package docstring).

Every floating-point step the method performs in fp32 is done in numpy
float32 (IEEE-754, correctly rounded division and multiplication, subnormals
kept).  Every narrowing to E4M3 / E2M1 / bf16 goes through ``formats`` (one
round-to-nearest-even from the exact value).

Parity status
-------------
* ``e8m0_scale_exp`` (exponent-first, 0.75 threshold): pinned by the
  worked table of vLLM PR #43557 ("Root Cause": vecMax 2.7/5.5/1.2 -> 126/127/
  125) and by the clip-zone table ("Why This Helps Precision").
* ``quant_mxfp4``: the scale rule above + the E2M1 cast (pinned in formats) +
  the PR's saturation statement (a scaled element between 6 and 7 is clipped
  to E2M1's largest value, 6).
* ``quant_fp8_block``: the scale example "amax 22.4 -> scale 0.05 -> 448" and
  the E4M3 cast pins (200.04 -> 208, subnormal edges).
* ``quant_int4_rtn``, ``quant_nvfp4``: parity unpinned beyond invariants (the
  pages print no algorithm for them; the readings are stated below).
"""

import numpy as np

from . import formats as F

F32 = np.float32


def _blocks(x, g):
    x = np.asarray(x)
    assert x.shape[-1] % g == 0, "the block size must divide the row length"
    return x.reshape(x.shape[:-1] + (x.shape[-1] // g, g))


def _as_f32(x_bits_or_f32):
    """Accept bf16 bit patterns (uint16) or float32 values; return float32."""
    x = np.asarray(x_bits_or_f32)
    if x.dtype == np.uint16:
        return F.bf16_decode(x).astype(F32)       # exact widening
    return x.astype(F32)


def pack_nibbles(codes):
    """Two 4-bit codes per byte along the last axis, even index in the low nibble."""
    c = np.asarray(codes).astype(np.uint8) & 0xF
    return (c[..., 0::2] | (c[..., 1::2] << 4)).astype(np.uint8)


def unpack_nibbles(packed):
    p = np.asarray(packed).astype(np.uint8)
    out = np.empty(p.shape[:-1] + (p.shape[-1] * 2,), dtype=np.uint8)
    out[..., 0::2] = p & 0xF
    out[..., 1::2] = p >> 4
    return out


# ----------------------------------------------------------------------------
# E8M0 shared exponent
# ----------------------------------------------------------------------------

def e8m0_scale_exp(vecMax):
    """Scale exponent for one MX block from the fp32 block maximum.

    vLLM PR #43557, "Fix: Exponent-First with 0.75-Threshold Rounding".  The
    rule works on vecMax's binade: write vecMax = f * 2**E with the
    significand f in [1, 2).  The exponent is rounded up to E + 1 when the
    fraction part of f is at least 0.75 (f >= 1.75 -- the point where
    adding half a unit of the third mantissa bit carries into the exponent),
    and the scale is the biased result minus 2 (E2M1 tops out in the 2**2
    binade), never below 0.  Formulated here with frexp in float64: frexp
    gives vecMax = m * 2**e with m in [0.5, 1), so f = 2m and E = e - 1.
    Subnormal and zero maxima have biased exponents <= 2 and clamp to 0.
    """
    v = np.asarray(vecMax, dtype=F32).astype(np.float64)
    m, e = np.frexp(v)
    biased = (e.astype(np.int64) - 1) + 127 + (2.0 * m >= 1.75)
    return np.where((v > 0) & (biased > 2), biased - 2, 0).astype(np.uint8)


def e8m0_scale_exp_old(vecMax):
    """The rule the PR replaced: biased exponent of vecMax/6 (negative pin only).

    "Root Cause": ``vecMax * reciprocal_approximate_ftz(6.0f)`` then ``>> 23``.
    Computed here with an exact division; the pinned table values do not
    depend on the reciprocal's last bit.
    """
    q = (np.asarray(vecMax, dtype=np.float64) / 6.0).astype(F32)
    return ((F.bits_from_f32(q) >> 23) & 0xFF).astype(np.uint8)


def e8m0_scale_exp_ocp(vecMax):
    """Strict OCP MX variant from the PR's comparison table: biased_exp(vecMax) - 2."""
    b = ((F.bits_from_f32(np.asarray(vecMax, dtype=F32)) >> 23) & 0xFF).astype(np.int64)
    return np.where(b > 2, b - 2, 0).astype(np.uint8)


def e8m0_scale_exp_ceil(vecMax):
    """SGLang MXFP4QuantizeUtil variant: ceil(max(log2(amax/6), -127)) + 127.

    "Numerics" page, "MXFP4 and the block-scaled family".  Documented variant,
    not the path's rule (it never clips, at up to one binade of headroom).
    """
    v = np.asarray(vecMax, dtype=np.float64)
    with np.errstate(divide="ignore"):
        e = np.ceil(np.maximum(np.log2(v / 6.0), -127.0))
    return (e + 127).astype(np.uint8)


# ----------------------------------------------------------------------------
# a6: MXFP4 quantizer (activations with g=16 or 32; weights with g=32)
# ----------------------------------------------------------------------------

def quant_mxfp4(x, g):
    """MXFP4: per block of g along the last axis.

    1. vecMax = max |x| over the block (fp32; exact from bf16 or fp32 input).
    2. scale code se = e8m0_scale_exp(vecMax).
    3. each element t = x * 2**(127 - se), an exact power-of-two scaling
       (the PR's test plan asks for "exact division").
    4. code = E2M1 round-to-nearest-even with saturation at 6 (the PR: ratio
       in [6, 7) clips to 6.0).
    5. pack two codes per byte, even element in the low nibble.
    Returns (packed codes [..., K/2] uint8, scale codes [..., K/g] uint8).
    """
    xb = _blocks(_as_f32(x), g)
    vecMax = np.max(np.abs(xb), axis=-1)
    se = e8m0_scale_exp(vecMax)
    t = np.ldexp(xb.astype(np.float64), (127 - se.astype(np.int64))[..., None])
    codes = F.e2m1_encode(t).reshape(np.asarray(x).shape)
    return pack_nibbles(codes), se


# ----------------------------------------------------------------------------
# a7: FP8 E4M3 block quantizer (g=128 per 1x128 block; g=K is per-token)
# ----------------------------------------------------------------------------

def fp8_block_scale(amax):
    """scale = amax / 448 in fp32; an all-zero block gets scale 1.0.

    "Numerics" page, fp8 linear walk-through step 1 (amax -> fp32 -> / 448),
    which asks for an explicit all-zero-group rule and names s = 1.  The unstated minimum
    clamp (_FP8_MIN_SCALING_FACTOR) is not applied.
    """
    a = np.asarray(amax, dtype=F32)
    s = a / F32(448.0)
    return np.where(a == 0, F32(1.0), s).astype(F32)


def quant_fp8_block(x, g):
    """FP8 E4M3 per 1 x g block.

    1. a = max |x| over the block (fp32).
    2. s = a / 448 (fp32, correctly rounded; zero block -> 1.0).
    3. t = x / s (fp32 IEEE division, as in vLLM ``scaled_fp8_conversion``
       with a non-inverted scale).
    4. code = E4M3 round-to-nearest-even once from fp32, saturating at +-448
       (FreeToken PR #805: one rounding, never fp32 -> fp16 -> e4m3).
    Returns (codes [..., K] uint8, scales [..., K/g] float32).
    """
    xb = _blocks(_as_f32(x), g)
    s = fp8_block_scale(np.max(np.abs(xb), axis=-1))
    t = (xb / s[..., None]).astype(F32)
    codes = F.e4m3_encode(t).reshape(np.asarray(x).shape)
    return codes, s


# ----------------------------------------------------------------------------
# FP8 group scales for W4A8 with an FP8 x FP8 matmul ("Production-Ready W4A8",
# "Accurate W4A8 Kernel")
# ----------------------------------------------------------------------------

def fp8_group_scales(s_bits):
    """The page's W4A8 recipe for the bf16 group scales of an INT4 checkpoint.

    1. Quantize each output channel's row of bf16 group scales to FP8 with the
       same per-token quantizer the activations use: cs[n] = max_g |s[n,g]| /
       448 (fp32), code = E4M3(s[n,g] / cs[n]) (quant_fp8_block with the block
       = the whole row).
    2. Scale the FP8 scales by 1/8 so that every INT4 value times a scale
       stays inside the E4M3 range, and compensate by multiplying the channel
       scales by 8: s8 = E4M3(decode(code) / 8) (exact for codes >= 2^-3,
       otherwise one more E4M3 rounding), cs8 = cs * 8 (exact).
    Returns (s8 E4M3 codes [N, G] uint8, cs8 float32 [N]).
    """
    s = F.bf16_decode(s_bits).astype(F32)
    codes, cs = quant_fp8_block(s, s.shape[-1])
    s8 = F.e4m3_encode((F.e4m3_decode(codes).astype(F32) * F32(0.125)).astype(F32))
    return s8, (cs[..., 0] * F32(8.0)).astype(F32)


def fp8_lut_weights(packed, s8_codes, g=128):
    """Weights of the W4A8 FP8 matmul: E4M3(q * s8) for every INT4 value q
    and its group's FP8 scale -- the contents of the page's per-scale lookup
    table (a 4-bit q gives just 16 products s * w per scale), one E4M3
    round-to-nearest-even of the exact product.  Returns E4M3 codes [N, K]."""
    q = F.int4_decode(unpack_nibbles(packed)).astype(np.float64)
    s8 = F.e4m3_decode(s8_codes).astype(np.float64)
    N, K = q.shape
    prod = (q.reshape(N, K // g, g) * s8[..., None]).reshape(N, K)     # exact (<= 8 significant bits)
    return F.e4m3_encode(prod.astype(F32))


# ----------------------------------------------------------------------------
# weight quantizers (load-time; the GPU kernels consume their output)
# ----------------------------------------------------------------------------

def quant_int4_rtn(w, g):
    """Symmetric INT4 round-to-nearest with one bf16 scale per group of g.

    Reading of "Numerics" (affine map with z = 0; "symmetric INT8 can set
    z=0 and compute s = max|x|/127" -> /7 for int4, range [-8, 7]; all-zero
    group -> s = 1): s = bf16_RNE(absmax / 7) with the division in fp32;
    q = clamp(round_half_even(w / s), -8, 7) with w / s in fp32.  A group whose
    bf16 scale underflows to zero is treated as an all-zero group.
    Returns (packed [N, K/2] uint8, scales [N, K/g] bf16 bits uint16).
    parity unpinned (invariants only).
    """
    wb = _blocks(np.asarray(w, dtype=F32), g)
    absmax = np.max(np.abs(wb), axis=-1)
    s_bits = F.bf16_encode((absmax / F32(7.0)).astype(F32))
    s_val = F.bf16_decode(s_bits).astype(F32)
    zero = s_val == 0
    s_bits = np.where(zero, np.uint16(0x3F80), s_bits).astype(np.uint16)
    s_val = np.where(zero, F32(1.0), s_val).astype(F32)
    t = (wb / s_val[..., None]).astype(F32)
    q = np.clip(np.rint(t), -8, 7).astype(np.int64)
    q = np.where(zero[..., None], 0, q)
    return pack_nibbles((q & 0xF).reshape(np.asarray(w).shape)), s_bits


def quant_int4_zp(w, g):
    """Asymmetric INT4 with a zero point per group of g.

    "Numerics" gives the affine map x = s * (q - z) with an integer zero point
    z (z != 0: asymmetric) and vLLM's dequant line ``(iweights - zeros) *
    scales``, but prints no quantizer.  Reading (min-max, the plainest one):
    per group lo = min(w), hi = max(w); s = bf16_RNE((hi - lo) / 15) with the
    subtraction and division in fp32; a group with hi == lo, or whose bf16
    scale underflows to zero, gets s = 1 (the page's all-zero-group policy);
    z = clamp(round_half_even(-lo / s), 0, 15); q = clamp(round_half_even(w / s)
    + z, 0, 15), every division in fp32.  q and z are unsigned nibbles.
    Returns (packed [N, K/2] uint8 unsigned nibbles, scales [N, K/g] bf16 bits,
    zero points [N, K/g] uint8).  parity unpinned beyond its invariants.
    """
    wb = _blocks(np.asarray(w, dtype=F32), g)
    lo = np.min(wb, axis=-1)
    hi = np.max(wb, axis=-1)
    s_bits = F.bf16_encode(((hi - lo).astype(F32) / F32(15.0)).astype(F32))
    s_val = F.bf16_decode(s_bits).astype(F32)
    flat = s_val == 0
    s_bits = np.where(flat, np.uint16(0x3F80), s_bits).astype(np.uint16)
    s_val = np.where(flat, F32(1.0), s_val).astype(F32)
    z = np.clip(np.rint((-lo / s_val).astype(F32)), 0, 15).astype(np.int64)
    t = (wb / s_val[..., None]).astype(F32)
    q = np.clip(np.rint(t) + z[..., None], 0, 15).astype(np.int64)
    return pack_nibbles(q.reshape(np.asarray(w).shape)), s_bits, z.astype(np.uint8)


def quant_fp8_channel(w):
    """FP8 E4M3 with one fp32 scale per output channel (row of W [N, K]).

    Same arithmetic as the block quantizer with the block equal to the row
    (per-channel: a single scale for each output channel of the weight).
    Returns (codes [N, K] uint8, cs [N] float32).
    """
    w = np.asarray(w, dtype=F32)
    codes, s = quant_fp8_block(w, w.shape[-1])
    return codes, s[..., 0]


NVFP4_BLOCK = 16


def quant_nvfp4(w):
    """NVFP4: E2M1 codes, one E4M3 scale per 16 elements, one fp32 global scale.

    The pages fix the format (block of 16, E4M3 scale with mantissa bits, the
    "Numerics" MXFP4 section; decode "each 16-value E2M1 block and its E4M3
    scale", the 3090 article section 2.1) and, in the vLLM PR review, that
    elements are divided by the *dequantized* block scale.  Reading (parity
    unpinned beyond invariants):
      gs  = amax(W) / (448 * 6)                 fp32; all-zero W -> 1.0
      d   = 6 * gs                              fp32
      sb  = E4M3_RNE_sat(amax_block / d)        fp32 division, one rounding
      den = e4m3(sb) * gs                       fp32
      code= E2M1_RNE_sat(w / den)               fp32 division; sb == 0 -> 0
    Returns (packed [N, K/2] uint8, sb [N, K/16] uint8, gs float32 scalar).
    """
    w = np.asarray(w, dtype=F32)
    amax = F32(np.max(np.abs(w))) if w.size else F32(0)
    gs = F32(1.0) if amax == 0 else F32(amax / F32(2688.0))
    wb = _blocks(w, NVFP4_BLOCK)
    amax_b = np.max(np.abs(wb), axis=-1).astype(F32)
    d = F32(F32(6.0) * gs)
    sb = F.e4m3_encode((amax_b / d).astype(F32))
    den = (F.e4m3_decode(sb).astype(F32) * gs).astype(F32)
    safe = np.where(den == 0, F32(1.0), den).astype(F32)
    t = (wb / safe[..., None]).astype(F32)
    codes = F.e2m1_encode(t)
    codes = np.where((den == 0)[..., None], np.uint8(0), codes)
    return pack_nibbles(codes.reshape(w.shape)), sb, gs


def quant_mxfp4_weights(w, g=32):
    """MXFP4 weights: the same block quantizer on fp32 rows, OCP block of 32."""
    return quant_mxfp4(np.asarray(w, dtype=F32), g)
