"""Canonical dequantization and the fp64 reference products.

TEST INFRASTRUCTURE ONLY (see the package docstring).

Layouts (row-major, contiguous): W is [N, K] (output channel major, K
contiguous), X is [M, K] bf16, Y is [M, N] bf16.  Packed 4-bit codes hold two
elements per byte along K, even k in the low nibble.

Canonical dequantized weights (bf16 bit patterns, the bit-exact targets):
* INT4:  bf16_RNE(q * s).  The fp32 product is exact (a 4-bit integer times
  an 8-bit significand), so there is exactly one rounding.  This is the
  Cohere W4A8 article's recipe (INT4 weights turned into BF16 on the CUDA
  cores, the product taken in BF16) and the in-register dequant of the 3090
  article (section 4.1).
* FP8:   the E4M3 value in bf16 (exact: the 3090 article, section 4.1, notes
  that every E4M3 and E2M1 value has an exact 16-bit float form).  The fp32
  channel scale is applied to the accumulated row in the epilogue.
* MXFP4: bf16(e2m1 * 2**(c - 127)) -- exact for every code the quantizer
  emits (c <= 252).
* NVFP4: bf16(e2m1 * e4m3(sb)) -- exact; the fp32 global scale is applied in
  the epilogue.

Products: y64 = epilogue_scale * sum_k x[m,k] * w[n,k] in float64 (every
product of two bf16 values is exact in float64); the path's output is
bf16_RNE(y64).  ("Numerics": accumulate wide, narrow once at the store.)

Parity: the product is pinned by exact-arithmetic brute force on tiny inputs
(fractions), the dequantizers by the format pins and brute force over codes.
The MoE harness functions are readings (the pages name the steps but print no
formulas); ``swiglu_f32`` and ``moe_combine`` are pinned by mathematics:
SiLU(0) = 0, SiLU(v) - SiLU(-v) = v, the limits at +-inf, the Taylor value
near 0, agreement with a library logistic routine, the gate/up order, and an
exact-rational brute force of the weighted combine.
"""

import numpy as np

from . import formats as F
from . import quant as Q

F32 = np.float32


# ----------------------------------------------------------------------------
# canonical dequantization -> bf16 bit patterns [N, K]
# ----------------------------------------------------------------------------

def dequant_int4(packed, s_bits, g):
    q = F.int4_decode(Q.unpack_nibbles(packed)).astype(F32)
    s = F.bf16_decode(s_bits).astype(F32)
    with np.errstate(over="ignore"):       # beyond fp32's range: inf, as RNE to bf16 gives
        prod = (q.reshape(q.shape[:-1] + (-1, g)) * s[..., None]).astype(F32)   # exact
    return F.bf16_encode(prod.reshape(q.shape))


def dequant_int4_zp(packed, s_bits, z, g):
    """Canonical asymmetric INT4 dequant ("Numerics": x = s (q - z); vLLM's
    ``(iweights - zeros) * scales``): bf16_RNE((q - z) * s) with q, z unsigned
    nibbles.  q - z is an integer in [-15, 15] and s a bf16, so the fp32
    product is exact and there is one rounding."""
    q = Q.unpack_nibbles(packed).astype(np.int64)
    zz = np.asarray(z).astype(np.int64)
    d = (q.reshape(q.shape[:-1] + (-1, g)) - zz[..., None]).astype(F32)
    s = F.bf16_decode(s_bits).astype(F32)
    prod = (d * s[..., None]).astype(F32)                                     # exact
    return F.bf16_encode(prod.reshape(q.shape))


def dequant_fp8(codes):
    return F.bf16_encode(F.e4m3_decode(codes))


def dequant_mxfp4(packed, se, g=32):
    v = F.e2m1_decode(Q.unpack_nibbles(packed))
    v = v.reshape(v.shape[:-1] + (-1, g)) * F.e8m0_decode(se)[..., None]
    return F.bf16_encode(v.reshape(v.shape[:-2] + (-1,)))


def dequant_nvfp4(packed, sb):
    v = F.e2m1_decode(Q.unpack_nibbles(packed))
    g = Q.NVFP4_BLOCK
    v = v.reshape(v.shape[:-1] + (-1, g)) * F.e4m3_decode(sb)[..., None]
    return F.bf16_encode(v.reshape(v.shape[:-2] + (-1,)))


# ----------------------------------------------------------------------------
# weight-only products (W x A16): fp64 sum, one bf16 rounding
# ----------------------------------------------------------------------------

def gemm_bf16_f64(x_bits, w_bits, col_scale=None):
    """y64[m, n] = col_scale[n] * sum_k x[m,k] * w[n,k], all in float64."""
    x = F.bf16_decode(x_bits)
    w = F.bf16_decode(w_bits)
    y = x @ w.T
    if col_scale is not None:
        y = y * np.asarray(col_scale, dtype=np.float64)
    return y


def w8a8_f64(a_codes, a_s, w_codes, cs, g):
    """FP8 weights with per-channel scales times activations quantized to E4M3
    per 1 x g block (the activation quantizer of the FP8 GEMV prologue in
    FreeToken PR #805's list of native casts; here the a7 block rule):
    y64[m, n] = cs[n] * sum_b a_s[m, b] * sum_{k in block b} e4m3(a[m,k]) * e4m3(w[n,k]),
    everything in float64 (the block partial sums are exact products summed).
    a_codes [M, K], a_s [M, K/g], w_codes [N, K], cs [N]."""
    a = F.e4m3_decode(a_codes)
    w = F.e4m3_decode(w_codes)
    M, K = a.shape
    nb = K // g
    y = np.zeros((M, w.shape[0]))
    s = np.asarray(a_s, np.float64).reshape(M, nb)
    for b in range(nb):
        y += (a[:, b * g:(b + 1) * g] @ w[:, b * g:(b + 1) * g].T) * s[:, b:b + 1]
    return y * np.asarray(cs, np.float64)[None, :]


def qgemm_w4a16(x_bits, packed, s_bits, g):
    return gemm_bf16_f64(x_bits, dequant_int4(packed, s_bits, g))


def qgemm_w8a16(x_bits, codes, cs):
    return gemm_bf16_f64(x_bits, dequant_fp8(codes), cs)


def qgemm_mxfp4a16(x_bits, packed, se, g=32):
    return gemm_bf16_f64(x_bits, dequant_mxfp4(packed, se, g))


def qgemm_nvfp4a16(x_bits, packed, sb, gs):
    n = np.asarray(packed).shape[0]
    return gemm_bf16_f64(x_bits, dequant_nvfp4(packed, sb), np.full(n, float(gs)))


def w4a4_mxfp4_f64(x_bits, packed, se, g_act=32):
    """W4A4 with MXFP4 on both sides (the MXFP4 W4A4 MoE GEMM of vLLM PR
    #43557): the activations are quantized by the a6 rule (exponent-first
    0.75-threshold E8M0 scale, E2M1 RNE with saturation) per block of g_act,
    both operands decoded to their exact values, the product summed in
    float64.  Returns (y64, activation codes, activation scale codes)."""
    aq, ase = Q.quant_mxfp4(np.asarray(x_bits, np.uint16), g_act)
    a = F.e2m1_decode(Q.unpack_nibbles(aq))
    a = (a.reshape(a.shape[:-1] + (-1, g_act)) * F.e8m0_decode(ase)[..., None]).reshape(a.shape)
    w = F.e2m1_decode(Q.unpack_nibbles(packed))
    w = (w.reshape(w.shape[:-1] + (-1, 32)) * F.e8m0_decode(se)[..., None]).reshape(w.shape)
    return a.astype(np.float64) @ w.astype(np.float64).T, aq, ase


def to_bf16(y64):
    """The path's narrowing store: one round-to-nearest-even to bf16."""
    return F.bf16_encode(y64)


# ----------------------------------------------------------------------------
# W4A8 grouped GEMM
# ----------------------------------------------------------------------------

def w4a8_grouped_f64(a_codes, a_s, expert_off, packed, s_bits, g):
    """Rows sorted by expert; rows expert_off[e]..expert_off[e+1] use expert e.

    y64[r, n] = a_s[r] * sum_k e4m3(a[r,k]) * q_e[n,k] * s_e[n, k // g]
    with q * s exact (reading of the W4A8 config: INT4 g128 bf16 scales,
    per-token E4M3 activations with absmax/448 scales, fp32 accumulate).
    """
    a = F.e4m3_decode(a_codes)
    R = a.shape[0]
    E, N = np.asarray(packed).shape[:2]
    y = np.zeros((R, N))
    for e in range(E):
        r0, r1 = int(expert_off[e]), int(expert_off[e + 1])
        if r1 <= r0:
            continue
        q = F.int4_decode(Q.unpack_nibbles(packed[e]))
        s = F.bf16_decode(s_bits[e])
        w = (q.reshape(N, -1, g) * s[..., None]).reshape(N, -1)      # exact in fp64
        y[r0:r1] = (a[r0:r1] @ w.T) * np.asarray(a_s[r0:r1], np.float64)[:, None]
    return y


def w4a8_fp8s_grouped_f64(a_codes, a_s, expert_off, w8_codes, cs8):
    """W4A8 with FP8 group scales ("Production-Ready W4A8", "Accurate W4A8
    Kernel"): rows sorted by expert, expert e's weights are the E4M3 codes
    w8 = E4M3(q * s8) and its fp32 channel scales cs8;
    y64[r, n] = a_s[r] * cs8_e[n] * sum_k e4m3(a[r,k]) * e4m3(w8_e[n,k])
    (the per-token and per-channel scales applied in the epilogue, "outer
    vector scaling")."""
    a = F.e4m3_decode(a_codes)
    R = a.shape[0]
    E, N = np.asarray(w8_codes).shape[:2]
    y = np.zeros((R, N))
    for e in range(E):
        r0, r1 = int(expert_off[e]), int(expert_off[e + 1])
        if r1 <= r0:
            continue
        w = F.e4m3_decode(w8_codes[e])
        y[r0:r1] = (a[r0:r1] @ w.T) * np.asarray(a_s[r0:r1], np.float64)[:, None] \
            * np.asarray(cs8[e], np.float64)[None, :]
    return y


def swiglu_f32(gate_up_bits, inter):
    """h = SiLU(gate) * up from the bf16 projection output, in fp32.

    Reading (the pages name a fused SwiGLU kernel, FreeToken PR #805's
    ``_swiglu_kernel``, but give no formula): the first ``inter`` columns are
    the gate, the next ``inter`` the up projection; SiLU(v) = v / (1 + e^-v).
    Evaluated in float64 and rounded once to float32.
    Pinned by mathematics: SiLU(0) = 0; SiLU(v) - SiLU(-v) = v (sigmoid(v) +
    sigmoid(-v) = 1); SiLU(v) -> v and -> 0 at +-inf; the series x/2 + x^2/4
    near 0; v * expit(v) from a library logistic routine; the gate half first.
    """
    gu = F.bf16_decode(gate_up_bits)
    gate, up = gu[:, :inter], gu[:, inter:2 * inter]
    return (gate / (1.0 + np.exp(-gate)) * up).astype(F32)


def moe_layer(x_bits, route_rows, expert_off, w1, w2, g, inter):
    """W4A8 MoE layer over rows already grouped by expert.

    route_rows: [R] source token of each expert-sorted row; expert_off [E+1].
    w1 = (packed [E, 2I, H/2], scales [E, 2I, H/g]); w2 = (packed [E, H, I/2],
    scales [E, H, I/g]).
    Steps: per-token FP8 quant of x (block = H) -> gather rows -> grouped
    gate/up -> bf16 -> SwiGLU (fp32) -> per-row FP8 quant (block = I) ->
    grouped down -> bf16.  Returns (down_bits [R, H], gate_up_bits [R, 2I]).
    The weighted combine is applied by ``moe_combine``.
    """
    H = np.asarray(x_bits).shape[1]
    a8, a_s = Q.quant_fp8_block(x_bits, H)
    rows = np.asarray(route_rows)
    gu = to_bf16(w4a8_grouped_f64(a8[rows], a_s[rows, 0], expert_off, w1[0], w1[1], g))
    h = swiglu_f32(gu, inter)
    h8, h_s = Q.quant_fp8_block(h, inter)
    down = to_bf16(w4a8_grouped_f64(h8, h_s[:, 0], expert_off, w2[0], w2[1], g))
    return down, gu


def moe_layer_fp8s(x_bits, route_rows, expert_off, w1, w2, inter):
    """The MoE layer of ``moe_layer`` with both projections on the FP8
    group-scale recipe ("Production-Ready W4A8", "Accurate W4A8 Kernel"):
    w1 = (w8 codes [E, 2I, H], cs8 [E, 2I]) and w2 = (w8 [E, H, I], cs8 [E, H])
    as prepared by ``quant.fp8_group_scales`` and ``quant.fp8_lut_weights``.
    Same steps in the same order: per-token FP8 quant of x (block = H) ->
    gather -> grouped gate/up -> bf16 -> SwiGLU (fp32) -> per-row FP8 quant
    (block = I) -> grouped down -> bf16.  Returns (down_bits, gate_up_bits)."""
    H = np.asarray(x_bits).shape[1]
    a8, a_s = Q.quant_fp8_block(x_bits, H)
    rows = np.asarray(route_rows)
    gu = to_bf16(w4a8_fp8s_grouped_f64(a8[rows], a_s[rows, 0], expert_off, w1[0], w1[1]))
    h = swiglu_f32(gu, inter)
    h8, h_s = Q.quant_fp8_block(h, inter)
    down = to_bf16(w4a8_fp8s_grouped_f64(h8, h_s[:, 0], expert_off, w2[0], w2[1]))
    return down, gu


def moe_combine(down_bits, route_rows, route_weight, T):
    """out[t] = sum over t's rows of p * down (float64), one bf16 rounding.

    Reading of the MoE harness: each token's output is the sum of its routed
    rows' down projections weighted by their (not renormalised) routing
    probabilities.  Pinned by an exact-rational brute force on dyadic inputs
    (every product and partial sum exact), rounded once to bf16.
    """
    d = F.bf16_decode(down_bits)
    out = np.zeros((T, d.shape[1]))
    np.add.at(out, np.asarray(route_rows), d * np.asarray(route_weight, np.float64)[:, None])
    return to_bf16(out)
