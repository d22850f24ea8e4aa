"""Pins of the CPU oracle against what the pages and the mathematics fix.

No GPU.  Each test names the passage (page title + section/table) or the
mathematical fact it relies on; stored values live in tests/golden/ with their
citations.  None of these tests re-types an oracle formula and compares it
with itself: they use page values, brute force over all codes, exact rational
arithmetic, an independent formulation, or a library routine (torch's CPU
casts) as the other side.
"""

from fractions import Fraction

import numpy as np
import pytest
import torch

from oracle import formats as F
from oracle import gemm as G
from oracle import quant as Q
from tests.conftest import read_golden


# ----------------------------------------------------------------------------
# formats: max-finite closed form and page values
# ----------------------------------------------------------------------------

def _golden_max():
    return {r[0]: float(r[3]) for r in read_golden("max_finite.txt")}


def test_max_finite_closed_form_matches_page_values():
    g = _golden_max()
    # (2 - 2**-m) * 2**(2**e - 2 - B) for the IEEE formats
    assert F.ieee_max_finite(5, 10) == g["float16_e5m10"]
    assert F.ieee_max_finite(8, 7) == g["float16_e8m7"]
    assert F.ieee_max_finite(5, 2) == g["float8_e5m2"]
    # E4M3 extended range: (1 + 6/8) * 2**(15 - 7)
    assert (1 + 6 / 8) * 2.0 ** (15 - 7) == g["float8_e4m3fn"]


def test_decoders_reach_the_page_maxima_by_brute_force():
    g = _golden_max()
    e4 = F.e4m3_decode(np.arange(256))
    e5 = F.e5m2_decode(np.arange(256))
    e2 = F.e2m1_decode(np.arange(16))
    bf = F.bf16_decode(np.arange(65536, dtype=np.uint32))
    fp = F.fp16_decode(np.arange(65536, dtype=np.uint32))
    fin = lambda v: v[np.isfinite(v)]
    assert fin(e4).max() == g["float8_e4m3fn"] and fin(e4).min() == -g["float8_e4m3fn"]
    assert fin(e5).max() == g["float8_e5m2"]
    assert fin(bf).max() == g["float16_e8m7"]
    assert fin(fp).max() == g["float16_e5m10"]
    assert e2.max() == g["float4_e2m1"]
    i4 = F.int4_decode(np.arange(16))
    assert i4.max() == g["int4"] and i4.min() == g["int4_min"]


def test_e4m3_code_structure():
    v = F.e4m3_decode(np.arange(256))
    nan = np.isnan(v)
    assert list(np.nonzero(nan)[0]) == [0x7F, 0xFF]          # only S.1111.111
    assert not np.isinf(v).any()                               # 'fn': no infinities
    pos = v[1:0x7F]
    assert np.all(np.diff(pos) > 0) and len(pos) == 126        # monotone in the code
    assert pos[0] == 2.0 ** -9                                 # smallest subnormal
    assert np.signbit(v[0x80]) and v[0x80] == 0


def test_e2m1_page_lists():
    rows = {r[0]: [float(t) for t in r[1:]] for r in read_golden("e2m1_lists.txt")}
    assert list(F.e2m1_decode(np.arange(8))) == rows["values"]
    mids = (F.E2M1_MAGNITUDES[:-1] + F.E2M1_MAGNITUDES[1:]) / 2
    assert list(mids) == rows["bounds"]
    assert list(F.e2m1_decode(np.arange(8, 16))) == [-v for v in rows["values"]]


# ----------------------------------------------------------------------------
# brute force: every code round-trips; two formulations of RNE agree
# ----------------------------------------------------------------------------

def test_e4m3_all_256_codes_round_trip():
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)])
    assert np.array_equal(F.e4m3_encode(F.e4m3_decode(codes)), codes)


def test_e2m1_all_16_codes_round_trip():
    codes = np.arange(16)
    assert np.array_equal(F.e2m1_encode(F.e2m1_decode(codes)), codes)


def test_marlin_bit_trick_identity_pins_e4m3_decoder():
    """3090 article section 4.1: (q & 0x80008000) | ((q & 0x7F007F00) >> 1)
    turns an E4M3 byte (placed in the high byte of a 16-bit lane) into the fp16
    pattern of value * 2**-8; the bf16 variant shifts by 4 and gives value *
    2**-120.  numpy's float16 decoding is the independent side."""
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], dtype=np.uint32)
    q = codes << 8
    h16 = (q & 0x8000) | ((q & 0x7F00) >> 1)
    b16 = (q & 0x8000) | ((q & 0x7F00) >> 4)
    val = F.e4m3_decode(codes)
    assert np.array_equal(h16.astype(np.uint16).view(np.float16).astype(np.float64), val * 2.0 ** -8)
    bf = torch.from_numpy(b16.astype(np.int16)).view(torch.bfloat16).double().numpy()
    assert np.array_equal(bf, val * 2.0 ** -120)


def _e4m3_sweep():
    """FreeToken PR #805's sweep design: every grid value and midpoint, one fp32
    ulp either side of each midpoint, uniform samples over the range and over
    the subnormals, both signs."""
    g = F.E4M3_GRID
    mids = (g[:-1] + g[1:]) / 2
    m32 = mids.astype(np.float32)
    up = np.nextafter(m32, np.float32(np.inf))
    dn = np.nextafter(m32, np.float32(-np.inf))
    r = np.random.Generator(np.random.PCG64(7))
    uni = r.uniform(0, 448, 200000).astype(np.float32)
    sub = r.uniform(0, 2.0 ** -6, 100000).astype(np.float32)
    big = r.uniform(448, 1e4, 1000).astype(np.float32)
    x = np.concatenate([g, mids, up, dn, uni, sub, big, [0.0, 2.0 ** -10]]).astype(np.float32)
    return np.concatenate([x, -x])


def test_e4m3_grid_vs_binade_formulations_agree():
    x = _e4m3_sweep()
    a = F.e4m3_decode(F.e4m3_encode(x))
    b = F.e4m3_round_binade(x)
    assert np.array_equal(a, b)
    assert np.array_equal(np.signbit(a), np.signbit(b))


def test_e2m1_grid_vs_binade_formulations_agree():
    g = F.E2M1_GRID
    mids = (g[:-1] + g[1:]) / 2
    m32 = mids.astype(np.float32)
    r = np.random.Generator(np.random.PCG64(8))
    x = np.concatenate([g, mids, np.nextafter(m32, np.float32(9)), np.nextafter(m32, np.float32(-9)),
                        r.uniform(0, 8, 100000)]).astype(np.float32)
    x = np.concatenate([x, -x])
    assert np.array_equal(F.e2m1_decode(F.e2m1_encode(x)), F.e2m1_round_binade(x))


def test_e2m1_ties_go_to_the_even_code():
    ties = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0])
    assert list(F.e2m1_decode(F.e2m1_encode(ties))) == [0.0, 1.0, 1.0, 2.0, 2.0, 4.0, 4.0]
    assert list(F.e2m1_decode(F.e2m1_encode([6.5, 7.0, 100.0]))) == [6.0, 6.0, 6.0]


def test_e4m3_matches_torch_cpu_cast_in_range():
    """Library routine as the other side: torch's float32 -> float8_e4m3fn."""
    x = _e4m3_sweep()
    x = x[np.abs(x) <= 448]
    t = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(F.e4m3_encode(x), t)


def test_bf16_matches_torch_cpu_cast():
    r = np.random.Generator(np.random.PCG64(9))
    bits = r.integers(0, 2 ** 32, 500000, dtype=np.uint64).astype(np.uint32)
    x = bits.view(np.float32)
    x = x[np.isfinite(x)]
    x = np.concatenate([x, (np.arange(1, 2 ** 16, dtype=np.uint32) << 16 | 0x8000).view(np.float32)])
    x = x[np.isfinite(x)]
    t = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(F.bf16_encode(x), t)


def test_bf16_bit_rounding_agrees_with_binade_rounding():
    """The two bf16 formulations (bit-pattern carry, significand rounding in
    the binade) agree on random finite fp32 values, ties and near-ties."""
    r = np.random.Generator(np.random.PCG64(10))
    bits = r.integers(0, 2 ** 32, 400000, dtype=np.uint64).astype(np.uint32)
    bits = np.concatenate([bits, (bits & 0xFFFF0000) | 0x8000, (bits & 0xFFFF0000) | 0x7FFF,
                           (bits & 0xFFFF0000) | 0x8001])
    x = bits.view(np.float32)
    x = x[np.isfinite(x)]
    a = F.bf16_encode_f32(x)
    b = F.bf16_encode(x.astype(np.float64))
    assert np.array_equal(a, b)


# ----------------------------------------------------------------------------
# page values for the casts
# ----------------------------------------------------------------------------

def test_e4m3_cast_page_values():
    for inp, exp in ((float(a), float(b)) for a, b in read_golden("e4m3_cast.txt")):
        got = F.e4m3_decode(F.e4m3_encode(np.float32(inp)))
        assert got == exp and np.signbit(got) == np.signbit(exp), (inp, got, exp)


def test_double_rounding_bug_is_not_reproduced():
    """FreeToken PR #805: going through fp16 with truncation first, then E4M3
    rounding, turns 200.04 into 192 (the double-rounding bug)."""
    x = np.float32(200.04)
    h = np.float16(x)
    rtz = h if abs(float(h)) <= float(x) else np.nextafter(h, np.float16(0))
    assert F.e4m3_decode(F.e4m3_encode(np.float32(rtz))) == 192.0
    assert F.e4m3_decode(F.e4m3_encode(x)) == 208.0


def test_bf16_serial_sum_of_4096_ones():
    rows = {r[0]: float(r[1]) for r in read_golden("accumulation.txt")}
    s_bf16, s_f32 = 0.0, np.float32(0)
    for _ in range(int(rows["terms"])):
        s_bf16 = float(F.bf16_round(s_bf16 + 1.0))
        s_f32 = np.float32(s_f32 + np.float32(1))
    assert s_bf16 == rows["bf16_serial_sum"]
    assert float(s_f32) == rows["fp32_serial_sum"]


def test_70000_survives_bf16_not_fp16():
    v = float(dict(read_golden("overflow.txt"))["value"])
    assert np.isfinite(F.bf16_round(v))
    assert np.isinf(np.float16(v))
    # the binade rounding with fp16's parameters overflows past 65504 too
    assert F.round_binade(v, 11, -14) > F.ieee_max_finite(5, 10)


def test_bytes_per_param():
    rows = {r[0]: float(r[1]) for r in read_golden("bits_per_param.txt")}
    assert round(0.5 + 16 / 128 / 8, 3) == rows["int4_g128_bytes"]
    assert 4 + 8 / 32 == rows["mxfp4_bits"]


# ----------------------------------------------------------------------------
# E8M0 scale rule (vLLM PR #43557)
# ----------------------------------------------------------------------------

def test_e8m0_worked_table():
    for row in read_golden("e8m0_table.txt"):
        vmax, old_be, old_s, be, s, r_old, r_new = map(float, row)
        v = np.float32(vmax)
        se = int(Q.e8m0_scale_exp(v))
        assert se == be and 2.0 ** (se - 127) == s
        assert round(vmax / 2.0 ** (se - 127), 6) == r_new
        so = int(Q.e8m0_scale_exp_old(v))
        assert so == old_be and 2.0 ** (so - 127) == old_s
        assert round(vmax / 2.0 ** (so - 127), 6) == r_old


@pytest.mark.parametrize("k", [-20, -3, 0, 1, 5, 40])
def test_e8m0_threshold_edges(k):
    s = lambda m: int(Q.e8m0_scale_exp(np.float32(m * 2.0 ** k)))
    assert s(1.75) == 127 + k + 1 - 2          # significand 0.75 rounds the exponent up
    assert s(1.7421875) == 127 + k - 2         # the bf16 just below does not
    # ratio 6.5 saturates to 6; ratio 6 lands exactly on 6
    for m, code in ((1.625, 7), (1.5, 7)):
        x = np.zeros(16, np.float32)
        x[0] = m * 2.0 ** k
        packed, se = Q.quant_mxfp4(x, 16)
        assert int(se[0]) == 127 + k - 2
        assert int(Q.unpack_nibbles(packed)[0]) == code


def test_clip_zone_fractions():
    rows = {r[0]: float(r[1]) for r in read_golden("clip_zones.txt")}
    r = np.random.Generator(np.random.PCG64(11))
    sig = 1.0 + r.integers(0, 2 ** 23, 200000) / 2.0 ** 23
    vmax = (sig * 2.0 ** r.integers(-10, 10, sig.size)).astype(np.float32)

    def clip_frac(se):
        ratio = vmax / np.ldexp(1.0, se.astype(np.int64) - 127)
        return np.mean(ratio > 6.0)

    assert abs(clip_frac(Q.e8m0_scale_exp(vmax)) - rows["threshold_0.75"]) < 0.01
    assert abs(clip_frac(Q.e8m0_scale_exp_ocp(vmax)) - rows["strict_ocp"]) < 0.01
    assert clip_frac(Q.e8m0_scale_exp_ceil(vmax)) == rows["threshold_0.5"]
    ratio = vmax / np.ldexp(1.0, Q.e8m0_scale_exp(vmax).astype(np.int64) - 127)
    assert ratio.max() < 7.0 and ratio.min() >= 3.5


def test_quant_mxfp4_brute_force_small():
    """Each element's code is the nearest of all 16 codes to x / 2**(se-127),
    ties to the even code, found by exhaustive search with exact fractions."""
    r = np.random.Generator(np.random.PCG64(12))
    x = (r.standard_normal((4, 64)) * 3).astype(np.float32)
    x[0, 5] = 0.0
    x[1, :16] = 0.0
    packed, se = Q.quant_mxfp4(x, 16)
    codes = Q.unpack_nibbles(packed)
    vals = [Fraction(float(v)) for v in F.e2m1_decode(np.arange(16))]
    for i in range(4):
        for j in range(64):
            blk = x[i, (j // 16) * 16:(j // 16) * 16 + 16]
            vmax = float(np.max(np.abs(blk)))
            e = int(se[i, j // 16])
            assert e == int(Q.e8m0_scale_exp(np.float32(vmax)))
            t = Fraction(float(x[i, j])) / Fraction(2) ** (e - 127)
            t = max(min(t, Fraction(6)), Fraction(-6))
            best = min(range(16), key=lambda c: (abs(vals[c] - t), c % 2, -c if t < 0 else c))
            got = int(codes[i, j])
            assert vals[got] == vals[best], (i, j, got, best)


# ----------------------------------------------------------------------------
# FP8 block quantizer
# ----------------------------------------------------------------------------

def test_fp8_scale_page_example():
    rows = {r[0]: float(r[1]) for r in read_golden("scale_example.txt")}
    x = np.zeros(128, np.float32)
    x[3] = np.float32(rows["amax"])
    x[7] = np.float32(-1.0)
    codes, s = Q.quant_fp8_block(x, 128)
    assert np.isclose(float(s[0]), rows["scale"], rtol=1e-6)
    assert F.e4m3_decode(codes[3]) == rows["largest_lands_on"]


def test_fp8_block_invariants():
    r = np.random.Generator(np.random.PCG64(13))
    x = r.standard_normal((16, 512)).astype(np.float32) * np.float32(3.0)
    x[2, 128:256] = 0.0
    codes, s = Q.quant_fp8_block(x, 128)
    dec = F.e4m3_decode(codes).reshape(16, 4, 128)
    xb = x.reshape(16, 4, 128).astype(np.float64)
    assert s[2, 1] == 1.0 and np.all(codes.reshape(16, 4, 128)[2, 1] == 0)
    for i in range(16):
        for b in range(4):
            if i == 2 and b == 1:
                continue
            j = np.argmax(np.abs(xb[i, b]))
            assert abs(dec[i, b, j]) == 448.0
            t = xb[i, b] / float(s[i, b])
            # one rounding: relative error <= 2**-4 for normals, abs <= 2**-10 below
            err = np.abs(dec[i, b] - t)
            assert np.all(err <= np.maximum(np.abs(t) * 2.0 ** -4, 2.0 ** -10) * (1 + 1e-6))


# ----------------------------------------------------------------------------
# weight quantizers (invariants only: parity unpinned)
# ----------------------------------------------------------------------------

def test_int4_rtn_invariants():
    r = np.random.Generator(np.random.PCG64(14))
    w = (r.standard_normal((8, 512)) * 0.02).astype(np.float32)
    w[3, 128:256] = 0
    packed, sb = Q.quant_int4_rtn(w, 128)
    q = F.int4_decode(Q.unpack_nibbles(packed)).reshape(8, 4, 128)
    s = F.bf16_decode(sb)
    assert sb[3, 1] == 0x3F80 and np.all(q[3, 1] == 0)
    wb = w.reshape(8, 4, 128).astype(np.float64)
    for i in range(8):
        for g in range(4):
            if i == 3 and g == 1:
                continue
            assert np.max(np.abs(q[i, g])) == 7
            assert np.all(np.abs(q[i, g] * s[i, g] - wb[i, g]) <= s[i, g] / 2 * (1 + 2.0 ** -7))


def test_int4_zp_worked_example():
    """A hand-derived group of 4 (g = 4) under the asymmetric reading of
    "Numerics" (x = s (q - z)): lo = -0.3, hi = 1.2, (hi - lo) / 15 = 0.1 in
    fp32, whose bf16 rounding is 0x3DCD = 0.10009765625; z = rint(0.3 / s) =
    rint(2.997..) = 3; q = rint(w / s) + z = (-3, 0, 4, 12) + 3 = (0, 3, 7, 15).
    Dequant (q - z) s = (-3, 0, 4, 12) * s = (-0.30029296875, 0, 0.400390625,
    1.201171875), whose bf16 roundings are (-0.30078125, 0, 0.400390625,
    1.203125) (0.201171875 * 128 = 25.75 rounds up to 26)."""
    w = np.array([[-0.3, 0.0, 0.45, 1.2]], np.float32)
    packed, sb, z = Q.quant_int4_zp(w, 4)
    assert int(sb[0, 0]) == 0x3DCD and int(z[0, 0]) == 3
    assert list(Q.unpack_nibbles(packed)[0]) == [0, 3, 7, 15]
    deq = F.bf16_decode(G.dequant_int4_zp(packed, sb, z, 4))[0]
    assert list(deq) == [-0.30078125, 0.0, 0.400390625, 1.203125]


def test_int4_zp_invariants():
    r = np.random.Generator(np.random.PCG64(17))
    w = (r.standard_normal((8, 512)) * 0.02 + 0.01).astype(np.float32)
    w[3, 64:128] = 0
    w[5, 0:64] = 0.25                                # constant nonzero group
    packed, sb, z = Q.quant_int4_zp(w, 64)
    q = Q.unpack_nibbles(packed).reshape(8, 8, 64).astype(np.int64)
    s = F.bf16_decode(sb)
    assert sb[3, 1] == 0x3F80 and z[3, 1] == 0 and np.all(q[3, 1] == 0)   # all-zero policy
    assert sb[5, 0] == 0x3F80                        # flat group: s = 1 as well
    assert np.all(z <= 15) and np.all(q <= 15)
    wb = w.reshape(8, 8, 64).astype(np.float64)
    for i in range(8):
        for g in range(8):
            if (i, g) in ((3, 1), (5, 0)):
                continue
            lo_i, hi_i = np.argmin(wb[i, g]), np.argmax(wb[i, g])
            assert q[i, g, lo_i] == 0 or z[i, g] == 0    # the minimum maps to code 0 (unless z clamps)
            err = np.abs((q[i, g] - int(z[i, g])) * s[i, g] - wb[i, g])
            assert np.all(err <= s[i, g] * (0.5 + 2.0 ** -6)), (i, g, err.max() / s[i, g])


def test_int4_zp_at_z8_is_the_symmetric_dequant():
    """With z = 8 and the unsigned nibble u = q + 8, s (u - z) is s q: the
    asymmetric dequant must reproduce the (separately pinned) symmetric one bit
    for bit, for every q in [-8, 7] and a spread of bf16 scales."""
    r = np.random.Generator(np.random.PCG64(18))
    s_bits = r.integers(0x2000, 0x5000, (32, 2)).astype(np.uint16)
    q = np.tile(np.arange(-8, 8), 16).reshape(1, 256).repeat(32, 0)
    sym = G.dequant_int4(Q.pack_nibbles(q & 0xF), s_bits, 128)
    asym = G.dequant_int4_zp(Q.pack_nibbles(q + 8), s_bits, np.full((32, 2), 8, np.uint8), 128)
    assert np.array_equal(sym, asym)


def test_dequant_int4_zp_is_one_rounding_of_the_exact_product():
    r = np.random.Generator(np.random.PCG64(19))
    s_bits = r.integers(0x3000, 0x4400, 16).astype(np.uint16)
    u = np.arange(16)
    for zv in range(16):
        packed = Q.pack_nibbles(np.tile(u, 4).reshape(1, 64).repeat(16, 0))
        deq = F.bf16_decode(G.dequant_int4_zp(packed, s_bits.reshape(16, 1), np.full((16, 1), zv, np.uint8), 64))
        for n in range(16):
            sv = Fraction(float(F.bf16_decode(s_bits[n])))
            for k in range(16):
                assert Fraction(float(deq[n, k])) == _nearest_bf16_fraction((int(u[k]) - zv) * sv)


def test_nvfp4_invariants():
    r = np.random.Generator(np.random.PCG64(15))
    w = (r.standard_normal((8, 256)) * 0.02).astype(np.float32)
    packed, sb, gs = Q.quant_nvfp4(w)
    assert np.isclose(float(gs), np.abs(w).max() / 2688.0, rtol=1e-6)
    i, j = np.unravel_index(np.argmax(np.abs(w)), w.shape)
    assert F.e4m3_decode(sb[i, j // 16]) == 448.0
    codes = Q.unpack_nibbles(packed)
    assert abs(F.e2m1_decode(codes[i, j])) == 6.0
    deq = F.e2m1_decode(codes) * np.repeat(F.e4m3_decode(sb), 16, axis=1) * float(gs)
    scale = np.repeat(F.e4m3_decode(sb), 16, axis=1) * float(gs)
    # one E2M1 rounding of w / scale (relative 2**-2 for normals) plus saturation at 6
    assert np.all(np.abs(deq - w) <= np.maximum(np.abs(w) * 0.25, 0.25 * scale) * 1.001 + 1e-12)


# ----------------------------------------------------------------------------
# dequantization and products: exact arithmetic as the other side
# ----------------------------------------------------------------------------

def _nearest_bf16_fraction(v):
    """Round an exact Fraction to bf16 by exhaustive search over the 2 neighbours."""
    f = float(v)                                     # within 1 ulp of double
    lo = F.bf16_decode(F.bf16_encode(np.float64(f)))
    cands = set()
    for base in (float(lo),):
        b = int(F.bf16_encode(np.float64(base)))
        for d in (-2, -1, 0, 1, 2):
            c = (b + d) & 0xFFFF
            cv = float(F.bf16_decode(np.uint16(c)))
            if np.isfinite(cv):
                cands.add((Fraction(cv), c))
    best = min(cands, key=lambda fc: (abs(fc[0] - v), (fc[1] & 1)))
    return best[0]


def test_dequant_int4_is_one_rounding_of_the_exact_product():
    r = np.random.Generator(np.random.PCG64(16))
    s_bits = r.integers(0x3000, 0x4400, 64).astype(np.uint16)
    q = np.arange(-8, 8)
    packed = Q.pack_nibbles(np.tile(q & 0xF, 8).reshape(1, 128).repeat(64, 0))
    deq = F.bf16_decode(G.dequant_int4(packed, s_bits.reshape(64, 1), 128))
    for n in range(64):
        s = Fraction(float(F.bf16_decode(s_bits[n])))
        for k in range(16):
            assert Fraction(float(deq[n, k])) == _nearest_bf16_fraction(int(q[k]) * s)


def test_gemm_f64_matches_exact_brute_force():
    """Dyadic x and w on tiny odd shapes: the fp64 product is exact, so it must
    equal a pure-Python Fraction sum; a transposed operand or dropped scale
    fails here (N != M != K)."""
    r = np.random.Generator(np.random.PCG64(17))
    M, N, K = 3, 5, 64
    x = (r.integers(-16, 16, (M, K)) / 8.0).astype(np.float32)
    w = (r.integers(-16, 16, (N, K)) / 4.0).astype(np.float32)
    cs = (r.integers(1, 9, N) / 2.0)
    xb = F.bf16_encode(x)
    wb = F.bf16_encode(w)
    y = G.gemm_bf16_f64(xb, wb, cs)
    for m in range(M):
        for n in range(N):
            ref = sum(Fraction(float(x[m, k])) * Fraction(float(w[n, k])) for k in range(K))
            assert Fraction(float(y[m, n])) == ref * Fraction(float(cs[n]))


def test_w8a8_matches_exact_brute_force():
    """E4M3 codes on both sides, per-block activation scales and per-channel
    weight scales that are powers of two: every term is exact, so the fp64
    oracle must equal a Fraction sum; swapping the block index, a transposed
    operand or a scale on the wrong axis fails (M != N, 3 blocks)."""
    r = np.random.Generator(np.random.PCG64(23))
    M, N, g, nb = 2, 3, 16, 3
    K = g * nb
    a = r.integers(0, 0x7F, (M, K)).astype(np.uint8) | (r.integers(0, 2, (M, K)) << 7).astype(np.uint8)
    w = r.integers(0, 0x7F, (N, K)).astype(np.uint8)
    a_s = 2.0 ** r.integers(-4, 4, (M, nb)).astype(np.float64)
    cs = 2.0 ** r.integers(-3, 3, N).astype(np.float64)
    y = G.w8a8_f64(a, a_s, w, cs, g)
    for m in range(M):
        for n in range(N):
            ref = Fraction(0)
            for b in range(nb):
                part = sum(Fraction(float(F.e4m3_decode(a[m, k]))) * Fraction(float(F.e4m3_decode(w[n, k])))
                           for k in range(b * g, (b + 1) * g))
                ref += part * Fraction(float(a_s[m, b]))
            assert Fraction(float(y[m, n])) == ref * Fraction(float(cs[n]))


def test_w4a8_grouped_matches_exact_brute_force():
    r = np.random.Generator(np.random.PCG64(18))
    E, N, K, g = 3, 4, 256, 128
    off = np.array([0, 2, 2, 5], dtype=np.int32)
    a = r.integers(0, 256, (5, K)).astype(np.uint8)
    a[(a & 0x7F) == 0x7F] = 0x10
    a_s = (r.integers(1, 5, 5) / 4.0).astype(np.float32)
    qn = r.integers(0, 16, (E, N, K)).astype(np.uint8)
    packed = Q.pack_nibbles(qn)
    s_bits = r.integers(0x3C00, 0x4000, (E, N, K // g)).astype(np.uint16)
    y = G.w4a8_grouped_f64(a, a_s, off, packed, s_bits, g)
    av = F.e4m3_decode(a)
    qv = F.int4_decode(qn)
    sv = F.bf16_decode(s_bits)
    for row in range(5):
        e = int(np.searchsorted(off, row, side="right") - 1)
        for n in range(N):
            ref = sum(Fraction(float(av[row, k])) * int(qv[e, n, k]) * Fraction(float(sv[e, n, k // g]))
                      for k in range(K))
            assert Fraction(float(y[row, n])) == ref * Fraction(float(a_s[row]))


def test_output_narrowing_is_a_single_rounding():
    """bf16(y64) must not go through fp32 (double rounding): y = 1 + 2**-8 +
    2**-30 rounds up in one step but ties-to-even down via fp32."""
    y = 1.0 + 2.0 ** -8 + 2.0 ** -30
    assert F.bf16_decode(G.to_bf16(np.float64(y))) == 1.0 + 2.0 ** -7
    y32 = np.float32(y)            # 1 + 2**-8 exactly (the 2**-30 is lost)
    assert F.bf16_decode(G.to_bf16(np.float64(y32))) == 1.0


# ----------------------------------------------------------------------------
# W4A8 with FP8 group scales ("Production-Ready W4A8", "Accurate W4A8 Kernel")
# ----------------------------------------------------------------------------

def _e4m3_values():
    codes = np.arange(256, dtype=np.uint8)
    vals = F.e4m3_decode(codes)
    fin = np.isfinite(vals)
    return codes[fin], vals[fin]


def test_fp8_group_scales_never_clip_int4_products():
    """The page scales the FP8 scales by 1/8 so that 'weights are guaranteed
    to be in FP8 range after multiplication by INT4 values': every finite E4M3
    scale divided by 8 times every INT4 value is within +-448."""
    codes, vals = _e4m3_values()
    s8 = F.e4m3_decode(F.e4m3_encode((vals.astype(np.float32) * np.float32(0.125)).astype(np.float32)))
    prod = np.abs(np.arange(-8, 8, dtype=np.float64)[:, None] * s8[None, :])
    assert prod.max() == 448.0                      # reached by q = -8 and the largest scale 448 / 8
    # without the 1/8 the same products overflow E4M3 (the clipping the page shows)
    assert (np.abs(np.arange(-8, 8)[:, None] * vals[None, :]) > 448).any()


def test_fp8_group_scales_worked_example():
    """One channel with bf16 group scales s, s/2, s/4, 0 (exact ratios):
    cs = s/448, the codes of 448, 224, 112, 0; after the 1/8: 56, 28, 14, 0;
    channel scale times 8 (reading of 'quantize each column of BF16 group-wise
    scales to FP8' with the activation quantizer, then 'scale the FP8 scales
    by 1/8 ... multiplying per-channel scales by eight')."""
    s = np.float32(0.02)
    row = np.array([[s, s / 2, s / 4, 0.0]], np.float32)
    bits = F.bf16_encode(row)
    s8, cs8 = Q.fp8_group_scales(bits)
    sb = F.bf16_decode(bits)[0, 0]
    assert list(F.e4m3_decode(s8)[0]) == [56.0, 28.0, 14.0, 0.0]
    assert float(cs8[0]) == float(np.float32(np.float32(sb) / np.float32(448.0)) * np.float32(8.0))
    # the E4M3 codes themselves, from the format definition: 56 = 1.75 * 2^5 -> e = 12, m = 6
    assert list(s8[0]) == [(12 << 3) | 6, (11 << 3) | 6, (10 << 3) | 6, 0]


def test_fp8_lut_weights_match_brute_force_nearest_code():
    """E4M3(q * s8) against a brute-force nearest-code search over all 256
    codes with ties to the even code (an independent formulation)."""
    codes, vals = _e4m3_values()
    order = np.argsort(vals, kind="stable")
    rng = np.random.Generator(np.random.PCG64(17))
    s8 = rng.choice(codes[(vals > 0) & (vals <= 56)], size=(3, 2)).astype(np.uint8)
    q = rng.integers(-8, 8, size=(3, 256))
    packed = Q.pack_nibbles(q.astype(np.int64))
    got = Q.fp8_lut_weights(packed, s8, g=128)
    for n in range(3):
        for k in range(256):
            x = Fraction(int(q[n, k])) * Fraction(float(F.e4m3_decode(s8[n, k // 128])))
            best = None
            for c in codes:
                v = Fraction(float(F.e4m3_decode(np.uint8(c))))
                d = abs(v - x)
                key = (d, int(c) & 1)                 # nearest, then the even code
                if best is None or key < best[0]:
                    best = (key, c)
            want = F.e4m3_decode(np.uint8(best[1]))
            assert F.e4m3_decode(got[n, k]) == want, (n, k, q[n, k])


def test_w4a8_fp8s_grouped_matches_exact_brute_force():
    """The grouped product with the outer per-token x per-channel scaling,
    against exact rational arithmetic."""
    rng = np.random.Generator(np.random.PCG64(23))
    E, N, K, off = 2, 3, 64, np.array([0, 2, 5], np.int32)
    a = rng.integers(0, 256, size=(5, K)).astype(np.uint8)
    a[(a & 0x7F) == 0x7F] = 0                         # no NaN codes
    a_s = rng.random(5).astype(np.float32)
    w8 = rng.integers(0, 256, size=(E, N, K)).astype(np.uint8)
    w8[(w8 & 0x7F) == 0x7F] = 0
    cs8 = rng.random((E, N)).astype(np.float32)
    y = G.w4a8_fp8s_grouped_f64(a, a_s, off, w8, cs8)
    for e in range(E):
        for r in range(off[e], off[e + 1]):
            for n in range(N):
                acc = sum(Fraction(float(F.e4m3_decode(a[r, k]))) * Fraction(float(F.e4m3_decode(w8[e, n, k])))
                          for k in range(K))
                want = acc * Fraction(float(a_s[r])) * Fraction(float(cs8[e, n]))
                assert abs(Fraction(y[r, n]) - want) <= abs(want) * Fraction(1, 2 ** 50)


def test_fp8_group_scale_recipe_stays_close_to_exact_w4a8():
    """Invariant: the recipe adds one E4M3 rounding per weight (3 mantissa
    bits), so on RTN-quantized N(0, 0.02) weights its output stays within a
    few percent of the exact W4A8 product."""
    from numerics_packed_int4_gb300 import inputs
    N, K, R = 64, 512, 32
    q, s = Q.quant_int4_rtn(inputs.weights_f32(N, K, seed=5), 128)
    s8, cs8 = Q.fp8_group_scales(s)
    w8 = Q.fp8_lut_weights(q, s8)
    a, a_s = Q.quant_fp8_block(F.bf16_decode(inputs.activations_bf16(R, K, seed=6)), K)
    off = np.array([0, R], np.int32)
    exact = G.w4a8_grouped_f64(a, a_s[:, 0], off, q[None], s[None], 128)
    recipe = G.w4a8_fp8s_grouped_f64(a, a_s[:, 0], off, w8[None], cs8[None])
    rel = np.linalg.norm(recipe - exact) / np.linalg.norm(exact)
    assert 1e-3 < rel < 5e-2


# ----------------------------------------------------------------------------
# W4A4 MXFP4 x MXFP4 (vLLM PR #43557's W4A4 GEMM, activations by the a6 rule)
# ----------------------------------------------------------------------------

E2M1_TABLE = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]     # the E2M1 magnitudes the pages list


def _e2m1_value(code):
    v = Fraction(E2M1_TABLE[code & 7]).limit_denominator(2)
    return -v if code & 8 else v


def _nibble(packed_row, k):
    b = int(packed_row[k // 2])
    return b & 0xF if k % 2 == 0 else b >> 4


def _mxfp4_weights(N, K, seed):
    r = np.random.Generator(np.random.PCG64(seed))
    w = (r.standard_normal((N, K)) * 0.02).astype(np.float32)
    return Q.quant_mxfp4_weights(w)


def test_w4a4_matches_exact_brute_force():
    """Both operands decoded by hand (E2M1 table, 2^(c-127) scales, nibble
    order even-k low) and summed as Fractions: the fp64 oracle must agree
    exactly (every term is a dyadic rational well inside fp64).  Two
    activation blocks per row, M != N, so a swapped block index or a
    transposed operand fails."""
    r = np.random.Generator(np.random.PCG64(31))
    M, N, K = 3, 4, 64
    x = F.bf16_encode((r.standard_normal((M, K)) * np.exp2(r.integers(-6, 6, (M, 1)))).astype(np.float32))
    wq, wse = _mxfp4_weights(N, K, 32)
    y, aq, ase = G.w4a4_mxfp4_f64(x, wq, wse)
    for m in range(M):
        for n in range(N):
            ref = Fraction(0)
            for k in range(K):
                a = _e2m1_value(_nibble(aq[m], k)) * Fraction(2) ** (int(ase[m, k // 32]) - 127)
                w = _e2m1_value(_nibble(wq[n], k)) * Fraction(2) ** (int(wse[n, k // 32]) - 127)
                ref += a * w
            assert Fraction(float(y[m, n])) == ref


def test_w4a4_on_representable_activations_is_the_w4a16_product():
    """Activations that already are MXFP4 values, each 32-block holding a
    6 * 2^e element (the rule's vecMax 6 * 2^e gives scale exponent e, so the
    quantizer returns them unchanged): W4A4 must equal the weight-only MXFP4
    product of the same bf16 activations, bit for bit in fp64."""
    r = np.random.Generator(np.random.PCG64(37))
    M, N, K = 5, 6, 128
    codes = r.integers(0, 16, (M, K)).astype(np.uint8)
    codes[:, ::32] = 7                                          # +6 in every block
    e = r.integers(-20, 10, (M, K // 32))
    vals = F.e2m1_decode(codes) * np.exp2(np.repeat(e, 32, axis=1))
    x = F.bf16_encode(vals.astype(np.float32))
    assert np.array_equal(F.bf16_decode(x), vals)               # representable in bf16
    wq, wse = _mxfp4_weights(N, K, 38)
    y, aq, ase = G.w4a4_mxfp4_f64(x, wq, wse)
    np.testing.assert_array_equal(ase, (e + 127).astype(np.uint8))
    np.testing.assert_array_equal(Q.unpack_nibbles(aq), codes)   # -0 keeps its sign code
    np.testing.assert_array_equal(y, G.qgemm_mxfp4a16(x, wq, wse))


@pytest.mark.parametrize("j", [-9, -1, 3, 12])
def test_w4a4_commutes_with_power_of_two_activation_scaling(j):
    """Scaling the activations by 2^j moves every block scale by j and leaves
    the E2M1 codes alone, so the product scales by exactly 2^j."""
    r = np.random.Generator(np.random.PCG64(41))
    M, N, K = 4, 3, 96
    xf = r.standard_normal((M, K)).astype(np.float32)
    wq, wse = _mxfp4_weights(N, K, 42)
    y0, aq0, ase0 = G.w4a4_mxfp4_f64(F.bf16_encode(xf), wq, wse)
    y1, aq1, ase1 = G.w4a4_mxfp4_f64(F.bf16_encode(np.ldexp(xf, j)), wq, wse)
    np.testing.assert_array_equal(aq1, aq0)
    np.testing.assert_array_equal(ase1.astype(int), ase0.astype(int) + j)
    np.testing.assert_array_equal(y1, np.ldexp(y0, j))


# ----------------------------------------------------------------------------
# MoE harness between the projections: SwiGLU and the weighted combine.
# The pages name a fused SwiGLU kernel (FreeToken PR #805's list of native
# kernels) but print no formula; these pins come from the mathematics of
# SiLU(v) = v * sigmoid(v) and of an exact weighted sum.
# ----------------------------------------------------------------------------

def _gate_up(gate, up):
    """[R, 2I] bf16 bit patterns with the gate columns first."""
    return F.bf16_encode(np.concatenate([np.asarray(gate, np.float32), np.asarray(up, np.float32)], 1))


def _bf16_grid(lo, hi):
    """Every finite bf16 value in [lo, hi] (as float32)."""
    v = F.bf16_decode(np.arange(65536, dtype=np.uint32)).astype(np.float64)
    v = v[np.isfinite(v) & (v >= lo) & (v <= hi)]
    return np.unique(v).astype(np.float32)


def test_silu_at_zero_is_zero():
    """SiLU(0) = 0 whatever the up value, and up = 0 zeroes any gate."""
    up = np.array([[1.0, -3.0, 250.0, 2.0 ** -20]], np.float32)
    h = G.swiglu_f32(_gate_up(np.zeros_like(up), up), 4)
    assert np.all(h == 0)
    h = G.swiglu_f32(_gate_up(np.array([[5.0, -5.0, 0.5, 100.0]], np.float32), np.zeros_like(up)), 4)
    assert np.all(h == 0)


def test_silu_odd_part_is_the_identity():
    """sigmoid(v) + sigmoid(-v) = 1, so SiLU(v) - SiLU(-v) = v exactly.  Each
    side is one fp32 rounding of the true value, so the fp32 difference is v
    within half an ulp of each side, over every bf16 value in [-30, 30]."""
    v = _bf16_grid(-30.0, 30.0)
    ones = np.ones((1, v.size), np.float32)
    hp = G.swiglu_f32(_gate_up(v[None, :], ones), v.size).astype(np.float64)[0]
    hn = G.swiglu_f32(_gate_up(-v[None, :], ones), v.size).astype(np.float64)[0]
    ulp = lambda a: np.spacing(np.abs(a).astype(np.float32)).astype(np.float64)
    assert np.all(np.abs((hp - hn) - v) <= 0.5 * (ulp(hp) + ulp(hn)) * 1.0001)


def test_silu_limits():
    """SiLU(v) -> v as v -> +inf and -> 0 as v -> -inf: for v >= 40, e^-v <
    2^-57 and the fp32 result is v itself; for v <= -40, |SiLU(v)| <= |v| e^v."""
    v = _bf16_grid(40.0, 3.0e38)
    v = v[:: max(1, v.size // 400)]
    h = G.swiglu_f32(_gate_up(v[None, :], np.ones((1, v.size), np.float32)), v.size)[0]
    assert np.array_equal(h, v)
    n = -v[v <= 80.0]
    h = G.swiglu_f32(_gate_up(n[None, :], np.ones((1, n.size), np.float32)), n.size)[0].astype(np.float64)
    assert np.all(h <= 0) and np.all(np.abs(h) <= np.abs(n) * np.exp(n.astype(np.float64)) * 1.0001)


@pytest.mark.parametrize("j", [10, 12, 16])
def test_silu_taylor_point(j):
    """Near 0, SiLU(x) = x/2 + x^2/4 - x^4/48 + ...  For x = 2^-j the quartic
    term is below half an fp32 ulp of x/2, so the fp32 result is exactly
    2^-(j+1) + 2^-(2j+2).  A sign error in the exponent gives x/2 - x^2/4, a
    GELU-style gate x/2 + 0.399 x^2: both miss this value."""
    x = np.float32(2.0 ** -j)
    h = G.swiglu_f32(_gate_up([[x]], [[1.0]]), 1)[0, 0]
    assert h == np.float32(2.0 ** -(j + 1) + 2.0 ** -(2 * j + 2))


def test_silu_matches_the_logistic_routine():
    """SiLU(v) = v * expit(v), with scipy's logistic function as the
    independent routine (every bf16 value in [-60, 60], unit up)."""
    special = pytest.importorskip("scipy.special")
    v = _bf16_grid(-60.0, 60.0)
    h = G.swiglu_f32(_gate_up(v[None, :], np.ones((1, v.size), np.float32)), v.size)[0]
    ref = (v.astype(np.float64) * special.expit(v.astype(np.float64))).astype(np.float32)
    assert np.array_equal(h, ref)


def test_swiglu_takes_the_gate_from_the_first_half():
    """gate = [50, 0], up = [3, 7]: SiLU(50) * 3 = 150 and SiLU(0) * 7 = 0.
    With the halves swapped the row would be [SiLU(3) * 50, SiLU(7) * 0] =
    [142.88.., 0]; with the up projection ignored, [50, 0]."""
    h = G.swiglu_f32(_gate_up([[50.0, 0.0]], [[3.0, 7.0]]), 2)
    assert h.tolist() == [[150.0, 0.0]]
    # the product is formed in wide precision and rounded once: SiLU(v) * u
    # with u = 3 for v where the fp32 SiLU times 3 would round differently
    v = _bf16_grid(0.5, 8.0)
    h = G.swiglu_f32(_gate_up(v[None, :], np.full((1, v.size), 3.0, np.float32)), v.size)[0]
    ref = [float(Fraction(float(x)) * 3 / (1 + Fraction(np.exp(-np.float64(x))))) for x in v]
    assert np.array_equal(h, np.array(ref, np.float64).astype(np.float32))


def test_moe_combine_matches_exact_brute_force():
    """out[t] = bf16(sum over the rows routed from t of p * down[row]): dyadic
    rows and weights (every product and sum exact as a Fraction), rows in a
    scrambled order, one token with no rows, weights not renormalised.  The
    exact sum rounded once to bf16 (nearest, ties to even, by search) must be
    the oracle's output; a dropped weight, a wrong row index or a second
    rounding fails it."""
    r = np.random.Generator(np.random.PCG64(23))
    T, H, R = 5, 24, 8
    route_rows = np.array([3, 0, 1, 3, 0, 4, 1, 3])           # token 2 gets no row
    weight = r.integers(1, 64, R) / 64.0                       # dyadic, not summing to 1
    down = F.bf16_encode((r.integers(-512, 512, (R, H)) / 8.0).astype(np.float32) +
                         np.float32(2.0 ** -9))                # 13-bit values: bf16 rounds some
    out = F.bf16_decode(G.moe_combine(down, route_rows, weight, T))
    dv = F.bf16_decode(down)
    for t in range(T):
        for h in range(H):
            acc = sum((Fraction(float(weight[i])) * Fraction(float(dv[i, h]))
                       for i in range(R) if route_rows[i] == t), Fraction(0))
            assert Fraction(float(out[t, h])) == _nearest_bf16_fraction(acc)
    assert np.all(out[2] == 0)
