// In-register weight decode: packed low-bit codes -> bf16x2 pairs.
//
// Every routine produces the canonical dequantized weight bit for bit:
//   INT4   bf16_RNE(q * s): the nibble becomes the exact bf16 integer q with
//          the magic-number trick ((u | 0x4300) - 136 with u = q + 8), then one
//          bf16 multiply by the group scale rounds the exact product once; with
//          a zero point, bf16_RNE((u - z) * s) the same way ((u | 0x4300) -
//          (128 + z));
//   E4M3   exact: sign and the 7 exponent/mantissa bits move into bf16
//          position with shift/and/or (the FP8 -> FP16 bit trick described in
//          "Your 3090 Isn't Missing Anything...", section 4.1, with the bf16
//          shift of 4) and one exact multiply by 2^120 restores the bias;
//   E2M1   exact: the three magnitude bits land in the bf16 exponent/mantissa
//          field (value * 2^-126, subnormal code included) and one exact
//          multiply by 2^126 restores the bias; the block scale (a power of
//          two for MXFP4, an E4M3 value for NVFP4) is one more exact multiply.
// No table lookups; shifts, lop3 and packed bf16 arithmetic only.
//
// Pair order: the "kperm" forms return, for the 8 k-values k0..k7 held by one
// 32-bit word (4-bit formats) or two words (E4M3), the pairs used directly as
// mma.sync A fragments.  Callers that need natural k order use the
// *_natural helpers (one prmt per pair).
#pragma once

#include "qg_common.cuh"

namespace qg {

constexpr uint32_t kBf16x2_136 = 0x43084308u;     // 136.0 in both lanes
constexpr uint32_t kBf16x2_2p120 = 0x7B807B80u;   // 2^120
constexpr uint32_t kBf16x2_2p126 = 0x7E807E80u;   // 2^126

// lop3 truth tables: a = 0xF0, b = 0xCC, c = 0xAA
constexpr int kLutAndXor = 0x6A;   // (a & b) ^ c
constexpr int kLutAndOr = 0xEA;    // (a & b) | c

// ---- INT4 -------------------------------------------------------------------
// p[i] = (k_i, k_{i+4}) for i = 0..3
QG_DEVICE void int4x8_kperm(uint32_t v, uint32_t s2, uint32_t (&p)[4]) {
  p[0] = lop3<kLutAndXor>(v, 0x000F000Fu, 0x43084308u);   // 0x4300 | (nibble ^ 8)
  p[1] = lop3<kLutAndXor>(v >> 4, 0x000F000Fu, 0x43084308u);
  p[2] = lop3<kLutAndXor>(v >> 8, 0x000F000Fu, 0x43084308u);
  p[3] = lop3<kLutAndXor>(v >> 12, 0x000F000Fu, 0x43084308u);
#pragma unroll
  for (int i = 0; i < 4; ++i) p[i] = bf16x2_mul(bf16x2_sub(p[i], kBf16x2_136), s2);
}

// Natural k order straight from the nibbles, for operands stored to tensor
// memory: byte b of v holds (k_2b, k_2b+1) and byte b of v >> 4 has k_2b+1 in
// its low nibble, so one prmt puts k_2b under the low half's magic and k_2b+1
// under the high half's; then the same (u | 0x4300) - 136 and one multiply by
// the scale as int4x8_kperm.  p[b] = (k_2b, k_2b+1) for b = 0..3.
QG_DEVICE void int4x8_nat(uint32_t v, uint32_t s2, uint32_t (&p)[4]) {
  const uint32_t v4 = v >> 4;
#pragma unroll
  for (int b = 0; b < 4; ++b) {
    const uint32_t t = prmt(v, v4, (uint32_t)(b | ((4 + b) << 8)));
    p[b] = bf16x2_mul(bf16x2_sub(lop3<kLutAndXor>(t, 0x000F000Fu, 0x43084308u), kBf16x2_136), s2);
  }
}

// ---- INT4 with a zero point -----------------------------------------------------
// Unsigned nibble u, group zero point z and scale s: (u | 0x4300) is the exact
// bf16 128 + u; subtracting zb2 = bf16x2(128 + z) leaves the exact integer
// u - z in [-15, 15], and one bf16 multiply by s rounds (u - z) * s once --
// the canonical bf16_RNE((q - z) * s), at the cost of the symmetric decode.
QG_DEVICE uint32_t bf16x2_zero128(uint32_t z) { return (0x4300u | (z & 0xFu)) * 0x00010001u; }
// Natural-order form (see int4x8_nat) with a zero point: zb2 = bf16x2(128 + z).
QG_DEVICE void int4zp_x8_nat(uint32_t v, uint32_t s2, uint32_t zb2, uint32_t (&p)[4]) {
  const uint32_t v4 = v >> 4;
#pragma unroll
  for (int b = 0; b < 4; ++b) {
    const uint32_t t = prmt(v, v4, (uint32_t)(b | ((4 + b) << 8)));
    p[b] = bf16x2_mul(bf16x2_sub(lop3<kLutAndOr>(t, 0x000F000Fu, 0x43004300u), zb2), s2);
  }
}
// p[i] = (k_i, k_{i+4}) for i = 0..3
QG_DEVICE void int4zp_x8_kperm(uint32_t v, uint32_t s2, uint32_t zb2, uint32_t (&p)[4]) {
  p[0] = lop3<kLutAndOr>(v, 0x000F000Fu, 0x43004300u);      // 0x4300 | nibble = 128 + u
  p[1] = lop3<kLutAndOr>(v >> 4, 0x000F000Fu, 0x43004300u);
  p[2] = lop3<kLutAndOr>(v >> 8, 0x000F000Fu, 0x43004300u);
  p[3] = lop3<kLutAndOr>(v >> 12, 0x000F000Fu, 0x43004300u);
#pragma unroll
  for (int i = 0; i < 4; ++i) p[i] = bf16x2_mul(bf16x2_sub(p[i], zb2), s2);
}

// ---- fp16 forms (W4A8: exact products on a 16-bit MMA) ------------------------
QG_DEVICE uint32_t f16x2_sub(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}
QG_DEVICE uint32_t f16x2_mul(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}
// two E4M3 codes (low byte first) -> f16x2 (low half first), exact
QG_DEVICE uint32_t e4m3x2_to_f16x2(uint32_t two) {
  uint32_t d;
  const uint16_t in = (uint16_t)two;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(d) : "h"(in));
  return d;
}
QG_DEVICE uint16_t f32_to_f16_bits(float f) {
  uint16_t r;
  asm("cvt.rn.f16.f32 %0, %1;" : "=h"(r) : "f"(f));
  return r;
}

// Natural-order fp16 form (see int4x8_nat): p[b] = (k_2b, k_2b+1) * scale.
QG_DEVICE void int4x8_nat_f16(uint32_t v, uint32_t s2, uint32_t (&p)[4]) {
  const uint32_t v4 = v >> 4;
#pragma unroll
  for (int b = 0; b < 4; ++b) {
    const uint32_t t = prmt(v, v4, (uint32_t)(b | ((4 + b) << 8)));
    p[b] = f16x2_mul(f16x2_sub(lop3<kLutAndXor>(t, 0x000F000Fu, 0x64086408u), 0x64086408u), s2);
  }
}

// ---- E2M1 -------------------------------------------------------------------
// p[i] = (k_i, k_{i+4}) for i = 0..3, each e2m1 * scale (exact)
// The E2M1 bit patterns only: p[i] = (k_i, k_{i+4}) * 2^-126 (exact, the
// 0.5 code a bf16 subnormal).
QG_DEVICE void e2m1x8_kperm_raw(uint32_t v, uint32_t (&p)[4]) {
  const uint32_t MAG = 0x01C001C0u, SGN = 0x80008000u;
  p[0] = lop3<kLutAndOr>(v << 6, MAG, (v << 12) & SGN);
  p[1] = lop3<kLutAndOr>(v << 2, MAG, (v << 8) & SGN);
  p[2] = lop3<kLutAndOr>(v >> 2, MAG, (v << 4) & SGN);
  p[3] = lop3<kLutAndOr>(v >> 6, MAG, v & SGN);
}
QG_DEVICE void e2m1x8_kperm(uint32_t v, uint32_t scale2, uint32_t (&p)[4]) {
  e2m1x8_kperm_raw(v, p);
#pragma unroll
  for (int i = 0; i < 4; ++i) p[i] = bf16x2_mul(bf16x2_mul(p[i], kBf16x2_2p126), scale2);
}
// One multiply by a folded factor f2 = 2^126 * (block scale) * 2^-j: the caller
// guarantees f2 is a normal bf16 and undoes 2^-j on the accumulated row.
QG_DEVICE void e2m1x8_kperm_folded(uint32_t v, uint32_t f2, uint32_t (&p)[4]) {
  e2m1x8_kperm_raw(v, p);
#pragma unroll
  for (int i = 0; i < 4; ++i) p[i] = bf16x2_mul(p[i], f2);
}

// ---- E4M3 -------------------------------------------------------------------
// w holds bytes k0..k3: p02 = (k0, k2), p13 = (k1, k3), exact values
QG_DEVICE void e4m3x4_kperm(uint32_t w, uint32_t& p02, uint32_t& p13) {
  const uint32_t SGN = 0x80008000u, EM = 0x07F007F0u;
  p13 = lop3<kLutAndOr>(w, SGN, (w >> 4) & EM);
  const uint32_t w8 = w << 8;
  p02 = lop3<kLutAndOr>(w8, SGN, (w8 >> 4) & EM);
  p13 = bf16x2_mul(p13, kBf16x2_2p120);
  p02 = bf16x2_mul(p02, kBf16x2_2p120);
}

// ---- scales -> bf16x2 ----------------------------------------------------------
QG_DEVICE uint32_t bf16x2_splat(uint32_t b) { return (b & 0xFFFFu) * 0x00010001u; }

// E8M0 code c -> bf16 2^(c-127) (c = 0 is the subnormal 2^-127; 255 is NaN)
QG_DEVICE uint32_t e8m0_to_bf16x2(uint32_t c) {
  const uint32_t b = c == 0 ? 0x0040u : (c == 255 ? 0x7FC0u : (c << 7));
  return bf16x2_splat(b);
}

// E4M3 code -> bf16 (exact)
QG_DEVICE uint32_t e4m3_to_bf16x2(uint32_t c) {
  return bf16x2_splat(__float_as_uint(e4m3_to_f32(c & 0xFFu)) >> 16);
}

// FP4 block scales folded into the E2M1 decode, so that each weight pair
// costs one bf16 multiply instead of two (the E2M1 bit pattern is the value
// times 2^-126):
//  * MXFP4: f = 2^126 * 2^(c-127) = 2^(c-1), a normal bf16 for codes c <= 128
//    (blocks with magnitudes below 12 -- every code a weight block of unit
//    order gets); a warp whose rows hold a larger code takes the two-multiply
//    decode for that slab or segment.  Exact either way.
//  * NVFP4: f = 2^126 * e4m3(sb) * 2^-9 (at most 448 * 2^117 < 2^126), the
//    weight comes out times 2^-9 exactly (never below 2^-19, so normal) and
//    the epilogue multiplies the row by 2^9 with the global scale.
constexpr float kNvfp4Unfold = 512.f;
QG_DEVICE uint32_t mxfp4_fold(uint32_t c) { return c <= 128u ? bf16x2_splat((c + 126u) << 7) : 0u; }
QG_DEVICE uint32_t nvfp4_fold_x2(uint32_t two_codes) {     // (lo code, hi code) -> bf16x2 folded factors
  const uint32_t h = e4m3x2_to_f16x2(two_codes);         // exact
  float lo, hi;
  asm("{\n .reg .b16 a, b;\n mov.b32 {a, b}, %2;\n cvt.f32.f16 %0, a;\n cvt.f32.f16 %1, b;\n}"
      : "=f"(lo), "=f"(hi) : "r"(h));
  const float k = 1.6615349947311448e35f;                 // 2^117
  uint32_t d;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(hi * k), "f"(lo * k));   // exact products
  return d;
}

// ---- natural order ---------------------------------------------------------
// (k0,k1),(k2,k3),(k4,k5),(k6,k7) from the (k_i, k_{i+4}) pairs
QG_DEVICE void kperm4_to_natural(const uint32_t (&p)[4], uint32_t (&o)[4]) {
  o[0] = prmt(p[0], p[1], 0x5410u);
  o[1] = prmt(p[2], p[3], 0x5410u);
  o[2] = prmt(p[0], p[1], 0x7632u);
  o[3] = prmt(p[2], p[3], 0x7632u);
}

}  // namespace qg
