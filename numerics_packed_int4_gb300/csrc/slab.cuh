// One weight row's 64-k slab, as the tensor-core kernels consume it: the
// packed codes arrive in shared memory (TMA), the thread that owns the row
// fetches the slab's scales from global memory and decodes the 64 weights
// into 32 bf16 pairs in natural k order, ready for tcgen05.st into the A
// operand's tensor-memory slot.
//
// Formats (the canonical dequantized weight of each is in dequant.cuh):
//   SF_INT4   INT4, one bf16 scale per group of g (g a power of two >= 32)
//   SF_INT4Z  the same with an unsigned nibble and a zero point per group
//   SF_FP8    E4M3, the per-channel fp32 scale applied in the epilogue
//   SF_MXFP4  E2M1 with an E8M0 scale per 32 k
//   SF_NVFP4  E2M1 with an E4M3 scale per 16 k, the fp32 global scale
//             applied in the epilogue
#pragma once

#include "dequant.cuh"

namespace qg {

enum SlabFmt { SF_INT4 = 0, SF_INT4Z = 1, SF_FP8 = 2, SF_MXFP4 = 3, SF_NVFP4 = 4 };

constexpr int kSlabK = 64;             // k per slab (one 128-byte swizzle row of bf16)

template <int WF> struct SlabTraits {
  static constexpr int WROW = WF == SF_FP8 ? kSlabK : kSlabK / 2;   // packed bytes per row per slab
  static constexpr bool EPI_SCALE = WF == SF_FP8 || WF == SF_NVFP4;  // scale applied to the accumulated row
};

// Scale and zero-point rows of output channel n.
template <int WF>
QG_DEVICE void slab_rows(const void* ws, const uint8_t* wz, int K, int lg, size_t n, const uint8_t*& srow,
                         const uint8_t*& zrow) {
  const uint8_t* wsb = static_cast<const uint8_t*>(ws);
  if constexpr (WF == SF_INT4 || WF == SF_INT4Z) {
    const size_t r = n * (size_t)(K >> lg);
    srow = wsb + 2 * r;
    if constexpr (WF == SF_INT4Z) zrow = wz + r;
  } else if constexpr (WF == SF_MXFP4) {
    srow = wsb + n * (size_t)(K / 32);
  } else if constexpr (WF == SF_NVFP4) {
    srow = wsb + n * (size_t)(K / 16);
  }
}

// The scales of slab s of a row.  INT4: the bf16 scales of the slab's two
// 32-k halves in v0 and v1 (bits 0-15), their zero points in bits 16-19 with
// SF_INT4Z; one load when both halves lie in one group (g >= 64).  FP4: the
// slab's block-scale codes in v0 (MXFP4: two, NVFP4: four, lowest k first).
template <int WF>
QG_DEVICE void slab_scales(const uint8_t* srow, const uint8_t* zrow, int s, int lg, uint32_t& v0, uint32_t& v1) {
  v0 = v1 = 0u;
  if constexpr (WF == SF_INT4 || WF == SF_INT4Z) {
    const uint16_t* sr = reinterpret_cast<const uint16_t*>(srow);
    const int g0 = (s * kSlabK) >> lg, g1 = (s * kSlabK + 32) >> lg;
    v0 = __ldg(sr + g0);
    if constexpr (WF == SF_INT4Z) v0 |= (uint32_t)__ldg(zrow + g0) << 16;
    if (g1 == g0) {
      v1 = v0;
    } else {
      v1 = __ldg(sr + g1);
      if constexpr (WF == SF_INT4Z) v1 |= (uint32_t)__ldg(zrow + g1) << 16;
    }
  } else if constexpr (WF == SF_MXFP4) {
    v0 = __ldg(reinterpret_cast<const uint16_t*>(srow) + s);
  } else if constexpr (WF == SF_NVFP4) {
    v0 = __ldg(reinterpret_cast<const uint32_t*>(srow) + s);
  }
}

// The packed words of one row's slab: 8 words of 8 nibbles (4-bit formats) or
// 16 words of 4 E4M3 codes, lowest k first.
template <int WF> struct SlabWords {
  uint32_t w[WF == SF_FP8 ? 16 : 8];
};

// Slab words from a stage whose rows hold exactly one slab: 4-bit rows of 32
// bytes stored plainly, FP8 rows of 64 bytes in the 64-byte swizzle (16-byte
// chunk c of row r at c ^ ((r >> 1) & 3)).
template <int WF>
QG_DEVICE void load_slab_words(const uint8_t* wrow, int row, SlabWords<WF>& sw) {
  if constexpr (WF == SF_FP8) {
    const int x = (row >> 1) & 3;
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      const uint4 w4 = *reinterpret_cast<const uint4*>(wrow + 16 * (c ^ x));
      sw.w[4 * c] = w4.x; sw.w[4 * c + 1] = w4.y; sw.w[4 * c + 2] = w4.z; sw.w[4 * c + 3] = w4.w;
    }
  } else {
#pragma unroll
    for (int c = 0; c < 2; ++c) {
      const uint4 w4 = *reinterpret_cast<const uint4*>(wrow + 16 * c);
      sw.w[4 * c] = w4.x; sw.w[4 * c + 1] = w4.y; sw.w[4 * c + 2] = w4.z; sw.w[4 * c + 3] = w4.w;
    }
  }
}

// Decode a slab's words: out[i] = (k_2i, k_2i+1) in bf16.  The FP4 block
// scales are folded into the E2M1 decode (dequant.cuh): NVFP4 weights come out
// times 2^-9 exactly (the caller multiplies the accumulated row by
// kNvfp4Unfold), MXFP4 weights exactly, with one multiply per pair when every
// row of the warp has block codes <= 128.  Warp-collective for MXFP4.
template <int WF>
QG_DEVICE void decode_slab_words(const SlabWords<WF>& sw, uint32_t v0, uint32_t v1, uint32_t (&out)[32]) {
  if constexpr (WF == SF_FP8) {
#pragma unroll
    for (int i = 0; i < 16; ++i) {               // bytes k0..k3 -> (k0, k1), (k2, k3), exact
      uint32_t p02, p13;
      e4m3x4_kperm(sw.w[i], p02, p13);
      out[2 * i] = prmt(p02, p13, 0x5410u);
      out[2 * i + 1] = prmt(p02, p13, 0x7632u);
    }
  } else if constexpr (WF == SF_INT4 || WF == SF_INT4Z) {
    const uint32_t s2a = bf16x2_splat(v0), s2b = bf16x2_splat(v1);
    const uint32_t z2a = bf16x2_zero128(v0 >> 16), z2b = bf16x2_zero128(v1 >> 16);
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      uint32_t nat[4];
      if constexpr (WF == SF_INT4Z)
        int4zp_x8_nat(sw.w[j], j < 4 ? s2a : s2b, j < 4 ? z2a : z2b, nat);
      else
        int4x8_nat(sw.w[j], j < 4 ? s2a : s2b, nat);
      out[4 * j + 0] = nat[0]; out[4 * j + 1] = nat[1];
      out[4 * j + 2] = nat[2]; out[4 * j + 3] = nat[3];
    }
  } else {
    // words of 8 E2M1 codes; block scale: MXFP4 per 32 k (words j / 4), NVFP4 per 16 (j / 2)
    auto put = [&](int j, const uint32_t (&pq)[4]) {
      uint32_t nat[4];
      kperm4_to_natural(pq, nat);
      out[4 * j + 0] = nat[0]; out[4 * j + 1] = nat[1];
      out[4 * j + 2] = nat[2]; out[4 * j + 3] = nat[3];
    };
    if constexpr (WF == SF_NVFP4) {
      const uint32_t f01 = nvfp4_fold_x2(v0 & 0xFFFFu), f23 = nvfp4_fold_x2(v0 >> 16);
      const uint32_t f[4] = {prmt(f01, f01, 0x1010u), prmt(f01, f01, 0x3232u),
                             prmt(f23, f23, 0x1010u), prmt(f23, f23, 0x3232u)};
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        uint32_t pq[4];
        e2m1x8_kperm_folded(sw.w[j], f[j >> 1], pq);
        put(j, pq);
      }
    } else {
      const uint32_t c0 = v0 & 0xFFu, c1 = (v0 >> 8) & 0xFFu;
      if (__all_sync(0xffffffffu, c0 <= 128u && c1 <= 128u)) {
        const uint32_t f0 = mxfp4_fold(c0), f1 = mxfp4_fold(c1);
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          uint32_t pq[4];
          e2m1x8_kperm_folded(sw.w[j], j < 4 ? f0 : f1, pq);
          put(j, pq);
        }
      } else {
        const uint32_t s0 = e8m0_to_bf16x2(c0), s1 = e8m0_to_bf16x2(c1);
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          uint32_t pq[4];
          e2m1x8_kperm(sw.w[j], j < 4 ? s0 : s1, pq);
          put(j, pq);
        }
      }
    }
  }
}

// Decode the row's slab from a one-slab-per-row stage (load_slab_words layout).
template <int WF>
QG_DEVICE void decode_slab(const uint8_t* wrow, int row, uint32_t v0, uint32_t v1, uint32_t (&out)[32]) {
  SlabWords<WF> sw;
  load_slab_words<WF>(wrow, row, sw);
  decode_slab_words<WF>(sw, v0, v1, out);
}

}  // namespace qg
