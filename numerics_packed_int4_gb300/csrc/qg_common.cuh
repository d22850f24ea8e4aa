// Shared device/host helpers for the sm_103a kernels behind include/qgemm.h.
//
// Numerics contract (no fast-math, no flush-to-zero; the build passes
// -ftz=false -prec-div=true -prec-sqrt=true):
//   * bf16 inputs widen to fp32 exactly;
//   * every narrowing to E4M3 / E2M1 uses the hardware cvt.rn.satfinite
//     conversions (one round-to-nearest-even from fp32, saturating), the cast
//     FreeToken PR #805 asks for;
//   * every fp32 division that decides a code is IEEE correctly rounded.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

#include "qgemm.h"

#define QG_HOST_DEVICE __host__ __device__ __forceinline__
#define QG_DEVICE __device__ __forceinline__

namespace qg {

// ---------------------------------------------------------------------------
// host-side status plumbing (abi.cu)
// ---------------------------------------------------------------------------
qg_status set_error(qg_status st, const char* fmt, ...);
qg_status check_launch(const char* what);
unsigned int* device_error_word();      // per-device error word (nullptr on failure)
int sm_count();                         // SMs of the current device
uint32_t wait_limit();                  // iteration cap for device-side spin waits

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Raise a kernel's dynamic shared memory limit once per (kernel, device), so
// that later launches -- including ones inside CUDA-graph capture -- issue no
// attribute calls.
bool ensure_smem_attr(const void* kernel, int bytes);
template <typename K>
inline bool ensure_smem(K kernel, int bytes) {
  return ensure_smem_attr(reinterpret_cast<const void*>(kernel), bytes);
}

// device error codes written into the error word
enum : unsigned int { DEV_ERR_NONE = 0, DEV_ERR_TIMEOUT = 1 };

// ---------------------------------------------------------------------------
// small device helpers
// ---------------------------------------------------------------------------
QG_DEVICE float bf16_lo_to_f32(uint32_t v) { return __uint_as_float(v << 16); }
QG_DEVICE float bf16_hi_to_f32(uint32_t v) { return __uint_as_float(v & 0xFFFF0000u); }
QG_DEVICE float bf16_bits_to_f32(uint16_t v) { return __uint_as_float(uint32_t(v) << 16); }

// fp32 -> bf16 bits, round to nearest even (hardware cvt)
QG_DEVICE uint16_t f32_to_bf16_bits(float f) {
  uint16_t r;
  asm("cvt.rn.bf16.f32 %0, %1;" : "=h"(r) : "f"(f));
  return r;
}

// two fp32 -> packed E4M3x2, RNE, satfinite.  'hi' lands in bits 15..8.
QG_DEVICE uint16_t f32x2_to_e4m3x2(float hi, float lo) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

// two fp32 -> packed E2M1x2 in one byte, RNE, satfinite.  'hi' lands in bits 7..4.
QG_DEVICE uint32_t f32x2_to_e2m1x2(float hi, float lo) {
  uint32_t r;
  asm("{ .reg .b8 t; cvt.rn.satfinite.e2m1x2.f32 t, %1, %2; cvt.u32.u8 %0, t; }"
      : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

// E4M3 code -> exact fp32 value (finite codes; 0x7F/0xFF give NaN)
// FP8 E4M3 block scale: absmax / 448 in IEEE fp32 (an all-zero block gets 1)
QG_DEVICE float fp8_scale(float amax) { return amax == 0.f ? 1.f : __fdiv_rn(amax, 448.f); }

QG_DEVICE float e4m3_to_f32(uint32_t c) {
  const uint32_t s = (c & 0x80u) << 24, E = (c >> 3) & 0xFu, Mn = c & 7u;
  if ((c & 0x7Fu) == 0x7Fu) return __uint_as_float(0x7FC00000u);
  if (E == 0) {                                   // subnormal: M * 2^-9 (signed zero kept)
    const float v = float(Mn) * 0.001953125f;
    return s ? -v : v;
  }
  return __uint_as_float(s | ((E + 120u) << 23) | (Mn << 20));
}

// 2^(127 - se) as an fp32 (se in [0, 253] gives a normal number)
QG_DEVICE float pow2_127_minus(uint32_t se) { return __uint_as_float((254u - se) << 23); }

// packed bf16x2 arithmetic (one IEEE rounding per lane, no flush)
QG_DEVICE uint32_t bf16x2_sub(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("sub.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}
QG_DEVICE uint32_t bf16x2_mul(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}
QG_DEVICE uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t d;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
  return d;
}
template <int IMM>
QG_DEVICE uint32_t lop3(uint32_t a, uint32_t b, uint32_t c) {
  uint32_t d;
  asm("lop3.b32 %0, %1, %2, %3, %4;" : "=r"(d) : "r"(a), "r"(b), "r"(c), "n"(IMM));
  return d;
}

// warp-level max over groups of G consecutive lanes (G power of two <= 32)
template <int G>
QG_DEVICE float group_max(float v) {
#pragma unroll
  for (int o = G / 2; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// streaming 16-byte global load that does not allocate in L1
QG_DEVICE uint4 ldg_stream(const void* p) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w) : "l"(p));
  return r;
}

}  // namespace qg
