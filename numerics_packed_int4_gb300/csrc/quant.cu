// Online activation quantizers, load-time weight quantizers and the MoE
// harness kernels.  All of them are HBM-streaming: each thread owns 8
// consecutive elements (one 16-byte bf16 load or two 16-byte fp32 loads), the
// quantization block is reduced with warp shuffles (blocks of <= 256) or a
// CTA reduction (larger blocks, e.g. per-token), and codes leave as one
// 4- or 8-byte store per thread.
#include <cfloat>

#include "dequant.cuh"

#define QG_REQUIRE(cond, st, ...) \
  do { if (!(cond)) return qg::set_error(st, __VA_ARGS__); } while (0)

namespace qg {
namespace {

constexpr int kThreads = 256;

// ---- loading 8 consecutive elements as fp32 --------------------------------
template <typename T> struct Load8;
template <> struct Load8<uint16_t> {          // bf16 bit patterns
  static QG_DEVICE void run(const uint16_t* p, float (&v)[8]) {
    const uint4 u = *reinterpret_cast<const uint4*>(p);
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) { v[2 * i] = bf16_lo_to_f32(w[i]); v[2 * i + 1] = bf16_hi_to_f32(w[i]); }
  }
};
template <> struct Load8<float> {
  static QG_DEVICE void run(const float* p, float (&v)[8]) {
    const float4 a = *reinterpret_cast<const float4*>(p);
    const float4 b = *reinterpret_cast<const float4*>(p + 4);
    v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w; v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
  }
};

QG_DEVICE float absmax8(const float (&v)[8]) {
  float m = 0.f;
#pragma unroll
  for (int i = 0; i < 8; ++i) m = fmaxf(m, fabsf(v[i]));
  return m;
}

// ---- E4M3 block step: s = amax/448 (zero -> 1), codes of x/s ---------------

QG_DEVICE uint2 fp8_codes8(const float (&v)[8], float s) {
  uint32_t c[4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
    c[i] = f32x2_to_e4m3x2(__fdiv_rn(v[2 * i + 1], s), __fdiv_rn(v[2 * i], s));
  return make_uint2(c[0] | (c[1] << 16), c[2] | (c[3] << 16));
}
// ---- MXFP4 block step -----------------------------------------------------------
// Exponent-first 0.75-threshold rule (vLLM PR #43557, "Fix"): take vecMax's
// exponent field, step it up by one when the significand is at least 1.75
// (its two leading fraction bits both set), then subtract E2M1's top binade
// (2) and clamp at 0.  vecMax >= 0 here (a maximum of magnitudes).
QG_DEVICE uint32_t e8m0_scale_exp(float vecMax) {
  const uint32_t u = __float_as_uint(vecMax);
  const uint32_t e = ((u >> 23) & 0xFFu) + (((u >> 21) & 3u) == 3u ? 1u : 0u);
  return e > 2u ? e - 2u : 0u;
}

QG_DEVICE uint32_t e2m1_codes8(const float (&v)[8], float mul) {
  uint32_t r = 0;
#pragma unroll
  for (int i = 0; i < 4; ++i)
    r |= f32x2_to_e2m1x2(__fmul_rn(v[2 * i + 1], mul), __fmul_rn(v[2 * i], mul)) << (8 * i);
  return r;
}

// ===========================================================================
// block size <= 256: GT = g/8 lanes per block, shuffles only
// ===========================================================================
// g <= 256: GT = g/8 consecutive lanes per block.  A CTA takes CPT slices of
// kThreads consecutive chunks; every thread loads its CPT chunks before any
// is quantized, so each thread keeps CPT 16-byte loads in flight (with one
// chunk per thread the divisions held the threads and too few bytes were in
// flight to cover the memory latency).
template <typename Tin, int GT, int CPT>
__global__ void __launch_bounds__(kThreads) fp8_block_small_kernel(
    const Tin* __restrict__ x, uint8_t* __restrict__ q, float* __restrict__ s,
    long long nchunks, int K) {
  float v[CPT][8];
#pragma unroll
  for (int j = 0; j < CPT; ++j) {
    const long long c = ((long long)blockIdx.x * CPT + j) * kThreads + threadIdx.x;
#pragma unroll
    for (int i = 0; i < 8; ++i) v[j][i] = 0.f;
    if (c < nchunks) Load8<Tin>::run(x + c * 8, v[j]);
  }
#pragma unroll
  for (int j = 0; j < CPT; ++j) {
    const long long c = ((long long)blockIdx.x * CPT + j) * kThreads + threadIdx.x;
    const float amax = group_max<GT>(absmax8(v[j]));
    const float sc = fp8_scale(amax);
    if (c < nchunks) {
      *reinterpret_cast<uint2*>(q + c * 8) = fp8_codes8(v[j], sc);
      if ((c % GT) == 0) s[c / GT] = sc;
    }
  }
}

template <typename Tin, int GT, int CPT>
__global__ void __launch_bounds__(kThreads) mxfp4_kernel(
    const Tin* __restrict__ x, uint8_t* __restrict__ q, uint8_t* __restrict__ se_out,
    long long nchunks) {
  float v[CPT][8];
#pragma unroll
  for (int j = 0; j < CPT; ++j) {          // every load in flight before any block is quantized
    const long long c = ((long long)blockIdx.x * CPT + j) * kThreads + threadIdx.x;
#pragma unroll
    for (int i = 0; i < 8; ++i) v[j][i] = 0.f;
    if (c < nchunks) Load8<Tin>::run(x + c * 8, v[j]);
  }
#pragma unroll
  for (int j = 0; j < CPT; ++j) {
    const long long c = ((long long)blockIdx.x * CPT + j) * kThreads + threadIdx.x;
    const float vecMax = group_max<GT>(absmax8(v[j]));
    const uint32_t se = e8m0_scale_exp(vecMax);
    if (c < nchunks) {
      *reinterpret_cast<uint32_t*>(q + c * 4) = e2m1_codes8(v[j], pow2_127_minus(se));
      if ((c % GT) == 0) se_out[c / GT] = uint8_t(se);
    }
  }
}

template <int GT>
__global__ void __launch_bounds__(kThreads) int4_rtn_kernel(
    const float* __restrict__ w, uint8_t* __restrict__ q, uint16_t* __restrict__ s,
    long long nchunks) {
  const long long c = blockIdx.x * (long long)kThreads + threadIdx.x;
  const bool live = c < nchunks;
  float v[8] = {0, 0, 0, 0, 0, 0, 0, 0};
  if (live) Load8<float>::run(w + c * 8, v);
  const float amax = group_max<GT>(absmax8(v));
  if (!live) return;
  uint16_t sb = f32_to_bf16_bits(__fdiv_rn(amax, 7.f));
  float sf = bf16_bits_to_f32(sb);
  uint32_t packed = 0;
  if (sf == 0.f) {
    sb = 0x3F80;                       // all-zero group policy: s = 1, q = 0
  } else {
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      float t = rintf(__fdiv_rn(v[i], sf));
      t = fminf(fmaxf(t, -8.f), 7.f);
      packed |= (uint32_t(int(t)) & 0xFu) << (4 * i);
    }
  }
  *reinterpret_cast<uint32_t*>(q + c * 4) = packed;
  if ((c % GT) == 0) s[c / GT] = sb;
}

// Asymmetric INT4 with a zero point per group ("Numerics": x = s (q - z)):
// lo / hi = min / max of the group, s = bf16_RNE((hi - lo) / 15) (fp32
// subtraction and division; a flat group, or one whose scale rounds to zero,
// gets s = 1), z = clamp(rint(-lo / s), 0, 15), q = clamp(rint(w / s) + z,
// 0, 15), unsigned nibbles.
template <int GT>
__global__ void __launch_bounds__(kThreads) int4_zp_kernel(
    const float* __restrict__ w, uint8_t* __restrict__ q, uint16_t* __restrict__ s, uint8_t* __restrict__ z,
    long long nchunks) {
  const long long c = blockIdx.x * (long long)kThreads + threadIdx.x;
  const bool live = c < nchunks;
  float v[8] = {0, 0, 0, 0, 0, 0, 0, 0};
  if (live) Load8<float>::run(w + c * 8, v);
  float mx = v[0], mn = v[0];
#pragma unroll
  for (int i = 1; i < 8; ++i) { mx = fmaxf(mx, v[i]); mn = fminf(mn, v[i]); }
  const float hi = group_max<GT>(mx);
  const float lo = -group_max<GT>(-mn);
  if (!live) return;
  uint16_t sb = f32_to_bf16_bits(__fdiv_rn(__fsub_rn(hi, lo), 15.f));
  float sf = bf16_bits_to_f32(sb);
  if (sf == 0.f) { sb = 0x3F80; sf = 1.f; }     // flat or all-zero group: s = 1
  const float zf = fminf(fmaxf(rintf(__fdiv_rn(-lo, sf)), 0.f), 15.f);
  uint32_t packed = 0;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const float t = fminf(fmaxf(rintf(__fdiv_rn(v[i], sf)) + zf, 0.f), 15.f);
    packed |= (uint32_t(int(t)) & 0xFu) << (4 * i);
  }
  *reinterpret_cast<uint32_t*>(q + c * 4) = packed;
  if ((c % GT) == 0) {
    s[c / GT] = sb;
    z[c / GT] = (uint8_t)int(zf);
  }
}

// ===========================================================================
// large blocks (g > 256, e.g. per-token / per-channel): one CTA per block
// ===========================================================================
QG_DEVICE float cta_max(float v, float* red) {
  v = group_max<32>(v);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if (lane == 0) red[warp] = v;
  __syncthreads();
  if (warp == 0) {
    v = lane < kThreads / 32 ? red[lane] : 0.f;
    v = group_max<32>(v);
    if (lane == 0) red[0] = v;
  }
  __syncthreads();
  const float r = red[0];
  __syncthreads();
  return r;
}

template <typename Tin>
__global__ void __launch_bounds__(kThreads) fp8_block_large_kernel(
    const Tin* __restrict__ x, uint8_t* __restrict__ q, float* __restrict__ s, int g) {
  __shared__ float red[kThreads / 32];
  const long long base = (long long)blockIdx.x * g;
  float m = 0.f;
  for (int c = threadIdx.x; c < g / 8; c += kThreads) {
    float v[8];
    Load8<Tin>::run(x + base + c * 8, v);
    m = fmaxf(m, absmax8(v));
  }
  const float sc = fp8_scale(cta_max(m, red));
  for (int c = threadIdx.x; c < g / 8; c += kThreads) {
    float v[8];
    Load8<Tin>::run(x + base + c * 8, v);
    *reinterpret_cast<uint2*>(q + base + c * 8) = fp8_codes8(v, sc);
  }
  if (threadIdx.x == 0) s[blockIdx.x] = sc;
}

// One block per CTA with the block's values kept in registers (CPT chunks of
// 8 per thread): one read of the input instead of two.
template <typename Tin, int CPT>
__global__ void __launch_bounds__(kThreads) fp8_block_reg_kernel(
    const Tin* __restrict__ x, uint8_t* __restrict__ q, float* __restrict__ s, int g) {
  __shared__ float red[kThreads / 32];
  const long long base = (long long)blockIdx.x * g;
  const int nc = g / 8;
  float v[CPT][8];
  float m = 0.f;
#pragma unroll
  for (int j = 0; j < CPT; ++j) {
    const int c = threadIdx.x + j * kThreads;
    if (c < nc) {
      Load8<Tin>::run(x + base + c * 8, v[j]);
      m = fmaxf(m, absmax8(v[j]));
    }
  }
  const float sc = fp8_scale(cta_max(m, red));
#pragma unroll
  for (int j = 0; j < CPT; ++j) {
    const int c = threadIdx.x + j * kThreads;
    if (c < nc) *reinterpret_cast<uint2*>(q + base + c * 8) = fp8_codes8(v[j], sc);
  }
  if (threadIdx.x == 0) s[blockIdx.x] = sc;
}

// ===========================================================================
// NVFP4 weights
// ===========================================================================
__global__ void __launch_bounds__(kThreads) amax_kernel(const float* __restrict__ w, long long nchunks,
                                                        unsigned int* __restrict__ out) {
  __shared__ float red[kThreads / 32];
  float m = 0.f;
  for (long long c = blockIdx.x * (long long)kThreads + threadIdx.x; c < nchunks;
       c += (long long)gridDim.x * kThreads) {
    float v[8];
    Load8<float>::run(w + c * 8, v);
    m = fmaxf(m, absmax8(v));
  }
  m = cta_max(m, red);
  if (threadIdx.x == 0) atomicMax(out, __float_as_uint(m));   // m >= 0: bits are ordered
}

QG_DEVICE float nvfp4_global_scale(float amax) { return amax == 0.f ? 1.f : __fdiv_rn(amax, 2688.f); }

__global__ void __launch_bounds__(kThreads) nvfp4_kernel(
    const float* __restrict__ w, uint8_t* __restrict__ q, uint8_t* __restrict__ sb_out,
    const float* __restrict__ amax_word, long long nchunks) {
  const long long c = blockIdx.x * (long long)kThreads + threadIdx.x;
  const bool live = c < nchunks;
  float v[8] = {0, 0, 0, 0, 0, 0, 0, 0};
  if (live) Load8<float>::run(w + c * 8, v);
  const float amax_b = group_max<2>(absmax8(v));
  if (!live) return;
  const float gs = nvfp4_global_scale(*amax_word);
  const float d = __fmul_rn(6.f, gs);
  const uint32_t sb = f32x2_to_e4m3x2(0.f, __fdiv_rn(amax_b, d)) & 0xFFu;
  const float den = __fmul_rn(e4m3_to_f32(sb), gs);
  uint32_t packed = 0;
  if (den != 0.f) {
    float t[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) t[i] = __fdiv_rn(v[i], den);
    packed = e2m1_codes8(t, 1.f);
  }
  *reinterpret_cast<uint32_t*>(q + c * 4) = packed;
  if ((c & 1) == 0) sb_out[c / 2] = uint8_t(sb);
}

__global__ void nvfp4_finalize_kernel(float* gs_word) {
  gs_word[0] = nvfp4_global_scale(gs_word[0]);
}

// ===========================================================================
// MoE harness
// ===========================================================================
// 8 E4M3 codes -> their 8 fp16 values (exact)
QG_DEVICE uint4 e4m3x8_to_f16x8(uint2 c) {
  return make_uint4(e4m3x2_to_f16x2(c.x & 0xFFFFu), e4m3x2_to_f16x2(c.x >> 16),
                    e4m3x2_to_f16x2(c.y & 0xFFFFu), e4m3x2_to_f16x2(c.y >> 16));
}

// Row gather of E4M3 codes and their row scales; F16: the destination takes
// the codes' fp16 values instead of the codes.
template <bool F16>
__global__ void __launch_bounds__(kThreads) gather_fp8_kernel(
    const uint8_t* __restrict__ src_q, const float* __restrict__ src_s,
    const int32_t* __restrict__ rows, void* __restrict__ dst_v, float* __restrict__ dst_s,
    int T, int K) {
  const int r = blockIdx.x;
  int t = rows[r];
  t = t < 0 ? 0 : (t >= T ? T - 1 : t);
  const uint4* src = reinterpret_cast<const uint4*>(src_q + (long long)t * K);
  if constexpr (F16) {
    uint4* dst = reinterpret_cast<uint4*>(static_cast<uint16_t*>(dst_v) + (long long)r * K);
    for (int i = threadIdx.x; i < K / 16; i += kThreads) {
      const uint4 c = src[i];
      dst[2 * i] = e4m3x8_to_f16x8(make_uint2(c.x, c.y));
      dst[2 * i + 1] = e4m3x8_to_f16x8(make_uint2(c.z, c.w));
    }
  } else {
    uint4* dst = reinterpret_cast<uint4*>(static_cast<uint8_t*>(dst_v) + (long long)r * K);
    for (int i = threadIdx.x; i < K / 16; i += kThreads) dst[i] = src[i];
  }
  if (threadIdx.x == 0) dst_s[r] = src_s[t];
}

// store of 8 codes, or (F16) of their fp16 values, at element offset o of a row
template <bool F16>
QG_DEVICE void store_codes8(void* q, long long o, uint2 codes) {
  if constexpr (F16) *reinterpret_cast<uint4*>(static_cast<uint16_t*>(q) + o) = e4m3x8_to_f16x8(codes);
  else *reinterpret_cast<uint2*>(static_cast<uint8_t*>(q) + o) = codes;
}

// h = SiLU(g) * u = (g * u) / (1 + e^-g) in fp32.  g and u are bf16, so
// p = g * u (16 significant bits) is exact.  The exponential is CUDA's accurate
// expf (not the fast intrinsic).  d = 1 + e is kept as an unevaluated sum
// d + dl (Knuth's TwoSum), and the quotient p / (d + dl) is formed from an
// approximate reciprocal with one correction from the exact remainder p - q*d
// (an FMA) -- the classic Newton/Markstein step -- so h is p / (d + dl) to
// about half an ulp: the only error left beyond one rounding is expf's, scaled
// by e / (1 + e) -- negligible where g is large and positive, which is where
// a row's largest |h| (and so its scale) usually comes from.  A code can
// still differ from the correctly rounded h's code where h / s lies within a
// few ulps of an E4M3 rounding boundary.  g -> -inf gives d = inf and h = +-0
// (the correction is skipped there); g -> +inf gives p / 1.
QG_DEVICE float rcp_approx(float x) {
  float r;
  asm("rcp.approx.f32 %0, %1;" : "=f"(r) : "f"(x));
  return r;
}
QG_DEVICE float silu_mul(float g, float u) {
  const float p = __fmul_rn(g, u);
  const float e = expf(-g);
  const float d = __fadd_rn(1.f, e);
  const float rc = rcp_approx(d);
  const float q = __fmul_rn(p, rc);
  if (isinf(d)) return q;                 // +-0
  const float bv = __fsub_rn(d, 1.f);
  const float dl = __fadd_rn(__fsub_rn(1.f, __fsub_rn(d, bv)), __fsub_rn(e, bv));   // (1 + e) - d, exact
  float r = __fmaf_rn(-q, d, p);          // p - q*d, exact
  r = __fmaf_rn(-q, dl, r);               // minus q*dl
  return __fmaf_rn(r, rc, q);
}

QG_DEVICE void swiglu8(const uint16_t* gu, int I, int c, float (&h)[8]) {
  float gv[8], uv[8];
  Load8<uint16_t>::run(gu + c * 8, gv);
  Load8<uint16_t>::run(gu + I + c * 8, uv);
#pragma unroll
  for (int i = 0; i < 8; ++i) h[i] = silu_mul(gv[i], uv[i]);
}

// One row per CTA with the row's SwiGLU values kept in registers: one read of
// gate/up, the per-row absmax, then the E4M3 codes (CPT chunks of 8 per thread,
// NT threads).
template <int NT>
QG_DEVICE float cta_max_nt(float v, float* red) {
  v = group_max<32>(v);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if (lane == 0) red[warp] = v;
  __syncthreads();
  if (warp == 0) {
    v = lane < NT / 32 ? red[lane] : 0.f;
    v = group_max<32>(v);
    if (lane == 0) red[0] = v;
  }
  __syncthreads();
  return red[0];
}

template <int CPT, int NT, bool F16>
__global__ void __launch_bounds__(NT) swiglu_quant_reg_kernel(
    const uint16_t* __restrict__ gate_up, void* __restrict__ q, float* __restrict__ s, int I) {
  __shared__ float red[NT / 32];
  const uint16_t* gu = gate_up + (long long)blockIdx.x * 2 * I;
  const int nc = I / 8;
  float h[CPT][8];
  float m = 0.f;
#pragma unroll
  for (int j = 0; j < CPT; ++j) {
    const int c = threadIdx.x + j * NT;
    if (c < nc) {
      swiglu8(gu, I, c, h[j]);
      m = fmaxf(m, absmax8(h[j]));
    }
  }
  const float sc = fp8_scale(cta_max_nt<NT>(m, red));
#pragma unroll
  for (int j = 0; j < CPT; ++j) {
    const int c = threadIdx.x + j * NT;
    if (c < nc) store_codes8<F16>(q, (long long)blockIdx.x * I + c * 8, fp8_codes8(h[j], sc));
  }
  if (threadIdx.x == 0) s[blockIdx.x] = sc;
}

template <bool F16>
__global__ void __launch_bounds__(kThreads) swiglu_quant_kernel(
    const uint16_t* __restrict__ gate_up, void* __restrict__ q, float* __restrict__ s, int I) {
  __shared__ float red[kThreads / 32];
  const uint16_t* gu = gate_up + (long long)blockIdx.x * 2 * I;
  float m = 0.f;
  for (int c = threadIdx.x; c < I / 8; c += kThreads) {
    float h[8];
    swiglu8(gu, I, c, h);
    m = fmaxf(m, absmax8(h));
  }
  const float sc = fp8_scale(cta_max(m, red));
  for (int c = threadIdx.x; c < I / 8; c += kThreads) {
    float h[8];
    swiglu8(gu, I, c, h);
    store_codes8<F16>(q, (long long)blockIdx.x * I + c * 8, fp8_codes8(h, sc));
  }
  if (threadIdx.x == 0) s[blockIdx.x] = sc;
}

__global__ void __launch_bounds__(kThreads) combine_kernel(
    const uint16_t* __restrict__ down, const int32_t* __restrict__ row_of,
    const float* __restrict__ weight, uint16_t* __restrict__ out, int topk, int R, int H) {
  const int t = blockIdx.y;
  const int c = blockIdx.x * kThreads + threadIdx.x;
  if (c >= H / 8) return;
  float acc[8] = {0, 0, 0, 0, 0, 0, 0, 0};
  for (int j = 0; j < topk; ++j) {
    int r = row_of[t * topk + j];
    if (r < 0 || r >= R) continue;
    const float p = weight[t * topk + j];
    float d[8];
    Load8<uint16_t>::run(down + (long long)r * H + c * 8, d);
#pragma unroll
    for (int i = 0; i < 8; ++i) acc[i] = __fmaf_rn(p, d[i], acc[i]);
  }
  uint32_t o[4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
    o[i] = uint32_t(f32_to_bf16_bits(acc[2 * i])) | (uint32_t(f32_to_bf16_bits(acc[2 * i + 1])) << 16);
  *reinterpret_cast<uint4*>(out + (long long)t * H + c * 8) = make_uint4(o[0], o[1], o[2], o[3]);
}

// ---- FP8 group scales of the W4A8 FP8 x FP8 path (one warp per row) --------
// Production-Ready W4A8, "Accurate W4A8 Kernel": the per-token FP8 quantizer
// applied to each output channel's row of bf16 group scales, then the FP8
// scales times 1/8 and the channel scale times 8.
__global__ void __launch_bounds__(kThreads) w4a8_fp8_scales_kernel(
    const uint16_t* __restrict__ w_s, uint8_t* __restrict__ s8, float* __restrict__ cs8, int rows, int G) {
  const long long row = ((long long)blockIdx.x * kThreads + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (row >= rows) return;
  const uint16_t* src = w_s + row * G;
  float m = 0.f;
  for (int g = lane; g < G; g += 32) m = fmaxf(m, fabsf(bf16_bits_to_f32(src[g])));
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  const float cs = fp8_scale(m);
  for (int g = lane; g < G; g += 32) {
    const uint32_t code = f32x2_to_e4m3x2(0.f, __fdiv_rn(bf16_bits_to_f32(src[g]), cs)) & 0xFFu;
    const float eighth = e4m3_to_f32(code) * 0.125f;                 // exact in fp32
    s8[(long long)g * rows + row] = uint8_t(f32x2_to_e4m3x2(0.f, eighth) & 0xFFu);   // group-major
  }
  if (lane == 0) cs8[row] = cs * 8.f;
}

// ---- launch helpers ----------------------------------------------------------
inline unsigned grid_for(long long nchunks) { return unsigned((nchunks + kThreads - 1) / kThreads); }
constexpr int kFp8Cpt = 2;             // chunks per thread of the small-block FP8 quantizer
constexpr int kMxCpt = 2;              // and of the MXFP4 quantizer
inline unsigned grid_cpt(long long nchunks, int cpt) {
  return unsigned((nchunks + (long long)kThreads * cpt - 1) / ((long long)kThreads * cpt));
}

template <typename Tin>
qg_status launch_fp8_block(const Tin* x, uint8_t* q, float* s, int g, long long rows, int K,
                           cudaStream_t st, const char* name) {
  const long long nchunks = rows * (long long)K / 8;
  if (nchunks == 0) return QG_OK;
  const long long nblocks = rows * (long long)(K / g);
  switch (g) {
    case 8:   fp8_block_small_kernel<Tin, 1, kFp8Cpt><<<grid_cpt(nchunks, kFp8Cpt), kThreads, 0, st>>>(x, q, s, nchunks, K); break;
    case 16:  fp8_block_small_kernel<Tin, 2, kFp8Cpt><<<grid_cpt(nchunks, kFp8Cpt), kThreads, 0, st>>>(x, q, s, nchunks, K); break;
    case 32:  fp8_block_small_kernel<Tin, 4, kFp8Cpt><<<grid_cpt(nchunks, kFp8Cpt), kThreads, 0, st>>>(x, q, s, nchunks, K); break;
    case 64:  fp8_block_small_kernel<Tin, 8, kFp8Cpt><<<grid_cpt(nchunks, kFp8Cpt), kThreads, 0, st>>>(x, q, s, nchunks, K); break;
    case 128: fp8_block_small_kernel<Tin, 16, kFp8Cpt><<<grid_cpt(nchunks, kFp8Cpt), kThreads, 0, st>>>(x, q, s, nchunks, K); break;
    case 256: fp8_block_small_kernel<Tin, 32, kFp8Cpt><<<grid_cpt(nchunks, kFp8Cpt), kThreads, 0, st>>>(x, q, s, nchunks, K); break;
    default: {
      if (nblocks > 0x7FFFFFFFLL) return set_error(QG_ERR_UNSUPPORTED_SHAPE, "%s: too many blocks", name);
      const int cpt = (g / 8 + kThreads - 1) / kThreads;      // chunks of 8 per thread
      const unsigned nb = unsigned(nblocks);
      if (cpt <= 2)      fp8_block_reg_kernel<Tin, 2><<<nb, kThreads, 0, st>>>(x, q, s, g);
      else if (cpt <= 4) fp8_block_reg_kernel<Tin, 4><<<nb, kThreads, 0, st>>>(x, q, s, g);
      else if (cpt <= 8) fp8_block_reg_kernel<Tin, 8><<<nb, kThreads, 0, st>>>(x, q, s, g);
      else               fp8_block_large_kernel<Tin><<<nb, kThreads, 0, st>>>(x, q, s, g);
    }
  }
  return check_launch(name);
}

template <typename Tin>
qg_status launch_mxfp4(const Tin* x, uint8_t* q, uint8_t* se, int g, long long rows, int K,
                       cudaStream_t st, const char* name) {
  const long long nchunks = rows * (long long)K / 8;
  if (nchunks == 0) return QG_OK;
  if (g == 16) mxfp4_kernel<Tin, 2, kMxCpt><<<grid_cpt(nchunks, kMxCpt), kThreads, 0, st>>>(x, q, se, nchunks);
  else         mxfp4_kernel<Tin, 4, kMxCpt><<<grid_cpt(nchunks, kMxCpt), kThreads, 0, st>>>(x, q, se, nchunks);
  return check_launch(name);
}

bool is_pow2_block(int g) { return g == 8 || g == 16 || g == 32 || g == 64 || g == 128 || g == 256; }

}  // namespace
}  // namespace qg

using qg::aligned16;

extern "C" {

qg_status quant_act_fp8_block(const uint16_t* x, uint8_t* q, float* s, int g, int M, int K,
                              qg_stream_t stream) {
  QG_REQUIRE(x && q && s, QG_ERR_INVALID_ARG, "quant_act_fp8_block: NULL pointer");
  QG_REQUIRE(M >= 0 && K > 0 && g > 0, QG_ERR_INVALID_ARG, "quant_act_fp8_block: bad sizes");
  QG_REQUIRE(K % g == 0 && g % 8 == 0, QG_ERR_UNSUPPORTED_SHAPE,
             "quant_act_fp8_block: need K %% g == 0 and g %% 8 == 0 (K=%d g=%d)", K, g);
  QG_REQUIRE(aligned16(x) && aligned16(q) && (reinterpret_cast<uintptr_t>(s) & 3) == 0,
             QG_ERR_MISALIGNED, "quant_act_fp8_block: misaligned pointer");
  return qg::launch_fp8_block(x, q, s, g, M, K, reinterpret_cast<cudaStream_t>(stream),
                              "quant_act_fp8_block");
}

qg_status quant_act_mxfp4(const uint16_t* x, uint8_t* q, uint8_t* s_e8m0, int g, int M, int K,
                          qg_stream_t stream) {
  QG_REQUIRE(x && q && s_e8m0, QG_ERR_INVALID_ARG, "quant_act_mxfp4: NULL pointer");
  QG_REQUIRE(M >= 0 && K > 0, QG_ERR_INVALID_ARG, "quant_act_mxfp4: bad sizes");
  QG_REQUIRE(g == 16 || g == 32, QG_ERR_UNSUPPORTED_SHAPE, "quant_act_mxfp4: g must be 16 or 32");
  QG_REQUIRE(K % g == 0, QG_ERR_UNSUPPORTED_SHAPE, "quant_act_mxfp4: K %% g != 0");
  QG_REQUIRE(aligned16(x) && (reinterpret_cast<uintptr_t>(q) & 3) == 0, QG_ERR_MISALIGNED,
             "quant_act_mxfp4: misaligned pointer");
  return qg::launch_mxfp4(x, q, s_e8m0, g, M, K, reinterpret_cast<cudaStream_t>(stream),
                          "quant_act_mxfp4");
}

qg_status qg_quantize_weights_int4(const float* w, uint8_t* w_q, uint16_t* w_s, int g, int N, int K,
                                   qg_stream_t stream) {
  QG_REQUIRE(w && w_q && w_s, QG_ERR_INVALID_ARG, "qg_quantize_weights_int4: NULL pointer");
  QG_REQUIRE(N >= 0 && K > 0, QG_ERR_INVALID_ARG, "qg_quantize_weights_int4: bad sizes");
  QG_REQUIRE(qg::is_pow2_block(g) && K % g == 0, QG_ERR_UNSUPPORTED_SHAPE,
             "qg_quantize_weights_int4: g must be a power of two in [8, 256] dividing K");
  QG_REQUIRE(aligned16(w) && (reinterpret_cast<uintptr_t>(w_q) & 3) == 0, QG_ERR_MISALIGNED,
             "qg_quantize_weights_int4: misaligned pointer");
  const long long nchunks = (long long)N * K / 8;
  if (nchunks == 0) return QG_OK;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  const unsigned grid = qg::grid_for(nchunks);
  switch (g / 8) {
    case 1:  qg::int4_rtn_kernel<1><<<grid, qg::kThreads, 0, st>>>(w, w_q, w_s, nchunks); break;
    case 2:  qg::int4_rtn_kernel<2><<<grid, qg::kThreads, 0, st>>>(w, w_q, w_s, nchunks); break;
    case 4:  qg::int4_rtn_kernel<4><<<grid, qg::kThreads, 0, st>>>(w, w_q, w_s, nchunks); break;
    case 8:  qg::int4_rtn_kernel<8><<<grid, qg::kThreads, 0, st>>>(w, w_q, w_s, nchunks); break;
    case 16: qg::int4_rtn_kernel<16><<<grid, qg::kThreads, 0, st>>>(w, w_q, w_s, nchunks); break;
    default: qg::int4_rtn_kernel<32><<<grid, qg::kThreads, 0, st>>>(w, w_q, w_s, nchunks); break;
  }
  return qg::check_launch("qg_quantize_weights_int4");
}

qg_status qg_quantize_weights_int4_zp(const float* w, uint8_t* w_q, uint16_t* w_s, uint8_t* w_z, int g, int N,
                                      int K, qg_stream_t stream) {
  QG_REQUIRE(w && w_q && w_s && w_z, QG_ERR_INVALID_ARG, "qg_quantize_weights_int4_zp: NULL pointer");
  QG_REQUIRE(N >= 0 && K > 0, QG_ERR_INVALID_ARG, "qg_quantize_weights_int4_zp: bad sizes");
  QG_REQUIRE(qg::is_pow2_block(g) && K % g == 0, QG_ERR_UNSUPPORTED_SHAPE,
             "qg_quantize_weights_int4_zp: g must be a power of two in [8, 256] dividing K");
  QG_REQUIRE(aligned16(w) && (reinterpret_cast<uintptr_t>(w_q) & 3) == 0, QG_ERR_MISALIGNED,
             "qg_quantize_weights_int4_zp: misaligned pointer");
  const long long nchunks = (long long)N * K / 8;
  if (nchunks == 0) return QG_OK;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  const unsigned grid = qg::grid_for(nchunks);
  switch (g / 8) {
    case 1:  qg::int4_zp_kernel<1><<<grid, qg::kThreads, 0, st>>>(w, w_q, w_s, w_z, nchunks); break;
    case 2:  qg::int4_zp_kernel<2><<<grid, qg::kThreads, 0, st>>>(w, w_q, w_s, w_z, nchunks); break;
    case 4:  qg::int4_zp_kernel<4><<<grid, qg::kThreads, 0, st>>>(w, w_q, w_s, w_z, nchunks); break;
    case 8:  qg::int4_zp_kernel<8><<<grid, qg::kThreads, 0, st>>>(w, w_q, w_s, w_z, nchunks); break;
    case 16: qg::int4_zp_kernel<16><<<grid, qg::kThreads, 0, st>>>(w, w_q, w_s, w_z, nchunks); break;
    default: qg::int4_zp_kernel<32><<<grid, qg::kThreads, 0, st>>>(w, w_q, w_s, w_z, nchunks); break;
  }
  return qg::check_launch("qg_quantize_weights_int4_zp");
}

qg_status qg_quantize_weights_fp8(const float* w, uint8_t* w_e4m3, float* w_cs, int N, int K,
                                  qg_stream_t stream) {
  QG_REQUIRE(w && w_e4m3 && w_cs, QG_ERR_INVALID_ARG, "qg_quantize_weights_fp8: NULL pointer");
  QG_REQUIRE(N >= 0 && K > 0, QG_ERR_INVALID_ARG, "qg_quantize_weights_fp8: bad sizes");
  QG_REQUIRE(K % 8 == 0, QG_ERR_UNSUPPORTED_SHAPE, "qg_quantize_weights_fp8: K %% 8 != 0");
  QG_REQUIRE(aligned16(w) && aligned16(w_e4m3), QG_ERR_MISALIGNED,
             "qg_quantize_weights_fp8: misaligned pointer");
  return qg::launch_fp8_block(w, w_e4m3, w_cs, K, N, K, reinterpret_cast<cudaStream_t>(stream),
                              "qg_quantize_weights_fp8");
}

qg_status qg_quantize_weights_mxfp4(const float* w, uint8_t* w_e2m1, uint8_t* w_e8m0, int g, int N,
                                    int K, qg_stream_t stream) {
  QG_REQUIRE(w && w_e2m1 && w_e8m0, QG_ERR_INVALID_ARG, "qg_quantize_weights_mxfp4: NULL pointer");
  QG_REQUIRE(N >= 0 && K > 0, QG_ERR_INVALID_ARG, "qg_quantize_weights_mxfp4: bad sizes");
  QG_REQUIRE(g == 32 && K % 32 == 0, QG_ERR_UNSUPPORTED_SHAPE,
             "qg_quantize_weights_mxfp4: g must be 32 and divide K");
  QG_REQUIRE(aligned16(w) && (reinterpret_cast<uintptr_t>(w_e2m1) & 3) == 0, QG_ERR_MISALIGNED,
             "qg_quantize_weights_mxfp4: misaligned pointer");
  return qg::launch_mxfp4(w, w_e2m1, w_e8m0, g, N, K, reinterpret_cast<cudaStream_t>(stream),
                          "qg_quantize_weights_mxfp4");
}

qg_status qg_quantize_weights_nvfp4(const float* w, uint8_t* w_e2m1, uint8_t* w_e4m3,
                                    float* global_scale, int N, int K, qg_stream_t stream) {
  QG_REQUIRE(w && w_e2m1 && w_e4m3 && global_scale, QG_ERR_INVALID_ARG,
             "qg_quantize_weights_nvfp4: NULL pointer");
  QG_REQUIRE(N >= 0 && K > 0, QG_ERR_INVALID_ARG, "qg_quantize_weights_nvfp4: bad sizes");
  QG_REQUIRE(K % 16 == 0, QG_ERR_UNSUPPORTED_SHAPE, "qg_quantize_weights_nvfp4: K %% 16 != 0");
  QG_REQUIRE(aligned16(w) && (reinterpret_cast<uintptr_t>(w_e2m1) & 3) == 0 &&
                 (reinterpret_cast<uintptr_t>(global_scale) & 3) == 0,
             QG_ERR_MISALIGNED, "qg_quantize_weights_nvfp4: misaligned pointer");
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (cudaMemsetAsync(global_scale, 0, sizeof(float), st) != cudaSuccess)
    return qg::set_error(QG_ERR_CUDA, "qg_quantize_weights_nvfp4: memset failed");
  const long long nchunks = (long long)N * K / 8;
  if (nchunks > 0) {
    const unsigned g1 = unsigned(std::min<long long>(qg::grid_for(nchunks), 4LL * qg::sm_count()));
    qg::amax_kernel<<<g1, qg::kThreads, 0, st>>>(w, nchunks, reinterpret_cast<unsigned int*>(global_scale));
    qg::nvfp4_kernel<<<qg::grid_for(nchunks), qg::kThreads, 0, st>>>(w, w_e2m1, w_e4m3, global_scale, nchunks);
  }
  qg::nvfp4_finalize_kernel<<<1, 1, 0, st>>>(global_scale);
  return qg::check_launch("qg_quantize_weights_nvfp4");
}

qg_status qg_moe_gather_fp8(const uint8_t* src_q, const float* src_s, const int32_t* route_rows,
                            uint8_t* dst_q, float* dst_s, int R, int T, int K, qg_stream_t stream) {
  QG_REQUIRE(src_q && src_s && route_rows && dst_q && dst_s, QG_ERR_INVALID_ARG,
             "qg_moe_gather_fp8: NULL pointer");
  QG_REQUIRE(R >= 0 && T > 0 && K > 0, QG_ERR_INVALID_ARG, "qg_moe_gather_fp8: bad sizes");
  QG_REQUIRE(K % 16 == 0, QG_ERR_UNSUPPORTED_SHAPE, "qg_moe_gather_fp8: K %% 16 != 0");
  QG_REQUIRE(aligned16(src_q) && aligned16(dst_q), QG_ERR_MISALIGNED, "qg_moe_gather_fp8: misaligned");
  if (R == 0) return QG_OK;
  qg::gather_fp8_kernel<false><<<R, qg::kThreads, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
      src_q, src_s, route_rows, dst_q, dst_s, T, K);
  return qg::check_launch("qg_moe_gather_fp8");
}

qg_status qg_moe_gather_fp8_f16(const uint8_t* src_q, const float* src_s, const int32_t* route_rows,
                                uint16_t* dst_f16, float* dst_s, int R, int T, int K, qg_stream_t stream) {
  QG_REQUIRE(src_q && src_s && route_rows && dst_f16 && dst_s, QG_ERR_INVALID_ARG,
             "qg_moe_gather_fp8_f16: NULL pointer");
  QG_REQUIRE(R >= 0 && T > 0 && K > 0, QG_ERR_INVALID_ARG, "qg_moe_gather_fp8_f16: bad sizes");
  QG_REQUIRE(K % 16 == 0, QG_ERR_UNSUPPORTED_SHAPE, "qg_moe_gather_fp8_f16: K %% 16 != 0");
  QG_REQUIRE(aligned16(src_q) && aligned16(dst_f16), QG_ERR_MISALIGNED, "qg_moe_gather_fp8_f16: misaligned");
  if (R == 0) return QG_OK;
  qg::gather_fp8_kernel<true><<<R, qg::kThreads, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
      src_q, src_s, route_rows, dst_f16, dst_s, T, K);
  return qg::check_launch("qg_moe_gather_fp8_f16");
}

}  // extern "C"

namespace qg {
template <bool F16>
qg_status swiglu_quant_launch(const uint16_t* gate_up, void* q, float* s, int R, int I, qg_stream_t stream,
                              const char* name) {
  QG_REQUIRE(gate_up && q && s, QG_ERR_INVALID_ARG, "%s: NULL pointer", name);
  QG_REQUIRE(R >= 0 && I > 0, QG_ERR_INVALID_ARG, "%s: bad sizes", name);
  QG_REQUIRE(I % 8 == 0, QG_ERR_UNSUPPORTED_SHAPE, "%s: I %% 8 != 0", name);
  QG_REQUIRE(aligned16(gate_up) && aligned16(q), QG_ERR_MISALIGNED, "%s: misaligned", name);
  if (R == 0) return QG_OK;
  const cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  const int cpt = (I / 8 + kThreads - 1) / kThreads;    // chunks per thread
  const int cpt512 = (I / 8 + 511) / 512;
  if (cpt <= 1)         swiglu_quant_reg_kernel<1, kThreads, F16><<<R, kThreads, 0, st>>>(gate_up, q, s, I);
  else if (cpt <= 2)    swiglu_quant_reg_kernel<2, kThreads, F16><<<R, kThreads, 0, st>>>(gate_up, q, s, I);
  else if (cpt512 <= 2) swiglu_quant_reg_kernel<2, 512, F16><<<R, 512, 0, st>>>(gate_up, q, s, I);
  else if (cpt512 <= 4) swiglu_quant_reg_kernel<4, 512, F16><<<R, 512, 0, st>>>(gate_up, q, s, I);
  else               swiglu_quant_kernel<F16><<<R, kThreads, 0, st>>>(gate_up, q, s, I);
  return check_launch(name);
}
}  // namespace qg

extern "C" {

qg_status qg_swiglu_quant_fp8(const uint16_t* gate_up, uint8_t* q, float* s, int R, int I,
                              qg_stream_t stream) {
  return qg::swiglu_quant_launch<false>(gate_up, q, s, R, I, stream, "qg_swiglu_quant_fp8");
}

qg_status qg_swiglu_quant_fp8_f16(const uint16_t* gate_up, uint16_t* q_f16, float* s, int R, int I,
                                  qg_stream_t stream) {
  return qg::swiglu_quant_launch<true>(gate_up, q_f16, s, R, I, stream, "qg_swiglu_quant_fp8_f16");
}

qg_status qg_moe_combine(const uint16_t* down, const int32_t* row_of, const float* weight,
                         uint16_t* out, int T, int topk, int R, int H, qg_stream_t stream) {
  QG_REQUIRE(down && row_of && weight && out, QG_ERR_INVALID_ARG, "qg_moe_combine: NULL pointer");
  QG_REQUIRE(T >= 0 && topk > 0 && R >= 0 && H > 0, QG_ERR_INVALID_ARG, "qg_moe_combine: bad sizes");
  QG_REQUIRE(H % 8 == 0, QG_ERR_UNSUPPORTED_SHAPE, "qg_moe_combine: H %% 8 != 0");
  QG_REQUIRE(aligned16(down) && aligned16(out), QG_ERR_MISALIGNED, "qg_moe_combine: misaligned");
  if (T == 0) return QG_OK;
  dim3 grid((H / 8 + qg::kThreads - 1) / qg::kThreads, T);
  qg::combine_kernel<<<grid, qg::kThreads, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
      down, row_of, weight, out, topk, R, H);
  return qg::check_launch("qg_moe_combine");
}

qg_status qg_w4a8_fp8_scales(const uint16_t* w_s, uint8_t* w_s8, float* w_cs8, int rows, int G,
                             qg_stream_t stream) {
  QG_REQUIRE(w_s && w_s8 && w_cs8, QG_ERR_INVALID_ARG, "qg_w4a8_fp8_scales: NULL pointer");
  QG_REQUIRE(rows >= 0 && G > 0, QG_ERR_INVALID_ARG, "qg_w4a8_fp8_scales: bad sizes");
  if (rows == 0) return QG_OK;
  const long long threads = (long long)rows * 32;
  qg::w4a8_fp8_scales_kernel<<<unsigned((threads + qg::kThreads - 1) / qg::kThreads), qg::kThreads, 0,
                              reinterpret_cast<cudaStream_t>(stream)>>>(w_s, w_s8, w_cs8, rows, G);
  return qg::check_launch("qg_w4a8_fp8_scales");
}

}  // extern "C"
