// Decode (M <= 16) weight-only GEMV for the four weight formats, plus the
// test-only canonical dequantization export.
//
// Design ("Your 3090 Isn't Missing Anything...", section 4.3: at M = 1 DRAM
// bandwidth sets the time; the dequant must stay off the critical path):
//   * A CTA of 8 warps owns rg 16-row groups (16 * rg output channels); the
//     kWarps / rg warps of a row group take interleaved K segments and their
//     partial sums are reduced through shared memory.  The grid is sized to
//     a single wave.  When the activation slice would leave room for only one
//     CTA per SM (M <= 8) or would not fit (M > 8), the K range is split over
//     a thread-block cluster (1..8 CTAs) reduced through distributed shared
//     memory -- no global scratch, no atomics, deterministic.
//   * Each warp streams the packed words of its two rows per lane (g and g+8
//     of the mma group) through a private 4- to 6-deep cp.async.cg ring in
//     shared memory (16-byte, L1-bypassing), and decodes them in registers
//     into mma.sync m16n8k16 A fragments (weights are the M = 16 side,
//     activations the N = 8 side, so one mma covers 256 weights).
//   * The activation slice is staged once per CTA in shared memory with the k
//     order permuted to match the decode's pair order, one pad chunk per 8.
//   * Programmatic dependent launch: a CTA triggers its dependent at once,
//     issues its weight prologue, and waits for the previous kernel only
//     before it reads X (weights and scales must not be the previous decode
//     kernel's output -- stated in the header).
//   * FP4 block scales are folded into the E2M1 decode (one multiply per
//     pair; dequant.cuh), the NVFP4 weights then carrying 2^-9, undone with
//     the global scale.
//   * fp32 accumulation; the FP8 channel scale / NVFP4 global scale is
//     applied to the reduced row; one bf16 rounding at the store.
//   * W8A8 (FP8 weights, activations quantized here): the prologue quantizes
//     the CTA's activation slice per 1 x 128 block with the quant_act_fp8_block
//     rule and stages the codes' exact bf16 values; each block's partial sums
//     are scaled into the accumulator by the block scale at the block's end.
#include <algorithm>

#include "dequant.cuh"

#define QG_REQUIRE(cond, st, ...) \
  do { if (!(cond)) return qg::set_error(st, __VA_ARGS__); } while (0)

namespace qg {
namespace {

enum Fmt { F_INT4 = 0, F_FP8 = 1, F_MXFP4 = 2, F_NVFP4 = 3, F_INT4Z = 4, F_FP8A8 = 5 };
// FP8 weights (one byte per weight)
constexpr bool fp8_weights(int f) { return f == F_FP8 || f == F_FP8A8; }
constexpr int kActBlock = 128;         // F_FP8A8: activation quantization block (1 x 128)

constexpr int kWarps = 8;
// Weight segments in flight per warp (cp.async ring) and the scale prefetch
// distance, per activation-tile count: with two 8-column tiles (M > 8) the
// activation slice takes much of the shared memory, and a 4-deep ring leaves
// room for more CTAs per SM (M = 16, INT4 14336x4096: 25.8 -> 18.5 us;
// a 4-deep ring at M = 1 costs 10.0 -> 11.4 us).
template <int MT> struct RingCfg {
  static constexpr int RING = MT == 2 ? 4 : 6;
  static constexpr int PFS = MT == 2 ? 2 : 3;   // divides RING
  static_assert(RING % PFS == 0, "the scale ring index u % PFS must equal s % PFS");
};

template <int FMT> struct FmtTraits;
template <> struct FmtTraits<F_INT4>  { static constexpr int KSEG = 128, CPL = 4; };
template <> struct FmtTraits<F_INT4Z> { static constexpr int KSEG = 128, CPL = 4; };
template <> struct FmtTraits<F_MXFP4> { static constexpr int KSEG = 128, CPL = 4; };
template <> struct FmtTraits<F_NVFP4> { static constexpr int KSEG = 128, CPL = 4; };
template <> struct FmtTraits<F_FP8>   { static constexpr int KSEG = 64,  CPL = 2; };
template <> struct FmtTraits<F_FP8A8> { static constexpr int KSEG = 64,  CPL = 2; };

struct GemvArgs {
  const uint8_t* w;        // packed weights [N][row_bytes]
  const void* scales;      // per-format scale array (or channel scales for FP8)
  const uint8_t* zeros;    // INT4 zero points [N][K/g] (F_INT4Z) or nullptr
  const float* gscale;     // NVFP4 global scale (device scalar) or nullptr
  const uint16_t* x;       // [M][K] bf16
  uint16_t* y;             // [M][N] bf16
  int M, N, K, g;
  int lg;                  // log2(g) for INT4 (g is a power of two)
  int nseg;                // K / KSEG
  int ncp;                 // X smem row pitch in 16-byte chunks
  int rg;                  // 16-row groups per CTA (warps split K by kWarps / rg)
};

// Staged activation chunk c (16 bytes) sits at c + c / 8: one pad chunk per
// 8 keeps the lanes' 16-byte reads bank-conflict free, and a lane's chunks
// for one segment are consecutive, so they are addressed from one base.
QG_DEVICE int xpad(int c) { return c + (c >> 3); }

QG_DEVICE void mma_bf16(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                        uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Per-lane scale state for one segment of one row.
struct Scale { uint32_t a, b; };

// Scale row of output channel n (bytes), and the scale of segment 'seg' for lane t.
template <int FMT>
QG_DEVICE const uint8_t* scale_row(const GemvArgs& p, int n) {
  const uint8_t* base = static_cast<const uint8_t*>(p.scales);
  if constexpr (FMT == F_INT4 || FMT == F_INT4Z) return base + (size_t)n * (size_t)(p.K >> p.lg) * 2;
  if constexpr (FMT == F_MXFP4) return base + (size_t)n * (size_t)(p.K / 32);
  if constexpr (FMT == F_NVFP4) return base + (size_t)n * (size_t)(p.K / 16);
  return base;
}

// Zero-point row of output channel n (F_INT4Z only).
template <int FMT>
QG_DEVICE const uint8_t* zero_row(const GemvArgs& p, int n) {
  if constexpr (FMT == F_INT4Z) return p.zeros + (size_t)n * (size_t)(p.K >> p.lg);
  return nullptr;
}

// G1: INT4 with g == 128, one group per segment: the group index is the
// segment index.  load_scale fetches the raw scale (and zero-point) codes of
// a segment; finish_scale turns them into the decode's operands.  The GEMV
// prefetches raw codes a few segments ahead and finishes them only when the
// segment is decoded, so no warp waits on a prefetch.  FOLD: the GEMV's
// folded FP4 factors in s.b (MXFP4; 0 when the code is above 128) and s.a
// (NVFP4, both codes of the segment); without FOLD the raw codes (the
// canonical dequant export).
template <int FMT, bool G1>
QG_DEVICE Scale load_scale(const GemvArgs& p, const uint8_t* srow, const uint8_t* zrow, int seg, int t) {
  Scale s{0u, 0u};
  if constexpr (G1 && FMT == F_INT4) {
    s.a = __ldg(reinterpret_cast<const uint16_t*>(srow) + seg);
  } else if constexpr (G1 && FMT == F_INT4Z) {
    s.a = __ldg(reinterpret_cast<const uint16_t*>(srow) + seg);
    s.b = __ldg(zrow + seg);
  } else if constexpr (FMT == F_INT4) {
    const int grp = (seg * 128 + 32 * t) >> p.lg;
    s.a = __ldg(reinterpret_cast<const uint16_t*>(srow) + grp);
  } else if constexpr (FMT == F_INT4Z) {
    const int grp = (seg * 128 + 32 * t) >> p.lg;
    s.a = __ldg(reinterpret_cast<const uint16_t*>(srow) + grp);
    s.b = __ldg(zrow + grp);
  } else if constexpr (FMT == F_MXFP4) {
    s.a = __ldg(srow + seg * 4 + t);
  } else if constexpr (FMT == F_NVFP4) {
    s.a = __ldg(reinterpret_cast<const uint16_t*>(srow + seg * 8 + 2 * t));
  }
  return s;
}
template <int FMT, bool FOLD = false>
QG_DEVICE Scale finish_scale(Scale s) {
  if constexpr (FMT == F_INT4) {
    s.a = bf16x2_splat(s.a);
  } else if constexpr (FMT == F_INT4Z) {
    s.a = bf16x2_splat(s.a);
    s.b = bf16x2_zero128(s.b);
  } else if constexpr (FMT == F_MXFP4) {
    if constexpr (FOLD) s.b = mxfp4_fold(s.a);
  } else if constexpr (FMT == F_NVFP4) {
    if constexpr (FOLD) s.a = nvfp4_fold_x2(s.a);
  }
  return s;
}

// Programmatic dependent launch: let the next kernel in the stream start its
// prologue now, and wait for the previous kernel's results before touching
// any input.
QG_DEVICE void pdl_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
QG_DEVICE void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }


// Decode chunk j (8 k-values) of the lane's 16-byte word into A pairs:
// a[0], a[1] for the first mma (lo / hi k-slots), a[2], a[3] for the second.
// FOLD (FP4 formats, scales from load_scale<..., true>): MXFP4 with
// FAST = every row of the warp has its folded factor, NVFP4 always.
template <int FMT, bool FOLD = false, bool FAST = false>
QG_DEVICE void decode_chunk(const uint4& w, const Scale& s, int j, uint32_t (&a)[4]) {
  const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
  if constexpr (FMT == F_INT4) {
    int4x8_kperm(ww[j], s.a, a);
  } else if constexpr (FMT == F_INT4Z) {
    int4zp_x8_kperm(ww[j], s.a, s.b, a);
  } else if constexpr (FMT == F_MXFP4 && FOLD && FAST) {
    e2m1x8_kperm_folded(ww[j], s.b, a);
  } else if constexpr (FMT == F_MXFP4) {
    e2m1x8_kperm(ww[j], e8m0_to_bf16x2(s.a), a);
  } else if constexpr (FMT == F_NVFP4 && FOLD) {
    e2m1x8_kperm_folded(ww[j], prmt(s.a, s.a, j < 2 ? 0x1010u : 0x3232u), a);
  } else if constexpr (FMT == F_NVFP4) {
    e2m1x8_kperm(ww[j], e4m3_to_bf16x2(j < 2 ? (s.a & 0xFFu) : (s.a >> 8)), a);
  } else {
    e4m3x4_kperm(ww[2 * j], a[0], a[1]);
    e4m3x4_kperm(ww[2 * j + 1], a[2], a[3]);
  }
}

// X chunk permutation matching decode_chunk's pair order
template <int FMT>
QG_DEVICE uint4 perm_x(const uint4& u) {
  if constexpr (fp8_weights(FMT))   // (0,2,1,3,4,6,5,7)
    return make_uint4(prmt(u.x, u.y, 0x5410u), prmt(u.x, u.y, 0x7632u),
                      prmt(u.z, u.w, 0x5410u), prmt(u.z, u.w, 0x7632u));
  else                          // (0,4,1,5,2,6,3,7)
    return make_uint4(prmt(u.x, u.z, 0x5410u), prmt(u.x, u.z, 0x7632u),
                      prmt(u.y, u.w, 0x5410u), prmt(u.y, u.w, 0x7632u));
}

QG_DEVICE uint32_t smem_u32(const void* p) { return static_cast<uint32_t>(__cvta_generic_to_shared(p)); }

// 16-byte asynchronous global -> shared copy that bypasses L1 (cp.async.cg)
QG_DEVICE void cp_async16(uint32_t dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" :: "r"(dst), "l"(src) : "memory");
}
QG_DEVICE void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
QG_DEVICE void cp_async_wait() { asm volatile("cp.async.wait_group %0;" :: "n"(N) : "memory"); }

QG_DEVICE void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\nbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

QG_DEVICE float ld_dsmem_f32(uint32_t local_addr, uint32_t rank) {
  uint32_t remote;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(local_addr), "r"(rank));
  float v;
  asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(remote) : "memory");
  return v;
}

template <int FMT, int MT, bool G1>
__global__ void __launch_bounds__(kWarps * 32) gemv_kernel(const GemvArgs p) {
  using Tr = FmtTraits<FMT>;
  constexpr int kRing = RingCfg<MT>::RING, kPFS = RingCfg<MT>::PFS;
  extern __shared__ __align__(16) uint4 smem[];
  const int M = p.M;
  const int MP = MT * 8;
  const int RG = p.rg, KW = kWarps / p.rg;          // row groups x k-split warps
  const int rows_cta = 16 * RG;
  uint4* wring = smem;                                                      // [kWarps][kRing][2][32]
  uint4* xs = smem + (size_t)kWarps * kRing * 64;                           // [M][ncp]
  float* red = reinterpret_cast<float*>(xs + (size_t)M * p.ncp);            // [kWarps][16][MP]
  float* rsum = red + kWarps * 16 * MP;                                     // [rows_cta][MP]
  float* xsc = rsum + 16 * RG * MP;          // F_FP8A8: activation block scales [M][nblk]

  // k range of this CTA (cluster split) and of this warp (warp split)
  const int ks = gridDim.x, kr = blockIdx.x;
  const int seg_lo = (int)((long long)p.nseg * kr / ks);
  const int seg_hi = (int)((long long)p.nseg * (kr + 1) / ks);
  const int nseg_cta = seg_hi - seg_lo;
  const int k0 = seg_lo * Tr::KSEG;
  const int nchunk = nseg_cta * Tr::KSEG / 8;
  const size_t row_bytes = fp8_weights(FMT) ? (size_t)p.K : (size_t)p.K / 2;
  const int row0 = blockIdx.y * rows_cta;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, t = lane & 3;
  const int rg = warp / KW, kw = warp - rg * KW;
  const int s_lo = (int)((long long)nseg_cta * kw / KW);
  const int s_hi = (int)((long long)nseg_cta * (kw + 1) / KW);
  const int nseg = s_hi - s_lo;                     // this warp's segments (relative to seg_lo)
  const int nb = row0 + rg * 16;
  const int n0 = min(nb + g, p.N - 1), n1 = min(nb + g + 8, p.N - 1);
  const uint8_t* sr0 = scale_row<FMT>(p, n0);
  const uint8_t* sr1 = scale_row<FMT>(p, n1);
  const uint8_t* zr0 = zero_row<FMT>(p, n0);
  const uint8_t* zr1 = zero_row<FMT>(p, n1);
  const uint8_t* w0 = p.w + (size_t)n0 * row_bytes + (size_t)(seg_lo + s_lo) * 64 + 16 * t;
  const uint8_t* w1 = p.w + (size_t)n1 * row_bytes + (size_t)(seg_lo + s_lo) * 64 + 16 * t;

  const int col0 = min(g, M - 1), col1 = min(8 + g, M - 1);
  // this lane's activation chunks: segment s, chunk j at xq0[s * kPadSeg + j]
  // (KSEG / 8 is a multiple of 8, so the pad count of a segment is KSEG / 64)
  constexpr int kPadSeg = Tr::KSEG / 8 + Tr::KSEG / 64;
  const int lane_chunk = t * Tr::CPL;
  const uint4* xq0 = xs + col0 * p.ncp + s_lo * kPadSeg + xpad(lane_chunk);
  const uint4* xq1 = xs + col1 * p.ncp + s_lo * kPadSeg + xpad(lane_chunk);

  // Start the next kernel in the stream now.  This grid's weight stream is
  // issued before waiting for the previous kernel (qgemm.h: weights are never
  // written by the decode kernels, the only kernels that start early); the
  // activations are read only after the wait.
  pdl_launch_dependents();
  // Each lane streams its own two 16-byte words per segment through a private
  // ring of kRing segments in shared memory (cp.async; the lane reads back
  // only what it copied, so no cross-lane synchronization is needed).
  uint4* ring = wring + (size_t)warp * kRing * 64 + lane;          // [kRing][2][32] uint4 per warp
  const uint32_t ring_s = smem_u32(ring);
#pragma unroll
  for (int u = 0; u < kRing; ++u) {
    if (u < nseg) {
      cp_async16(ring_s + (uint32_t)(u * 64) * 16u, w0 + 64 * u);
      cp_async16(ring_s + (uint32_t)(u * 64 + 32) * 16u, w1 + 64 * u);
    }
    cp_async_commit();
  }
  Scale sa[kPFS], sb[kPFS];
#pragma unroll
  for (int u = 0; u < kPFS; ++u) {
    if (u < nseg) {
      sa[u] = load_scale<FMT, G1>(p, sr0, zr0, seg_lo + s_lo + u, t);
      sb[u] = load_scale<FMT, G1>(p, sr1, zr1, seg_lo + s_lo + u, t);
    }
  }

  // ---- previous kernel done: its outputs (our activations) are visible ------
  pdl_wait();
  // ---- stage the activation slice, permuted and swizzled -------------------
  // F_FP8A8 then quantizes it in place, per 1 x 128 block of the whole row
  // (the quant_act_fp8_block rule: s = absmax / 448, code = E4M3_RNE_sat(x /
  // s)), keeping the codes' exact bf16 values; the block maxima are gathered
  // while staging (a partly covered block's maximum includes its elements
  // outside this CTA's k range) and the scales go to xsc.
  const int blk0 = k0 / kActBlock;
  const int nblk = (k0 + nchunk * 8 + kActBlock - 1) / kActBlock - blk0;
  unsigned int* xmax = reinterpret_cast<unsigned int*>(xsc + M * nblk);     // [M][nblk] |x| maxima (bits)
  if constexpr (FMT == F_FP8A8) {
    for (int i = threadIdx.x; i < M * nblk; i += kWarps * 32) xmax[i] = 0u;
    __syncthreads();
  }
  for (int i = threadIdx.x; i < M * nchunk; i += kWarps * 32) {
    const int m = i / nchunk, c = i - m * nchunk;
    const uint4 u = __ldg(reinterpret_cast<const uint4*>(p.x + (size_t)m * p.K + k0 + 8 * c));
    xs[m * p.ncp + xpad(c)] = perm_x<FMT>(u);
    if constexpr (FMT == F_FP8A8) {
      const float a = fmaxf(fmaxf(fmaxf(fabsf(bf16_lo_to_f32(u.x)), fabsf(bf16_hi_to_f32(u.x))),
                                  fmaxf(fabsf(bf16_lo_to_f32(u.y)), fabsf(bf16_hi_to_f32(u.y)))),
                            fmaxf(fmaxf(fabsf(bf16_lo_to_f32(u.z)), fabsf(bf16_hi_to_f32(u.z))),
                                  fmaxf(fabsf(bf16_lo_to_f32(u.w)), fabsf(bf16_hi_to_f32(u.w)))));
      atomicMax(&xmax[m * nblk + (k0 + 8 * c) / kActBlock - blk0], __float_as_uint(a));   // a >= 0
    }
  }
  if constexpr (FMT == F_FP8A8) {
    // the parts of the first and last blocks outside this CTA's k range
    const int kend = k0 + nchunk * 8;
    const int head = k0 - blk0 * kActBlock, tail = (blk0 + nblk) * kActBlock - kend;
    for (int i = threadIdx.x; i < M * (head + tail) / 8; i += kWarps * 32) {
      const int per = (head + tail) / 8, m = i / per, c = i - m * per;
      const int k = c < head / 8 ? blk0 * kActBlock + 8 * c : kend + 8 * (c - head / 8);
      const uint4 u = __ldg(reinterpret_cast<const uint4*>(p.x + (size_t)m * p.K + k));
      const float a = fmaxf(fmaxf(fmaxf(fabsf(bf16_lo_to_f32(u.x)), fabsf(bf16_hi_to_f32(u.x))),
                                  fmaxf(fabsf(bf16_lo_to_f32(u.y)), fabsf(bf16_hi_to_f32(u.y)))),
                            fmaxf(fmaxf(fabsf(bf16_lo_to_f32(u.z)), fabsf(bf16_hi_to_f32(u.z))),
                                  fmaxf(fabsf(bf16_lo_to_f32(u.w)), fabsf(bf16_hi_to_f32(u.w)))));
      atomicMax(&xmax[m * nblk + k / kActBlock - blk0], __float_as_uint(a));
    }
    __syncthreads();
    for (int i = threadIdx.x; i < M * nblk; i += kWarps * 32) xsc[i] = fp8_scale(__uint_as_float(xmax[i]));
    __syncthreads();
    for (int i = threadIdx.x; i < M * nchunk; i += kWarps * 32) {
      const int m = i / nchunk, c = i - m * nchunk;
      const float sc = xsc[m * nblk + (k0 + 8 * c) / kActBlock - blk0];
      uint4& xv = xs[m * p.ncp + xpad(c)];
      uint32_t w[4] = {xv.x, xv.y, xv.z, xv.w};
#pragma unroll
      for (int j = 0; j < 4; ++j) {          // elementwise, so the staged (permuted) order is fine
        const uint32_t code = f32x2_to_e4m3x2(__fdiv_rn(bf16_hi_to_f32(w[j]), sc), __fdiv_rn(bf16_lo_to_f32(w[j]), sc));
        w[j] = (__float_as_uint(e4m3_to_f32(code & 0xFFu)) >> 16) | (__float_as_uint(e4m3_to_f32(code >> 8)) & 0xFFFF0000u);
      }
      xv = make_uint4(w[0], w[1], w[2], w[3]);
    }
  }
  __syncthreads();

  float acc[MT][4];
#pragma unroll
  for (int i = 0; i < MT; ++i) acc[i][0] = acc[i][1] = acc[i][2] = acc[i][3] = 0.f;
  // F_FP8A8: the current activation block's partial sums, scaled into acc at
  // each block boundary (the products inside a block are exact in fp32)
  float accb[MT][4];
#pragma unroll
  for (int i = 0; i < MT; ++i) accb[i][0] = accb[i][1] = accb[i][2] = accb[i][3] = 0.f;
  float (&acc_mma)[MT][4] = (FMT == F_FP8A8) ? accb : acc;

  for (int s0 = 0; s0 < nseg; s0 += kRing) {
#pragma unroll
    for (int u = 0; u < kRing; ++u) {
      const int s = s0 + u;
      if (s < nseg) {
        cp_async_wait<kRing - 1>();
        const uint4 wa = ring[u * 64];
        const uint4 wb = ring[u * 64 + 32];
        const int sn = s + kRing;
        if (sn < nseg) {
          cp_async16(ring_s + (uint32_t)(u * 64) * 16u, w0 + 64 * sn);
          cp_async16(ring_s + (uint32_t)(u * 64 + 32) * 16u, w1 + 64 * sn);
        }
        cp_async_commit();
        const int us = u % kPFS;
        const Scale s_a = finish_scale<FMT, true>(sa[us]), s_b = finish_scale<FMT, true>(sb[us]);
        if (s + kPFS < nseg) {
          sa[us] = load_scale<FMT, G1>(p, sr0, zr0, seg_lo + s_lo + s + kPFS, t);
          sb[us] = load_scale<FMT, G1>(p, sr1, zr1, seg_lo + s_lo + s + kPFS, t);
        }
        const uint4* xs0 = xq0 + s * kPadSeg;
        const uint4* xs1 = xq1 + s * kPadSeg;
        auto chunks = [&](auto fast) {
#pragma unroll
          for (int j = 0; j < Tr::CPL; ++j) {
            uint32_t ag[4], ah[4];
            decode_chunk<FMT, true, decltype(fast)::value>(wa, s_a, j, ag);
            decode_chunk<FMT, true, decltype(fast)::value>(wb, s_b, j, ah);
            {
              const uint4 xf = xs0[j];
              mma_bf16(acc_mma[0], ag[0], ah[0], ag[1], ah[1], xf.x, xf.y);
              mma_bf16(acc_mma[0], ag[2], ah[2], ag[3], ah[3], xf.z, xf.w);
            }
            if constexpr (MT == 2) {
              const uint4 xf = xs1[j];
              mma_bf16(acc_mma[1], ag[0], ah[0], ag[1], ah[1], xf.x, xf.y);
              mma_bf16(acc_mma[1], ag[2], ah[2], ag[3], ah[3], xf.z, xf.w);
            }
          }
        };
        if constexpr (FMT == F_MXFP4) {
          // one multiply per pair when every row of the warp has its folded factor
          if (__all_sync(0xffffffffu, (s_a.b != 0u) && (s_b.b != 0u)))
            chunks(std::true_type{});
          else
            chunks(std::false_type{});
        } else {
          chunks(std::false_type{});
        }
        if constexpr (FMT == F_FP8A8) {
          // block boundary (two 64-k segments per block) or the end of this
          // warp's range: acc += partial * block scale of each column m
          const int gseg = seg_lo + s_lo + s;
          if ((gseg & 1) || s == nseg - 1) {
            const int bl = (gseg >> 1) - blk0;
#pragma unroll
            for (int i = 0; i < MT; ++i) {
              const float x0 = xsc[min(8 * i + 2 * t, M - 1) * nblk + bl];
              const float x1 = xsc[min(8 * i + 2 * t + 1, M - 1) * nblk + bl];
              acc[i][0] = fmaf(accb[i][0], x0, acc[i][0]); acc[i][1] = fmaf(accb[i][1], x1, acc[i][1]);
              acc[i][2] = fmaf(accb[i][2], x0, acc[i][2]); acc[i][3] = fmaf(accb[i][3], x1, acc[i][3]);
              accb[i][0] = accb[i][1] = accb[i][2] = accb[i][3] = 0.f;
            }
          }
        }
      }
    }
  }
  cp_async_wait<0>();

  // ---- per-warp partials -> shared memory, reduce the k-split warps ---------
  {
    float* rw = red + warp * 16 * MP;
#pragma unroll
    for (int i = 0; i < MT; ++i) {
      const int m = 8 * i + 2 * t;
      rw[g * MP + m] = acc[i][0];
      rw[g * MP + m + 1] = acc[i][1];
      rw[(g + 8) * MP + m] = acc[i][2];
      rw[(g + 8) * MP + m + 1] = acc[i][3];
    }
  }
  __syncthreads();
  for (int i = threadIdx.x; i < rows_cta * MP; i += kWarps * 32) {
    const int r = i / MP, m = i - r * MP;
    const int rgi = r >> 4, rr = r & 15;
    float v = 0.f;
    for (int q = 0; q < KW; ++q) v += red[((rgi * KW + q) * 16 + rr) * MP + m];
    rsum[i] = v;
  }
  if (ks > 1) cluster_sync(); else __syncthreads();

  // ---- cluster reduction of this CTA's share of rows, epilogue, store --------
  const int rows_per = rows_cta / ks;
  const int rbeg = kr * rows_per;
  for (int i = threadIdx.x; i < rows_per * M; i += kWarps * 32) {
    const int m = i / rows_per, r = rbeg + (i - m * rows_per);
    const int n = row0 + r;
    float v;
    if (ks > 1) {
      const uint32_t a = smem_u32(rsum + r * MP + m);
      v = 0.f;
      for (int q = 0; q < ks; ++q) v += ld_dsmem_f32(a, q);
    } else {
      v = rsum[r * MP + m];
    }
    if (n < p.N) {
      if constexpr (fp8_weights(FMT)) v *= __ldg(static_cast<const float*>(p.scales) + n);
      if constexpr (FMT == F_NVFP4) v *= __ldg(p.gscale) * kNvfp4Unfold;   // 2^9 exactly (folded decode)
      p.y[(size_t)m * p.N + n] = f32_to_bf16_bits(v);
    }
  }
  if (ks > 1) cluster_sync();
}

// ---------------------------------------------------------------------------
// test-only canonical dequantization (same decode routines, natural order)
// ---------------------------------------------------------------------------
template <int FMT>
__global__ void dequant_kernel(const uint8_t* __restrict__ w, const void* __restrict__ scales,
                               const uint8_t* __restrict__ zeros, int g, uint16_t* __restrict__ out, int N,
                               int K) {
  using Tr = FmtTraits<FMT>;
  const int t = threadIdx.x & 3;              // position inside a 64-byte segment
  const long long lane_id = (blockIdx.x * (long long)blockDim.x + threadIdx.x) >> 2;
  const int nseg = K / Tr::KSEG;
  const long long total = (long long)N * nseg;
  if (lane_id >= total) return;
  const int n = int(lane_id / nseg), seg = int(lane_id % nseg);
  const size_t row_bytes = fp8_weights(FMT) ? (size_t)K : (size_t)K / 2;
  const uint4 wv = *reinterpret_cast<const uint4*>(w + (size_t)n * row_bytes + seg * 64 + 16 * t);
  GemvArgs p{};
  p.scales = scales; p.zeros = zeros; p.K = K; p.g = g; p.lg = 31 - __clz(g);
  const Scale s = finish_scale<FMT>(load_scale<FMT, false>(p, scale_row<FMT>(p, n), zero_row<FMT>(p, n), seg, t));
  uint16_t* o = out + (size_t)n * K + (size_t)seg * Tr::KSEG + t * Tr::CPL * 8;
#pragma unroll
  for (int j = 0; j < Tr::CPL; ++j) {
    uint32_t a[4], nat[4];
    decode_chunk<FMT>(wv, s, j, a);
    if constexpr (FMT == F_FP8) {       // a = (0,2),(1,3),(4,6),(5,7)
      nat[0] = prmt(a[0], a[1], 0x5410u); nat[1] = prmt(a[0], a[1], 0x7632u);
      nat[2] = prmt(a[2], a[3], 0x5410u); nat[3] = prmt(a[2], a[3], 0x7632u);
    } else {
      kperm4_to_natural(a, nat);
    }
    *reinterpret_cast<uint4*>(o + 8 * j) = make_uint4(nat[0], nat[1], nat[2], nat[3]);
  }
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------
template <int FMT, int MT>
qg_status launch_gemv_t(const GemvArgs& a0, cudaStream_t st, const char* name) {
  using Tr = FmtTraits<FMT>;
  GemvArgs a = a0;
  a.nseg = a.K / Tr::KSEG;
  const int row_groups = (a.N + 15) / 16;
  constexpr bool kInt4 = FMT == F_INT4 || FMT == F_INT4Z;
  auto kern = (kInt4 && a.g == 128) ? gemv_kernel<FMT, MT, kInt4> : gemv_kernel<FMT, MT, false>;
  auto smem_for = [&](int ks, int rg) {
    const int nseg_max = (a.nseg + ks - 1) / ks;
    const int nch = nseg_max * Tr::KSEG / 8;
    int ncp = nch + nch / 8;                          // padded row (one pad chunk per 8)
    const int want = fp8_weights(FMT) ? 1 : 2;        // bank-conflict-free pitch (mod 8)
    while ((ncp & 7) != want) ++ncp;
    a.ncp = ncp;
    const size_t xsc_bytes = FMT == F_FP8A8 ? (size_t)a.M * (nseg_max * Tr::KSEG / kActBlock + 2) * 8 : 0;
    return (size_t)kWarps * RingCfg<MT>::RING * 64 * 16 + (size_t)a.M * ncp * 16 +
           (size_t)(kWarps * 16 + 16 * rg) * MT * 8 * 4 + xsc_bytes;
  };
  // K split over a cluster when the activation slice would leave room for
  // only one CTA per SM: for one activation tile (M <= 8) above 96 KB of
  // shared memory (M = 4, K = 14336: 13.7 -> 12.6 us INT4, 16.8 -> 14.8 us
  // FP8), for two tiles only when it does not fit (a split there costs more
  // than it gains: M = 16 14336x4096 25.9 -> 38.1 us at a 96 KB target)
  int ks = 1;
  const size_t smem_target = MT == 1 ? 96 * 1024 : 200 * 1024;
  while (smem_for(ks, 8) > smem_target && ks < 8) ks *= 2;
  if (smem_for(ks, 8) > 220 * 1024)
    return set_error(QG_ERR_UNSUPPORTED_SHAPE, "%s: activation slice too large for one CTA", name);
  // rows per CTA: the fewest that keep every CTA resident in one wave
  const int cap_sm = sm_count();
  int rg = 1;
  for (;;) {
    const size_t smem = smem_for(ks, rg);
    if (!ensure_smem(kern, (int)smem)) return set_error(QG_ERR_CUDA, "%s: cannot set shared memory size", name);
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kWarps * 32, smem) != cudaSuccess)
      per_sm = 1;
    const long long ctas = (long long)((row_groups + rg - 1) / rg) * ks;
    const bool kw_ok = (kWarps / rg) <= (a.nseg + ks - 1) / ks;
    if ((ctas <= (long long)per_sm * cap_sm / ks * ks && kw_ok) || rg == kWarps) break;
    rg *= 2;
  }
  a.rg = rg;
  const size_t smem = smem_for(ks, rg);
  const int rb = (row_groups + rg - 1) / rg;

  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(ks, rb, 1);
  cfg.blockDim = dim3(kWarps * 32, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = ks;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  const cudaError_t e = cudaLaunchKernelEx(&cfg, kern, a);
  if (e != cudaSuccess) return set_error(QG_ERR_CUDA, "%s: launch failed: %s", name, cudaGetErrorString(e));
  return QG_OK;
}

template <int FMT>
qg_status launch_gemv(const GemvArgs& a, cudaStream_t st, const char* name) {
  // M <= 8: one 8-column activation tile; 9..16: two.  Larger M is processed
  // in slices of 16 rows.
  if (a.M <= 8) return launch_gemv_t<FMT, 1>(a, st, name);
  return launch_gemv_t<FMT, 2>(a, st, name);
}

template <int FMT>
qg_status run_weight_only(GemvArgs a, cudaStream_t st, const char* name) {
  const int M = a.M;
  for (int m0 = 0; m0 < M; m0 += 16) {
    GemvArgs s = a;
    s.M = std::min(16, M - m0);
    s.x = a.x + (size_t)m0 * a.K;
    s.y = a.y + (size_t)m0 * a.N;
    const qg_status r = launch_gemv<FMT>(s, st, name);
    if (r != QG_OK) return r;
  }
  return QG_OK;
}

qg_status check_common(const void* w, const void* x, const void* y, int M, int N, int K, const char* name) {
  QG_REQUIRE(w && x && y, QG_ERR_INVALID_ARG, "%s: NULL pointer", name);
  QG_REQUIRE(M >= 0 && N > 0 && K > 0, QG_ERR_INVALID_ARG, "%s: bad sizes M=%d N=%d K=%d", name, M, N, K);
  QG_REQUIRE(N % 8 == 0 && K % 128 == 0, QG_ERR_UNSUPPORTED_SHAPE,
             "%s: need N %% 8 == 0 and K %% 128 == 0 (N=%d K=%d)", name, N, K);
  QG_REQUIRE(aligned16(w) && aligned16(x) && aligned16(y), QG_ERR_MISALIGNED, "%s: misaligned pointer", name);
  return QG_OK;
}

// The dense entries (W4A16, W4A16 with zero points, W8A16, FP4A16, W4A4)
// take any K that is a multiple of 32 (and of g); K % 128 == 0 runs on the
// fast kernels, anything else on gemm_any_k_kernel.
qg_status check_common_k32(const void* w, const void* x, const void* y, int M, int N, int K, const char* name) {
  QG_REQUIRE(w && x && y, QG_ERR_INVALID_ARG, "%s: NULL pointer", name);
  QG_REQUIRE(M >= 0 && N > 0 && K > 0, QG_ERR_INVALID_ARG, "%s: bad sizes M=%d N=%d K=%d", name, M, N, K);
  QG_REQUIRE(N % 8 == 0 && K % 32 == 0, QG_ERR_UNSUPPORTED_SHAPE,
             "%s: need N %% 8 == 0 and K %% 32 == 0 (N=%d K=%d)", name, N, K);
  QG_REQUIRE(aligned16(w) && aligned16(x) && aligned16(y), QG_ERR_MISALIGNED, "%s: misaligned pointer", name);
  return QG_OK;
}

// E2M1 code (4 bits) -> its value: sign, then 0, 0.5 or 2^(e-1) * (1 + m/2)
QG_DEVICE float e2m1_value(uint32_t x) {
  const uint32_t m = x & 7u, e = m >> 1, man = m & 1u;
  const uint32_t bits = e ? ((e + 126u) << 23) | (man << 22) : (man ? 0x3F000000u : 0u);
  return __uint_as_float(bits | ((x & 8u) << 28));
}
// 2^(se - 127) exactly (se = 0 gives the fp32 subnormal 2^-127)
QG_DEVICE float e8m0_value(uint32_t se) { return __uint_as_float(se ? se << 23 : 0x00400000u); }

// The general path for K % 128 != 0: one thread per output, the canonical
// dequantized weight of every k (INT4: bf16_RNE(q * s), exact fp32 product;
// zero points: bf16_RNE((u - z) * s); FP8, MXFP4, NVFP4: the exact values),
// fp32 accumulation in k order, the format's epilogue scale (FP8 channel,
// NVFP4 global), one bf16 rounding.  It is there for the shapes the fast
// kernels' 128-k segments do not cover, not for speed.
struct AnyK {
  const uint8_t* w;                      // packed codes, rows of K (FP8) or K/2 bytes
  const void* s;                         // bf16 [N][K/g] (INT4), E8M0 / E4M3 bytes [N][K/g] (FP4)
  const uint8_t* z;                      // zero points [N][K/g] (INT4 with zero points)
  const float* cs;                       // FP8 channel scales [N]
  const float* gs;                       // NVFP4 global scale
  const uint16_t* x;
  uint16_t* y;
  int M, N, K, g;
};
template <int FMT>
__global__ void gemm_any_k_kernel(const AnyK p) {
  const int n = blockIdx.x * blockDim.x + threadIdx.x, m = blockIdx.y;
  if (n >= p.N) return;
  const uint16_t* xr = p.x + (size_t)m * p.K;
  const size_t sg = (size_t)n * (p.K / p.g);
  float acc = 0.f;
  for (int k = 0; k < p.K; ++k) {
    float w;
    if constexpr (FMT == F_FP8) {
      w = e4m3_to_f32(__ldg(p.w + (size_t)n * p.K + k));
    } else {
      const uint32_t b = __ldg(p.w + (size_t)n * (p.K / 2) + k / 2), u = (k & 1) ? b >> 4 : b & 15u;
      if constexpr (FMT == F_INT4 || FMT == F_INT4Z) {
        const float sc = bf16_bits_to_f32(__ldg(reinterpret_cast<const uint16_t*>(p.s) + sg + k / p.g));
        const int q = FMT == F_INT4 ? (u >= 8u ? (int)u - 16 : (int)u) : (int)u - (int)__ldg(p.z + sg + k / p.g);
        w = bf16_bits_to_f32(f32_to_bf16_bits((float)q * sc));
      } else {
        const uint32_t c = __ldg(reinterpret_cast<const uint8_t*>(p.s) + sg + k / p.g);
        w = e2m1_value(u) * (FMT == F_MXFP4 ? e8m0_value(c) : e4m3_to_f32(c));
      }
    }
    acc = fmaf(bf16_bits_to_f32(__ldg(xr + k)), w, acc);
  }
  if constexpr (FMT == F_FP8) acc = __fmul_rn(acc, __ldg(p.cs + n));
  if constexpr (FMT == F_NVFP4) acc = __fmul_rn(acc, __ldg(p.gs));
  p.y[(size_t)m * p.N + n] = f32_to_bf16_bits(acc);
}
template <int FMT>
qg_status run_any_k(const AnyK& a, cudaStream_t st, const char* name) {
  for (int m0 = 0; m0 < a.M; m0 += 65535) {          // the grid's y extent is at most 65535 rows
    AnyK s = a;
    s.M = std::min(65535, a.M - m0);
    s.x = a.x + (size_t)m0 * a.K;
    s.y = a.y + (size_t)m0 * a.N;
    gemm_any_k_kernel<FMT><<<dim3((s.N + 127) / 128, s.M), 128, 0, st>>>(s);
    const qg_status r = check_launch(name);
    if (r != QG_OK) return r;
  }
  return QG_OK;
}

// MXFP4 codes with one E8M0 code per G elements (G = 16 or 32) -> their exact
// bf16 values, natural k order (the W4A4 expansion): a thread takes 8 codes
// (within one block); each value is the E2M1 value times 2^(se - 127), exact
// in fp32 and in bf16 (at most two significant bits, at least 2^-128).
template <int G>
__global__ void mxfp4_expand_kernel(const uint8_t* __restrict__ q, const uint8_t* __restrict__ se,
                                    uint16_t* __restrict__ out, long long n8) {
  const long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x;
  if (i >= n8) return;
  const uint32_t w = __ldg(reinterpret_cast<const uint32_t*>(q) + i);
  const float f = e8m0_value(__ldg(se + i / (G / 8)));
  uint32_t o[4];
#pragma unroll
  for (int b = 0; b < 4; ++b)                     // elements 2b, 2b + 1: the low nibble first
    o[b] = (uint32_t)f32_to_bf16_bits(e2m1_value((w >> (8 * b)) & 0xFu) * f) |
           ((uint32_t)f32_to_bf16_bits(e2m1_value((w >> (8 * b + 4)) & 0xFu) * f) << 16);
  reinterpret_cast<uint4*>(out)[i] = make_uint4(o[0], o[1], o[2], o[3]);
}

}  // namespace

// block-scaled FP4 W4A4 (gemm_fp4.cu)
qg_status w4a4_mxfp4_bs(const uint8_t* w_e2m1, const uint8_t* w_e8m0, const uint8_t* a_e2m1,
                        const uint8_t* a_e8m0, int g_act, uint16_t* y, int M, int N, int K, cudaStream_t st,
                        bool* handled);

// entry for the prefill path (gemm_tc.cu) when it declines a shape; w_z
// (zero points) selects the asymmetric format
qg_status gemv_w4a16_any_m(const uint8_t* w_q, const uint16_t* w_s, const uint8_t* w_z, int g,
                           const uint16_t* x, uint16_t* y, int M, int N, int K, cudaStream_t st,
                           const char* name) {
  GemvArgs a{};
  a.w = w_q; a.scales = w_s; a.zeros = w_z; a.x = x; a.y = y; a.M = M; a.N = N; a.K = K; a.g = g;
  a.lg = 0;
  while ((1 << a.lg) < g) ++a.lg;
  return w_z ? run_weight_only<F_INT4Z>(a, st, name) : run_weight_only<F_INT4>(a, st, name);
}

}  // namespace qg

using qg::aligned16;

// prefill dispatcher lives in gemm_tc.cu (wf: 0 INT4, 1 INT4 with zero points, 2 FP8, 3 MXFP4, 4 NVFP4)
namespace qg {
qg_status prefill_tc(int wf, const uint8_t* w_q, const void* w_s, const uint8_t* w_z, const float* cs,
                     const float* gs, int g, const uint16_t* x, uint16_t* y, int M, int N, int K,
                     cudaStream_t st, bool* handled, const char* name);
}

extern "C" {

qg_status qgemm_w4a16(const uint8_t* w_q, const uint16_t* w_s, int g, const uint16_t* x, uint16_t* y,
                      int M, int N, int K, qg_stream_t stream) {
  qg_status r = qg::check_common_k32(w_q, x, y, M, N, K, "qgemm_w4a16");
  if (r != QG_OK) return r;
  QG_REQUIRE(w_s, QG_ERR_INVALID_ARG, "qgemm_w4a16: NULL scales");
  QG_REQUIRE(g >= 32 && (g & (g - 1)) == 0 && K % g == 0, QG_ERR_UNSUPPORTED_SHAPE,
             "qgemm_w4a16: need g a power of two >= 32 dividing K (g=%d)", g);
  if (M == 0) return QG_OK;
  if (K % 128 != 0)
    return qg::run_any_k<qg::F_INT4>({w_q, w_s, nullptr, nullptr, nullptr, x, y, M, N, K, g},
                                     reinterpret_cast<cudaStream_t>(stream), "qgemm_w4a16");
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (M > 16) {
    bool handled = false;
    r = qg::prefill_tc(0, w_q, w_s, nullptr, nullptr, nullptr, g, x, y, M, N, K, st, &handled, "qgemm_w4a16");
    if (handled) return r;
  }
  return qg::gemv_w4a16_any_m(w_q, w_s, nullptr, g, x, y, M, N, K, st, "qgemm_w4a16");
}

qg_status qgemm_w4a16_zp(const uint8_t* w_q, const uint16_t* w_s, const uint8_t* w_z, int g,
                         const uint16_t* x, uint16_t* y, int M, int N, int K, qg_stream_t stream) {
  qg_status r = qg::check_common_k32(w_q, x, y, M, N, K, "qgemm_w4a16_zp");
  if (r != QG_OK) return r;
  QG_REQUIRE(w_s && w_z, QG_ERR_INVALID_ARG, "qgemm_w4a16_zp: NULL scales or zero points");
  QG_REQUIRE(g >= 32 && (g & (g - 1)) == 0 && K % g == 0, QG_ERR_UNSUPPORTED_SHAPE,
             "qgemm_w4a16_zp: need g a power of two >= 32 dividing K (g=%d)", g);
  if (M == 0) return QG_OK;
  if (K % 128 != 0)
    return qg::run_any_k<qg::F_INT4Z>({w_q, w_s, w_z, nullptr, nullptr, x, y, M, N, K, g},
                                      reinterpret_cast<cudaStream_t>(stream), "qgemm_w4a16_zp");
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (M > 16) {
    bool handled = false;
    r = qg::prefill_tc(1, w_q, w_s, w_z, nullptr, nullptr, g, x, y, M, N, K, st, &handled, "qgemm_w4a16_zp");
    if (handled) return r;
  }
  return qg::gemv_w4a16_any_m(w_q, w_s, w_z, g, x, y, M, N, K, st, "qgemm_w4a16_zp");
}

qg_status qgemm_w8a16(const uint8_t* w_e4m3, const float* w_cs, const uint16_t* x, uint16_t* y,
                      int M, int N, int K, qg_stream_t stream) {
  qg_status r = qg::check_common_k32(w_e4m3, x, y, M, N, K, "qgemm_w8a16");
  if (r != QG_OK) return r;
  QG_REQUIRE(w_cs, QG_ERR_INVALID_ARG, "qgemm_w8a16: NULL channel scales");
  if (M == 0) return QG_OK;
  if (K % 128 != 0)
    return qg::run_any_k<qg::F_FP8>({w_e4m3, nullptr, nullptr, w_cs, nullptr, x, y, M, N, K, 1},
                                    reinterpret_cast<cudaStream_t>(stream), "qgemm_w8a16");
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (M > 16) {
    bool handled = false;
    r = qg::prefill_tc(2, w_e4m3, nullptr, nullptr, w_cs, nullptr, K, x, y, M, N, K, st, &handled, "qgemm_w8a16");
    if (handled) return r;
  }
  qg::GemvArgs a{};
  a.w = w_e4m3; a.scales = w_cs; a.x = x; a.y = y; a.M = M; a.N = N; a.K = K; a.g = K;
  return qg::run_weight_only<qg::F_FP8>(a, st, "qgemm_w8a16");
}

qg_status qgemm_w8a8(const uint8_t* w_e4m3, const float* w_cs, const uint16_t* x, uint16_t* y,
                     int M, int N, int K, qg_stream_t stream) {
  qg_status r = qg::check_common(w_e4m3, x, y, M, N, K, "qgemm_w8a8");
  if (r != QG_OK) return r;
  QG_REQUIRE(w_cs, QG_ERR_INVALID_ARG, "qgemm_w8a8: NULL channel scales");
  if (M == 0) return QG_OK;
  qg::GemvArgs a{};
  a.w = w_e4m3; a.scales = w_cs; a.x = x; a.y = y; a.M = M; a.N = N; a.K = K; a.g = K;
  return qg::run_weight_only<qg::F_FP8A8>(a, reinterpret_cast<cudaStream_t>(stream), "qgemm_w8a8");
}

qg_status qgemm_fp4a16(const uint8_t* w_e2m1, const uint8_t* w_bs, int scale_fmt, int g,
                       const float* global_scale, const uint16_t* x, uint16_t* y, int M, int N, int K,
                       qg_stream_t stream) {
  qg_status r = qg::check_common_k32(w_e2m1, x, y, M, N, K, "qgemm_fp4a16");
  if (r != QG_OK) return r;
  QG_REQUIRE(w_bs, QG_ERR_INVALID_ARG, "qgemm_fp4a16: NULL block scales");
  qg::GemvArgs a{};
  a.w = w_e2m1; a.scales = w_bs; a.x = x; a.y = y; a.M = M; a.N = N; a.K = K; a.g = g;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (scale_fmt == QG_SCALE_E8M0) {
    QG_REQUIRE(g == 32, QG_ERR_UNSUPPORTED_SHAPE, "qgemm_fp4a16: MXFP4 needs g == 32");
    QG_REQUIRE(global_scale == nullptr, QG_ERR_INVALID_ARG, "qgemm_fp4a16: MXFP4 takes no global scale");
    if (M == 0) return QG_OK;
    if (K % 128 != 0)
      return qg::run_any_k<qg::F_MXFP4>({w_e2m1, w_bs, nullptr, nullptr, nullptr, x, y, M, N, K, 32}, st,
                                        "qgemm_fp4a16");
    if (M > 16) {
      bool handled = false;
      r = qg::prefill_tc(3, w_e2m1, w_bs, nullptr, nullptr, nullptr, g, x, y, M, N, K, st, &handled, "qgemm_fp4a16");
      if (handled) return r;
    }
    return qg::run_weight_only<qg::F_MXFP4>(a, st, "qgemm_fp4a16");
  }
  if (scale_fmt == QG_SCALE_E4M3) {
    QG_REQUIRE(g == 16, QG_ERR_UNSUPPORTED_SHAPE, "qgemm_fp4a16: NVFP4 needs g == 16");
    QG_REQUIRE(global_scale != nullptr, QG_ERR_INVALID_ARG, "qgemm_fp4a16: NVFP4 needs a global scale");
    QG_REQUIRE((reinterpret_cast<uintptr_t>(global_scale) & 3) == 0, QG_ERR_MISALIGNED,
               "qgemm_fp4a16: misaligned global scale");
    a.gscale = global_scale;
    if (M == 0) return QG_OK;
    if (K % 128 != 0)
      return qg::run_any_k<qg::F_NVFP4>({w_e2m1, w_bs, nullptr, nullptr, global_scale, x, y, M, N, K, 16}, st,
                                        "qgemm_fp4a16");
    if (M > 16) {
      bool handled = false;
      r = qg::prefill_tc(4, w_e2m1, w_bs, nullptr, nullptr, global_scale, g, x, y, M, N, K, st, &handled,
                         "qgemm_fp4a16");
      if (handled) return r;
    }
    return qg::run_weight_only<qg::F_NVFP4>(a, st, "qgemm_fp4a16");
  }
  return qg::set_error(QG_ERR_INVALID_ARG, "qgemm_fp4a16: unknown scale format %d", scale_fmt);
}

namespace qg {
namespace {
// W4A4: for M > 16 the block-scaled FP4 tensor cores (gemm_fp4.cu), when K
// is a multiple of 256 and both scale arrays are 8-byte aligned; otherwise
// the MXFP4 activations (blocks of g_act) are expanded to bf16 (exact) into
// a_work and the MXFP4-weight GEMM (qgemm_fp4a16) runs on them.
qg_status w4a4_impl(const uint8_t* w_e2m1, const uint8_t* w_e8m0, const uint8_t* a_e2m1, const uint8_t* a_e8m0,
                    int g_act, uint16_t* a_work, uint16_t* y, int M, int N, int K, qg_stream_t stream,
                    const char* name) {
  QG_REQUIRE(a_e2m1 && a_e8m0 && a_work && w_e8m0, QG_ERR_INVALID_ARG, "%s: NULL pointer", name);
  qg_status r = check_common_k32(w_e2m1, a_work, y, M, N, K, name);
  if (r != QG_OK) return r;
  QG_REQUIRE(aligned16(a_e2m1), QG_ERR_MISALIGNED, "%s: misaligned activation codes", name);
  if (M == 0) return QG_OK;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (M > 16) {
    bool handled = false;
    r = w4a4_mxfp4_bs(w_e2m1, w_e8m0, a_e2m1, a_e8m0, g_act, y, M, N, K, st, &handled);
    if (handled) return r;
  }
  const long long n8 = (long long)M * K / 8;
  if (g_act == 32)
    mxfp4_expand_kernel<32><<<unsigned((n8 + 255) / 256), 256, 0, st>>>(a_e2m1, a_e8m0, a_work, n8);
  else
    mxfp4_expand_kernel<16><<<unsigned((n8 + 255) / 256), 256, 0, st>>>(a_e2m1, a_e8m0, a_work, n8);
  r = check_launch(name);
  if (r != QG_OK) return r;
  return qgemm_fp4a16(w_e2m1, w_e8m0, QG_SCALE_E8M0, 32, nullptr, a_work, y, M, N, K, stream);
}
}  // namespace
}  // namespace qg

qg_status qgemm_w4a4_mxfp4(const uint8_t* w_e2m1, const uint8_t* w_e8m0, const uint8_t* a_e2m1,
                           const uint8_t* a_e8m0, uint16_t* a_work, uint16_t* y, int M, int N, int K,
                           qg_stream_t stream) {
  return qg::w4a4_impl(w_e2m1, w_e8m0, a_e2m1, a_e8m0, 32, a_work, y, M, N, K, stream, "qgemm_w4a4_mxfp4");
}

qg_status qgemm_w4a4_mxfp4_g(const uint8_t* w_e2m1, const uint8_t* w_e8m0, const uint8_t* a_e2m1,
                             const uint8_t* a_e8m0, int g_act, uint16_t* a_work, uint16_t* y, int M, int N,
                             int K, qg_stream_t stream) {
  QG_REQUIRE(g_act == 16 || g_act == 32, QG_ERR_UNSUPPORTED_SHAPE, "qgemm_w4a4_mxfp4_g: g_act must be 16 or 32");
  return qg::w4a4_impl(w_e2m1, w_e8m0, a_e2m1, a_e8m0, g_act, a_work, y, M, N, K, stream, "qgemm_w4a4_mxfp4_g");
}

qg_status qg_dequant_weights(int fmt, const uint8_t* w, const void* scales, int g, uint16_t* w_out,
                             int N, int K, qg_stream_t stream) {
  QG_REQUIRE(w && w_out, QG_ERR_INVALID_ARG, "qg_dequant_weights: NULL pointer");
  QG_REQUIRE(N >= 0 && K > 0, QG_ERR_INVALID_ARG, "qg_dequant_weights: bad sizes");
  QG_REQUIRE(K % 128 == 0, QG_ERR_UNSUPPORTED_SHAPE, "qg_dequant_weights: K %% 128 != 0");
  QG_REQUIRE(aligned16(w) && aligned16(w_out), QG_ERR_MISALIGNED, "qg_dequant_weights: misaligned");
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  const int threads = 256;
  auto grid = [&](int kseg) {
    const long long lanes = (long long)N * (K / kseg) * 4;
    return unsigned((lanes + threads - 1) / threads);
  };
  if (N == 0) return QG_OK;
  switch (fmt) {
    case QG_FMT_INT4:
      QG_REQUIRE(scales && g >= 32 && (g & (g - 1)) == 0 && K % g == 0, QG_ERR_UNSUPPORTED_SHAPE,
                 "qg_dequant_weights: INT4 needs scales and g a power of two >= 32");
      qg::dequant_kernel<qg::F_INT4><<<grid(128), threads, 0, st>>>(w, scales, nullptr, g, w_out, N, K);
      break;
    case QG_FMT_FP8:
      qg::dequant_kernel<qg::F_FP8><<<grid(64), threads, 0, st>>>(w, scales, nullptr, g, w_out, N, K);
      break;
    case QG_FMT_MXFP4:
      QG_REQUIRE(scales, QG_ERR_INVALID_ARG, "qg_dequant_weights: NULL scales");
      qg::dequant_kernel<qg::F_MXFP4><<<grid(128), threads, 0, st>>>(w, scales, nullptr, 32, w_out, N, K);
      break;
    case QG_FMT_NVFP4:
      QG_REQUIRE(scales, QG_ERR_INVALID_ARG, "qg_dequant_weights: NULL scales");
      qg::dequant_kernel<qg::F_NVFP4><<<grid(128), threads, 0, st>>>(w, scales, nullptr, 16, w_out, N, K);
      break;
    default:
      return qg::set_error(QG_ERR_INVALID_ARG, "qg_dequant_weights: unknown format %d", fmt);
  }
  return qg::check_launch("qg_dequant_weights");
}

qg_status qg_dequant_weights_int4_zp(const uint8_t* w_q, const uint16_t* w_s, const uint8_t* w_z, int g,
                                     uint16_t* w_out, int N, int K, qg_stream_t stream) {
  QG_REQUIRE(w_q && w_s && w_z && w_out, QG_ERR_INVALID_ARG, "qg_dequant_weights_int4_zp: NULL pointer");
  QG_REQUIRE(N >= 0 && K > 0, QG_ERR_INVALID_ARG, "qg_dequant_weights_int4_zp: bad sizes");
  QG_REQUIRE(K % 128 == 0 && g >= 32 && (g & (g - 1)) == 0 && K % g == 0, QG_ERR_UNSUPPORTED_SHAPE,
             "qg_dequant_weights_int4_zp: need K %% 128 == 0 and g a power of two >= 32");
  QG_REQUIRE(aligned16(w_q) && aligned16(w_out), QG_ERR_MISALIGNED, "qg_dequant_weights_int4_zp: misaligned");
  if (N == 0) return QG_OK;
  const int threads = 256;
  const long long lanes = (long long)N * (K / 128) * 4;
  qg::dequant_kernel<qg::F_INT4Z><<<unsigned((lanes + threads - 1) / threads), threads, 0,
                                    reinterpret_cast<cudaStream_t>(stream)>>>(w_q, w_s, w_z, g, w_out, N, K);
  return qg::check_launch("qg_dequant_weights_int4_zp");
}

}  // extern "C"
