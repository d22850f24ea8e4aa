// W4A8 grouped (MoE) GEMM with FP8 group scales on an FP8 x FP8 tensor-core
// matmul (Production-Ready W4A8, "Accurate W4A8 Kernel").
//
// Semantics: y[r,n] = bf16( a_s[r] * cs8[n] * sum_k e4m3(a[r,k]) * w8[n,k] )
// with w8 = E4M3(q[n,k] * s8[n,k/128]) -- the page's per-scale lookup table
// of the 16 products of an FP8 scale with the INT4 values, here formed by
// arithmetic: q * s8 is exact in fp16 (at most 8 significant bits) and one
// cvt.rn.satfinite rounds it to E4M3 (the 1/8 pre-scaling of s8 keeps every
// product inside +-448).  fp32 accumulation; the per-token and per-channel
// scales are applied in the epilogue ("outer vector scaling").
//
// tcgen05.mma.cta_group::1.kind::f8f6f4, E4M3 x E4M3, M = 128 channels,
// N = 256 activation rows, K = 32:
//   A operand  = the E4M3 weights, written by 16 dequant warps into 8 slots of
//                tensor memory (128 k = 32 columns per slot);
//   B operand  = the E4M3 activations, TMA-loaded straight into shared memory
//                in the 128-byte swizzled K-major layout (a 128-k slab is one
//                128-byte row) -- no conversion and no second copy;
//   D          = fp32 accumulator in TMEM columns 0-255.
// Roles: warp 0 TMA for the packed weights (8 stages), warp 1 TMEM + MMA
// issuer, warp 2 TMA for the activations (5 stages), warps 3-18 dequant and
// epilogue, warp 19 scheduler (waits for each slab's operands and publishes
// the ready count the issuer polls, as in the prefill kernel).  One CTA per
// 128-channel x 256-row tile of one expert, located on the device from
// expert_off.  Every wait is bounded.
#include "dequant.cuh"
#include "tc_common.cuh"

namespace qg {

bool make_u8_tmap(CUtensorMap* m, const void* base, int rows, int cols, int box_rows, int box_cols);
bool make_u8_tmap_sw128(CUtensorMap* m, const void* base, int rows, int cols, int box_rows, int box_cols);

namespace {

constexpr int fTW = 128;                 // weight rows per tile (MMA M)
constexpr int fTT = 256;                 // activation rows per tile (MMA N)
constexpr int fBK = 128;                 // k per slab: one 128-byte row of E4M3, one scale group
constexpr int fXStages = 5;              // activation stages (<= fSlots: released through a_empty)
constexpr int fSlots = 8;                // TMEM A slots and packed-weight stages
constexpr int fDeqWarps = 16;
constexpr int fDeq0 = 3;
constexpr int fSchedWarp = fDeq0 + fDeqWarps;
constexpr int fThreads = (fSchedWarp + 1) * 32;
constexpr int fXStage = fTT * fBK;       // 32 KB E4M3 activations
constexpr int fWStage = fTW * fBK / 2;   // 8 KB packed INT4
constexpr uint32_t fTmemCols = 512;
constexpr uint32_t fACol0 = 256;
constexpr uint32_t fACols = fBK / 4;     // 32 columns: 128 E4M3 codes per lane
constexpr uint32_t fDrainCap = 1u << 21;
static_assert(fXStages <= fSlots, "activation stages are released through the A-slot barriers");

struct Fp8sArgs {
  const float* a_s;
  const int32_t* off;
  const uint8_t* s8;                     // [E*N][K/128] E4M3
  const float* cs8;                      // [E*N]
  uint16_t* y;
  int R, E, N, K;
  int tiles_w;
  unsigned int* err;
  uint32_t cap;
};

struct __align__(8) Fp8sTail {
  uint64_t x_full[fXStages];
  uint64_t w_full[fSlots];
  uint64_t w_empty[fSlots];
  uint64_t a_full[fSlots];
  uint64_t a_empty[fSlots];
  uint64_t acc_full;
  uint64_t drain;
  uint32_t tmem_base;
  int abort;
  unsigned int ready;
};

QG_DEVICE uint32_t f16x2_sub_(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}
QG_DEVICE uint32_t f16x2_mul_(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}
// two fp16 (low half first) -> two E4M3 codes (low byte first), RNE, satfinite
QG_DEVICE uint32_t f16x2_to_e4m3x2(uint32_t h2) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f16x2 %0, %1;" : "=h"(r) : "r"(h2));
  return r;
}
// one E4M3 code -> fp16x2 with the value in both halves (exact)
QG_DEVICE uint32_t e4m3_to_f16x2_splat(uint32_t code) {
  uint32_t d;
  const uint16_t two = (uint16_t)(code | (code << 8));
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(d) : "h"(two));
  return d;
}

// 8 INT4 codes (k0..k7, even k in the low nibble) -> 8 E4M3 codes of q * s in
// natural k order (two words).  (1024 + (nib ^ 8)) - 1032 is the exact integer
// q in fp16; q * s is exact (<= 8 significant bits); one rounding to E4M3.
QG_DEVICE void int4x8_to_e4m3x8(uint32_t v, uint32_t s2, uint32_t& lo, uint32_t& hi) {
  uint32_t p[4];
  p[0] = lop3<kLutAndXor>(v, 0x000F000Fu, 0x64086408u);            // (k0, k4)
  p[1] = lop3<kLutAndXor>(v >> 4, 0x000F000Fu, 0x64086408u);       // (k1, k5)
  p[2] = lop3<kLutAndXor>(v >> 8, 0x000F000Fu, 0x64086408u);       // (k2, k6)
  p[3] = lop3<kLutAndXor>(v >> 12, 0x000F000Fu, 0x64086408u);      // (k3, k7)
  uint32_t c[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) c[i] = f16x2_to_e4m3x2(f16x2_mul_(f16x2_sub_(p[i], 0x64086408u), s2));
  // c[i] = [e(k_i), e(k_{i+4})] in its low 16 bits
  const uint32_t t01 = c[0] | (c[1] << 16), t23 = c[2] | (c[3] << 16);
  lo = prmt(t01, t23, 0x6420u);                                    // e(k0) e(k1) e(k2) e(k3)
  hi = prmt(t01, t23, 0x7531u);                                    // e(k4) e(k5) e(k6) e(k7)
}

__global__ void __launch_bounds__(fThreads, 1)
moe_fp8s_kernel(const __grid_constant__ CUtensorMap tmap_a, const __grid_constant__ CUtensorMap tmap_w,
                const Fp8sArgs p) {
  // ---- tile: expert, weight tile, row tile (before any setup) ----
  int tile = blockIdx.x, e = -1, r0 = 0, r_end = 0, wt = 0;
  for (int i = 0; i < p.E; ++i) {
    const int a = __ldg(p.off + i), b = __ldg(p.off + i + 1);
    const int nt = b > a ? (b - a + fTT - 1) / fTT : 0;
    const int cnt = nt * p.tiles_w;
    if (tile < cnt) {
      e = i;
      wt = tile / nt;
      r0 = a + (tile - wt * nt) * fTT;
      r_end = b;
      break;
    }
    tile -= cnt;
  }
  if (e < 0) return;
  const int n0 = wt * fTW;
  const int nslab = p.K / fBK;

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* xs = smem;                                    // [fXStages][32 KB] E4M3, swizzled
  uint8_t* wsm = xs + fXStages * fXStage;                // [fSlots][8 KB] INT4
  Fp8sTail* tl = reinterpret_cast<Fp8sTail*>(wsm + fSlots * fWStage);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < fXStages; ++s) mbar_init(&tl->x_full[s], 1);
    for (int s = 0; s < fSlots; ++s) {
      mbar_init(&tl->w_full[s], 1);
      mbar_init(&tl->w_empty[s], fDeqWarps / 2);
      mbar_init(&tl->a_full[s], fDeqWarps / 2);
      mbar_init(&tl->a_empty[s], 1);
    }
    mbar_init(&tl->acc_full, 1);
    mbar_init(&tl->drain, 1);
    tl->abort = 0;
    tl->ready = 0;
    mbar_fence_init();
    tma_prefetch_desc(&tmap_a);
    tma_prefetch_desc(&tmap_w);
  }
  if (warp == 1) tmem_alloc(&tl->tmem_base, fTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tl->tmem_base;
  volatile int* abort = &tl->abort;

  if (warp == 0) {
    // ---------------- TMA producer: packed weights ----------------
    if (lane == 0) {
      int issued = 0;
      for (int s = 0; s < nslab; ++s) {
        const int st = s % fSlots, r = s / fSlots;
        if (r > 0 && !mbar_wait(&tl->w_empty[st], (r - 1) & 1, p.cap, abort, p.err)) break;
        mbar_arrive_expect_tx(&tl->w_full[st], fWStage);
        tma_load_2d(wsm + st * fWStage, &tmap_w, &tl->w_full[st], s * (fBK / 2), e * p.N + n0);
        issued = s + 1;
      }
      if (*abort) {
        for (int s = max(0, issued - fSlots); s < issued; ++s)
          mbar_wait(&tl->w_full[s % fSlots], (s / fSlots) & 1, fDrainCap, abort, nullptr);
      }
    }
  } else if (warp == 2) {
    // ---------------- TMA producer: E4M3 activations ----------------
    if (lane == 0) {
      int issued = 0;
      for (int s = 0; s < nslab; ++s) {
        const int st = s % fXStages, sp = s - fXStages;   // stage last held slab sp
        if (sp >= 0 && !mbar_wait(&tl->a_empty[sp % fSlots], (sp / fSlots) & 1, p.cap, abort, p.err)) break;
        mbar_arrive_expect_tx(&tl->x_full[st], fXStage);
        tma_load_2d(xs + st * fXStage, &tmap_a, &tl->x_full[st], s * fBK, r0);
        issued = s + 1;
      }
      if (*abort) {
        for (int s = max(0, issued - fXStages); s < issued; ++s)
          mbar_wait(&tl->x_full[s % fXStages], (s / fXStages) & 1, fDrainCap, abort, nullptr);
      }
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer ----------------
    if (lane == 0) {
      // kind::f8f6f4: fp32 D, E4M3 A and B (format 0), both K-major
      const uint32_t idesc = (1u << 4) | ((uint32_t)(fTT >> 3) << 17) | ((uint32_t)(fTW >> 4) << 24);
      bool any = false;
      unsigned int ready = 0;
      for (int s = 0; s < nslab; ++s) {
        const int st = s % fXStages, sa = s % fSlots;
        if (!wait_count(&tl->ready, (unsigned)s, ready, p.cap * 4, abort, p.err)) break;
        tc_fence_after();
        const uint64_t bdesc = sw128_kmajor_desc(smem_addr(xs + st * fXStage));
#pragma unroll
        for (int j = 0; j < fBK / 32; ++j)       // K = 32 per MMA: 32 bytes of each operand row
          asm volatile(
              "{\n .reg .pred p;\n setp.ne.u32 p, %4, 0;\n"
              " tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], [%1], %2, %3, p;\n}"
              :: "r"(tmem), "r"(tmem + fACol0 + sa * fACols + 8 * j), "l"(bdesc + 2 * j), "r"(idesc),
                 "r"((s | j) != 0 ? 1u : 0u)
              : "memory");
        tc_commit(&tl->a_empty[sa]);                   // frees the A slot and the activation stage
        any = true;
      }
      if (!*abort) {
        tc_commit(&tl->acc_full);
      } else if (any) {
        tc_commit(&tl->drain);
        mbar_wait(&tl->drain, 0, fDrainCap, abort, nullptr);
      }
    }
  } else if (warp == fSchedWarp) {
    // ---------------- scheduler ----------------
    if (lane == 0) {
      for (int s = 0; s < nslab; ++s) {
        if (!mbar_wait(&tl->a_full[s % fSlots], (s / fSlots) & 1, p.cap, abort, p.err)) break;
        if (!mbar_wait(&tl->x_full[s % fXStages], (s / fXStages) & 1, p.cap, abort, p.err)) break;
        publish_count(&tl->ready, (unsigned)(s + 1));
      }
    }
  } else {
    // ---------------- dequant producers, then the epilogue ----------------
    // Thread = one weight row (TMEM lane) x one 64-k half of a 128-k slab; the
    // two sets of 8 warps take alternate slabs.  A slab is one scale group.
    const int dw = warp - fDeq0;
    const int q = warp & 3, h = (dw >> 2) & 1, par = dw >> 3;
    const int row = 32 * q + lane;
    const int n = min(n0 + row, p.N - 1);
    const int ng = p.K / fBK;
    const uint8_t* srow = p.s8 + ((size_t)e * p.N + n) * ng;
    const uint32_t lane_base = tmem + ((uint32_t)(32 * q) << 16) + fACol0 + 16 * h;
    uint32_t sc_next = par < nslab ? __ldg(srow + par) : 0u;
    for (int s = par; s < nslab; s += 2) {
      const int sa = s % fSlots, ra = s / fSlots;
      const uint32_t s2 = e4m3_to_f16x2_splat(sc_next);
      if (s + 2 < nslab) sc_next = __ldg(srow + s + 2);
      if (!mbar_wait_warp(&tl->w_full[sa], ra & 1, p.cap, abort, p.err)) break;
      const uint8_t* wrow = wsm + sa * fWStage + row * (fBK / 2) + 32 * h;
      const uint4 wa = *reinterpret_cast<const uint4*>(wrow);
      const uint4 wb = *reinterpret_cast<const uint4*>(wrow + 16);
      const uint32_t v[8] = {wa.x, wa.y, wa.z, wa.w, wb.x, wb.y, wb.z, wb.w};
      uint32_t out[16];
#pragma unroll
      for (int j = 0; j < 8; ++j) int4x8_to_e4m3x8(v[j], s2, out[2 * j], out[2 * j + 1]);
      mbar_arrive_warp(&tl->w_empty[sa]);           // packed slab decoded: its stage may be refilled
      if (ra > 0) {
        if (!mbar_wait_warp(&tl->a_empty[sa], (ra - 1) & 1, p.cap, abort, p.err)) break;
        tc_fence_after();
      }
      tmem_st16(lane_base + sa * fACols, out);
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive_warp(&tl->a_full[sa]);
    }

    // epilogue: warp covers lane quarter q and 64 of the 256 activation rows
    const int cq = dw >> 2;
    if (mbar_wait_warp(&tl->acc_full, 0, p.cap, abort, p.err)) {
      tc_fence_after();
      const int nn = n0 + row;
      const float cs = nn < p.N ? __ldg(p.cs8 + (size_t)e * p.N + nn) : 0.f;
#pragma unroll 1
      for (int i = 0; i < 2; ++i) {
        uint32_t v[32];
        tmem_ld32(tmem + ((uint32_t)(32 * q) << 16) + 64 * cq + 32 * i, v);
        tmem_wait_ld();
        const int mb = r0 + 64 * cq + 32 * i;
        if (nn < p.N) {
#pragma unroll
          for (int c = 0; c < 32; ++c) {
            const int m = mb + c;
            if (m < r_end) p.y[(size_t)m * p.N + nn] = f32_to_bf16_bits(__uint_as_float(v[c]) * __ldg(p.a_s + m) * cs);
          }
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, fTmemCols);
  }
}

}  // namespace

}  // namespace qg

extern "C" qg_status qgemm_w4a8_grouped_fp8s(const uint8_t* a_e4m3, const float* a_s, const int32_t* expert_off,
                                             const uint8_t* w_q, const uint8_t* w_s8, const float* w_cs8,
                                             uint16_t* y, int R, int E, int N, int K, qg_stream_t stream) {
  using namespace qg;
  if (!(a_e4m3 && a_s && expert_off && w_q && w_s8 && w_cs8 && y))
    return set_error(QG_ERR_INVALID_ARG, "qgemm_w4a8_grouped_fp8s: NULL pointer");
  if (!(R >= 0 && E >= 1 && N > 0 && K > 0)) return set_error(QG_ERR_INVALID_ARG, "qgemm_w4a8_grouped_fp8s: bad sizes");
  if (!(K % fBK == 0 && N % 16 == 0))
    return set_error(QG_ERR_UNSUPPORTED_SHAPE, "qgemm_w4a8_grouped_fp8s: need K %% 128 == 0 and N %% 16 == 0");
  if (!(aligned16(a_e4m3) && aligned16(w_q) && aligned16(y)))
    return set_error(QG_ERR_MISALIGNED, "qgemm_w4a8_grouped_fp8s: misaligned pointer");
  if (R == 0) return QG_OK;
  CUtensorMap tmap_a, tmap_w;
  if (!make_u8_tmap_sw128(&tmap_a, a_e4m3, R, K, fTT, fBK))
    return set_error(QG_ERR_CUDA, "qgemm_w4a8_grouped_fp8s: cannot encode the activation tensor map");
  if (!make_u8_tmap(&tmap_w, w_q, E * N, K / 2, fTW, fBK / 2))
    return set_error(QG_ERR_CUDA, "qgemm_w4a8_grouped_fp8s: cannot encode the weight tensor map");
  unsigned int* err = device_error_word();
  if (!err) return set_error(QG_ERR_CUDA, "qgemm_w4a8_grouped_fp8s: no device error word");
  Fp8sArgs a{};
  a.a_s = a_s; a.off = expert_off; a.s8 = w_s8; a.cs8 = w_cs8; a.y = y;
  a.R = R; a.E = E; a.N = N; a.K = K;
  a.tiles_w = (N + fTW - 1) / fTW;
  a.err = err;
  a.cap = wait_limit();
  const int smem = fXStages * fXStage + fSlots * fWStage + (int)sizeof(Fp8sTail) + 1024;
  if (!ensure_smem(moe_fp8s_kernel, smem)) return set_error(QG_ERR_CUDA, "qgemm_w4a8_grouped_fp8s: smem attribute");
  const long long tiles = ((long long)(R + fTT - 1) / fTT + E) * a.tiles_w;
  moe_fp8s_kernel<<<(unsigned)tiles, fThreads, smem, reinterpret_cast<cudaStream_t>(stream)>>>(tmap_a, tmap_w, a);
  return check_launch("qgemm_w4a8_grouped_fp8s");
}
