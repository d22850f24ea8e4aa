// W4A8 grouped (MoE) GEMM with exact bf16 group scales on the fp16 tensor
// cores, for both forms of the activations: E4M3 codes (qgemm_w4a8_grouped,
// from 256 rows) and fp16 re-encodings of those codes handed over by the
// caller (qgemm_w4a8_grouped_f16act).
//
// Semantics (Production-Ready W4A8): y[r,n] = a_s[r] * sum_k e4m3(a[r,k]) *
// q[n,k] * s[n,k/128], every product exact, fp32 accumulation, one bf16
// rounding at the store.  Every E4M3 value is exact in fp16, so the fp16
// form of the activations is a lossless encoding and both forms give the
// same bits.  The weights are formed as fp16(q * s * 2^e_n) -- exact: q * s
// has at most 11 significant bits, and the per-row power of two e_n puts the
// row's largest scale in [2^11, 2^12) -- and the epilogue multiplies by
// 2^-e_n and the token scale.  No per-group promotion is needed.
//
// tcgen05.mma.cta_group::1.kind::f16 (fp16 A and B), M = 128 channels,
// N = 256 activation rows, K = 16:
//   A operand  = the fp16 weights, written by 16 dequant warps into 8 slots
//                of tensor memory (64 k = 32 columns per slot);
//   B operand  = the fp16 activations in the 128-byte swizzled K-major
//                layout (64 k per 128-byte row, 32 KB per stage): TMA-loaded
//                as they are (fp16 input, 6 stages), or converted from the
//                E4M3 codes by the dequant sets (E4M3 input, 4 stages, the
//                codes TMA-loaded into a 4-stage staging ring);
//   D          = fp32 accumulator in TMEM columns 0-255.
// Persistent, one CTA per SM over the (expert, 128-channel block, 256-row
// block) tile list with row blocks inner, the rings running on across tiles
// and the epilogue of a tile overlapping the next tile's MMAs.  Roles: warp 0
// TMA for the packed weights, warp 1 TMEM + MMA issuer, warp 2 TMA for the
// activations, warps 3-18 dequant (four sets of four, one warp per TMEM lane
// quarter, a thread decoding its row's 64-k slab, each set taking every
// fourth slab; with E4M3 input the set also converts its slab's codes) and
// the epilogue, warp 19 scheduler (waits for each slab's operands and
// publishes the ready count the issuer polls).  Every wait is bounded.
#include <algorithm>

#include "dequant.cuh"
#include "tc_common.cuh"

namespace qg {

bool make_u8_tmap(CUtensorMap* m, const void* base, int rows, int cols, int box_rows, int box_cols);
bool make_bf16_tmap(CUtensorMap* m, const void* base, int rows, int cols, int box_rows, int box_cols);
bool make_u8_tmap_swizzled(CUtensorMap* m, const void* base, int rows, int cols, int box_rows, int box_cols);

namespace {

constexpr int hTW = 128;                 // weight rows per tile (MMA M)
constexpr int hTT = 256;                 // activation rows per tile (MMA N)
constexpr int hBK = 64;                  // k per slab: one 128-byte row of fp16
constexpr int hXStages = 6;              // activation stages (<= hSlots: released through a_empty)
constexpr int hXStagesE = 4;             // fp16 stages written by the dequant sets (E4M3 input)
constexpr int hEStages = 4;              // E4M3 staging stages (E4M3 input)
constexpr int hSlots = 8;                // TMEM A slots (and packed-weight stages, fp16 input)
constexpr int hWStagesE = 4;             // packed-weight stages, E4M3 input
constexpr int hDeqWarps = 16;            // four sets of 4 (one per TMEM lane quarter)
constexpr int hDeqSet = 4;
constexpr int hDeqSets = hDeqWarps / hDeqSet;
constexpr int hDeq0 = 3;
constexpr int hSchedWarp = hDeq0 + hDeqWarps;
constexpr int hThreads = (hSchedWarp + 1) * 32;
constexpr int hXStage = hTT * hBK * 2;   // 32 KB fp16 activations
constexpr int hWStage = hTW * hBK / 2;   // 4 KB packed INT4
constexpr int hEStage = hTT * hBK;       // 16 KB E4M3 activations (64-byte swizzled rows)
constexpr uint32_t hTmemCols = 512;
constexpr uint32_t hACol0 = 256;
constexpr uint32_t hACols = hBK / 2;     // 32 columns: 64 fp16 per lane
constexpr uint32_t hDrainCap = 1u << 21;
static_assert(hXStages <= hSlots && hXStagesE <= hSlots, "activation stages are released through the A-slot barriers");
// E4M3 input: the set converting slab g waits on staging stage g % hEStages
// for the phase of slab g.  A parity wait is only sound if the stage's
// previous phase (slab g - hEStages) has completed, and that is guaranteed
// only when the same set converted slab g - hEStages: with 4 sets and 3
// staging stages a set can pass the wait on the previous phase's parity and
// the phases of the barrier pair mix (a build with 3 stages faulted).
static_assert(hEStages % hDeqSets == 0, "E4M3 staging ring: a multiple of the dequant sets");
static_assert(hWStagesE % hDeqSets == 0 && hSlots % hDeqSets == 0, "packed-weight ring: the same rule");

struct F16Args {
  const float* a_s;
  const int32_t* off;
  const uint16_t* ws;                    // [E*N][K/128] bf16
  const int8_t* we;                      // [E*N] row exponent shifts (qg_w4a8_row_shifts) or nullptr
  uint16_t* y;
  int R, E, N, K;
  int tiles_w;
  unsigned int* err;
  uint32_t cap;
};

struct __align__(8) F16Tail {
  uint64_t x_full[hXStages];
  uint64_t w_full[hSlots];                // the first nW used
  uint64_t w_empty[hSlots];
  uint64_t a_full[hSlots];
  uint64_t a_empty[hSlots];
  uint64_t e_full[hEStages];             // E4M3 input: staging stage loaded
  uint64_t e_empty[hEStages];            // E4M3 input: staging stage converted
  uint64_t acc_full;
  uint64_t acc_empty;
  uint64_t drain;
  uint32_t tmem_base;
  int abort;
  unsigned int ready;
};

struct HTile {
  int e, r0, r_end, n0;
};
QG_DEVICE void expert_rows(const F16Args& p, int i, int& a, int& b) {
  a = min(max(__ldg(p.off + i), 0), p.R);
  b = min(max(__ldg(p.off + i + 1), a), p.R);
}
QG_DEVICE int tile_count(const F16Args& p) {
  int n = 0;
  for (int i = 0; i < p.E; ++i) {
    int a, b;
    expert_rows(p, i, a, b);
    n += (b - a + hTT - 1) / hTT * p.tiles_w;
  }
  return n;
}
QG_DEVICE HTile tile_at(const F16Args& p, int t) {
  for (int i = 0; i < p.E; ++i) {
    int a, b;
    expert_rows(p, i, a, b);
    const int nt = (b - a + hTT - 1) / hTT;
    const int cnt = nt * p.tiles_w;
    if (t < cnt) {
      const int wt = t / nt;
      return HTile{i, a + (t - wt * nt) * hTT, b, wt * hTW};
    }
    t -= cnt;
  }
  return HTile{0, 0, 0, 0};
}

// Per-row power of two: the row's largest |scale| lands in [2^11, 2^12), so
// every fp16 product q * s * 2^ex is exact and in range.  A group scale more
// than 2^24 below its row's largest would turn subnormal in fp16; RTN scales
// of one weight row never spread that far.
QG_DEVICE int row_exponent(const uint16_t* srow, int ng) {
  float smax = 0.f;
  int i = 0;
  if ((reinterpret_cast<uintptr_t>(srow) & 15u) == 0) {
    for (; i + 8 <= ng; i += 8) {
      const uint4 u = __ldg(reinterpret_cast<const uint4*>(srow + i));
      const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
      for (int c = 0; c < 4; ++c)
        smax = fmaxf(smax, fmaxf(fabsf(bf16_lo_to_f32(w[c])), fabsf(bf16_hi_to_f32(w[c]))));
    }
  }
  for (; i < ng; ++i) smax = fmaxf(smax, fabsf(bf16_bits_to_f32(__ldg(srow + i))));
  if (!(smax > 0.f)) return 0;
  int e2;
  frexpf(smax, &e2);                       // smax = m * 2^e2, m in [0.5, 1)
  return min(max(12 - e2, -100), 100);
}

// kE8: the activations arrive as E4M3 codes.  warp 2 then TMA-loads them
// into a 64-byte swizzled staging ring, and the dequant set that writes slab
// g's A slot also converts slab g's codes to fp16 (exact) into the 128-byte
// swizzled B layout, once slab g - hXStagesE's MMAs have released the stage;
// its A-slot arrival then covers both operands.
template <bool kE8>
__global__ void __launch_bounds__(hThreads, 1)
moe_f16_kernel(const __grid_constant__ CUtensorMap tmap_a, const __grid_constant__ CUtensorMap tmap_w,
               const F16Args p) {
  constexpr int nX = kE8 ? hXStagesE : hXStages;
  // how far a dequant set may produce into tile e + 1 before the epilogue of
  // tile e: its waits reach back hSlots slabs (A slot), with E4M3 input nX
  // (fp16 stage), and must not wait on MMAs of tile e + 1
  constexpr int kRun = kE8 ? nX : hSlots;
  constexpr int nW = kE8 ? hWStagesE : hSlots;           // packed-weight stages
  const int ntiles_total = tile_count(p);
  const int ntiles = ((int)blockIdx.x < ntiles_total)
                         ? (ntiles_total - (int)blockIdx.x + (int)gridDim.x - 1) / (int)gridDim.x : 0;
  if (ntiles == 0) return;
  const int nslab = p.K / hBK;
  const int total = ntiles * nslab;
  auto tile_of = [&](int i) { return tile_at(p, (int)blockIdx.x + i * (int)gridDim.x); };

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* xs = smem;                                    // [nX][32 KB] fp16, swizzled
  uint8_t* es = xs + nX * hXStage;                       // E4M3 input: [hEStages][16 KB]
  uint8_t* wsm = es + (kE8 ? hEStages * hEStage : 0);    // [nW][4 KB] INT4
  F16Tail* tl = reinterpret_cast<F16Tail*>(wsm + nW * hWStage);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < hXStages; ++s) mbar_init(&tl->x_full[s], 1);
    for (int s = 0; s < hEStages; ++s) {
      mbar_init(&tl->e_full[s], 1);
      mbar_init(&tl->e_empty[s], hDeqSet);
    }
    for (int s = 0; s < hSlots; ++s) {
      mbar_init(&tl->w_full[s], 1);
      mbar_init(&tl->w_empty[s], hDeqSet);
      mbar_init(&tl->a_full[s], hDeqSet);
      mbar_init(&tl->a_empty[s], 1);
    }
    mbar_init(&tl->acc_full, 1);
    mbar_init(&tl->acc_empty, hDeqWarps);
    mbar_init(&tl->drain, 1);
    tl->abort = 0;
    tl->ready = 0;
    mbar_fence_init();
    tma_prefetch_desc(&tmap_a);
    tma_prefetch_desc(&tmap_w);
  }
  if (warp == 1) tmem_alloc(&tl->tmem_base, hTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tl->tmem_base;
  volatile int* abort = &tl->abort;

  if (warp == 0) {
    // ---------------- TMA producer: packed weights ----------------
    if (lane == 0) {
      int issued = 0, s = 0, i = 0;
      HTile t = tile_of(0);
      for (int g = 0; g < total; ++g, ++s) {
        if (s == nslab) { s = 0; t = tile_of(++i); }
        const int st = g % nW, r = g / nW;
        if (r > 0 && !mbar_wait(&tl->w_empty[st], (r - 1) & 1, p.cap, abort, p.err)) break;
        mbar_arrive_expect_tx(&tl->w_full[st], hWStage);
        tma_load_2d(wsm + st * hWStage, &tmap_w, &tl->w_full[st], s * (hBK / 2), t.e * p.N + t.n0);
        issued = g + 1;
      }
      if (*abort) {
        for (int g = max(0, issued - nW); g < issued; ++g)
          mbar_drain(&tl->w_full[g % nW], (g / nW) & 1, hDrainCap);
      }
    }
  } else if (warp == 2 && kE8) {
    // ---------------- TMA producer: E4M3 activations ----------------
    if (lane == 0) {
      int issued = 0, s = 0, i = 0;
      HTile t = tile_of(0);
      for (int g = 0; g < total; ++g, ++s) {
        if (s == nslab) { s = 0; t = tile_of(++i); }
        const int st = g % hEStages, r = g / hEStages;
        if (r > 0 && !mbar_wait(&tl->e_empty[st], (r - 1) & 1, p.cap, abort, p.err)) break;
        mbar_arrive_expect_tx(&tl->e_full[st], hEStage);
        tma_load_2d(es + st * hEStage, &tmap_a, &tl->e_full[st], s * hBK, t.r0);
        issued = g + 1;
      }
      if (*abort) {
        for (int g = max(0, issued - hEStages); g < issued; ++g)
          mbar_drain(&tl->e_full[g % hEStages], (g / hEStages) & 1, hDrainCap);
      }
    }
  } else if (warp == 2) {
    // ---------------- TMA producer: fp16 activations ----------------
    if (lane == 0) {
      int issued = 0, s = 0, i = 0;
      HTile t = tile_of(0);
      for (int g = 0; g < total; ++g, ++s) {
        if (s == nslab) { s = 0; t = tile_of(++i); }
        const int st = g % hXStages, gp = g - hXStages;   // stage last held slab gp
        if (gp >= 0 && !mbar_wait(&tl->a_empty[gp % hSlots], (gp / hSlots) & 1, p.cap, abort, p.err)) break;
        mbar_arrive_expect_tx(&tl->x_full[st], hXStage);
        tma_load_2d(xs + st * hXStage, &tmap_a, &tl->x_full[st], s * hBK, t.r0);
        issued = g + 1;
      }
      if (*abort) {
        for (int g = max(0, issued - hXStages); g < issued; ++g)
          mbar_drain(&tl->x_full[g % hXStages], (g / hXStages) & 1, hDrainCap);
      }
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer ----------------
    if (lane == 0) {
      const uint32_t idesc = idesc_f16_f32(hTW, hTT);
      bool any = false;
      unsigned int ready = 0;
      int g = 0;
      for (int i = 0; i < ntiles && !*abort; ++i) {
        if (i > 0) {              // the accumulator is free once the epilogue has read the previous tile
          if (!mbar_wait(&tl->acc_empty, (i - 1) & 1, p.cap, abort, p.err)) break;
          tc_fence_after();
        }
        bool ok = true;
        for (int s = 0; s < nslab; ++s, ++g) {
          const int st = g % nX, sa = g % hSlots;
          if (!wait_count(&tl->ready, (unsigned)g, ready, p.cap * 4, abort, p.err)) { ok = false; break; }
          tc_fence_after();
          const uint64_t bdesc = sw128_kmajor_desc(smem_addr(xs + st * hXStage));
#pragma unroll
          for (int j = 0; j < hBK / 16; ++j)
            tc_mma_ts(tmem, tmem + hACol0 + sa * hACols + 8 * j, bdesc + 2 * j, idesc, (s | j) != 0);
          tc_commit(&tl->a_empty[sa]);                   // frees the A slot and the activation stage
          any = true;
        }
        if (!ok) break;
        tc_commit(&tl->acc_full);
      }
      if (*abort && any) {
        tc_commit(&tl->drain);
        mbar_drain(&tl->drain, 0, hDrainCap);
      }
    }
  } else if (warp == hSchedWarp) {
    // ---------------- scheduler ----------------
    if (lane == 0) {
      for (int g = 0; g < total; ++g) {
        if (!mbar_wait(&tl->a_full[g % hSlots], (g / hSlots) & 1, p.cap, abort, p.err)) break;
        if (!kE8 && !mbar_wait(&tl->x_full[g % hXStages], (g / hXStages) & 1, p.cap, abort, p.err)) break;
        publish_count(&tl->ready, (unsigned)(g + 1));
      }
    }
  } else {
    // ---------------- dequant producers, then the epilogues ----------------
    // The epilogue of tile e runs once this warp is about to produce the slab
    // hSlots past the start of tile e+1 (no slot it needs is then held by a
    // tile-(e+1) MMA, which waits for the epilogue).
    const int dw = warp - hDeq0;
    const int q = warp & 3, set = dw >> 2;
    const int row = 32 * q + lane;
    const int cq = set;                              // epilogue: 64 of the 256 activation rows
    const int ng = p.K / 128;
    const uint32_t lane_base = tmem + ((uint32_t)(32 * q) << 16) + hACol0;
    // scale cursor: tile index, slab in the tile, this thread's scale row and
    // the row's fp16 exponent shift for that tile
    struct Cur { int i, s; const uint16_t* srow; float up; };
    auto set_row = [&](Cur& c) {
      if (c.i < ntiles) {
        const HTile t = tile_of(c.i);
        const size_t r = (size_t)t.e * p.N + min(t.n0 + row, p.N - 1);
        c.srow = p.ws + r * ng;
        c.up = ldexpf(1.f, p.we ? (int)__ldg(p.we + r) : row_exponent(c.srow, ng));
      }
    };
    auto advance = [&](Cur& c, int by) {
      c.s += by;
      while (c.s >= nslab) { c.s -= nslab; ++c.i; set_row(c); }
    };
    // fp16x2 splat of fp16(s * 2^e) for the slab's group (exact)
    auto scale_of = [&](const Cur& c) -> uint32_t {
      if (c.i >= ntiles) return 0u;
      return bf16x2_splat(f32_to_f16_bits(bf16_bits_to_f32(__ldg(c.srow + ((c.s * hBK) >> 7))) * c.up));
    };
    auto epilogue = [&](int e) -> bool {
      if (!mbar_wait_warp(&tl->acc_full, e & 1, p.cap, abort, p.err)) return false;
      tc_fence_after();
      const HTile t = tile_of(e);
      const int nn = t.n0 + row;
      const int mb = t.r0 + 64 * cq;
      const size_t rr = (size_t)t.e * p.N + min(nn, p.N - 1);
      const float down = ldexpf(1.f, -(p.we ? (int)__ldg(p.we + rr) : row_exponent(p.ws + rr * ng, ng)));
      const float as_lo = mb + lane < t.r_end ? __ldg(p.a_s + mb + lane) : 0.f;
      const float as_hi = mb + 32 + lane < t.r_end ? __ldg(p.a_s + mb + 32 + lane) : 0.f;
      uint32_t packed[32];
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        uint32_t v[32];
        tmem_ld32(tmem + ((uint32_t)(32 * q) << 16) + 64 * cq + 32 * i, v);
        tmem_wait_ld();
        const float as = i ? as_hi : as_lo;
#pragma unroll
        for (int c = 0; c < 16; ++c) {
          const float lo = __uint_as_float(v[2 * c]) * down * __shfl_sync(0xffffffffu, as, 2 * c);
          const float hi = __uint_as_float(v[2 * c + 1]) * down * __shfl_sync(0xffffffffu, as, 2 * c + 1);
          packed[16 * i + c] = f32_to_bf16_bits(lo) | (f32_to_bf16_bits(hi) << 16);
        }
      }
      tc_fence_before();
      mbar_arrive_warp(&tl->acc_empty);              // the next tile's MMAs may overwrite it
      // lanes 2i, 2i+1 (channels n, n+1) swap halves: 4-byte stores
      const bool odd = lane & 1;
      const uint32_t sel = odd ? 0x3276u : 0x5410u;
      const int n2 = nn & ~1;                        // N is even: a pair is in range or out as a whole
#pragma unroll
      for (int c = 0; c < 32; ++c) {
        const uint32_t w = prmt(packed[c], __shfl_xor_sync(0xffffffffu, packed[c], 1), sel);
        const int m = mb + 2 * c + (odd ? 1 : 0);
        if (n2 < p.N && m < t.r_end) *reinterpret_cast<uint32_t*>(p.y + (size_t)m * p.N + n2) = w;
      }
      return true;
    };
    int e_next = 0;
    bool ok = true;
    Cur pf{0, 0, nullptr, 1.f};
    set_row(pf);
    advance(pf, set);
    uint32_t sc_cur = scale_of(pf);
    advance(pf, hDeqSets);
    uint32_t sc_nxt = scale_of(pf);
    for (int g = set; g < total; g += hDeqSets) {
      while (e_next < ntiles - 1 && g >= (e_next + 1) * nslab + kRun) {
        if (!(ok = epilogue(e_next))) break;
        ++e_next;
      }
      if (!ok) break;
      const int sa = g % hSlots, ra = g / hSlots, sw = g % nW;
      const uint32_t s2 = sc_cur;
      sc_cur = sc_nxt;
      advance(pf, hDeqSets);                         // pf now at this set's slab after the next
      sc_nxt = scale_of(pf);
      if (!mbar_wait_warp(&tl->w_full[sw], (g / nW) & 1, p.cap, abort, p.err)) { ok = false; break; }
      const uint4 wa = *reinterpret_cast<const uint4*>(wsm + sw * hWStage + row * (hBK / 2));
      const uint4 wb = *reinterpret_cast<const uint4*>(wsm + sw * hWStage + row * (hBK / 2) + 16);
      const uint32_t v[8] = {wa.x, wa.y, wa.z, wa.w, wb.x, wb.y, wb.z, wb.w};
      uint32_t out[32];
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        uint32_t nat[4];
        int4x8_nat_f16(v[j], s2, nat);
        out[4 * j + 0] = nat[0]; out[4 * j + 1] = nat[1];
        out[4 * j + 2] = nat[2]; out[4 * j + 3] = nat[3];
      }
      mbar_arrive_warp(&tl->w_empty[sw]);            // packed slab decoded: its stage may be refilled
      if (kE8) {
        // slab g - nX's MMAs complete (and with them slab g - hSlots's): the
        // fp16 stage and the A slot are both free
        if (g >= nX) {
          const int gp = g - nX;
          if (!mbar_wait_warp(&tl->a_empty[gp % hSlots], (gp / hSlots) & 1, p.cap, abort, p.err)) { ok = false; break; }
          tc_fence_after();
        }
      } else if (ra > 0) {
        if (!mbar_wait_warp(&tl->a_empty[sa], (ra - 1) & 1, p.cap, abort, p.err)) { ok = false; break; }
        tc_fence_after();
      }
      {
        const uint32_t (&o0)[16] = *reinterpret_cast<const uint32_t(*)[16]>(&out[0]);
        const uint32_t (&o1)[16] = *reinterpret_cast<const uint32_t(*)[16]>(&out[16]);
        tmem_st16(lane_base + sa * hACols, o0);
        tmem_st16(lane_base + sa * hACols + 16, o1);
      }
      if (kE8) {
        // slab g's E4M3 codes -> fp16 B stage.  Task (row r, 16 codes j): the
        // codes are chunk j of r's 64-byte staging row (64-byte swizzle: at
        // chunk j ^ ((r >> 1) & 3)); their fp16 values are chunks 2j, 2j + 1
        // of r's 128-byte B row (128-byte swizzle: chunk c at c ^ (r & 7)).
        // Eight consecutive lanes take eight consecutive rows: conflict-free.
        const int se = g % hEStages;
        if (!mbar_wait_warp(&tl->e_full[se], (g / hEStages) & 1, p.cap, abort, p.err)) {
          tmem_wait_st();
          ok = false;
          break;
        }
        const uint8_t* eb = es + se * hEStage;
        uint8_t* xb = xs + (g % nX) * hXStage;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const int j = i & 3, r = 128 * (i >> 2) + row;
          const uint4 c = *reinterpret_cast<const uint4*>(eb + r * hBK + 16 * (j ^ ((r >> 1) & 3)));
          const uint4 lo = make_uint4(e4m3x2_to_f16x2(c.x), e4m3x2_to_f16x2(c.x >> 16),
                                      e4m3x2_to_f16x2(c.y), e4m3x2_to_f16x2(c.y >> 16));
          const uint4 hi = make_uint4(e4m3x2_to_f16x2(c.z), e4m3x2_to_f16x2(c.z >> 16),
                                      e4m3x2_to_f16x2(c.w), e4m3x2_to_f16x2(c.w >> 16));
          *reinterpret_cast<uint4*>(xb + r * 2 * hBK + 16 * ((2 * j) ^ (r & 7))) = lo;
          *reinterpret_cast<uint4*>(xb + r * 2 * hBK + 16 * ((2 * j + 1) ^ (r & 7))) = hi;
        }
        fence_proxy_async_smem();                    // the tensor core reads the stage through the async proxy
        mbar_arrive_warp(&tl->e_empty[se]);
      }
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive_warp(&tl->a_full[sa]);
    }
    while (ok && e_next < ntiles) {
      if (!(ok = epilogue(e_next))) break;
      ++e_next;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, hTmemCols);
  }
}

// Row exponent shifts for qgemm_w4a8_grouped_f16act, one warp per row.
__global__ void row_shifts_kernel(const uint16_t* __restrict__ ws, int8_t* __restrict__ we, int rows, int G) {
  const long long row = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (row >= rows) return;
  const uint16_t* src = ws + row * G;
  float m = 0.f;
  for (int g = lane; g < G; g += 32) m = fmaxf(m, fabsf(bf16_bits_to_f32(src[g])));
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  if (lane == 0) {
    int ex = 0;
    if (m > 0.f) {
      int e2;
      frexpf(m, &e2);
      ex = min(max(12 - e2, -100), 100);
    }
    we[row] = (int8_t)ex;
  }
}

// E4M3 codes -> fp16 values (exact), 8 per thread
__global__ void e4m3_to_f16_kernel(const uint8_t* __restrict__ q, uint16_t* __restrict__ out, long long n8) {
  const long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x;
  if (i >= n8) return;
  const uint2 c = __ldg(reinterpret_cast<const uint2*>(q) + i);
  const uint4 h = make_uint4(e4m3x2_to_f16x2(c.x & 0xFFFFu), e4m3x2_to_f16x2(c.x >> 16),
                             e4m3x2_to_f16x2(c.y & 0xFFFFu), e4m3x2_to_f16x2(c.y >> 16));
  reinterpret_cast<uint4*>(out)[i] = h;
}

}  // namespace

}  // namespace qg

extern "C" qg_status qgemm_w4a8_grouped_f16act(const uint16_t* a_f16, const float* a_s, const int32_t* expert_off,
                                               const uint8_t* w_q, const uint16_t* w_s, const int8_t* w_e, int g,
                                               uint16_t* y, int R, int E, int N, int K, qg_stream_t stream) {
  using namespace qg;
  if (!(a_f16 && a_s && expert_off && w_q && w_s && y))
    return set_error(QG_ERR_INVALID_ARG, "qgemm_w4a8_grouped_f16act: NULL pointer");
  if (!(R >= 0 && E >= 1 && N > 0 && K > 0))
    return set_error(QG_ERR_INVALID_ARG, "qgemm_w4a8_grouped_f16act: bad sizes");
  if (!(g == 128 && K % 128 == 0 && N % 16 == 0))
    return set_error(QG_ERR_UNSUPPORTED_SHAPE, "qgemm_w4a8_grouped_f16act: need g == 128, K %% 128 == 0, N %% 16 == 0");
  if (!(aligned16(a_f16) && aligned16(w_q) && aligned16(y)))
    return set_error(QG_ERR_MISALIGNED, "qgemm_w4a8_grouped_f16act: misaligned pointer");
  if (R == 0) return QG_OK;
  CUtensorMap tmap_a, tmap_w;
  if (!make_bf16_tmap(&tmap_a, a_f16, R, K, hTT, hBK))     // a 16-bit copy: the element type is not read
    return set_error(QG_ERR_CUDA, "qgemm_w4a8_grouped_f16act: cannot encode the activation tensor map");
  if (!make_u8_tmap(&tmap_w, w_q, E * N, K / 2, hTW, hBK / 2))
    return set_error(QG_ERR_CUDA, "qgemm_w4a8_grouped_f16act: cannot encode the weight tensor map");
  unsigned int* err = device_error_word();
  if (!err) return set_error(QG_ERR_CUDA, "qgemm_w4a8_grouped_f16act: no device error word");
  F16Args a{};
  a.a_s = a_s; a.off = expert_off; a.ws = w_s; a.we = w_e; a.y = y;
  a.R = R; a.E = E; a.N = N; a.K = K;
  a.tiles_w = (N + hTW - 1) / hTW;
  a.err = err;
  a.cap = wait_limit();
  const int smem = hXStages * hXStage + hSlots * hWStage + (int)sizeof(F16Tail) + 1024;
  if (!ensure_smem(moe_f16_kernel<false>, smem))
    return set_error(QG_ERR_CUDA, "qgemm_w4a8_grouped_f16act: smem attribute");
  const long long bound = ((long long)(R + hTT - 1) / hTT + E) * a.tiles_w;
  const int grid = (int)std::min<long long>(bound, (long long)sm_count());
  moe_f16_kernel<false><<<grid, hThreads, smem, reinterpret_cast<cudaStream_t>(stream)>>>(tmap_a, tmap_w, a);
  return check_launch("qgemm_w4a8_grouped_f16act");
}

namespace qg {
// The E4M3-activation entry qgemm_w4a8_grouped on the same kernel, converting
// the codes to fp16 in shared memory (arguments validated by the caller:
// g == 128, K % 128 == 0, N % 16 == 0, 16-byte aligned pointers).  The
// result is bit-identical to qgemm_w4a8_grouped_f16act on the fp16 copy.
qg_status moe_w4a8_e4m3_f16(const uint8_t* a_e4m3, const float* a_s, const int32_t* expert_off, const uint8_t* w_q,
                            const uint16_t* w_s, uint16_t* y, int R, int E, int N, int K, cudaStream_t st) {
  CUtensorMap tmap_a, tmap_w;
  if (!make_u8_tmap_swizzled(&tmap_a, a_e4m3, R, K, hTT, hBK))      // 64-byte rows: 64-byte swizzle
    return set_error(QG_ERR_CUDA, "qgemm_w4a8_grouped: cannot encode the activation tensor map");
  if (!make_u8_tmap(&tmap_w, w_q, E * N, K / 2, hTW, hBK / 2))
    return set_error(QG_ERR_CUDA, "qgemm_w4a8_grouped: cannot encode the weight tensor map");
  unsigned int* err = device_error_word();
  if (!err) return set_error(QG_ERR_CUDA, "qgemm_w4a8_grouped: no device error word");
  F16Args a{};
  a.a_s = a_s; a.off = expert_off; a.ws = w_s; a.we = nullptr; a.y = y;
  a.R = R; a.E = E; a.N = N; a.K = K;
  a.tiles_w = (N + hTW - 1) / hTW;
  a.err = err;
  a.cap = wait_limit();
  const int smem = hXStagesE * hXStage + hEStages * hEStage + hWStagesE * hWStage + (int)sizeof(F16Tail) + 1024;
  if (!ensure_smem(moe_f16_kernel<true>, smem)) return set_error(QG_ERR_CUDA, "qgemm_w4a8_grouped: smem attribute");
  const long long bound = ((long long)(R + hTT - 1) / hTT + E) * a.tiles_w;
  const int grid = (int)std::min<long long>(bound, (long long)sm_count());
  moe_f16_kernel<true><<<grid, hThreads, smem, st>>>(tmap_a, tmap_w, a);
  return check_launch("qgemm_w4a8_grouped (tcgen05, E4M3 converted in shared memory)");
}
}  // namespace qg

extern "C" qg_status qg_w4a8_row_shifts(const uint16_t* w_s, int8_t* w_e, int rows, int G, qg_stream_t stream) {
  using namespace qg;
  if (!(w_s && w_e)) return set_error(QG_ERR_INVALID_ARG, "qg_w4a8_row_shifts: NULL pointer");
  if (!(rows >= 0 && G > 0)) return set_error(QG_ERR_INVALID_ARG, "qg_w4a8_row_shifts: bad sizes");
  if (rows == 0) return QG_OK;
  const long long threads = (long long)rows * 32;
  row_shifts_kernel<<<unsigned((threads + 255) / 256), 256, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
      w_s, w_e, rows, G);
  return check_launch("qg_w4a8_row_shifts");
}

extern "C" qg_status qg_e4m3_to_f16(const uint8_t* q, uint16_t* out, long long n, qg_stream_t stream) {
  using namespace qg;
  if (!(q && out)) return set_error(QG_ERR_INVALID_ARG, "qg_e4m3_to_f16: NULL pointer");
  if (n < 0) return set_error(QG_ERR_INVALID_ARG, "qg_e4m3_to_f16: bad size");
  if (n % 8 != 0) return set_error(QG_ERR_UNSUPPORTED_SHAPE, "qg_e4m3_to_f16: n %% 8 != 0");
  if (!((reinterpret_cast<uintptr_t>(q) & 7u) == 0 && aligned16(out)))
    return set_error(QG_ERR_MISALIGNED, "qg_e4m3_to_f16: misaligned pointer");
  if (n == 0) return QG_OK;
  const long long n8 = n / 8;
  e4m3_to_f16_kernel<<<unsigned((n8 + 255) / 256), 256, 0, reinterpret_cast<cudaStream_t>(stream)>>>(q, out, n8);
  return check_launch("qg_e4m3_to_f16");
}
