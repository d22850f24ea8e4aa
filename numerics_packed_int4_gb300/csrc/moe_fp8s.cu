// W4A8 grouped (MoE) GEMM with FP8 group scales on an FP8 x FP8 tensor-core
// matmul (Production-Ready W4A8, "Accurate W4A8 Kernel").
//
// Semantics: y[r,n] = bf16( a_s[r] * cs8[n] * sum_k e4m3(a[r,k]) * w8[n,k] )
// with w8 = E4M3(q[n,k] * s8[n,k/128]).  The page builds, per FP8 scale, a
// lookup table of its 16 products with the INT4 values; here each dequant
// thread builds that table in registers once per (channel, 128-k group) --
// q * s8 is exact in fp16 (at most 8 significant bits) and one
// cvt.rn.satfinite rounds it to E4M3, the 1/8 pre-scaling of s8 keeping every
// product inside +-448 -- and looks the INT4 codes up with byte permutes:
//   P = {E4M3(j*s8)}, j = 0..7     two registers, every byte's sign bit clear
//   N = {E4M3((j-8)*s8)}, j = 0..7 two registers, every byte's sign bit set
// A nibble j < 8 selects P[j]; a nibble 8 + j selects N[j].  prmt picks byte
// (nibble & 7) of a register pair, and replicates that byte's sign bit when
// the nibble's top bit is set, so prmt(P, nibble) is P[j] or 0x00 and
// prmt(N, nibble ^ 8) is N[j] or 0xFF; a third permute of the constant 0x55
// times 3 gives the 0xFF byte mask of the negative nibbles, and one lop3
// merges.  fp32 accumulation; the per-token and per-channel scales are
// applied in the epilogue (the page's outer-vector scaling step).
//
// tcgen05.mma.cta_group::1.kind::f8f6f4, E4M3 x E4M3, M = 128 channels,
// N = 256 activation rows, K = 32:
//   A operand  = the E4M3 weights, written by 16 dequant warps into 8 slots of
//                tensor memory (128 k = 32 columns per slot);
//   B operand  = the E4M3 activations, TMA-loaded straight into shared memory
//                in the 128-byte swizzled K-major layout (a 128-k slab is one
//                128-byte row) -- no conversion and no second copy;
//   D          = fp32 accumulator in TMEM columns 0-255.
// Persistent: one CTA per SM walks the tiles blockIdx.x, + gridDim.x, ... of
// the list (expert, 128-channel block, 256-row block) -- row blocks of one
// expert inner, so concurrently running CTAs share a weight block -- located
// on the device from expert_off.  Every role counts the k-slabs of all of the
// CTA's tiles in one sequence, so the rings run on from one tile into the
// next, and the epilogue of a tile overlaps the next tile's MMAs (the dequant
// warps read the accumulator once they have produced the next tile's first 8
// slabs, release it, then scale and store).
// Roles: warp 0 TMA for the packed weights (8 stages, 64-byte swizzled), warp
// 1 TMEM + MMA issuer, warp 2 TMA for the activations (5 stages), warps 3-18
// dequant and epilogue, warp 19 scheduler (waits for each slab's operands and
// publishes the ready count the issuer polls, so that the issuing thread
// never waits on an mbarrier with MMAs in flight).  Every wait is bounded.
#include <algorithm>

#include "dequant.cuh"
#include "tc_common.cuh"

namespace qg {

bool make_u8_tmap_swizzled(CUtensorMap* m, const void* base, int rows, int cols, int box_rows, int box_cols);

namespace {

constexpr int fTW = 128;                 // weight rows per tile (MMA M)
constexpr int fTT = 256;                 // activation rows per tile (MMA N)
constexpr int fBK = 128;                 // k per slab: one 128-byte row of E4M3, one scale group
constexpr int fXStages = 5;              // activation stages (<= fSlots: released through a_empty)
constexpr int fSlots = 8;                // TMEM A slots and packed-weight stages
constexpr int fDeqWarps = 16;            // four sets of 4 (one per TMEM lane quarter)
constexpr int fDeqSet = 4;
constexpr int fDeqSets = fDeqWarps / fDeqSet;
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
  const uint8_t* s8;                     // [K/128][E*N] E4M3 (group-major)
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
  uint64_t acc_full;                     // one phase per tile: its MMAs completed
  uint64_t acc_empty;                    // one phase per tile: the epilogue has read the accumulator
  uint64_t drain;
  uint32_t tmem_base;
  int abort;
  unsigned int ready;
};

// Tile t of the list -> expert, first row, end of the expert's rows, first
// channel.  Offsets are clamped into [0, R] so that no store leaves y.
struct FTile {
  int e, r0, r_end, n0;
};
QG_DEVICE void expert_rows(const Fp8sArgs& p, int i, int& a, int& b) {
  a = min(max(__ldg(p.off + i), 0), p.R);
  b = min(max(__ldg(p.off + i + 1), a), p.R);
}
QG_DEVICE int tile_count(const Fp8sArgs& p) {
  int n = 0;
  for (int i = 0; i < p.E; ++i) {
    int a, b;
    expert_rows(p, i, a, b);
    n += (b - a + fTT - 1) / fTT * p.tiles_w;
  }
  return n;
}
QG_DEVICE FTile tile_at(const Fp8sArgs& p, int t) {
  for (int i = 0; i < p.E; ++i) {
    int a, b;
    expert_rows(p, i, a, b);
    const int nt = (b - a + fTT - 1) / fTT;
    const int cnt = nt * p.tiles_w;
    if (t < cnt) {
      const int wt = t / nt;
      return FTile{i, a + (t - wt * nt) * fTT, b, wt * fTW};
    }
    t -= cnt;
  }
  return FTile{0, 0, 0, 0};
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

// The table of one FP8 scale s (fp16x2 splat): P[j] = E4M3(j*s) and
// N[j] = E4M3((j-8)*s), j = 0..7, four bytes per register.  The fp16x2
// constants are the integer pairs (0,1) (2,3) (4,5) (6,7) and (-8,-7) (-6,-5)
// (-4,-3) (-2,-1).
struct Lut {
  uint32_t p_lo, p_hi, n_lo, n_hi;
};
QG_DEVICE Lut lut_build(uint32_t s2) {
  const uint32_t c0 = f16x2_to_e4m3x2(f16x2_mul(0x3C000000u, s2));
  const uint32_t c1 = f16x2_to_e4m3x2(f16x2_mul(0x42004000u, s2));
  const uint32_t c2 = f16x2_to_e4m3x2(f16x2_mul(0x45004400u, s2));
  const uint32_t c3 = f16x2_to_e4m3x2(f16x2_mul(0x47004600u, s2));
  const uint32_t d0 = f16x2_to_e4m3x2(f16x2_mul(0xC700C800u, s2));
  const uint32_t d1 = f16x2_to_e4m3x2(f16x2_mul(0xC500C600u, s2));
  const uint32_t d2 = f16x2_to_e4m3x2(f16x2_mul(0xC200C400u, s2));
  const uint32_t d3 = f16x2_to_e4m3x2(f16x2_mul(0xBC00C000u, s2));
  return Lut{c0 | (c1 << 16), c2 | (c3 << 16), d0 | (d1 << 16), d2 | (d3 << 16)};
}
// Four INT4 codes (the low 4 nibbles of sel; fsel = sel ^ 0x8888) -> four
// E4M3 codes of q * s, nibble i -> byte i.
QG_DEVICE uint32_t lut4(uint32_t sel, uint32_t fsel, const Lut& t) {
  const uint32_t a = prmt(t.p_lo, t.p_hi, sel);                     // P[j] at q >= 0, 0x00 at q < 0
  const uint32_t b = prmt(t.n_lo, t.n_hi, fsel);                    // N[j] at q < 0, 0xFF at q >= 0
  const uint32_t m = prmt(0x55555555u, 0x55555555u, fsel) * 3u;     // 0xFF at q < 0, 0x00 at q >= 0
  return lop3<0xF8>(a, b, m);                                       // a | (b & m)
}

__global__ void __launch_bounds__(fThreads, 1)
moe_fp8s_kernel(const __grid_constant__ CUtensorMap tmap_a, const __grid_constant__ CUtensorMap tmap_w,
                const Fp8sArgs p) {
  // ---- persistent: tiles blockIdx.x, + gridDim.x, ... of the tile list ----
  const int ntiles_total = tile_count(p);
  const int ntiles = ((int)blockIdx.x < ntiles_total)
                         ? (ntiles_total - (int)blockIdx.x + (int)gridDim.x - 1) / (int)gridDim.x : 0;
  if (ntiles == 0) return;
  const int nslab = p.K / fBK;
  const int total = ntiles * nslab;
  auto tile_of = [&](int i) { return tile_at(p, (int)blockIdx.x + i * (int)gridDim.x); };

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
      mbar_init(&tl->w_empty[s], fDeqSet);
      mbar_init(&tl->a_full[s], fDeqSet);
      mbar_init(&tl->a_empty[s], 1);
    }
    mbar_init(&tl->acc_full, 1);
    mbar_init(&tl->acc_empty, fDeqWarps);
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
      int issued = 0, s = 0, i = 0;
      FTile t = tile_of(0);
      for (int g = 0; g < total; ++g, ++s) {
        if (s == nslab) { s = 0; t = tile_of(++i); }
        const int st = g % fSlots, r = g / fSlots;
        if (r > 0 && !mbar_wait(&tl->w_empty[st], (r - 1) & 1, p.cap, abort, p.err)) break;
        mbar_arrive_expect_tx(&tl->w_full[st], fWStage);
        tma_load_2d(wsm + st * fWStage, &tmap_w, &tl->w_full[st], s * (fBK / 2), t.e * p.N + t.n0);
        issued = g + 1;
      }
      if (*abort) {
        for (int g = max(0, issued - fSlots); g < issued; ++g)
          mbar_drain(&tl->w_full[g % fSlots], (g / fSlots) & 1, fDrainCap);
      }
    }
  } else if (warp == 2) {
    // ---------------- TMA producer: E4M3 activations ----------------
    if (lane == 0) {
      int issued = 0, s = 0, i = 0;
      FTile t = tile_of(0);
      for (int g = 0; g < total; ++g, ++s) {
        if (s == nslab) { s = 0; t = tile_of(++i); }
        const int st = g % fXStages, gp = g - fXStages;   // stage last held slab gp
        if (gp >= 0 && !mbar_wait(&tl->a_empty[gp % fSlots], (gp / fSlots) & 1, p.cap, abort, p.err)) break;
        mbar_arrive_expect_tx(&tl->x_full[st], fXStage);
        tma_load_2d(xs + st * fXStage, &tmap_a, &tl->x_full[st], s * fBK, t.r0);
        issued = g + 1;
      }
      if (*abort) {
        for (int g = max(0, issued - fXStages); g < issued; ++g)
          mbar_drain(&tl->x_full[g % fXStages], (g / fXStages) & 1, fDrainCap);
      }
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer ----------------
    if (lane == 0) {
      // kind::f8f6f4: fp32 D, E4M3 A and B (format 0), both K-major
      const uint32_t idesc = (1u << 4) | ((uint32_t)(fTT >> 3) << 17) | ((uint32_t)(fTW >> 4) << 24);
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
          const int st = g % fXStages, sa = g % fSlots;
          if (!wait_count(&tl->ready, (unsigned)g, ready, p.cap * 4, abort, p.err)) { ok = false; break; }
          tc_fence_after();
          const uint64_t bdesc = sw128_kmajor_desc(smem_addr(xs + st * fXStage));
#pragma unroll
          for (int j = 0; j < fBK / 32; ++j)     // K = 32 per MMA: 32 bytes of each operand row
            asm volatile(
                "{\n .reg .pred p;\n setp.ne.u32 p, %4, 0;\n"
                " tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], [%1], %2, %3, p;\n}"
                :: "r"(tmem), "r"(tmem + fACol0 + sa * fACols + 8 * j), "l"(bdesc + 2 * j), "r"(idesc),
                   "r"((s | j) != 0 ? 1u : 0u)
                : "memory");
          tc_commit(&tl->a_empty[sa]);                   // frees the A slot and the activation stage
          any = true;
        }
        if (!ok) break;
        tc_commit(&tl->acc_full);
      }
      if (*abort && any) {
        tc_commit(&tl->drain);
        mbar_drain(&tl->drain, 0, fDrainCap);
      }
    }
  } else if (warp == fSchedWarp) {
    // ---------------- scheduler ----------------
    if (lane == 0) {
      for (int g = 0; g < total; ++g) {
        if (!mbar_wait(&tl->a_full[g % fSlots], (g / fSlots) & 1, p.cap, abort, p.err)) break;
        if (!mbar_wait(&tl->x_full[g % fXStages], (g / fXStages) & 1, p.cap, abort, p.err)) break;
        publish_count(&tl->ready, (unsigned)(g + 1));
      }
    }
  } else {
    // ---------------- dequant producers, then the epilogues ----------------
    // Thread = one weight row (TMEM lane) of a 128-k slab; the four sets of 4
    // warps (one per TMEM lane quarter) take every fourth slab, so each has
    // four slab periods for its wait-load-decode-store chain and builds the
    // table of a (channel, group) once.  A slab is one scale group.
    // The epilogue of tile e runs once this warp is about to produce the slab
    // fSlots past the start of tile e+1: the MMAs then hold fSlots slabs of
    // tile e+1 to work on while it stores, and no slot this warp needs is
    // held by a tile-(e+1) MMA (which waits for the epilogue).
    const int dw = warp - fDeq0;
    const int q = warp & 3, set = dw >> 2;
    const int row = 32 * q + lane;
    const int cq = set;                              // epilogue: 64 of the 256 activation rows
    const uint32_t lane_base = tmem + ((uint32_t)(32 * q) << 16) + fACol0;
    const int wsw = (row >> 1) & 3;
    // scale cursor: tile index, slab in the tile, this thread's scale row
    struct Cur { int i, s; const uint8_t* srow; };
    // group-major scales: the scale of channel r, group s is s8[s * E*N + r],
    // so a warp's 32 channels read 32 consecutive bytes
    const size_t sstride = (size_t)p.E * p.N;
    auto set_row = [&](Cur& c) {
      if (c.i < ntiles) {
        const FTile t = tile_of(c.i);
        c.srow = p.s8 + (size_t)t.e * p.N + min(t.n0 + row, p.N - 1);
      }
    };
    auto advance = [&](Cur& c, int by) {
      c.s += by;
      while (c.s >= nslab) { c.s -= nslab; ++c.i; set_row(c); }
    };
    auto scale_of = [&](const Cur& c) -> uint32_t { return c.i < ntiles ? __ldg(c.srow + c.s * sstride) : 0u; };
    // epilogue of tile e: TMEM -> registers, scaled by the token and channel
    // scales and rounded to bf16 pairs -> (accumulator free) -> Y.  Lane l
    // fetches the token scales of rows l and 32 + l of this warp's 64; the
    // others come by shuffle.  Lanes 2i and 2i+1 (channels n, n+1) then swap
    // halves so that each stores 4 bytes: the even lane token m's (n, n+1),
    // the odd lane token m+1's.
    auto epilogue = [&](int e) -> bool {
      if (!mbar_wait_warp(&tl->acc_full, e & 1, p.cap, abort, p.err)) return false;
      tc_fence_after();
      const FTile t = tile_of(e);
      const int nn = t.n0 + row;
      const int mb = t.r0 + 64 * cq;
      const float cs = nn < p.N ? __ldg(p.cs8 + (size_t)t.e * p.N + nn) : 0.f;
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
        for (int c = 0; c < 16; ++c) {        // (acc * token scale) * channel scale, a pair at a time
          float lo, hi;
          fmul2(lo, hi, __uint_as_float(v[2 * c]), __uint_as_float(v[2 * c + 1]),
                __shfl_sync(0xffffffffu, as, 2 * c), __shfl_sync(0xffffffffu, as, 2 * c + 1));
          fmul2(lo, hi, lo, hi, cs, cs);
          packed[16 * i + c] = f32x2_to_bf16x2(lo, hi);
        }
      }
      tc_fence_before();
      mbar_arrive_warp(&tl->acc_empty);              // the next tile's MMAs may overwrite it
      const bool odd = lane & 1;
      const uint32_t sel = odd ? 0x3276u : 0x5410u;
      const int n2 = nn & ~1;                        // N is even: a pair is in range or out as a whole
      const int m0 = mb + (odd ? 1 : 0);
      const bool full = mb + 64 <= t.r_end && n2 < p.N;
      uint32_t* yp = reinterpret_cast<uint32_t*>(p.y + (size_t)m0 * p.N + n2);   // rows m0, m0 + 2, ...
#pragma unroll
      for (int c = 0; c < 32; ++c) {
        const uint32_t w = prmt(packed[c], __shfl_xor_sync(0xffffffffu, packed[c], 1), sel);
        if (full || (n2 < p.N && m0 + 2 * c < t.r_end)) yp[(size_t)c * p.N] = w;
      }
      return true;
    };
    int e_next = 0;                                  // next tile whose epilogue this warp owes
    bool ok = true;
    Cur pf{0, 0, nullptr};
    set_row(pf);
    advance(pf, set);
    uint32_t sc_cur = scale_of(pf);
    advance(pf, fDeqSets);
    uint32_t sc_nxt = scale_of(pf);
    for (int g = set; g < total; g += fDeqSets) {
      while (e_next < ntiles - 1 && g >= (e_next + 1) * nslab + fSlots) {
        if (!(ok = epilogue(e_next))) break;
        ++e_next;
      }
      if (!ok) break;
      const int sa = g % fSlots, ra = g / fSlots;
      const Lut tab = lut_build(e4m3_to_f16x2_splat(sc_cur));
      sc_cur = sc_nxt;
      advance(pf, fDeqSets);                         // pf now at this set's slab after the next
      sc_nxt = scale_of(pf);
      if (!mbar_wait_warp(&tl->w_full[sa], ra & 1, p.cap, abort, p.err)) { ok = false; break; }
      // this row's 64 packed bytes; 64-byte swizzled stage: 16-byte chunk c
      // of the row sits at chunk c ^ ((row >> 1) & 3)
      const uint8_t* wrow = wsm + sa * fWStage + row * (fBK / 2);
      uint32_t v[16];
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const uint4 w4 = *reinterpret_cast<const uint4*>(wrow + 16 * (c ^ wsw));
        v[4 * c] = w4.x; v[4 * c + 1] = w4.y; v[4 * c + 2] = w4.z; v[4 * c + 3] = w4.w;
      }
      uint32_t out[32];
#pragma unroll
      for (int j = 0; j < 16; ++j) {                 // 8 INT4 codes (k0..k7, k0 lowest) -> 8 E4M3 codes
        const uint32_t f = v[j] ^ 0x88888888u;
        out[2 * j] = lut4(v[j], f, tab);
        out[2 * j + 1] = lut4(v[j] >> 16, f >> 16, tab);
      }
      mbar_arrive_warp(&tl->w_empty[sa]);            // packed slab decoded: its stage may be refilled
      if (ra > 0) {
        if (!mbar_wait_warp(&tl->a_empty[sa], (ra - 1) & 1, p.cap, abort, p.err)) { ok = false; break; }
        tc_fence_after();
      }
      {
        const uint32_t (&o0)[16] = *reinterpret_cast<const uint32_t(*)[16]>(&out[0]);
        const uint32_t (&o1)[16] = *reinterpret_cast<const uint32_t(*)[16]>(&out[16]);
        tmem_st16(lane_base + sa * fACols, o0);
        tmem_st16(lane_base + sa * fACols + 16, o1);
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
  if (!make_u8_tmap_swizzled(&tmap_a, a_e4m3, R, K, fTT, fBK))
    return set_error(QG_ERR_CUDA, "qgemm_w4a8_grouped_fp8s: cannot encode the activation tensor map");
  if (!make_u8_tmap_swizzled(&tmap_w, w_q, E * N, K / 2, fTW, fBK / 2))
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
  // the tile count depends on expert_off (device memory): one CTA per SM, or
  // fewer when even the longest possible tile list is shorter
  const long long bound = ((long long)(R + fTT - 1) / fTT + E) * a.tiles_w;
  const int grid = (int)std::min<long long>(bound, (long long)sm_count());
  moe_fp8s_kernel<<<grid, fThreads, smem, reinterpret_cast<cudaStream_t>(stream)>>>(tmap_a, tmap_w, a);
  return check_launch("qgemm_w4a8_grouped_fp8s");
}
