// W4A8 grouped (MoE) GEMM with exact bf16 group scales on the FP8 tensor
// cores: the E4M3-activation entry qgemm_w4a8_grouped (Production-Ready W4A8:
// INT4 weights, per-token FP8 activations, group-wise bf16 weight scales,
// fp32 accumulation, per-token scale in the epilogue).
//
//   y[r,n] = a_s[r] * sum_g s[n,g] * ( sum_{k in g} e4m3(a[r,k]) * q[n,k] )
//
// Every INT4 value q in [-8, 7] is exactly an E4M3 value, so the inner sums
// are FP8 x FP8 tensor-core products of exact operands (tcgen05.mma
// kind::f8f6f4, fp32 accumulation): no rounding happens before the
// accumulator.  The bf16 group scale cannot be folded into the 8-bit weights
// without a rounding, so each 128-k group is accumulated on its own and then
// "promoted": the warps read the group's accumulator and add s[n,g] times it
// into fp32 running sums held in registers -- the per-group promotion of the
// page's W4A8 GEMM, here with the group partials in tensor memory.
//
// Tile: 128 output channels (MMA M, TMEM lanes) x 128 activation rows of one
// expert (MMA N).  Tensor memory (512 columns): three group accumulators of
// 128 columns (the MMAs of group g+1 and g+2 run while group g is promoted)
// and four weight slots of 32 columns (128 E4M3 codes per lane).
//   A operand = E4M3(q), written from registers (tcgen05.st) by 16 dequant
//               warps: the packed nibbles are mapped to E4M3 codes with byte
//               permutes from a constant 16-entry table (three prmt and one
//               lop3 per four weights);
//   B operand = the E4M3 activations, TMA-loaded straight into the 128-byte
//               swizzled K-major layout (a 128-k slab is one 128-byte row);
//   D         = fp32, one accumulator per group.
// Persistent: one CTA per SM walks the tiles blockIdx.x, + gridDim.x, ... of
// the list (expert, 128-channel block, 128-row block), row blocks inner, found
// on the device from expert_off.  Every role counts the k-slabs of all of the
// CTA's tiles in one sequence g, and every ring index and barrier phase
// derives from g.
//   warp 0      TMA for the packed weights (8 stages, 64-byte swizzled)
//   warp 1      TMEM allocation and MMA issuer (one lane)
//   warp 2      TMA for the activations (8 stages)
//   warps 3-10  dequant: two sets of 4 (one warp per TMEM lane quarter), set
//               s taking the slabs g = s mod 2 into weight slot g mod 4, as far
//               ahead of the MMAs as the slots allow
//   warps 11-26 promotion: lane quarter x 32 of the 128 rows each, for every
//               group; at a tile's last group they apply the token scale and
//               store.  They do nothing else, so a group accumulator is
//               released as soon as its MMAs complete
//   warp 27     scheduler: waits for each slab's operands and for the group
//               accumulator it will overwrite to be promoted, and publishes
//               the ready count the issuer polls (the issuer waits on no
//               mbarrier while its MMAs are in flight)
// Every wait is bounded; on expiry the CTA records a timeout in the device
// error word, drains what it issued, frees its tensor memory and returns.
// Measured on GB300 (MoE config, R = 8192): about 1 PFLOP/s.  What bounds it
// is the per-group round trip -- MMA completion, promotion, release of the
// accumulator, re-issue -- against only three accumulators of tensor memory:
// removing every promotion load and weight-slot store gained about 10 %, and
// 192-row tiles (two accumulators) or one commit instead of three per slab
// changed nothing.
#include <algorithm>

#include "dequant.cuh"
#include "tc_common.cuh"

namespace qg {

bool make_u8_tmap_swizzled(CUtensorMap* m, const void* base, int rows, int cols, int box_rows, int box_cols);

namespace {

constexpr int pTW = 128;                 // channels per tile (MMA M)
constexpr int pTT = 128;                 // activation rows per tile (MMA N)
constexpr int pBK = 128;                 // k per slab: one scale group, one 128-byte E4M3 row
constexpr int pXStages = 8;              // activation stages
constexpr int pWStages = 8;              // packed-weight stages
constexpr int pSlots = 4;                // weight slots in tensor memory (one per dequant set)
constexpr int pBufs = 3;                 // group accumulators in tensor memory
constexpr int pDone = 8;                 // slab-completion barriers (>= pXStages, even)
constexpr int pDeqWarps = 8;             // two sets of 4 (one warp per TMEM lane quarter)
constexpr int pDeqSet = 4;
constexpr int pDeqSets = pDeqWarps / pDeqSet;
constexpr int pProWarps = 16;            // promotion: 4 lane quarters x 4 column groups
constexpr int pProCols = pTT / 4;        // accumulator columns (activation rows) per promotion warp
constexpr int pDeq0 = 3;
constexpr int pPro0 = pDeq0 + pDeqWarps;
constexpr int pSchedWarp = pPro0 + pProWarps;
constexpr int pThreads = (pSchedWarp + 1) * 32;
constexpr int pXStage = pTT * pBK;       // 16 KB E4M3 activations
constexpr int pWStage = pTW * pBK / 2;   // 8 KB packed INT4
constexpr uint32_t pTmemCols = 512;
constexpr uint32_t pACol0 = pBufs * pTT; // weight slots after the accumulators
constexpr uint32_t pACols = pBK / 4;     // 32 columns: 128 E4M3 codes per lane
constexpr uint32_t pDrainCap = 1u << 21;
static_assert(pSlots % pDeqSets == 0, "a slot is always written by the same dequant set");
static_assert(pProCols % 16 == 0 && pProCols <= 64, "promotion columns per warp");
static_assert(pACol0 + pSlots * pACols <= pTmemCols, "tensor memory budget");
// Waiters of the done ring: the activation producer (slab g - pXStages, every
// slab in order), each dequant set (slab g - pSlots for its own slabs: with
// pDone and pDeqSets even a set only ever waits on its own entries, each of
// their phases in order) and the promotion warps (every slab in order, never
// more than pBufs behind the MMAs) -- none can fall a whole ring behind.
static_assert(pDone >= pXStages && pDone % pDeqSets == 0 && pSlots % pDeqSets == 0, "done ring");

struct Fp8pArgs {
  const float* a_s;
  const int32_t* off;
  const uint16_t* ws;                    // [E][N][K/128] bf16
  uint16_t* y;
  int R, E, N, K;
  int tiles_w;
  unsigned int* err;
  uint32_t cap;
};

struct __align__(8) Fp8pTail {
  uint64_t x_full[pXStages];
  uint64_t w_full[pWStages];
  uint64_t w_empty[pWStages];
  uint64_t a_full[pSlots];
  uint64_t done[pDone];                  // slab g's MMAs completed (one commit per slab, entry g % pDone)
  uint64_t g_empty[pBufs];               // every promoting warp has read the group's accumulator
  uint64_t drain;
  uint32_t tmem_base;
  int abort;
  unsigned int ready;
};

// Tile t of the list -> expert, first row, end of the expert's rows, first
// channel.  Offsets are clamped into [0, R] so that no access leaves A or y.
struct PTile {
  int e, r0, r_end, n0;
};
QG_DEVICE void expert_rows(const Fp8pArgs& p, int i, int& a, int& b) {
  a = min(max(__ldg(p.off + i), 0), p.R);
  b = min(max(__ldg(p.off + i + 1), a), p.R);
}
QG_DEVICE int tile_count(const Fp8pArgs& p) {
  int n = 0;
  for (int i = 0; i < p.E; ++i) {
    int a, b;
    expert_rows(p, i, a, b);
    n += (b - a + pTT - 1) / pTT * p.tiles_w;
  }
  return n;
}
QG_DEVICE PTile tile_at(const Fp8pArgs& p, int t) {
  for (int i = 0; i < p.E; ++i) {
    int a, b;
    expert_rows(p, i, a, b);
    const int nt = (b - a + pTT - 1) / pTT;
    const int cnt = nt * p.tiles_w;
    if (t < cnt) {
      const int wt = t / nt;
      return PTile{i, a + (t - wt * nt) * pTT, b, wt * pTW};
    }
    t -= cnt;
  }
  return PTile{0, 0, 0, 0};
}

// Four INT4 codes (two's complement nibbles; the low 4 nibbles of sel,
// fsel = sel ^ 0x8888) -> their E4M3 codes, nibble i -> byte i.  The table
// P[j] = E4M3(j), N[j] = E4M3(j - 8), j = 0..7: a nibble below 8 selects
// P[j]; 8 + j selects N[j].  prmt picks byte (nibble & 7) of a register pair
// and, when the selector's top bit is set, replicates that byte's sign bit
// instead: prmt(P, nibble) is P[j] or 0x00, prmt(N, nibble ^ 8) is N[j] or
// 0xFF, a third permute gives the 0xFF mask of the negative nibbles, and one
// lop3 merges (a | (b & m)).
constexpr uint32_t kP_lo = 0x44403800u, kP_hi = 0x4E4C4A48u;   // 0, 1, 2, 3 | 4, 5, 6, 7
constexpr uint32_t kN_lo = 0xCACCCED0u, kN_hi = 0xB8C0C4C8u;   // -8, -7, -6, -5 | -4, -3, -2, -1
QG_DEVICE uint32_t int4x4_to_e4m3(uint32_t sel, uint32_t fsel) {
  const uint32_t a = prmt(kP_lo, kP_hi, sel);
  const uint32_t b = prmt(kN_lo, kN_hi, fsel);
  const uint32_t m = prmt(0x55555555u, 0x55555555u, fsel) * 3u;
  return lop3<0xF8>(a, b, m);
}

// 16 consecutive 32-bit columns of this thread's TMEM lane
QG_DEVICE void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr) : "memory");
}

__global__ void __launch_bounds__(pThreads, 1)
moe_fp8p_kernel(const __grid_constant__ CUtensorMap tmap_a, const __grid_constant__ CUtensorMap tmap_w,
                const Fp8pArgs p) {
  const int ntiles_total = tile_count(p);
  const int ntiles = ((int)blockIdx.x < ntiles_total)
                         ? (ntiles_total - (int)blockIdx.x + (int)gridDim.x - 1) / (int)gridDim.x : 0;
  if (ntiles == 0) return;
  const int nslab = p.K / pBK;
  const int total = ntiles * nslab;
  auto tile_of = [&](int i) { return tile_at(p, (int)blockIdx.x + i * (int)gridDim.x); };

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* xs = smem;                                    // [pXStages][16 KB] E4M3, 128-byte swizzled
  uint8_t* wsm = xs + pXStages * pXStage;                // [pWStages][8 KB] INT4, 64-byte swizzled
  Fp8pTail* tl = reinterpret_cast<Fp8pTail*>(wsm + pWStages * pWStage);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < pXStages; ++s) {
      mbar_init(&tl->x_full[s], 1);
    }
    for (int s = 0; s < pWStages; ++s) {
      mbar_init(&tl->w_full[s], 1);
      mbar_init(&tl->w_empty[s], pDeqSet);
    }
    for (int s = 0; s < pSlots; ++s) {
      mbar_init(&tl->a_full[s], pDeqSet);
    }
    for (int d = 0; d < pDone; ++d) mbar_init(&tl->done[d], 1);
    for (int b = 0; b < pBufs; ++b) {
      mbar_init(&tl->g_empty[b], pProWarps);
    }
    mbar_init(&tl->drain, 1);
    tl->abort = 0;
    tl->ready = 0;
    mbar_fence_init();
    tma_prefetch_desc(&tmap_a);
    tma_prefetch_desc(&tmap_w);
  }
  if (warp == 1) tmem_alloc(&tl->tmem_base, pTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tl->tmem_base;
  volatile int* abort = &tl->abort;

  if (warp == 0) {
    // ---------------- TMA producer: packed weights ----------------
    if (lane == 0) {
      int issued = 0, s = 0, i = 0;
      PTile t = tile_of(0);
      for (int g = 0; g < total; ++g, ++s) {
        if (s == nslab) { s = 0; t = tile_of(++i); }
        const int st = g % pWStages, r = g / pWStages;
        if (r > 0 && !mbar_wait(&tl->w_empty[st], (r - 1) & 1, p.cap, abort, p.err)) break;
        mbar_arrive_expect_tx(&tl->w_full[st], pWStage);
        tma_load_2d(wsm + st * pWStage, &tmap_w, &tl->w_full[st], s * (pBK / 2), t.e * p.N + t.n0);
        issued = g + 1;
      }
      if (*abort) {
        for (int g = max(0, issued - pWStages); g < issued; ++g)
          mbar_drain(&tl->w_full[g % pWStages], (g / pWStages) & 1, pDrainCap);
      }
    }
  } else if (warp == 2) {
    // ---------------- TMA producer: E4M3 activations ----------------
    if (lane == 0) {
      int issued = 0, s = 0, i = 0;
      PTile t = tile_of(0);
      for (int g = 0; g < total; ++g, ++s) {
        if (s == nslab) { s = 0; t = tile_of(++i); }
        const int st = g % pXStages;
        const int gp = g - pXStages;                     // the stage last held slab gp
        if (gp >= 0 && !mbar_wait(&tl->done[gp % pDone], (gp / pDone) & 1, p.cap, abort, p.err)) break;
        mbar_arrive_expect_tx(&tl->x_full[st], pXStage);
        tma_load_2d(xs + st * pXStage, &tmap_a, &tl->x_full[st], s * pBK, t.r0);
        issued = g + 1;
      }
      if (*abort) {
        for (int g = max(0, issued - pXStages); g < issued; ++g)
          mbar_drain(&tl->x_full[g % pXStages], (g / pXStages) & 1, pDrainCap);
      }
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer ----------------
    if (lane == 0) {
      // kind::f8f6f4: fp32 D, E4M3 A and B (format 0), both K-major, M = 128, N = 128
      const uint32_t idesc = (1u << 4) | ((uint32_t)(pTT >> 3) << 17) | ((uint32_t)(pTW >> 4) << 24);
      bool any = false;
      unsigned int ready = 0;
      for (int g = 0; g < total; ++g) {
        const int st = g % pXStages, sa = g % pSlots, b = g % pBufs;
        if (!wait_count(&tl->ready, (unsigned)g, ready, p.cap * 4, abort, p.err)) break;
        tc_fence_after();
        const uint64_t bdesc = sw128_kmajor_desc(smem_addr(xs + st * pXStage));
        const uint32_t d = tmem + (uint32_t)(b * pTT);
#pragma unroll
        for (int j = 0; j < pBK / 32; ++j)       // K = 32 per MMA: 32 bytes of each operand row
          asm volatile(
              "{\n .reg .pred p;\n setp.ne.u32 p, %4, 0;\n"
              " tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], [%1], %2, %3, p;\n}"
              :: "r"(d), "r"(tmem + pACol0 + sa * pACols + 8 * j), "l"(bdesc + 2 * j), "r"(idesc),
                 "r"(j != 0 ? 1u : 0u)
              : "memory");
        // one commit per slab: its completion frees the weight slot and the
        // activation stage and makes the group's partial readable
        tc_commit(&tl->done[g % pDone]);
        any = true;
      }
      if (*abort && any) {
        tc_commit(&tl->drain);
        mbar_drain(&tl->drain, 0, pDrainCap);
      }
    }
  } else if (warp == pSchedWarp) {
    // ---------------- scheduler ----------------
    if (lane == 0) {
      for (int g = 0; g < total; ++g) {
        if (!mbar_wait(&tl->a_full[g % pSlots], (g / pSlots) & 1, p.cap, abort, p.err)) break;
        if (!mbar_wait(&tl->x_full[g % pXStages], (g / pXStages) & 1, p.cap, abort, p.err)) break;
        if (g >= pBufs &&
            !mbar_wait(&tl->g_empty[g % pBufs], ((g - pBufs) / pBufs) & 1, p.cap, abort, p.err)) break;
        publish_count(&tl->ready, (unsigned)(g + 1));
      }
    }
  } else if (warp < pPro0) {
    // ---------------- dequant: set s takes the slabs g = s mod 2 ----------------
    // Thread = one weight row (TMEM lane) of a 128-k slab.  The sets run ahead
    // of the MMAs as far as the weight slots allow (slot g mod 4, freed by the
    // MMAs of slab g - 4), never waiting on the promotion.
    const int dw = warp - pDeq0;
    const int q = warp & 3, set = dw >> 2;
    const int row = 32 * q + lane;
    const uint32_t lane_addr = (uint32_t)(32 * q) << 16;
    const int wsw = (row >> 1) & 3;
    for (int g = set; g < total; g += pDeqSets) {
      const int sw = g % pWStages, rw = g / pWStages, sa = g % pSlots, ra = g / pSlots;
      if (!mbar_wait_warp(&tl->w_full[sw], rw & 1, p.cap, abort, p.err)) break;
      // this row's 64 packed bytes; 64-byte swizzled stage: 16-byte chunk c
      // of the row sits at chunk c ^ ((row >> 1) & 3)
      const uint8_t* wrow = wsm + sw * pWStage + row * (pBK / 2);
      uint32_t v[16];
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const uint4 w4 = *reinterpret_cast<const uint4*>(wrow + 16 * (c ^ wsw));
        v[4 * c] = w4.x; v[4 * c + 1] = w4.y; v[4 * c + 2] = w4.z; v[4 * c + 3] = w4.w;
      }
      mbar_arrive_warp(&tl->w_empty[sw]);                // packed slab read: its stage may be refilled
      if (ra > 0) {
        const int gp = g - pSlots;                       // the slot last held slab gp
        if (!mbar_wait_warp(&tl->done[gp % pDone], (gp / pDone) & 1, p.cap, abort, p.err)) break;
        tc_fence_after();
      }
      const uint32_t at = tmem + lane_addr + pACol0 + (uint32_t)(sa * pACols);
#pragma unroll
      for (int h = 0; h < 2; ++h) {                      // 64 k at a time: 16 columns
        uint32_t out[16];
#pragma unroll
        for (int j = 0; j < 8; ++j) {                    // 8 INT4 codes (k0..k7, k0 lowest) -> 8 E4M3 codes
          const uint32_t w = v[8 * h + j], f = w ^ 0x88888888u;
          out[2 * j] = int4x4_to_e4m3(w, f);
          out[2 * j + 1] = int4x4_to_e4m3(w >> 16, f >> 16);
        }
        tmem_st16(at + 16 * h, out);
      }
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive_warp(&tl->a_full[sa]);
    }
  } else {
    // ---------------- promotion and the epilogue ----------------
    // Warp = lane quarter q (32 channels) x column group cq (32 of the 128
    // rows).  For every group: read the group's accumulator, release it, add
    // s[n, g] times it into the running sums; at a tile's last group apply
    // the token scale and store.
    const int pw = warp - pPro0;
    const int q = warp & 3, cq = pw >> 2;
    const int row = 32 * q + lane;                       // channel within the tile (TMEM lane)
    const uint32_t lane_addr = (uint32_t)(32 * q) << 16;
    const int ng = p.K / pBK;                            // scale groups per row
    float sum[pProCols];
#pragma unroll
    for (int c = 0; c < pProCols; ++c) sum[c] = 0.f;
    int ti = 0, s = 0;                                   // tile index and slab of the group promoted next
    PTile t = tile_of(0);
    const uint16_t* srow = p.ws + ((size_t)t.e * p.N + min(t.n0 + row, p.N - 1)) * ng;
    // The next group's scale is fetched one group ahead and kept raw: it is
    // widened only after that group's wait, so no group stalls on its load.
    uint32_t raw = __ldg(srow);
    for (int g = 0; g < total; ++g) {
      // next group's scale (the next tile's first when this group ends the tile)
      uint32_t raw_next = 0;
      PTile t_next = t;
      const uint16_t* srow_next = srow;
      if (s + 1 < nslab) {
        raw_next = __ldg(srow + s + 1);
      } else if (ti + 1 < ntiles) {
        t_next = tile_of(ti + 1);
        srow_next = p.ws + ((size_t)t_next.e * p.N + min(t_next.n0 + row, p.N - 1)) * ng;
        raw_next = __ldg(srow_next);
      }
      const int b = g % pBufs;
      if (!mbar_wait_warp(&tl->done[g % pDone], (g / pDone) & 1, p.cap, abort, p.err)) break;
      tc_fence_after();
      const float sc = __uint_as_float(raw << 16);
#pragma unroll
      for (int h = 0; h < pProCols / 16; ++h) {
        uint32_t v[16];
        tmem_ld16(tmem + lane_addr + (uint32_t)(b * pTT + pProCols * cq + 16 * h), v);
        tmem_wait_ld();
#pragma unroll
        for (int c = 0; c < 16; c += 2)                  // two fused multiply-adds per packed op
          ffma2(sum[16 * h + c], sum[16 * h + c + 1], sc, sc, __uint_as_float(v[c]), __uint_as_float(v[c + 1]),
                sum[16 * h + c], sum[16 * h + c + 1]);
      }
      tc_fence_before();
      mbar_arrive_warp(&tl->g_empty[b]);                 // the accumulator may take group g + 3
      if (s + 1 == nslab) {
        // tile done: token scale, one bf16 rounding, store; lane l holds the
        // token scales of rows pProCols * cq + l (+ 32), the others come by shuffle
        const int mb = t.r0 + pProCols * cq;
        const int nn = t.n0 + row;
        const float as0 = mb + lane < t.r_end ? __ldg(p.a_s + mb + lane) : 0.f;
        const float as1 = lane + 32 < pProCols && mb + 32 + lane < t.r_end ? __ldg(p.a_s + mb + 32 + lane) : 0.f;
#pragma unroll
        for (int c = 0; c < pProCols; ++c) {
          const float a_sc = __shfl_sync(0xffffffffu, c < 32 ? as0 : as1, c & 31);
          if (nn < p.N && mb + c < t.r_end)
            p.y[(size_t)(mb + c) * p.N + nn] = f32_to_bf16_bits(__fmul_rn(sum[c], a_sc));
          sum[c] = 0.f;
        }
        s = 0;
        ++ti;
        t = t_next;
        srow = srow_next;
      } else {
        ++s;
      }
      raw = raw_next;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, pTmemCols);
  }
}

}  // namespace

// Launch for qgemm_w4a8_grouped (arguments validated by the caller).
qg_status moe_w4a8_fp8p(const uint8_t* a_e4m3, const float* a_s, const int32_t* expert_off, const uint8_t* w_q,
                        const uint16_t* w_s, uint16_t* y, int R, int E, int N, int K, cudaStream_t st) {
  CUtensorMap tmap_a, tmap_w;
  if (!make_u8_tmap_swizzled(&tmap_a, a_e4m3, R, K, pTT, pBK))
    return set_error(QG_ERR_CUDA, "qgemm_w4a8_grouped: cannot encode the activation tensor map");
  if (!make_u8_tmap_swizzled(&tmap_w, w_q, E * N, K / 2, pTW, pBK / 2))
    return set_error(QG_ERR_CUDA, "qgemm_w4a8_grouped: cannot encode the weight tensor map");
  unsigned int* err = device_error_word();
  if (!err) return set_error(QG_ERR_CUDA, "qgemm_w4a8_grouped: no device error word");
  Fp8pArgs a{};
  a.a_s = a_s; a.off = expert_off; a.ws = w_s; a.y = y;
  a.R = R; a.E = E; a.N = N; a.K = K;
  a.tiles_w = (N + pTW - 1) / pTW;
  a.err = err;
  a.cap = wait_limit();
  const int smem = pXStages * pXStage + pWStages * pWStage + (int)sizeof(Fp8pTail) + 1024;
  if (!ensure_smem(moe_fp8p_kernel, smem)) return set_error(QG_ERR_CUDA, "qgemm_w4a8_grouped: smem attribute");
  // the tile count depends on expert_off (device memory): one CTA per SM, or
  // fewer when even the longest possible tile list is shorter
  const long long bound = ((long long)(R + pTT - 1) / pTT + E) * a.tiles_w;
  const int grid = (int)std::min<long long>(bound, (long long)sm_count());
  moe_fp8p_kernel<<<grid, pThreads, smem, st>>>(tmap_a, tmap_w, a);
  return check_launch("qgemm_w4a8_grouped (tcgen05)");
}

}  // namespace qg
