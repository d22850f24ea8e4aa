// W4A4 GEMM on the block-scaled FP4 tensor cores: MXFP4 activations (the
// exponent-first 0.75-threshold quantizer, blocks of 32) times MXFP4 weights
// (E2M1 codes with one E8M0 scale per 32 k), fp32 accumulation, one bf16
// rounding -- the product of vLLM PR #43557's MXFP4 W4A4 GEMM, and the FP4
// tensor-core rate the 3090 article (section 5) points at.
//
//   y[m,n] = sum_k (e2m1(a[m,k]) * 2^(sa[m,k/32]-127)) * (e2m1(w[n,k]) * 2^(sw[n,k/32]-127))
//
// tcgen05.mma.cta_group::1.kind::mxf4.block_scale.scale_vec::2X applies both
// scales inside the MMA: every product is exact and the partial sums are
// fp32, so the result is the exact-product sum up to the order of the fp32
// additions -- no dequantization, no conversion, no second copy.
//
// Orientation D[n, m] = sum_k W[n,k] X[m,k] (weights are the M side):
//   A operand = packed E2M1 weights, 128 channels x 256 k per stage (128-byte
//               rows), TMA-loaded straight into the 128-byte swizzled K-major
//               layout;
//   B operand = packed E2M1 activations, 256 tokens x 256 k, the same way;
//   scale factors = E8M0 codes in tensor memory, written from registers
//               (tcgen05.st) by four warps: an operand's codes fill a group of
//               columns, row 32c + l in column c, lane l (all four lane
//               quarters hold the same words), one 32-bit word = a row's codes
//               of 4 consecutive 32-k blocks; the MMA of k-quarter j (64 k)
//               reads bytes 0-1 (scale-factor ID 0, j even) or 2-3 (ID 2, j
//               odd) of the group for pair p = j / 2: four columns for the 128
//               weight rows at slot column 4p, eight for the 256 token rows at
//               slot column 8 + 8p (24 of a slot's 32 columns per 256-k slab).
//               With 16-element activation blocks (kA16) the same kernel runs
//               kind::mxf4nvf4.block_scale.scale_vec::4X: one word of four
//               16-element codes per row and MMA at ID 0 -- the token codes as
//               they are in memory, each 32-element weight code written twice
//               -- four columns per MMA for the weights (slot column 4j),
//               eight for the tokens (16 + 8j), 48 per slab;
//   D         = fp32, one 128 x 256 accumulator (256 columns): the epilogue
//               packs it to bf16 in registers and releases it before storing.
// One MMA instruction covers 128 x 256 x 64: an issue costs about the same
// at N = 256 as at N = 128, so the wide tile halves the instructions per flop.
// Persistent: one CTA per SM walks the tiles blockIdx.x, + gridDim.x, ... of
// 256 tokens x 128 channels (every channel tile of a token tile in turn, so a
// token tile's activations are read once).  Every role counts the k-slabs of
// all its tiles in one sequence g.
//   warp 0      TMA for both operands (one elected lane; 4 stages of 48 KB)
//   warp 1      TMEM allocation and MMA issuer (one lane)
//   warp 2      scheduler: waits for each slab's operands and scale factors,
//               publishes the ready count the issuer polls
//   warps 3-6   scale factors (lane quarter = warp % 4): bring the codes of
//               2 slabs at a time into shared memory (two TMA loads, or
//               8-byte cp.async when a code row's stride is not a multiple of
//               16 bytes; one row per lane straight from global memory would
//               cost a wavefront per row), and store each slab's words into
//               their lane quarter
//   warps 7-14  epilogue: lane quarter = warp % 4, token half = (warp - 7) / 4;
//               bf16 in registers, then 16-token pieces staged in shared
//               memory and written by TMA tile stores
// Every wait is bounded; on expiry the CTA records a timeout in the device
// error word, drains what it issued, frees its tensor memory and returns.
#include <algorithm>

#include "tc_common.cuh"

namespace qg {

bool make_u8_tmap(CUtensorMap* m, const void* base, int rows, int cols, int box_rows, int box_cols);
bool make_u8_tmap_swizzled(CUtensorMap* m, const void* base, int rows, int cols, int box_rows, int box_cols);

namespace {

constexpr int bTW = 128;                 // channels per tile (MMA M)
constexpr int bTT = 256;                 // tokens per tile (MMA N)
constexpr int bBK = 256;                 // k per slab: 128 packed bytes per row
constexpr int bStages = 4;               // operand stages (A + B)
constexpr int bSfSlots = 8;              // scale-factor slots in tensor memory (at most)
constexpr int bDone = 16;                // slab-completion barriers
constexpr int bABytes = bTW * bBK / 2;   // 16 KB of weights per stage
constexpr int bBBytes = bTT * bBK / 2;   // 32 KB of activations per stage
constexpr int bStageBytes = bABytes + bBBytes;
constexpr int bSfWarp0 = 3, bSfWarps = 4, bEpiWarp0 = bSfWarp0 + bSfWarps, bEpiWarps = 8;
constexpr int bThreads = (bEpiWarp0 + bEpiWarps) * 32;
constexpr uint32_t bTmemCols = 512;
constexpr uint32_t bSfCol0 = bTT;        // scale-factor slots follow the accumulator
static_assert(bSfCol0 % 32 == 0, "slots aligned: every store and code group aligned to its width");
constexpr int bChunk = 2;                // slabs of codes per shared-memory chunk
constexpr int bSfRowBytes = 8 * bChunk;  // weight codes per row of a chunk (32-element blocks): 16 bytes
constexpr int bPieceTok = 16;            // tokens per staged output piece (TMA store box: 128 channels x 16 tokens)
constexpr int bPieceBytes = bPieceTok * bTW * 2;

// What depends on the activations' block size (32, or 16 with kA16):
template <bool kA16> struct Fp4Cfg {
  static constexpr int kAScB = kA16 ? 16 : 8;                  // activation codes per row and slab
  static constexpr int kARowB = kAScB * bChunk;                // activation code bytes per row of a chunk
  static constexpr uint32_t kSlotCols = kA16 ? 48 : 32;        // tensor-memory columns per slab
  static constexpr int kSlots = kA16 ? 5 : 8;                  // slots in the ring
  static constexpr int kBufBytes = bTW * bSfRowBytes + bTT * kARowB;   // one chunk of codes
  static constexpr int kXchBytes = 2 * kBufBytes;              // two chunk buffers
  static constexpr int kPieces = kBufBytes / 8;                // 8-byte cp.async pieces per chunk
  static constexpr int kStgBufs = kA16 ? 1 : 2;                // staged output pieces in flight per token half
  static constexpr int kStgBytes = 2 * kStgBufs * bPieceBytes;
  static_assert(kPieces % (bSfWarps * 32) == 0, "chunk copy divides over the scale-factor threads");
  static_assert(kSlots <= bSfSlots && bDone > kSlots, "slab-completion ring covers every reuse distance");
  static_assert(bSfCol0 + kSlots * kSlotCols <= bTmemCols && kSlotCols % 16 == 0, "tensor memory budget");
};
constexpr uint32_t bDrainCap = 1u << 21;
static_assert(bDone >= bStages, "slab-completion ring covers every reuse distance");
static_assert(bEpiWarps * 32 * 128 == bTW * bTT, "each epilogue thread owns 128 outputs");

struct Fp4Args {
  const uint8_t* w_sf;                   // [N][K/32] E8M0
  const uint8_t* a_sf;                   // [M][K/32] E8M0 ([M][K/16] with 16-element activation blocks)
  uint16_t* y;                           // [M][N] bf16
  int M, N, K;
  int tiles_t, tiles_w;
  unsigned int* err;
  uint32_t cap;
};

struct __align__(8) Fp4Tail {
  uint64_t full[bStages];                // both operands of the stage landed (TMA bytes)
  uint64_t sf_full[bSfSlots];            // the slot's scale factors stored (4 warps)
  uint64_t done[bDone];                  // slab g's MMAs completed (entry g % bDone)
  uint64_t sf_tma[2];                    // a chunk of scale-factor codes landed (TMA bytes)
  uint64_t acc_full;                     // the tile's MMAs completed (one phase per tile)
  uint64_t acc_empty;                    // the epilogue has read the accumulator (8 warps)
  uint64_t drain;
  uint32_t tmem_base;
  int abort;
  unsigned int ready;
};

// Instruction descriptor of the block-scaled kinds (kind::mxf4 here):
//   bits 4-5  B scale-factor ID      bits 7-9   A format (E2M1 = 1)
//   bits 10-12 B format (E2M1 = 1)   bits 15/16 A/B major (0 = K-major)
//   bits 17-22 N >> 3                bit 23     scale type (1 = UE8M0)
//   bits 24-28 M >> 4                bits 29-30 A scale-factor ID
//   bit 31     K size (0 = 64 for dense FP4)
QG_HOST_DEVICE uint32_t idesc_mxf4(int M, int N, uint32_t sf_id) {
  return (sf_id << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(N >> 3) << 17) | (1u << 23) |
         ((uint32_t)(M >> 4) << 24) | (sf_id << 29);
}

QG_DEVICE void mma_mxf4(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc, uint32_t sfa,
                        uint32_t sfb, bool accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.u32 p, %6, 0;\n"
      " tcgen05.mma.cta_group::1.kind::mxf4.block_scale.scale_vec::2X [%0], %1, %2, %3, [%4], [%5], p;\n}"
      :: "r"(d_tmem), "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(sfa), "r"(sfb), "r"(accumulate ? 1u : 0u)
      : "memory");
}

// 16 consecutive 32-bit columns of this thread's TMEM lane
QG_DEVICE void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr) : "memory");
}

QG_DEVICE void cp_async8(void* dst, const void* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 8;"
               :: "r"(smem_addr(dst)), "l"(__cvta_generic_to_global(src)) : "memory");
}
QG_DEVICE void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
QG_DEVICE void cp_async_wait() { asm volatile("cp.async.wait_group %0;" :: "n"(N) : "memory"); }
QG_DEVICE void named_bar_sync(int id, int nthreads) {
  asm volatile("bar.sync %0, %1;" :: "r"(id), "r"(nthreads) : "memory");
}

QG_DEVICE void tma_store_2d(const CUtensorMap* m, const void* src, int x, int y) {
  asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%2, %3}], [%1];"
               :: "l"(reinterpret_cast<uint64_t>(m)), "r"(smem_addr(src)), "r"(x), "r"(y) : "memory");
}
QG_DEVICE void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
template <int N>
QG_DEVICE void bulk_wait_read() { asm volatile("cp.async.bulk.wait_group.read %0;" :: "n"(N) : "memory"); }
QG_DEVICE void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

QG_DEVICE void tmem_st8(uint32_t taddr, const uint32_t (&r)[8]) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};"
               :: "r"(taddr), "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7])
               : "memory");
}

// The same with four scale factors per row and MMA (16-element blocks), one
// 32-bit word of codes at scale-factor ID 0.
QG_DEVICE void mma_mxf4nvf4_4x(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc, uint32_t sfa,
                               uint32_t sfb, bool accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.u32 p, %6, 0;\n"
      " tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], %1, %2, %3, [%4], [%5], p;\n}"
      :: "r"(d_tmem), "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(sfa), "r"(sfb), "r"(accumulate ? 1u : 0u)
      : "memory");
}

QG_DEVICE void tile_origin(const Fp4Args& p, int tile, int& m0, int& n0) {
  m0 = (tile / p.tiles_w) * bTT;         // every channel tile of a token tile in turn
  n0 = (tile % p.tiles_w) * bTW;
}

template <bool kTmaSf, bool kA16>
__global__ void __launch_bounds__(bThreads, 1)
w4a4_bs_kernel(const __grid_constant__ CUtensorMap tmap_w, const __grid_constant__ CUtensorMap tmap_a,
               const __grid_constant__ CUtensorMap tmap_y, const __grid_constant__ CUtensorMap tmap_wsf,
               const __grid_constant__ CUtensorMap tmap_asf, const Fp4Args p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  using Cfg = Fp4Cfg<kA16>;
  Fp4Tail* tl = reinterpret_cast<Fp4Tail*>(smem + bStages * bStageBytes + Cfg::kXchBytes + Cfg::kStgBytes);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  const int nslab = p.K / bBK;
  const int ntiles_total = p.tiles_t * p.tiles_w;
  const int ntiles = ((int)blockIdx.x < ntiles_total)
                         ? (ntiles_total - (int)blockIdx.x + (int)gridDim.x - 1) / (int)gridDim.x : 0;
  if (ntiles == 0) return;
  const int total = ntiles * nslab;
  auto tile_of = [&](int i) { return (int)blockIdx.x + i * (int)gridDim.x; };

  if (threadIdx.x == 0) {
    for (int s = 0; s < bStages; ++s) mbar_init(&tl->full[s], 1);
    for (int s = 0; s < bSfSlots; ++s) mbar_init(&tl->sf_full[s], bSfWarps);
    for (int d = 0; d < bDone; ++d) mbar_init(&tl->done[d], 1);
    mbar_init(&tl->sf_tma[0], 1);
    mbar_init(&tl->sf_tma[1], 1);
    mbar_init(&tl->acc_full, 1);
    mbar_init(&tl->acc_empty, bEpiWarps);
    mbar_init(&tl->drain, 1);
    tl->abort = 0;
    tl->ready = 0;
    mbar_fence_init();
    tma_prefetch_desc(&tmap_w);
    tma_prefetch_desc(&tmap_a);
    tma_prefetch_desc(&tmap_y);
  }
  if (warp == 1) tmem_alloc(&tl->tmem_base, bTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tl->tmem_base;
  volatile int* abort = &tl->abort;

  if (warp == 0) {
    // ---------------- TMA producer: weights and activations of each slab ----------------
    if (lane == 0) {
      int issued = 0, s = 0, i = 0, m0 = 0, n0 = 0;
      tile_origin(p, tile_of(0), m0, n0);
      for (int g = 0; g < total; ++g, ++s) {
        if (s == nslab) { s = 0; tile_origin(p, tile_of(++i), m0, n0); }
        const int st = g % bStages, gp = g - bStages;   // the stage last held slab gp
        if (gp >= 0 && !mbar_wait(&tl->done[gp % bDone], (gp / bDone) & 1, p.cap, abort, p.err)) break;
        uint8_t* stage = smem + st * bStageBytes;
        mbar_arrive_expect_tx(&tl->full[st], bStageBytes);
        tma_load_2d(stage, &tmap_w, &tl->full[st], s * (bBK / 2), n0);
        tma_load_2d(stage + bABytes, &tmap_a, &tl->full[st], s * (bBK / 2), m0);
        issued = g + 1;
      }
      if (*abort) {     // let every copy already issued land before the CTA moves on
        for (int g = max(0, issued - bStages); g < issued; ++g)
          mbar_drain(&tl->full[g % bStages], (g / bStages) & 1, bDrainCap);
      }
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer ----------------
    if (lane == 0) {
      const uint32_t idesc[2] = {idesc_mxf4(bTW, bTT, 0), idesc_mxf4(bTW, bTT, 2)};   // bytes 0-1, bytes 2-3
      bool any = false;
      unsigned int ready = 0;
      int g = 0;
      for (int i = 0; i < ntiles && !*abort; ++i) {
        if (i >= 1) {             // the accumulator is free once the epilogue has read tile i - 1
          if (!mbar_wait(&tl->acc_empty, (i - 1) & 1, p.cap, abort, p.err)) break;
          tc_fence_after();
        }
        bool ok = true;
        for (int s = 0; s < nslab; ++s, ++g) {
          const int st = g % bStages, ss = g % Cfg::kSlots;
          if (!wait_count(&tl->ready, (unsigned)g, ready, p.cap * 4, abort, p.err)) { ok = false; break; }
          tc_fence_after();
          const uint32_t stage = smem_addr(smem + st * bStageBytes);
          const uint64_t adesc = sw128_kmajor_desc(stage), bdesc = sw128_kmajor_desc(stage + bABytes);
          const uint32_t sf = tmem + bSfCol0 + (uint32_t)ss * Cfg::kSlotCols;
#pragma unroll
          for (int j = 0; j < bBK / 64; ++j) {    // K = 64 per MMA: 32 packed bytes of each operand row
            if constexpr (kA16)                   // one word of four 16-element codes per row and MMA
              mma_mxf4nvf4_4x(tmem, adesc + 2 * j, bdesc + 2 * j, idesc[0], sf + 4u * j, sf + 16u + 8u * j,
                              (s | j) != 0);
            else
              mma_mxf4(tmem, adesc + 2 * j, bdesc + 2 * j, idesc[j & 1], sf + 4u * (j >> 1), sf + 8u + 8u * (j >> 1),
                       (s | j) != 0);
          }
          tc_commit(&tl->done[g % bDone]);              // frees the stage and the scale-factor slot
          any = true;
        }
        if (!ok) break;
        tc_commit(&tl->acc_full);
      }
      if (*abort && any) {
        tc_commit(&tl->drain);
        mbar_drain(&tl->drain, 0, bDrainCap);
      }
    }
  } else if (warp == 2) {
    // ---------------- scheduler ----------------
    if (lane == 0) {
      for (int g = 0; g < total; ++g) {
        if (!mbar_wait(&tl->full[g % bStages], (g / bStages) & 1, p.cap, abort, p.err)) break;
        if (!mbar_wait(&tl->sf_full[g % Cfg::kSlots], (g / Cfg::kSlots) & 1, p.cap, abort, p.err)) break;
        publish_count(&tl->ready, (unsigned)(g + 1));
      }
    }
  } else if (warp >= bSfWarp0 && warp < bEpiWarp0) {
    // ---------------- scale factors: E8M0 codes -> tensor memory ----------------
    // The MMAs of k-quarters 2p and 2p + 1 read an operand's codes from a
    // group of columns, row 32c + l in column c, lane l, the same words in
    // all four lane quarters, bytes 0-1 and 2-3 of a word that holds the
    // row's codes of 4 consecutive 32-k blocks: four columns for the 128
    // weight rows (A, slot column 4p), eight for the 256 token rows (B, slot
    // column 8 + 8p), so every address is aligned to its group's width.
    // Thread (quarter, lane l) stores the slab's 8 codes of weight rows
    // 32c + l (c < 4) and token rows 32c + l (c < 8) as they are in memory.
    // The codes arrive in chunks of 2 slabs per tile, 384 rows x 16 bytes
    // (weight rows first) in one of two shared-memory buffers, the next chunk
    // in flight while the current one is stored: with K % 512 == 0 two TMA
    // loads issued by one lane (16-byte rows: the row stride is a multiple of
    // 16), otherwise 8-byte cp.async by all 128 threads.  Each thread reads
    // its 12 rows 16 bytes at a time (conflict-free).  A slab's slot was last
    // used 8 slabs earlier, always in an earlier chunk, so the waits never
    // depend on the chunk being stored.  Rows past the matrix read zero codes
    // (TMA fill) or the last row's (cp.async): their operand rows are zero
    // and their results are not stored.
    const int q = warp & 3, tid = threadIdx.x - bSfWarp0 * 32;
    const uint32_t lane_addr = (uint32_t)(32 * q) << 16;
    const size_t sf_row = (size_t)(p.K / 32), sf_row_a = (size_t)(p.K / (kA16 ? 16 : 32));
    uint8_t* sfb = smem + bStages * bStageBytes;
    const int nch = (nslab + bChunk - 1) / bChunk, nunits = ntiles * nch;
    const bool issuer = kTmaSf && tid == 0;
    auto issue = [&](int u) {
      const int i = u / nch, k = u % nch;
      int m0, n0;
      tile_origin(p, tile_of(i), m0, n0);
      uint8_t* buf = sfb + (u & 1) * Cfg::kBufBytes;
      if constexpr (kTmaSf) {
        mbar_arrive_expect_tx(&tl->sf_tma[u & 1], Cfg::kBufBytes);
        tma_load_2d(buf, &tmap_wsf, &tl->sf_tma[u & 1], bSfRowBytes * k, n0);
        tma_load_2d(buf + bTW * bSfRowBytes, &tmap_asf, &tl->sf_tma[u & 1], Cfg::kARowB * k, m0);
      } else {
#pragma unroll
        for (int e = 0; e < Cfg::kPieces / (bSfWarps * 32); ++e) {
          // pieces 0 .. 2 * bTW - 1: weight rows, two per row; then the token
          // rows, kARowB / 8 per row; a piece whose slab lies past the row is
          // skipped (its codes are never read)
          const int t = tid + bSfWarps * 32 * e;
          const bool wpiece = t < 2 * bTW;
          const int tt = wpiece ? t : t - 2 * bTW, per = wpiece ? 2 : Cfg::kARowB / 8;
          const int row = tt / per, j = tt % per, rb = wpiece ? 8 : Cfg::kAScB;
          if (bChunk * k + 8 * j / rb < nslab) {
            const uint8_t* src = wpiece ? p.w_sf + (size_t)min(n0 + row, p.N - 1) * sf_row + bSfRowBytes * k
                                        : p.a_sf + (size_t)min(m0 + row, p.M - 1) * sf_row_a + Cfg::kARowB * k;
            uint8_t* dst = wpiece ? buf + row * bSfRowBytes : buf + bTW * bSfRowBytes + row * Cfg::kARowB;
            cp_async8(dst + 8 * j, src + 8 * j);
          }
        }
        cp_async_commit();
      }
    };
    bool live = true;            // every warp runs every iteration: the barrier counts stay equal
    int issued = 0;              // chunks the TMA lane has issued (it stops once its warp gave up)
    if (nunits > 0 && (issuer || !kTmaSf)) {
      issue(0);
      issued = 1;
    }
    for (int u = 0; u < nunits; ++u) {
      if (u + 1 < nunits) {
        if (!kTmaSf || (issuer && live)) {
          issue(u + 1);
          issued = u + 2;
        }
      } else if (!kTmaSf) {
        cp_async_commit();
      }
      if constexpr (kTmaSf) {
        if (live) live = mbar_wait_warp(&tl->sf_tma[u & 1], (u >> 1) & 1, p.cap, abort, p.err);
      } else {
        cp_async_wait<1>();                                      // this thread's copies of chunk u landed
        named_bar_sync(1, bSfWarps * 32);
      }
      const int i = u / nch, k = u % nch;
      const uint8_t* buf = sfb + (u & 1) * Cfg::kBufBytes;
      const uint8_t* abuf = buf + bTW * bSfRowBytes;             // token rows, kARowB bytes each
      uint4 wr[4], ar[8];                                        // rows 32c + l: both slabs' weight codes
#pragma unroll
      for (int c = 0; c < 4; ++c) wr[c] = *reinterpret_cast<const uint4*>(buf + (32 * c + lane) * bSfRowBytes);
      if constexpr (!kA16) {                                     // both slabs' token codes
#pragma unroll
        for (int c = 0; c < 8; ++c) ar[c] = *reinterpret_cast<const uint4*>(abuf + (32 * c + lane) * Cfg::kARowB);
      }
      // Both slabs of the chunk go out after one wait: the MMAs complete in
      // order, so the chunk's last slab's slot being free (slab g1 - 8 done)
      // frees the others; one wait::st then covers all the stores.
      const int s0 = bChunk * k, ns = min(bChunk, nslab - s0), g0 = i * nslab + s0, g1 = g0 + ns - 1;
      const int gp = g1 - Cfg::kSlots;
      if (live && gp >= 0) {
        live = mbar_wait_warp(&tl->done[gp % bDone], (gp / bDone) & 1, p.cap, abort, p.err);
        if (live) tc_fence_after();
      }
#pragma unroll
      for (int j = 0; j < bChunk; ++j) {
        if (j >= ns) break;
        const uint32_t at = tmem + lane_addr + bSfCol0 + (uint32_t)((g0 + j) % Cfg::kSlots) * Cfg::kSlotCols;
        if constexpr (!kA16) {
          // one 32-bit word = a row's codes of 4 consecutive 32-k blocks: the
          // MMAs of k-quarters 2p and 2p + 1 read its bytes 0-1 and 2-3
          uint32_t cols[24];
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            cols[c] = j == 0 ? wr[c].x : wr[c].z;
            cols[4 + c] = j == 0 ? wr[c].y : wr[c].w;
          }
#pragma unroll
          for (int c = 0; c < 8; ++c) {
            cols[8 + c] = j == 0 ? ar[c].x : ar[c].z;
            cols[16 + c] = j == 0 ? ar[c].y : ar[c].w;
          }
          if (live) {
            tmem_st16(at, *reinterpret_cast<const uint32_t(*)[16]>(&cols[0]));
            tmem_st8(at + 16u, *reinterpret_cast<const uint32_t(*)[8]>(&cols[16]));
          }
        } else {
          // one word per row and MMA, four codes of 16-element blocks: the
          // token codes as they are in memory; each weight code (a 32-element
          // block) covers two of them, so it is written twice
          uint32_t cols[48];
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            const uint32_t lo = j == 0 ? wr[c].x : wr[c].z, hi = j == 0 ? wr[c].y : wr[c].w;
            cols[c] = prmt(lo, 0u, 0x1100u);
            cols[4 + c] = prmt(lo, 0u, 0x3322u);
            cols[8 + c] = prmt(hi, 0u, 0x1100u);
            cols[12 + c] = prmt(hi, 0u, 0x3322u);
          }
#pragma unroll
          for (int c = 0; c < 8; ++c) {
            const uint4 a = *reinterpret_cast<const uint4*>(abuf + (32 * c + lane) * Cfg::kARowB + Cfg::kAScB * j);
            cols[16 + c] = a.x;
            cols[24 + c] = a.y;
            cols[32 + c] = a.z;
            cols[40 + c] = a.w;
          }
          if (live) {
#pragma unroll
            for (int h = 0; h < 3; ++h) tmem_st16(at + 16u * h, *reinterpret_cast<const uint32_t(*)[16]>(&cols[16 * h]));
          }
        }
      }
      if (live) {
        tmem_wait_st();
        tc_fence_before();
        for (int j = 0; j < ns; ++j) mbar_arrive_warp(&tl->sf_full[(g0 + j) % Cfg::kSlots]);
      }
      named_bar_sync(1, bSfWarps * 32);                          // buffer u & 1 is refilled by chunk u + 2
    }
    if constexpr (kTmaSf) {
      if (issuer && *abort)      // let the chunks still in flight land before the CTA moves on
        for (int u = max(0, issued - 2); u < issued; ++u) mbar_drain(&tl->sf_tma[u & 1], (u >> 1) & 1, bDrainCap);
    } else {
      cp_async_wait<0>();
    }
  } else {
    // ---------------- epilogue: TMEM -> bf16 -> Y ----------------
    // Eight warps: lane quarter warp % 4 (channel rows 32q .. 32q + 31), token
    // half h (accumulator columns 128h .. 128h + 127).  A thread packs its
    // 128 results to bf16 in registers and releases the accumulator; the
    // half then writes 16 tokens at a time into one of two staging buffers
    // ([token][128 channels], 32 consecutive channels per warp store) and one
    // lane issues the TMA tile store, which clips rows and channels past the
    // matrix.  (Per-thread global stores, 64 bytes per warp instruction,
    // held the tensor pipe back by about a sixth.)
    const int q = warp & 3, h = (warp - bEpiWarp0) >> 2, row = 32 * q + lane;
    const uint32_t lane_addr = (uint32_t)(32 * q) << 16;
    uint8_t* stg = smem + bStages * bStageBytes + Cfg::kXchBytes + h * Cfg::kStgBufs * bPieceBytes;
    const bool leader = warp == bEpiWarp0 + 4 * h && lane == 0;
    int piece = 0;
    for (int i = 0; i < ntiles; ++i) {
      if (!mbar_wait_warp(&tl->acc_full, i & 1, p.cap, abort, p.err)) break;
      tc_fence_after();
      uint32_t pk[64];
#pragma unroll
      for (int c0 = 0; c0 < 128; c0 += 16) {
        uint32_t v[16];
        tmem_ld16(tmem + lane_addr + (uint32_t)(128 * h + c0), v);
        tmem_wait_ld();
#pragma unroll
        for (int c = 0; c < 16; c += 2)
          pk[(c0 + c) / 2] = f32_to_bf16_bits(__uint_as_float(v[c])) |
                             ((uint32_t)f32_to_bf16_bits(__uint_as_float(v[c + 1])) << 16);
      }
      tc_fence_before();
      mbar_arrive_warp(&tl->acc_empty);                  // the MMAs of tile i + 1 may overwrite it
      int m0, n0;
      tile_origin(p, tile_of(i), m0, n0);
      const int t0 = m0 + 128 * h;
#pragma unroll
      for (int pc = 0; pc < 128 / bPieceTok; ++pc) {
        const int tp = t0 + bPieceTok * pc;
        if (tp >= p.M) break;                          // the remaining pieces lie past the matrix too
        uint16_t* buf = reinterpret_cast<uint16_t*>(stg + (piece % Cfg::kStgBufs) * bPieceBytes);
        if (leader) bulk_wait_read<Cfg::kStgBufs - 1>();   // the store issued from this buffer has read it
        named_bar_sync(2 + h, 128);
#pragma unroll
        for (int c = 0; c < bPieceTok; ++c)
          buf[c * bTW + row] = (uint16_t)(pk[(bPieceTok * pc + c) / 2] >> (16 * (c & 1)));
        fence_proxy_async_smem();
        named_bar_sync(2 + h, 128);
        if (leader) {
          tma_store_2d(&tmap_y, buf, 2 * n0, tp);
          bulk_commit();
        }
        ++piece;
      }
    }
    if (leader) bulk_wait_all();
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, bTmemCols);
  }
}

}  // namespace

// The W4A4 block-scaled launch (qgemm_w4a4_mxfp4 / _g for M > 16 and K % 256
// == 0; arguments validated by the caller).  g_act: the activations' block
// size, 32 or 16.  Declines (handled = false) when a scale array is not
// 8-byte aligned.
qg_status w4a4_mxfp4_bs(const uint8_t* w_e2m1, const uint8_t* w_e8m0, const uint8_t* a_e2m1,
                        const uint8_t* a_e8m0, int g_act, uint16_t* y, int M, int N, int K, cudaStream_t st,
                        bool* handled) {
  *handled = false;
  if (K % bBK != 0 || (g_act != 16 && g_act != 32) || (reinterpret_cast<uintptr_t>(w_e8m0) & 7) ||
      (reinterpret_cast<uintptr_t>(a_e8m0) & 7))
    return QG_OK;
  *handled = true;
  const bool a16 = g_act == 16;
  CUtensorMap tmap_w, tmap_a, tmap_y, tmap_wsf, tmap_asf;
  if (!make_u8_tmap_swizzled(&tmap_w, w_e2m1, N, K / 2, bTW, bBK / 2))
    return set_error(QG_ERR_CUDA, "qgemm_w4a4_mxfp4: cannot encode the weight tensor map");
  if (!make_u8_tmap_swizzled(&tmap_a, a_e2m1, M, K / 2, bTT, bBK / 2))
    return set_error(QG_ERR_CUDA, "qgemm_w4a4_mxfp4: cannot encode the activation tensor map");
  // Y as bytes [M][2N] (16-byte aligned, N % 8 == 0: checked by the caller):
  // a box of 128 channels x 16 tokens per store
  if (!make_u8_tmap(&tmap_y, y, M, 2 * N, bPieceTok, 2 * bTW))
    return set_error(QG_ERR_CUDA, "qgemm_w4a4_mxfp4: cannot encode the output tensor map");
  // Scale-factor codes by TMA: rows of K/32 (K/g_act) bytes need a 16-byte multiple
  const int arow = a16 ? Fp4Cfg<true>::kARowB : Fp4Cfg<false>::kARowB;
  const bool tma_sf = K % 512 == 0 && (reinterpret_cast<uintptr_t>(w_e8m0) & 15) == 0 &&
                      (reinterpret_cast<uintptr_t>(a_e8m0) & 15) == 0 &&
                      make_u8_tmap(&tmap_wsf, w_e8m0, N, K / 32, bTW, bSfRowBytes) &&
                      make_u8_tmap(&tmap_asf, a_e8m0, M, K / g_act, bTT, arow);
  if (!tma_sf) {
    memset(&tmap_wsf, 0, sizeof(tmap_wsf));
    memset(&tmap_asf, 0, sizeof(tmap_asf));
  }
  unsigned int* err = device_error_word();
  if (!err) return set_error(QG_ERR_CUDA, "qgemm_w4a4_mxfp4: no device error word");
  Fp4Args a{};
  a.w_sf = w_e8m0; a.a_sf = a_e8m0; a.y = y; a.M = M; a.N = N; a.K = K;
  a.tiles_t = (M + bTT - 1) / bTT;
  a.tiles_w = (N + bTW - 1) / bTW;
  a.err = err;
  a.cap = wait_limit();
  const int xch = a16 ? Fp4Cfg<true>::kXchBytes + Fp4Cfg<true>::kStgBytes
                      : Fp4Cfg<false>::kXchBytes + Fp4Cfg<false>::kStgBytes;
  const int smem = bStages * bStageBytes + xch + (int)sizeof(Fp4Tail) + 1024;
  auto kern = a16 ? (tma_sf ? w4a4_bs_kernel<true, true> : w4a4_bs_kernel<false, true>)
                  : (tma_sf ? w4a4_bs_kernel<true, false> : w4a4_bs_kernel<false, false>);
  if (!ensure_smem(kern, smem)) return set_error(QG_ERR_CUDA, "qgemm_w4a4_mxfp4: smem attribute");
  const long long tiles = (long long)a.tiles_t * a.tiles_w;
  const int grid = (int)std::min<long long>(tiles, (long long)sm_count());   // persistent: one CTA per SM
  kern<<<grid, bThreads, smem, st>>>(tmap_w, tmap_a, tmap_y, tmap_wsf, tmap_asf, a);
  return check_launch("qgemm_w4a4_mxfp4 (block-scaled)");
}

}  // namespace qg
