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
//   B operand = packed E2M1 activations, 128 tokens x 256 k, the same way;
//   scale factors = E8M0 codes in tensor memory, written from registers
//               (tcgen05.st) by four warps: for the MMA of k-quarter j (64 k,
//               two 32-k blocks) a 128-row operand's codes fill a group of
//               four columns, row 32c + l in column c, lane l (all four lane
//               quarters hold the same words), bytes 0 and 1 (scale-factor ID
//               0); A's group is column 8j of the slab's slot, B's 8j + 4, so
//               every scale-factor address is 4-column aligned;
//   D         = fp32, two 128-column accumulators (the epilogue of tile i
//               overlaps the MMAs of tile i + 1).
// Persistent: one CTA per SM walks the tiles blockIdx.x, + gridDim.x, ... of
// 128 tokens x 128 channels (every channel tile of a token tile in turn, so a
// token tile's activations are read once).  Every role counts the k-slabs of
// all its tiles in one sequence g.
//   warp 0      TMA for both operands (one elected lane; 6 stages of 32 KB)
//   warp 1      TMEM allocation and MMA issuer (one lane)
//   warp 2      scheduler: waits for each slab's operands and scale factors,
//               publishes the ready count the issuer polls
//   warps 3-10  scale factors: two sets of 4 (lane quarter = warp % 4) taking
//               alternate slabs, each loading its next slab's codes while it
//               stores the current one
//   warps 11-14 epilogue: lane quarter = warp % 4, TMEM -> bf16 -> Y
// Every wait is bounded; on expiry the CTA records a timeout in the device
// error word, drains what it issued, frees its tensor memory and returns.
#include <algorithm>

#include "tc_common.cuh"

namespace qg {

bool make_u8_tmap_swizzled(CUtensorMap* m, const void* base, int rows, int cols, int box_rows, int box_cols);

namespace {

constexpr int bTW = 128;                 // channels per tile (MMA M)
constexpr int bTT = 128;                 // tokens per tile (MMA N)
constexpr int bBK = 256;                 // k per slab: 128 packed bytes per row
constexpr int bStages = 6;               // operand stages (A + B)
constexpr int bSfSlots = 8;              // scale-factor slots in tensor memory
constexpr int bDone = 8;                 // slab-completion barriers
constexpr int bOpBytes = bTW * bBK / 2;  // 16 KB per operand per stage
constexpr int bStageBytes = 2 * bOpBytes;
constexpr int bSfWarp0 = 3, bSfSets = 2, bEpiWarp0 = bSfWarp0 + 4 * bSfSets;
constexpr int bThreads = (bEpiWarp0 + 4) * 32;
constexpr uint32_t bTmemCols = 512;
constexpr uint32_t bSfCol0 = 2 * bTT;    // scale-factor slots follow the two accumulators
constexpr uint32_t bSfCols = 32;         // per slot: MMA j reads A at +8j, B at +8j+4 (4-column aligned)
constexpr uint32_t bDrainCap = 1u << 21;
static_assert(bDone >= bStages && bDone >= bSfSlots, "slab-completion ring covers every reuse distance");
static_assert(bSfCol0 + bSfSlots * bSfCols <= bTmemCols, "tensor memory budget");
static_assert(bSfSlots % bSfSets == 0 && bDone % bSfSets == 0, "a set waits only on its own done entries, in order");

struct Fp4Args {
  const uint8_t* w_sf;                   // [N][K/32] E8M0
  const uint8_t* a_sf;                   // [M][K/32] E8M0
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
  uint64_t acc_full[2];                  // the tile's MMAs completed (one phase per use)
  uint64_t acc_empty[2];                 // the epilogue has read the accumulator (4 warps)
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

QG_DEVICE void tile_origin(const Fp4Args& p, int tile, int& m0, int& n0) {
  m0 = (tile / p.tiles_w) * bTT;         // every channel tile of a token tile in turn
  n0 = (tile % p.tiles_w) * bTW;
}

__global__ void __launch_bounds__(bThreads, 1)
w4a4_bs_kernel(const __grid_constant__ CUtensorMap tmap_w, const __grid_constant__ CUtensorMap tmap_a,
               const Fp4Args p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  Fp4Tail* tl = reinterpret_cast<Fp4Tail*>(smem + bStages * bStageBytes);
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
    for (int s = 0; s < bSfSlots; ++s) mbar_init(&tl->sf_full[s], 4);     // the 4 warps of the slot's set
    for (int d = 0; d < bDone; ++d) mbar_init(&tl->done[d], 1);
    for (int b = 0; b < 2; ++b) {
      mbar_init(&tl->acc_full[b], 1);
      mbar_init(&tl->acc_empty[b], 4);
    }
    mbar_init(&tl->drain, 1);
    tl->abort = 0;
    tl->ready = 0;
    mbar_fence_init();
    tma_prefetch_desc(&tmap_w);
    tma_prefetch_desc(&tmap_a);
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
        tma_load_2d(stage + bOpBytes, &tmap_a, &tl->full[st], s * (bBK / 2), m0);
        issued = g + 1;
      }
      if (*abort) {     // let every copy already issued land before the CTA moves on
        for (int g = max(0, issued - bStages); g < issued; ++g)
          mbar_wait(&tl->full[g % bStages], (g / bStages) & 1, bDrainCap, abort, nullptr);
      }
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer ----------------
    if (lane == 0) {
      const uint32_t idesc = idesc_mxf4(bTW, bTT, 0);
      bool any = false;
      unsigned int ready = 0;
      int g = 0;
      for (int i = 0; i < ntiles && !*abort; ++i) {
        const int b = i & 1;
        if (i >= 2) {             // the accumulator is free once the epilogue has read tile i - 2
          if (!mbar_wait(&tl->acc_empty[b], ((i - 2) >> 1) & 1, p.cap, abort, p.err)) break;
          tc_fence_after();
        }
        bool ok = true;
        for (int s = 0; s < nslab; ++s, ++g) {
          const int st = g % bStages, ss = g % bSfSlots;
          if (!wait_count(&tl->ready, (unsigned)g, ready, p.cap * 4, abort, p.err)) { ok = false; break; }
          tc_fence_after();
          const uint32_t stage = smem_addr(smem + st * bStageBytes);
          const uint64_t adesc = sw128_kmajor_desc(stage), bdesc = sw128_kmajor_desc(stage + bOpBytes);
          const uint32_t sf = tmem + bSfCol0 + (uint32_t)ss * bSfCols;
#pragma unroll
          for (int j = 0; j < bBK / 64; ++j)      // K = 64 per MMA: 32 packed bytes of each operand row
            mma_mxf4(tmem + (uint32_t)(b * bTT), adesc + 2 * j, bdesc + 2 * j, idesc,
                     sf + 8u * j, sf + 8u * j + 4u, (s | j) != 0);
          tc_commit(&tl->done[g % bDone]);              // frees the stage and the scale-factor slot
          any = true;
        }
        if (!ok) break;
        tc_commit(&tl->acc_full[b]);
      }
      if (*abort && any) {
        tc_commit(&tl->drain);
        mbar_wait(&tl->drain, 0, bDrainCap, abort, nullptr);
      }
    }
  } else if (warp == 2) {
    // ---------------- scheduler ----------------
    if (lane == 0) {
      for (int g = 0; g < total; ++g) {
        if (!mbar_wait(&tl->full[g % bStages], (g / bStages) & 1, p.cap, abort, p.err)) break;
        if (!mbar_wait(&tl->sf_full[g % bSfSlots], (g / bSfSlots) & 1, p.cap, abort, p.err)) break;
        publish_count(&tl->ready, (unsigned)(g + 1));
      }
    }
  } else if (warp >= bSfWarp0 && warp < bEpiWarp0) {
    // ---------------- scale factors: E8M0 codes -> tensor memory ----------------
    // The MMA of k-quarter j (64 k: two 32-k blocks) reads the codes of a
    // 128-row operand from a group of four columns: row 32c + l sits in column
    // c, lane l, bytes 0 and 1 (scale-factor ID 0); the same words are
    // written into all four lane quarters.  A's group for MMA j is column 8j
    // of the slab's slot, B's column 8j + 4, so every address is 4-column
    // aligned.  Thread (quarter, lane l) loads the slab's 8 codes of rows
    // l, 32 + l, 64 + l and 96 + l of both operands; the two sets take
    // alternate slabs (so a slot is always written by the same set) and load
    // their next slab's codes while storing the current one.
    const int q = warp & 3, set = (warp - bSfWarp0) >> 2;
    const uint32_t lane_addr = (uint32_t)(32 * q) << 16;
    const size_t sf_row = (size_t)(p.K / 32);
    // codes of slab gn (tile index i, slab s of the tile) for this thread's rows;
    // rows past the matrix take the last row's codes: their operand rows are
    // zero (TMA fill) and their results are not stored
    auto load = [&](int i, int s, uint2 (&wv)[4], uint2 (&av)[4]) {
      int m0, n0;
      tile_origin(p, tile_of(i), m0, n0);
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        wv[c] = __ldg(reinterpret_cast<const uint2*>(p.w_sf + (size_t)min(n0 + 32 * c + lane, p.N - 1) * sf_row + s * 8));
        av[c] = __ldg(reinterpret_cast<const uint2*>(p.a_sf + (size_t)min(m0 + 32 * c + lane, p.M - 1) * sf_row + s * 8));
      }
    };
    uint2 wv[4], av[4];
    if (set < total) load(set / nslab, set % nslab, wv, av);
    for (int g = set; g < total; g += bSfSets) {
      uint32_t cols[32];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const uint32_t w = j < 2 ? wv[c].x : wv[c].y, a = j < 2 ? av[c].x : av[c].y;
          cols[8 * j + c] = (w >> (16 * (j & 1))) & 0xFFFFu;       // blocks 2j, 2j + 1 of row 32c + l
          cols[8 * j + 4 + c] = (a >> (16 * (j & 1))) & 0xFFFFu;
        }
      }
      const int gn = g + bSfSets;                                // this set's next slab: load it now
      if (gn < total) load(gn / nslab, gn % nslab, wv, av);
      const int ss = g % bSfSlots, gp = g - bSfSlots;            // the slot last held slab gp
      if (gp >= 0) {
        if (!mbar_wait_warp(&tl->done[gp % bDone], (gp / bDone) & 1, p.cap, abort, p.err)) break;
        tc_fence_after();
      }
      {
        const uint32_t (&c0)[16] = *reinterpret_cast<const uint32_t(*)[16]>(&cols[0]);
        const uint32_t (&c1)[16] = *reinterpret_cast<const uint32_t(*)[16]>(&cols[16]);
        const uint32_t at = tmem + lane_addr + bSfCol0 + (uint32_t)ss * bSfCols;
        tmem_st16(at, c0);
        tmem_st16(at + 16, c1);
      }
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive_warp(&tl->sf_full[ss]);
    }
  } else {
    // ---------------- epilogue: TMEM -> bf16 -> Y ----------------
    const int q = warp & 3, row = 32 * q + lane;
    const uint32_t lane_addr = (uint32_t)(32 * q) << 16;
    for (int i = 0; i < ntiles; ++i) {
      const int b = i & 1;
      if (!mbar_wait_warp(&tl->acc_full[b], (i >> 1) & 1, p.cap, abort, p.err)) break;
      tc_fence_after();
      int m0, n0;
      tile_origin(p, tile_of(i), m0, n0);
      const int nn = n0 + row;
#pragma unroll 1
      for (int c0 = 0; c0 < bTT; c0 += 32) {
        uint32_t v[32];
        tmem_ld32(tmem + lane_addr + (uint32_t)(b * bTT + c0), v);
        tmem_wait_ld();
        if (c0 + 32 == bTT) {
          tc_fence_before();
          mbar_arrive_warp(&tl->acc_empty[b]);           // the MMAs of tile i + 2 may overwrite it
        }
        if (nn < p.N) {
#pragma unroll
          for (int c = 0; c < 32; ++c)
            if (m0 + c0 + c < p.M) p.y[(size_t)(m0 + c0 + c) * p.N + nn] = f32_to_bf16_bits(__uint_as_float(v[c]));
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, bTmemCols);
  }
}

}  // namespace

// The W4A4 block-scaled launch (qgemm_w4a4_mxfp4 for M > 16 and K % 256 == 0;
// arguments validated by the caller).  Declines (handled = false) when a
// scale array is not 8-byte aligned.
qg_status w4a4_mxfp4_bs(const uint8_t* w_e2m1, const uint8_t* w_e8m0, const uint8_t* a_e2m1,
                        const uint8_t* a_e8m0, uint16_t* y, int M, int N, int K, cudaStream_t st, bool* handled) {
  *handled = false;
  if (K % bBK != 0 || (reinterpret_cast<uintptr_t>(w_e8m0) & 7) || (reinterpret_cast<uintptr_t>(a_e8m0) & 7))
    return QG_OK;
  *handled = true;
  CUtensorMap tmap_w, tmap_a;
  if (!make_u8_tmap_swizzled(&tmap_w, w_e2m1, N, K / 2, bTW, bBK / 2))
    return set_error(QG_ERR_CUDA, "qgemm_w4a4_mxfp4: cannot encode the weight tensor map");
  if (!make_u8_tmap_swizzled(&tmap_a, a_e2m1, M, K / 2, bTT, bBK / 2))
    return set_error(QG_ERR_CUDA, "qgemm_w4a4_mxfp4: cannot encode the activation tensor map");
  unsigned int* err = device_error_word();
  if (!err) return set_error(QG_ERR_CUDA, "qgemm_w4a4_mxfp4: no device error word");
  Fp4Args a{};
  a.w_sf = w_e8m0; a.a_sf = a_e8m0; a.y = y; a.M = M; a.N = N; a.K = K;
  a.tiles_t = (M + bTT - 1) / bTT;
  a.tiles_w = (N + bTW - 1) / bTW;
  a.err = err;
  a.cap = wait_limit();
  const int smem = bStages * bStageBytes + (int)sizeof(Fp4Tail) + 1024;
  if (!ensure_smem(w4a4_bs_kernel, smem)) return set_error(QG_ERR_CUDA, "qgemm_w4a4_mxfp4: smem attribute");
  const long long tiles = (long long)a.tiles_t * a.tiles_w;
  const int grid = (int)std::min<long long>(tiles, (long long)sm_count());   // persistent: one CTA per SM
  w4a4_bs_kernel<<<grid, bThreads, smem, st>>>(tmap_w, tmap_a, a);
  return check_launch("qgemm_w4a4_mxfp4 (block-scaled)");
}

}  // namespace qg
