// Prefill (M > 16) weight-only GEMM on the 5th-generation tensor cores
// (tcgen05), one kernel template per weight format (slab.cuh): INT4 with group
// scales (symmetric or with zero points), FP8 E4M3 with channel scales, MXFP4
// and NVFP4.
//
// Orientation: the MMA computes Y^T tiles, D[n, m] = sum_k W[n,k] X[m,k].
//   * A operand = dequantized weights, 128 output channels x 16 k per MMA,
//     written straight from registers into tensor memory (tcgen05.st) by the
//     dequant warps -- the canonical bf16_RNE(q*s) never touches shared
//     memory.  ("Load INT4 weights and BF16 group scales from HBM into
//     registers, dequantize to BF16 using CUDA cores, multiply in BF16 on the
//     tensor cores", Production-Ready W4A8, "High-Performance W4A8 GEMM
//     Kernel"; the same scheme as the tcgen05 BF16 x NVFP4 kernel the 3090
//     article quotes in section 2.1.)
//   * B operand = activations, 256 tokens x 64 k per stage, TMA-loaded into
//     shared memory in the 128-byte swizzled K-major layout.
//   * D = fp32 accumulator in tensor memory, 128 lanes x 256 columns.
// Persistent: one CTA per SM walks the tiles blockIdx.x, + gridDim.x, ... of
// 256 tokens x 128 channels (raster: every channel tile of a token tile in turn), and
// every role counts the k-slabs of all its tiles in one sequence, so the
// rings simply continue from one tile into the next.
//   warp 0      TMA producer for the activations (one elected lane)
//   warp 1      TMEM allocator + MMA issuer (one elected lane)
//   warp 2      TMA producer for the packed weights, which runs ahead
//   warps 3..18 dequant producers (lane quarter = warp % 4, k half and slab
//               parity from (warp - 3) / 4), and the epilogue
//   warp 19     scheduler: waits for each k-slab's operands and publishes a
//               ready count that the MMA issuer polls
// The epilogue of a tile is done by the dequant warps once they have
// produced the first 8 slabs of the next tile: they read the accumulator
// into registers, release it (acc_empty, which the issuer waits for before
// the next tile's first MMA) and store while the MMAs of the next tile run
// (measured on GB300: 1.50 -> 1.61 PFLOP/s at M=8192, N=14336, K=4096).
// Three rings decouple them so that only the activation copy latency sits in
// front of the MMAs: 6 activation stages in shared memory (x_full: TMA bytes
// landed), 8 packed-weight stages (w_full / w_empty: the dequant warps holding
// that slab decoded it), and 8 dequantized-weight slots in tensor memory
// (a_full: the 8 dequant warps of that slab's parity stored it; a_empty: the
// MMAs of that slab completed -- one tcgen05.commit per slab, which also frees
// the slab's activation stage).
// The issuer waits on no mbarrier in the K loop: any shared-memory operation
// of the issuing thread stalls until the tensor core has taken the MMAs queued
// before it, so each wait there leaves the tensor pipe idle.  The scheduler
// warp does those waits and the issuer re-reads its counter only when the
// cached value runs out (measured on GB300: 1.06 -> 1.48 PFLOP/s at
// M=8192, N=14336, K=4096).
// Every wait is bounded; on expiry the CTA records a timeout in the device
// error word, drains its in-flight copies and MMAs, frees its tensor memory
// and returns.
#include <algorithm>

#include "slab.cuh"
#include "tc_common.cuh"

namespace qg {
namespace {

constexpr int kTileW = 128;            // weight rows (MMA M)
constexpr int kTileT = 256;            // tokens (MMA N)
constexpr int kBK = 64;                // k per stage (one 128-byte swizzle row of bf16)
constexpr int kStages = 6;             // activation stages (shared memory)
constexpr int kASlots = 8;             // dequantized-weight slots (tensor memory) and packed-weight stages
constexpr int kDeqWarps = 16;             // four sets of 4 (one per TMEM lane quarter)
constexpr int kDeqSet = 4;
constexpr int kDeqSets = kDeqWarps / kDeqSet;
constexpr int kDeq0 = 3;                            // first dequant warp
constexpr int kSchedWarp = kDeq0 + kDeqWarps;       // scheduler warp
constexpr int kThreadsTc = (kSchedWarp + 1) * 32;
constexpr int kXStageBytes = kTileT * kBK * 2;      // 32 KB activations

// Per weight format (SlabFmt): packed bytes per weight row per 64-k slab and
// activation stages (FP8's 8 KB weight stages leave room for 5).
static_assert(kBK == kSlabK, "one k-slab of the pipeline is one decoded slab");
template <int WF> struct PfTraits {
  static constexpr int WROW = SlabTraits<WF>::WROW;
  static constexpr int STAGES = WF == SF_FP8 ? 5 : 6;
  static constexpr int WSTAGE = kTileW * WROW;        // packed-weight stage bytes
};
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kACol0 = 256;                    // A slots follow the accumulator
constexpr uint32_t kACols = kBK / 2;                // 32 columns (2 bf16 per column)
constexpr uint32_t kDrainCap = 1u << 21;            // waits on work already issued (~2 s)

struct TcArgs {
  const uint8_t* wq;
  const void* ws;                      // INT4: [N][K/g] bf16; MXFP4: [N][K/32] E8M0; NVFP4: [N][K/16] E4M3
  const uint8_t* wz;                   // zero points [N][K/g] (asymmetric INT4) or nullptr
  const float* cs;                     // FP8: per-channel scales [N]
  const float* gs;                     // NVFP4: global scale (device scalar)
  uint16_t* y;
  int M, N, K, g, lg;
  int tiles_t, tiles_w, group_t;
  unsigned int* err;
  uint32_t cap;
};

struct __align__(8) TcSmemTail {
  uint64_t x_full[kStages];
  uint64_t w_full[kASlots];
  uint64_t w_empty[kASlots];
  uint64_t a_full[kASlots];
  uint64_t a_empty[kASlots];
  uint64_t acc_full;                   // all MMAs of the current tile done (one phase per tile)
  uint64_t acc_empty;                  // the epilogue has read the accumulator (one phase per tile)
  uint64_t drain;
  uint32_t tmem_base;
  int abort;
  unsigned int ready;                  // k-slabs (counted over all tiles of the CTA) whose operands are in place
};

// Grouped raster: group_t token tiles share a wave.  Tile index -> first token and channel.
QG_DEVICE void tile_origin(const TcArgs& p, int tile, int& m0, int& n0) {
  const int per_group = p.group_t * p.tiles_w;
  const int grp = tile / per_group;
  const int first_t = grp * p.group_t;
  const int gsize = min(p.group_t, p.tiles_t - first_t);
  const int within = tile - grp * per_group;
  m0 = (first_t + within % gsize) * kTileT;
  n0 = (within / gsize) * kTileW;
}

template <int WF>
__global__ void __launch_bounds__(kThreadsTc, 1)
w4a16_tc_kernel(const __grid_constant__ CUtensorMap tmap_x, const __grid_constant__ CUtensorMap tmap_w,
                const TcArgs p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  using Tr = PfTraits<WF>;
  constexpr int kSt = Tr::STAGES;
  uint8_t* xs = smem;                                                     // [kSt][32 KB]
  uint8_t* wsm = smem + kSt * kXStageBytes;                               // [kASlots][Tr::WSTAGE]
  TcSmemTail* tl = reinterpret_cast<TcSmemTail*>(wsm + kASlots * Tr::WSTAGE);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  // ---- persistent: this CTA computes tiles blockIdx.x, + gridDim.x, ... ----
  // Every role walks the same sequence of k-slabs over all of the CTA's tiles;
  // g counts them, and every ring index and barrier phase derives from g.
  const int nslab = p.K / kBK;
  const int ntiles_total = p.tiles_t * p.tiles_w;
  const int ntiles = (ntiles_total - (int)blockIdx.x + (int)gridDim.x - 1) / (int)gridDim.x;
  const int total = ntiles * nslab;
  auto tile_of = [&](int i) { return (int)blockIdx.x + i * (int)gridDim.x; };

  if (threadIdx.x == 0) {
    for (int s = 0; s < kSt; ++s) {
      mbar_init(&tl->x_full[s], 1);
    }
    for (int s = 0; s < kASlots; ++s) {
      mbar_init(&tl->w_full[s], 1);
      mbar_init(&tl->w_empty[s], kDeqSet);         // the set of 4 warps that read it
      mbar_init(&tl->a_full[s], kDeqSet);          // one arrival per warp of that set
      mbar_init(&tl->a_empty[s], 1);
    }
    mbar_init(&tl->acc_full, 1);
    mbar_init(&tl->acc_empty, kDeqWarps);          // every epilogue warp, once per tile
    mbar_init(&tl->drain, 1);
    tl->abort = 0;
    tl->ready = 0;
    mbar_fence_init();
    tma_prefetch_desc(&tmap_x);
    tma_prefetch_desc(&tmap_w);
  }
  if (warp == 1) tmem_alloc(&tl->tmem_base, kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tl->tmem_base;
  volatile int* abort = &tl->abort;

  if (warp == 0) {
    // ---------------- TMA producer: activations ----------------
    if (lane == 0) {
      int issued = 0, s = 0, i = 0, m0 = 0, n0 = 0;
      if (total > 0) tile_origin(p, tile_of(0), m0, n0);
      for (int g = 0; g < total; ++g, ++s) {
        if (s == nslab) { s = 0; tile_origin(p, tile_of(++i), m0, n0); }
        const int st = g % kSt, gp = g - kSt;           // stage last held slab gp
        if (gp >= 0 && !mbar_wait(&tl->a_empty[gp % kASlots], (gp / kASlots) & 1, p.cap, abort, p.err)) break;
        mbar_arrive_expect_tx(&tl->x_full[st], kXStageBytes);
        tma_load_2d(xs + st * kXStageBytes, &tmap_x, &tl->x_full[st], s * kBK, m0);
        issued = g + 1;
      }
      if (*abort) {     // let every copy already issued land before the CTA exits
        for (int g = max(0, issued - kSt); g < issued; ++g)
          mbar_drain(&tl->x_full[g % kSt], (g / kSt) & 1, kDrainCap);
      }
    }
  } else if (warp == 2) {
    // ---------------- TMA producer: packed weights (runs ahead) ----------------
    if (lane == 0) {
      int issued = 0, s = 0, i = 0, m0 = 0, n0 = 0;
      if (total > 0) tile_origin(p, tile_of(0), m0, n0);
      for (int g = 0; g < total; ++g, ++s) {
        if (s == nslab) { s = 0; tile_origin(p, tile_of(++i), m0, n0); }
        const int st = g % kASlots, r = g / kASlots;
        if (r > 0 && !mbar_wait(&tl->w_empty[st], (r - 1) & 1, p.cap, abort, p.err)) break;
        mbar_arrive_expect_tx(&tl->w_full[st], Tr::WSTAGE);
        tma_load_2d(wsm + st * Tr::WSTAGE, &tmap_w, &tl->w_full[st], s * Tr::WROW, n0);
        issued = g + 1;
      }
      if (*abort) {
        for (int g = max(0, issued - kASlots); g < issued; ++g)
          mbar_drain(&tl->w_full[g % kASlots], (g / kASlots) & 1, kDrainCap);
      }
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer ----------------
    if (lane == 0) {
      const uint32_t idesc = idesc_bf16_f32(kTileW, kTileT);
      bool any = false;
      unsigned int ready = 0;
      int g = 0;
      for (int i = 0; i < ntiles && !*abort; ++i) {
        // the accumulator is free once the epilogue has read the previous tile
        if (i > 0) {
          if (!mbar_wait(&tl->acc_empty, (i - 1) & 1, p.cap, abort, p.err)) break;
          tc_fence_after();
        }
        bool ok = true;
        for (int s = 0; s < nslab; ++s, ++g) {
          const int st = g % kSt, sa = g % kASlots;
          if (!wait_count(&tl->ready, (unsigned)g, ready, p.cap * 4, abort, p.err)) { ok = false; break; }
          tc_fence_after();
          const uint64_t bdesc = sw128_kmajor_desc(smem_addr(xs + st * kXStageBytes));
#pragma unroll
          for (int j = 0; j < kBK / 16; ++j)
            tc_mma_ts(tmem, tmem + kACol0 + sa * kACols + 8 * j, bdesc + 2 * j, idesc, (s | j) != 0);
          tc_commit(&tl->a_empty[sa]);                 // frees the A slot and the activation stage
          any = true;
        }
        if (!ok) break;
        tc_commit(&tl->acc_full);
      }
      if (*abort && any) {
        tc_commit(&tl->drain);                         // every MMA issued so far completes
        mbar_drain(&tl->drain, 0, kDrainCap);
      }
    }
  } else if (warp == kSchedWarp) {
    // ---------------- scheduler ----------------
    if (lane == 0) {
      for (int g = 0; g < total; ++g) {
        if (!mbar_wait(&tl->a_full[g % kASlots], (g / kASlots) & 1, p.cap, abort, p.err)) break;
        if (!mbar_wait(&tl->x_full[g % kSt], (g / kSt) & 1, p.cap, abort, p.err)) break;
        publish_count(&tl->ready, (unsigned)(g + 1));
      }
    }
  } else {
    // ---------------- dequant producers and the epilogue ----------------
    // Thread = one weight row (TMEM lane) of a 64-k slab; the four sets of 4
    // warps (one per TMEM lane quarter) take every fourth slab (g mod 4), so
    // each warp has four slab periods for its load-decode-store chain.  The
    // group scales (one per 32-k half: g may be 32) are fetched one own slab
    // ahead.  The epilogue of tile e runs once this warp is
    // about to produce the slab kASlots past the start of tile e+1: by then
    // the MMAs already have kASlots slabs of tile e+1 to work on while the
    // epilogue stores, and no slot this warp needs is held by a tile-(e+1) MMA
    // (which waits for the epilogue).
    const int dw = warp - kDeq0;
    const int q = warp & 3, set = dw >> 2;
    const int row = 32 * q + lane;
    const int cq = set;                             // epilogue: 64 of the 256 token columns
    const uint32_t lane_base = tmem + ((uint32_t)(32 * q) << 16) + kACol0;
    // scale cursor: tile index, slab in the tile, this thread's scale row
    // (and, with zero points, its zero-point row)
    struct Cur { int i, s; const uint8_t* srow; const uint8_t* zrow; };
    auto set_row = [&](Cur& c) {
      if (c.i < ntiles) {
        int m0, n0;
        tile_origin(p, tile_of(c.i), m0, n0);
        slab_rows<WF>(p.ws, p.wz, p.K, p.lg, (size_t)min(n0 + row, p.N - 1), c.srow, c.zrow);
      }
    };
    auto advance = [&](Cur& c, int by) {
      c.s += by;
      while (c.s >= nslab) { c.s -= nslab; ++c.i; set_row(c); }
    };
    auto scales_of = [&](const Cur& c, uint32_t& v0, uint32_t& v1) {
      v0 = v1 = 0u;
      if (c.i < ntiles) slab_scales<WF>(c.srow, c.zrow, c.s, p.lg, v0, v1);
    };
    // epilogue of tile e: TMEM -> registers -> (accumulator free) -> bf16 -> Y
    auto epilogue = [&](int e) -> bool {
      if (!mbar_wait_warp(&tl->acc_full, e & 1, p.cap, abort, p.err)) return false;
      tc_fence_after();
      uint32_t v[64];
      {
        uint32_t (&v0)[32] = *reinterpret_cast<uint32_t(*)[32]>(&v[0]);
        uint32_t (&v1)[32] = *reinterpret_cast<uint32_t(*)[32]>(&v[32]);
        tmem_ld32(tmem + ((uint32_t)(32 * q) << 16) + 64 * cq, v0);
        tmem_ld32(tmem + ((uint32_t)(32 * q) << 16) + 64 * cq + 32, v1);
      }
      tmem_wait_ld();
      tc_fence_before();
      mbar_arrive_warp(&tl->acc_empty);             // the MMAs of the next tile may overwrite it
      int m0, n0;
      tile_origin(p, tile_of(e), m0, n0);
      const int nn = n0 + row;
      const int mb = m0 + 64 * cq;
      if (nn < p.N) {
        // epilogue scale: FP8 per channel, NVFP4 global, none for INT4 / MXFP4
        float es = 1.f;
        if constexpr (WF == SF_FP8) es = __ldg(p.cs + nn);
        if constexpr (WF == SF_NVFP4) es = __ldg(p.gs) * kNvfp4Unfold;   // the slab decode's 2^-9 undone
#pragma unroll
        for (int c = 0; c < 64; ++c) {
          float val = __uint_as_float(v[c]);
          if constexpr (SlabTraits<WF>::EPI_SCALE) val *= es;
          if (mb + c < p.M) p.y[(size_t)(mb + c) * p.N + nn] = f32_to_bf16_bits(val);
        }
      }
      return true;
    };
    int e_next = 0;                                 // next tile whose epilogue this warp owes
    bool ok = true;
    Cur pf{0, 0, nullptr, nullptr};
    set_row(pf);
    advance(pf, set);
    uint32_t sc_cur0, sc_cur1, sc_nxt0, sc_nxt1;
    scales_of(pf, sc_cur0, sc_cur1);
    advance(pf, kDeqSets);
    scales_of(pf, sc_nxt0, sc_nxt1);
    for (int g = set; g < total; g += kDeqSets) {
      while (e_next < ntiles - 1 && g >= (e_next + 1) * nslab + kASlots) {
        if (!(ok = epilogue(e_next))) break;
        ++e_next;
      }
      if (!ok) break;
      const int sa = g % kASlots, ra = g / kASlots;
      const uint32_t v0 = sc_cur0, v1 = sc_cur1;
      sc_cur0 = sc_nxt0;
      sc_cur1 = sc_nxt1;
      advance(pf, kDeqSets);                        // pf now at this set's slab after the next
      scales_of(pf, sc_nxt0, sc_nxt1);
      if (!mbar_wait_warp(&tl->w_full[sa], ra & 1, p.cap, abort, p.err)) { ok = false; break; }
      uint32_t out[32];
      decode_slab<WF>(wsm + sa * Tr::WSTAGE + row * Tr::WROW, row, v0, v1, out);
      mbar_arrive_warp(&tl->w_empty[sa]);           // packed slab decoded: its stage may be refilled
      if (ra > 0) {
        if (!mbar_wait_warp(&tl->a_empty[sa], (ra - 1) & 1, p.cap, abort, p.err)) { ok = false; break; }
        tc_fence_after();
      }
      {
        const uint32_t (&o0)[16] = *reinterpret_cast<const uint32_t(*)[16]>(&out[0]);
        const uint32_t (&o1)[16] = *reinterpret_cast<const uint32_t(*)[16]>(&out[16]);
        tmem_st16(lane_base + sa * kACols, o0);
        tmem_st16(lane_base + sa * kACols + 16, o1);
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
    tmem_dealloc(tmem, kTmemCols);
  }
}

// ---- host: tensor map + launch -------------------------------------------------
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  if (!fn) {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess && q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(f);
  }
  return fn;
}

}  // namespace

// bf16 [rows][cols] row-major -> TMA map with a (box_cols x box_rows) box, 128-byte swizzle
// u8 [rows][cols] row-major -> TMA map with a (box_cols x box_rows) box, no swizzle
bool make_u8_tmap(CUtensorMap* m, const void* base, int rows, int cols, int box_rows, int box_cols) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)cols};
  const cuuint32_t box[2] = {(cuuint32_t)box_cols, (cuuint32_t)box_rows};
  const cuuint32_t estr[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Byte matrix staged in a swizzled shared-memory layout: 128-byte swizzle (the
// layout a K-major MMA operand descriptor reads; box_cols == 128) or 64-byte
// swizzle (box_cols == 64: 16-byte chunk c of row r lands at chunk
// c ^ ((r >> 1) & 3), so 8 consecutive rows read at one chunk offset hit 8
// different bank groups).
bool make_u8_tmap_swizzled(CUtensorMap* m, const void* base, int rows, int cols, int box_rows, int box_cols) {
  EncodeTiledFn fn = encode_fn();
  if (!fn || (box_cols != 128 && box_cols != 64)) return false;
  const cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)cols};
  const cuuint32_t box[2] = {(cuuint32_t)box_cols, (cuuint32_t)box_rows};
  const cuuint32_t estr[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, box_cols == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool make_bf16_tmap(CUtensorMap* m, const void* base, int rows, int cols, int box_rows, int box_cols) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)cols * 2};
  const cuuint32_t box[2] = {(cuuint32_t)box_cols, (cuuint32_t)box_rows};
  const cuuint32_t estr[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// The prefill dispatcher.  wf is a WFmt; w_s is the format's scale array
// (INT4 bf16 per group, MXFP4 E8M0 per 32, NVFP4 E4M3 per 16, unused for
// FP8), w_z the zero points (INT4Z), cs the FP8 channel scales, gs the NVFP4
// global scale.  Declines (handled = false) shapes for the decode kernel.
qg_status prefill_tc(int wf, const uint8_t* w_q, const void* w_s, const uint8_t* w_z, const float* cs,
                     const float* gs, int g, const uint16_t* x, uint16_t* y, int M, int N, int K,
                     cudaStream_t st, bool* handled, const char* name) {
  *handled = false;
  if (M <= 16 || K % kBK != 0) return QG_OK;
  if ((wf == SF_INT4 || wf == SF_INT4Z) && (g < 32 || (g & (g - 1)) != 0 || K % g != 0)) return QG_OK;
  // the FP4 block scales are read two (MXFP4) or four (NVFP4) codes at a time
  if (wf == SF_MXFP4 && (reinterpret_cast<uintptr_t>(w_s) & 1)) return QG_OK;
  if (wf == SF_NVFP4 && (reinterpret_cast<uintptr_t>(w_s) & 3)) return QG_OK;
  *handled = true;
  const int wrow = wf == SF_FP8 ? kBK : kBK / 2;        // packed bytes per row per slab
  CUtensorMap tmap, tmap_w;
  if (!make_bf16_tmap(&tmap, x, M, K, kTileT, kBK))
    return set_error(QG_ERR_CUDA, "%s: cannot encode the activation tensor map", name);
  const bool wok = wf == SF_FP8 ? make_u8_tmap_swizzled(&tmap_w, w_q, N, K, kTileW, wrow)
                                : make_u8_tmap(&tmap_w, w_q, N, K / 2, kTileW, wrow);
  if (!wok) return set_error(QG_ERR_CUDA, "%s: cannot encode the weight tensor map", name);
  unsigned int* err = device_error_word();
  if (!err) return set_error(QG_ERR_CUDA, "%s: no device error word", name);
  TcArgs a{};
  a.wq = w_q; a.ws = w_s; a.wz = w_z; a.cs = cs; a.gs = gs; a.y = y; a.M = M; a.N = N; a.K = K; a.g = g;
  a.lg = 0;
  while ((1 << a.lg) < g) ++a.lg;
  a.tiles_t = (M + kTileT - 1) / kTileT;
  a.tiles_w = (N + kTileW - 1) / kTileW;
  a.group_t = 1;          // token tiles per raster group (8 / 4 / 2 / 1: 1673 / 1690 / 1705 / 1705+ TFLOP/s)
  a.err = err;
  a.cap = wait_limit();
  const int stages = wf == SF_FP8 ? PfTraits<SF_FP8>::STAGES : PfTraits<SF_INT4>::STAGES;
  const int smem = stages * kXStageBytes + kASlots * kTileW * wrow + (int)sizeof(TcSmemTail) + 1024;
  void (*kern)(const __grid_constant__ CUtensorMap, const __grid_constant__ CUtensorMap, const TcArgs) = nullptr;
  switch (wf) {
    case SF_INT4: kern = w4a16_tc_kernel<SF_INT4>; break;
    case SF_INT4Z: kern = w4a16_tc_kernel<SF_INT4Z>; break;
    case SF_FP8: kern = w4a16_tc_kernel<SF_FP8>; break;
    case SF_MXFP4: kern = w4a16_tc_kernel<SF_MXFP4>; break;
    case SF_NVFP4: kern = w4a16_tc_kernel<SF_NVFP4>; break;
    default: return set_error(QG_ERR_INVALID_ARG, "%s: unknown prefill format %d", name, wf);
  }
  if (!ensure_smem(kern, smem)) return set_error(QG_ERR_CUDA, "%s: smem attribute", name);
  const long long tiles = (long long)a.tiles_t * a.tiles_w;
  const int grid = (int)std::min<long long>(tiles, (long long)sm_count());   // persistent: one CTA per SM
  kern<<<grid, kThreadsTc, smem, st>>>(tmap, tmap_w, a);
  return check_launch(name);
}

}  // namespace qg
