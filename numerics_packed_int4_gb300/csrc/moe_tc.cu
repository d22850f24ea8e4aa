// W4A8 grouped (MoE) GEMM on the 5th-generation tensor cores, one CTA pair
// (a cluster of two) per 256-channel x 256-row output tile of one expert.
//
// Semantics (Production-Ready W4A8): y[r,n] = a_s[r] * sum_k e4m3(a[r,k]) *
// q[n,k] * s[n, k/128], every product exact, fp32 accumulation, one bf16
// rounding at the store.  To keep that exactness on a 16-bit MMA, the
// weights are formed as fp16(q * s * 2^e_n): q is a 4-bit integer and s a
// bf16 (8 significant bits), so q * s has at most 11 significant bits and is
// exact in fp16; the per-row power of two e_n puts the row's largest scale in
// [2^11, 2^12) so every product stays inside fp16's range, and the epilogue
// multiplies by 2^-e_n exactly.  E4M3 activations are exact in fp16 too.
//
// Pair MMA (tcgen05.mma.cta_group::2, M = 256, N = 256, K = 16): each CTA
// holds 128 weight rows (A, dequantized into its own tensor memory) and 128
// of the 256 activation rows (B, fp16 in its own shared memory); each CTA's
// accumulator holds its 128 channels x all 256 rows.  Splitting B over the
// pair halves each SM's shared-memory traffic for the activations -- the E4M3
// copy, the converters' read and fp16 write, and the MMA read -- which bounds
// the single-CTA form of this kernel.
// Roles in each CTA:
//   warp 0       TMA producer for the CTA's packed weight rows (8 stages)
//   warp 1       TMEM allocation for the pair; in the even CTA one lane issues
//                the MMAs, one multicast tcgen05.commit per slab
//   warp 2       TMA producer for the CTA's 128 E4M3 activation rows (8 stages)
//   warps 3-18   dequant producers (four sets of 4, one warp per TMEM lane
//                quarter, each set taking every fourth slab; a thread decodes
//                its row's whole 64-k slab) into 8 tensor-memory slots, then
//                the epilogue
//   warps 19-22  converters: E4M3 stage -> fp16 stage in the 128-byte swizzled
//                K-major layout (cvt.rn.f16x2.e4m3x2), 8 stages
//   warp 23      scheduler (even CTA): waits for slab_full and publishes the
//                ready count that the MMA issuer polls
//   warps 24-27  relays (odd CTA): each takes every fourth slab, waits for the
//                CTA's local half_full and arrives on the even CTA's slab_full
// Barriers: slab_full (even CTA: its 4 dequant + 4 converter warps of the slab
// and one relay arrival), half_full (odd CTA: the same 8 local arrivals),
// a_empty (the pair's MMAs of the slab completed; frees the A slot and the
// fp16 stage in both CTAs), x_full / x_empty (E4M3 stage), w_full / w_empty
// (packed weights), acc_full.  The relays exist because the cross-CTA arrive
// needs cluster-scope release, which costs a few hundred nanoseconds; four
// relays in parallel keep it off the per-slab critical path, while each
// worker only releases at CTA scope.
// One pair computes one tile; tiles are located on the device from
// expert_off, so launching needs no host sync.  Every wait is bounded; on
// expiry the CTA records a timeout, drains what it issued, meets its peer at
// the final cluster barrier and frees its tensor memory.
#include <algorithm>
#include <cmath>

#include "dequant.cuh"
#include "tc_common.cuh"

namespace qg {

bool make_u8_tmap(CUtensorMap* m, const void* base, int rows, int cols, int box_rows, int box_cols);

namespace {

constexpr int mTW = 128;                 // weight rows per CTA (half of the MMA's M = 256)
constexpr int mTT = 256;                 // activation rows per pair (MMA N)
constexpr int mHT = mTT / 2;             // activation rows held by each CTA
constexpr int mBK = 64;                  // k per slab
constexpr int mSlots = 8;                // fp16 stages = TMEM A slots = packed-weight stages
constexpr int mXStages = 8;              // E4M3 stages
constexpr int mDeqWarps = 16;            // four sets of 4 (one per TMEM lane quarter)
constexpr int mDeqSet = 4;
constexpr int mDeqSets = mDeqWarps / mDeqSet;
constexpr int mCvtWarps = 4;
constexpr int mRelays = 4;
constexpr int mDeq0 = 3;
constexpr int mCvt0 = mDeq0 + mDeqWarps;
constexpr int mSchedWarp = mCvt0 + mCvtWarps;
constexpr int mRelay0 = mSchedWarp + 1;
constexpr int mThreads = (mRelay0 + mRelays) * 32;
constexpr int mBStage = mHT * mBK * 2;   // 16 KB fp16 activations (swizzled)
constexpr int mXStage = mHT * mBK;       // 8 KB E4M3 activations (TMA)
constexpr int mWStage = mTW * mBK / 2;   // 4 KB packed INT4 weights (TMA)
constexpr int mLocalArrivals = mDeqSet + mCvtWarps;   // per CTA per slab
constexpr uint32_t mTmemCols = 512;
constexpr uint32_t mACol0 = 256;
constexpr uint32_t mACols = mBK / 2;
constexpr uint32_t mDrainCap = 1u << 21;

struct MoeTcArgs {
  const float* a_s;
  const int32_t* off;
  const uint16_t* ws;
  uint16_t* y;
  int R, E, N, K;
  int tiles_w;                           // 256-channel pair tiles per expert
  unsigned int* err;
  uint32_t cap;
};

struct __align__(8) MoeTail {
  uint64_t slab_full[mSlots];            // even CTA
  uint64_t half_full[mSlots];            // odd CTA
  uint64_t a_empty[mSlots];
  uint64_t w_full[mSlots];
  uint64_t w_empty[mSlots];
  uint64_t x_full[mXStages];
  uint64_t x_empty[mXStages];
  uint64_t acc_full;
  uint64_t drain;
  uint32_t tmem_base;
  int abort;
  unsigned int ready;                    // k-slabs whose operands are in place in both CTAs
};

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(mThreads, 1)
moe_w4a8_tc_kernel(const __grid_constant__ CUtensorMap tmap_a, const __grid_constant__ CUtensorMap tmap_w,
                   const MoeTcArgs p) {
  // ---- tile of this pair: expert, weight pair tile, row tile (before any setup) ----
  int tile = blockIdx.x >> 1, e = -1, r0 = 0, r_end = 0, wt = 0;
  for (int i = 0; i < p.E; ++i) {
    const int a = __ldg(p.off + i), b = __ldg(p.off + i + 1);
    const int nt = b > a ? (b - a + mTT - 1) / mTT : 0;
    const int cnt = nt * p.tiles_w;
    if (tile < cnt) {
      e = i;
      wt = tile / nt;
      r0 = a + (tile - wt * nt) * mTT;
      r_end = b;
      break;
    }
    tile -= cnt;
  }
  if (e < 0) return;                     // both CTAs of the pair see the same tile
  const uint32_t rank = cluster_ctarank();
  const int n0 = wt * (2 * mTW) + (int)rank * mTW;     // this CTA's first channel
  const int nslab = p.K / mBK;

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* bs = smem;                                    // [mSlots][16 KB] fp16, swizzled
  uint8_t* as8 = bs + mSlots * mBStage;                  // [mXStages][8 KB] E4M3
  uint8_t* wsm = as8 + mXStages * mXStage;               // [mSlots][4 KB] INT4
  MoeTail* tl = reinterpret_cast<MoeTail*>(wsm + mSlots * mWStage);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < mSlots; ++s) {
      mbar_init(&tl->slab_full[s], mLocalArrivals + 1);   // local workers + one relay arrival
      mbar_init(&tl->half_full[s], mLocalArrivals);
      mbar_init(&tl->a_empty[s], 1);                      // the pair's multicast commit
      mbar_init(&tl->w_full[s], 1);
      mbar_init(&tl->w_empty[s], mDeqSet);
    }
    for (int s = 0; s < mXStages; ++s) {
      mbar_init(&tl->x_full[s], 1);
      mbar_init(&tl->x_empty[s], mCvtWarps);
    }
    mbar_init(&tl->acc_full, 1);
    mbar_init(&tl->drain, 1);
    tl->abort = 0;
    tl->ready = 0;
    mbar_fence_init();
    tma_prefetch_desc(&tmap_a);
    tma_prefetch_desc(&tmap_w);
  }
  if (warp == 1) tmem_alloc_pair(&tl->tmem_base, mTmemCols);
  tc_fence_before();
  cluster_sync_all();          // both CTAs' barriers exist before any remote arrive or multicast
  tc_fence_after();
  const uint32_t tmem = tl->tmem_base;
  volatile int* abort = &tl->abort;
  // per-slab "this CTA's operands are in place" barrier
  uint64_t* local_full = rank == 0 ? tl->slab_full : tl->half_full;

  if (warp == 0) {
    // ---------------- TMA producer: packed weights (runs ahead) ----------------
    if (lane == 0) {
      int issued = 0;
      for (int s = 0; s < nslab; ++s) {
        const int st = s % mSlots, r = s / mSlots;
        if (r > 0 && !mbar_wait(&tl->w_empty[st], (r - 1) & 1, p.cap, abort, p.err)) break;
        mbar_arrive_expect_tx(&tl->w_full[st], mWStage);
        tma_load_2d(wsm + st * mWStage, &tmap_w, &tl->w_full[st], s * (mBK / 2), e * p.N + n0);
        issued = s + 1;
      }
      if (*abort) {     // let every copy already issued land before the CTA moves on
        for (int s = max(0, issued - mSlots); s < issued; ++s)
          mbar_wait(&tl->w_full[s % mSlots], (s / mSlots) & 1, mDrainCap, abort, nullptr);
      }
    }
  } else if (warp == 2) {
    // ---------------- TMA producer: this CTA's E4M3 activation rows ----------------
    if (lane == 0) {
      int issued = 0;
      for (int s = 0; s < nslab; ++s) {
        const int st = s % mXStages, r = s / mXStages;
        if (r > 0 && !mbar_wait(&tl->x_empty[st], (r - 1) & 1, p.cap, abort, p.err)) break;
        mbar_arrive_expect_tx(&tl->x_full[st], mXStage);
        tma_load_2d(as8 + st * mXStage, &tmap_a, &tl->x_full[st], s * mBK, r0 + (int)rank * mHT);
        issued = s + 1;
      }
      if (*abort) {
        for (int s = max(0, issued - mXStages); s < issued; ++s)
          mbar_wait(&tl->x_full[s % mXStages], (s / mXStages) & 1, mDrainCap, abort, nullptr);
      }
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer (even CTA) ----------------
    if (rank == 0 && lane == 0) {
      const uint32_t idesc = idesc_f16_f32(2 * mTW, mTT);
      bool any = false;
      unsigned int ready = 0;
      for (int s = 0; s < nslab; ++s) {
        const int sa = s % mSlots;
        if (!wait_count(&tl->ready, (unsigned)s, ready, p.cap * 4, abort, p.err)) break;
        tc_fence_after();
        const uint64_t bdesc = sw128_kmajor_desc(smem_addr(bs + sa * mBStage));
#pragma unroll
        for (int j = 0; j < mBK / 16; ++j)
          tc_mma2_ts(tmem, tmem + mACol0 + sa * mACols + 8 * j, bdesc + 2 * j, idesc, (s | j) != 0);
        tc_commit_pair(&tl->a_empty[sa], 3);           // frees the A slots and fp16 stages of both CTAs
        any = true;
      }
      if (!*abort) {
        tc_commit_pair(&tl->acc_full, 3);
      } else if (any) {
        tc_commit_pair(&tl->drain, 1);
        mbar_wait(&tl->drain, 0, mDrainCap, abort, nullptr);
      }
    }
  } else if (warp == mSchedWarp) {
    // ---------------- scheduler (even CTA) ----------------
    if (rank == 0 && lane == 0) {
      for (int s = 0; s < nslab; ++s) {
        if (!mbar_wait_cluster(&tl->slab_full[s % mSlots], (s / mSlots) & 1, p.cap, abort, p.err)) break;
        publish_count(&tl->ready, (unsigned)(s + 1));
      }
    }
  } else if (warp >= mRelay0) {
    // ---------------- relays (odd CTA): half_full -> even CTA's slab_full ----------------
    if (rank == 1 && lane == 0) {
      for (int s = warp - mRelay0; s < nslab; s += mRelays) {
        if (!mbar_wait(&tl->half_full[s % mSlots], (s / mSlots) & 1, p.cap, abort, p.err)) break;
        mbar_arrive_remote(&tl->slab_full[s % mSlots], 0);
      }
    }
  } else if (warp >= mCvt0) {
    // ---------------- converters: E4M3 stage -> fp16 swizzled stage ----------------
    // Warp cw converts rows 32cw..32cw+31 of the CTA's 128; per i < 4 a lane
    // takes 16 bytes (chunk lane % 4) of row 32cw + 8i + lane / 4, so each
    // shared-memory access covers 8 whole rows (conflict-free on both sides).
    const int cw = warp - mCvt0, ch = lane & 3;
    for (int s = 0; s < nslab; ++s) {
      const int sx = s % mXStages, sb = s % mSlots, sp = s - mSlots;
      if (!mbar_wait_warp(&tl->x_full[sx], (s / mXStages) & 1, p.cap, abort, p.err)) break;
      uint4 cur[4];
      const uint8_t* xsrc = as8 + sx * mXStage + (32 * cw + (lane >> 2)) * mBK + 16 * ch;
#pragma unroll
      for (int i = 0; i < 4; ++i) cur[i] = *reinterpret_cast<const uint4*>(xsrc + 8 * i * mBK);
      mbar_arrive_warp(&tl->x_empty[sx]);           // E4M3 stage read: the copy may refill it
      // the fp16 stage last held slab sp: wait until the pair's MMAs of sp completed
      if (sp >= 0 && !mbar_wait_warp(&tl->a_empty[sp % mSlots], (sp / mSlots) & 1, p.cap, abort, p.err))
        break;
      uint8_t* stage = bs + sb * mBStage;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const uint32_t w[4] = {cur[i].x, cur[i].y, cur[i].z, cur[i].w};
        uint32_t h[8];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          h[2 * j] = e4m3x2_to_f16x2(w[j] & 0xFFFFu);
          h[2 * j + 1] = e4m3x2_to_f16x2(w[j] >> 16);
        }
        const int rr = 32 * cw + 8 * i + (lane >> 2);
        uint8_t* dst = stage + rr * 128;
        const int sw = rr & 7;
        *reinterpret_cast<uint4*>(dst + 16 * ((2 * ch) ^ sw)) = make_uint4(h[0], h[1], h[2], h[3]);
        *reinterpret_cast<uint4*>(dst + 16 * ((2 * ch + 1) ^ sw)) = make_uint4(h[4], h[5], h[6], h[7]);
      }
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");   // generic writes -> tensor core reads
      mbar_arrive_warp(&local_full[sb]);
    }
  } else {
    // ---------------- dequant producers, then the epilogue ----------------
    const int dw = warp - mDeq0;
    const int q = warp & 3, set = dw >> 2;
    const int row = 32 * q + lane;
    const int n = min(n0 + row, p.N - 1);
    const int ng = p.K / 128;
    const uint16_t* srow = p.ws + ((size_t)e * p.N + n) * ng;
    // per-row power of two: the row's largest scale lands in [2^11, 2^12)
    float smax = 0.f;
    {
      int i = 0;
      if ((reinterpret_cast<uintptr_t>(srow) & 15u) == 0) {
        for (; i + 64 <= ng; i += 64) {            // 8 independent 16-byte loads in flight
          uint4 u[8];
#pragma unroll
          for (int j = 0; j < 8; ++j) u[j] = __ldg(reinterpret_cast<const uint4*>(srow + i) + j);
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            const uint32_t w[4] = {u[j].x, u[j].y, u[j].z, u[j].w};
#pragma unroll
            for (int c = 0; c < 4; ++c)
              smax = fmaxf(smax, fmaxf(fabsf(bf16_lo_to_f32(w[c])), fabsf(bf16_hi_to_f32(w[c]))));
          }
        }
        for (; i + 8 <= ng; i += 8) {
          const uint4 u = __ldg(reinterpret_cast<const uint4*>(srow + i));
          const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
          for (int c = 0; c < 4; ++c)
            smax = fmaxf(smax, fmaxf(fabsf(bf16_lo_to_f32(w[c])), fabsf(bf16_hi_to_f32(w[c]))));
        }
      }
      for (; i < ng; ++i) smax = fmaxf(smax, fabsf(bf16_bits_to_f32(__ldg(srow + i))));
    }
    int ex = 0;
    if (smax > 0.f) {
      int e2;
      frexpf(smax, &e2);                       // smax = m * 2^e2, m in [0.5, 1)
      ex = min(max(12 - e2, -100), 100);
    }
    const float up = ldexpf(1.f, ex), down = ldexpf(1.f, -ex);
    const uint32_t lane_base = tmem + ((uint32_t)(32 * q) << 16) + mACol0;

    uint16_t sc_next = set < nslab ? __ldg(srow + (set * mBK) / 128) : 0;
    for (int s = set; s < nslab; s += mDeqSets) {
      const int sa = s % mSlots, ra = s / mSlots;
      const uint32_t s2 = bf16x2_splat(f32_to_f16_bits(bf16_bits_to_f32(sc_next) * up));
      if (s + mDeqSets < nslab) sc_next = __ldg(srow + ((s + mDeqSets) * mBK) / 128);
      if (!mbar_wait_warp(&tl->w_full[sa], ra & 1, p.cap, abort, p.err)) break;
      const uint4 wa = *reinterpret_cast<const uint4*>(wsm + sa * mWStage + row * (mBK / 2));
      const uint4 wb = *reinterpret_cast<const uint4*>(wsm + sa * mWStage + row * (mBK / 2) + 16);
      const uint32_t v[8] = {wa.x, wa.y, wa.z, wa.w, wb.x, wb.y, wb.z, wb.w};
      uint32_t out[32];
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        uint32_t nat[4];
        int4x8_nat_f16(v[j], s2, nat);
        out[4 * j + 0] = nat[0]; out[4 * j + 1] = nat[1];
        out[4 * j + 2] = nat[2]; out[4 * j + 3] = nat[3];
      }
      mbar_arrive_warp(&tl->w_empty[sa]);           // packed slab decoded: its stage may be refilled
      if (ra > 0) {
        if (!mbar_wait_warp(&tl->a_empty[sa], (ra - 1) & 1, p.cap, abort, p.err)) break;
        tc_fence_after();
      }
      {
        const uint32_t (&o0)[16] = *reinterpret_cast<const uint32_t(*)[16]>(&out[0]);
        const uint32_t (&o1)[16] = *reinterpret_cast<const uint32_t(*)[16]>(&out[16]);
        tmem_st16(lane_base + sa * mACols, o0);
        tmem_st16(lane_base + sa * mACols + 16, o1);
      }
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive_warp(&local_full[sa]);
    }

    // epilogue: warp covers lane quarter q and 64 of the 256 activation rows
    const int cq = dw >> 2;
    if (mbar_wait_warp(&tl->acc_full, 0, p.cap, abort, p.err)) {
      tc_fence_after();
      const int nn = n0 + row;
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
            if (m < r_end) {
              const float val = __uint_as_float(v[c]) * down * __ldg(p.a_s + m);
              p.y[(size_t)m * p.N + nn] = f32_to_bf16_bits(val);
            }
          }
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  cluster_sync_all();          // neither CTA frees TMEM or leaves while the pair's MMAs may still read it
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem, mTmemCols);
  }
}

}  // namespace

qg_status moe_w4a8_tc(const uint8_t* a_e4m3, const float* a_s, const int32_t* expert_off, const uint8_t* w_q,
                      const uint16_t* w_s, uint16_t* y, int R, int E, int N, int K, cudaStream_t st) {
  CUtensorMap tmap_a, tmap_w;
  if (!make_u8_tmap(&tmap_a, a_e4m3, R, K, mHT, mBK))
    return set_error(QG_ERR_CUDA, "qgemm_w4a8_grouped: cannot encode the activation tensor map");
  if (!make_u8_tmap(&tmap_w, w_q, E * N, K / 2, mTW, mBK / 2))
    return set_error(QG_ERR_CUDA, "qgemm_w4a8_grouped: cannot encode the weight tensor map");
  unsigned int* err = device_error_word();
  if (!err) return set_error(QG_ERR_CUDA, "qgemm_w4a8_grouped: no device error word");
  MoeTcArgs a{};
  a.a_s = a_s; a.off = expert_off; a.ws = w_s; a.y = y;
  a.R = R; a.E = E; a.N = N; a.K = K;
  a.tiles_w = (N + 2 * mTW - 1) / (2 * mTW);
  a.err = err;
  a.cap = wait_limit();
  const int smem = mSlots * mBStage + mXStages * mXStage + mSlots * mWStage + (int)sizeof(MoeTail) + 1024;
  if (!ensure_smem(moe_w4a8_tc_kernel, smem)) return set_error(QG_ERR_CUDA, "qgemm_w4a8_grouped: smem attribute");
  const long long pairs = ((long long)(R + mTT - 1) / mTT + E) * a.tiles_w;
  moe_w4a8_tc_kernel<<<(unsigned)(2 * pairs), mThreads, smem, st>>>(tmap_a, tmap_w, a);
  return check_launch("qgemm_w4a8_grouped (tcgen05)");
}

}  // namespace qg
