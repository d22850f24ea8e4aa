// W4A8 grouped (MoE) GEMM.
//
// Semantics (Production-Ready W4A8: INT4 weights, per-token FP8 activations,
// group-wise bf16 weight scales, per-token fp32 activation scale in the
// epilogue):  y[r,n] = a_s[r] * sum_g s[g,n] * sum_{k in g} e4m3(a[r,k]) * q[n,k].
// Both operands are exact in bf16 (an E4M3 value and a small integer), so
// each K-group is one exact-product, fp32-accumulated tensor-core partial;
// the group scale is applied to that partial in fp32 ("promotion"), and the
// activation scale once at the end.
//
// This version uses mma.sync m16n8k16 bf16 tiles: a CTA computes a 64-row x
// 128-column tile of one expert; both operands are decoded while staging a
// 128-wide K-group into shared memory (E4M3 -> bf16 bit trick, INT4 -> bf16
// integer magic number), double-buffered so the next group's global loads
// overlap this group's MMAs.  Expert tiles are found on the device from
// expert_off, so the launch needs no host synchronization.
#include "dequant.cuh"

#define QG_REQUIRE(cond, st, ...) \
  do { if (!(cond)) return qg::set_error(st, __VA_ARGS__); } while (0)

namespace qg {
namespace {

constexpr int BM = 64, BN = 128, BK = 128;
constexpr int kThreadsMoe = 256;
constexpr int LDS = BK + 8;      // bf16 row pitch in shared memory (conflict-free ldmatrix)

QG_DEVICE void mma16816(float (&c)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

QG_DEVICE void ldmatrix_x4(uint32_t (&r)[4], const void* p) {
  const uint32_t a = static_cast<uint32_t>(__cvta_generic_to_shared(p));
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]) : "r"(a));
}

struct MoeArgs {
  const uint8_t* a;          // [R][K] e4m3
  const float* a_s;          // [R]
  const int32_t* off;        // [E+1]
  const uint8_t* wq;         // [E][N][K/2]
  const uint16_t* ws;        // [E][N][K/128]
  uint16_t* y;               // [R][N]
  int R, E, N, K;
};

// raw global data for one K-group: A 64 x 128 bytes, B 128 x 64 bytes
struct Stage { uint4 a[2]; uint4 b[2]; };

QG_DEVICE void load_stage(const MoeArgs& p, int r0, int r_end, int e, int n0, int kg, Stage& st) {
  const int tid = threadIdx.x;
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const int idx = tid + i * kThreadsMoe;          // 512 x 16 B = 8 KB
    const int row = idx >> 3, c = idx & 7;
    const int r = min(r0 + row, r_end - 1);
    st.a[i] = __ldg(reinterpret_cast<const uint4*>(p.a + (size_t)r * p.K + kg * BK + 16 * c));
    const int n = min(n0 + row * 2 + (c >> 2), p.N - 1);   // 128 rows x 4 chunks
    const int cb = c & 3;
    st.b[i] = __ldg(reinterpret_cast<const uint4*>(p.wq + ((size_t)e * p.N + n) * (p.K / 2) +
                                                   kg * (BK / 2) + 16 * cb));
  }
}

QG_DEVICE void store_stage(const Stage& st, uint16_t* sa, uint16_t* sb) {
  const int tid = threadIdx.x;
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const int idx = tid + i * kThreadsMoe;
    const int row = idx >> 3, c = idx & 7;
    // A: 16 e4m3 -> 16 bf16 (exact)
    const uint32_t w[4] = {st.a[i].x, st.a[i].y, st.a[i].z, st.a[i].w};
    uint32_t o[8];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      uint32_t p02, p13;
      e4m3x4_kperm(w[j], p02, p13);
      o[2 * j] = prmt(p02, p13, 0x5410u);
      o[2 * j + 1] = prmt(p02, p13, 0x7632u);
    }
    uint4* da = reinterpret_cast<uint4*>(sa + row * LDS + 16 * c);
    da[0] = make_uint4(o[0], o[1], o[2], o[3]);
    da[1] = make_uint4(o[4], o[5], o[6], o[7]);
    // B: 32 int4 -> 32 bf16 integers (exact; the group scale is applied later)
    const int n = row * 2 + (c >> 2), cb = c & 3;
    const uint32_t v[4] = {st.b[i].x, st.b[i].y, st.b[i].z, st.b[i].w};
    uint4* db = reinterpret_cast<uint4*>(sb + n * LDS + 32 * cb);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      uint32_t pq[4], nat[4];
      int4x8_kperm(v[j], 0x3F803F80u, pq);       // scale 1.0: the exact integer
      kperm4_to_natural(pq, nat);
      db[j] = make_uint4(nat[0], nat[1], nat[2], nat[3]);
    }
  }
}

__global__ void __launch_bounds__(kThreadsMoe) moe_w4a8_kernel(const MoeArgs p) {
  extern __shared__ __align__(16) uint16_t smem_moe[];
  uint16_t* sA[2] = {smem_moe, smem_moe + BM * LDS};
  uint16_t* sB[2] = {smem_moe + 2 * BM * LDS, smem_moe + 2 * BM * LDS + BN * LDS};

  // ---- which expert / row tile is this CTA? ---------------------------------
  int tile = blockIdx.x, e = -1, r0 = 0, r_end = 0;
  for (int i = 0; i < p.E; ++i) {
    // offsets come from device memory: clamp them into [0, R] (and b >= a)
    // so that a malformed expert_off can never move a row outside A or y
    const int a = min(max(p.off[i], 0), p.R), b = min(max(p.off[i + 1], a), p.R);
    const int nt = b > a ? (b - a + BM - 1) / BM : 0;
    if (tile < nt) { e = i; r0 = a + tile * BM; r_end = b; break; }
    tile -= nt;
  }
  if (e < 0) return;
  const int n0 = blockIdx.y * BN;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int wm = warp >> 2, wn = warp & 3;          // 2 x 4 warps, 32 x 32 each
  const int g = lane >> 2, t = lane & 3;

  float acc[2][4][4], part[2][4][4];
#pragma unroll
  for (int i = 0; i < 2; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j)
#pragma unroll
      for (int k = 0; k < 4; ++k) acc[i][j][k] = 0.f;

  const int ngroups = p.K / BK;
  Stage st;
  load_stage(p, r0, r_end, e, n0, 0, st);
  store_stage(st, sA[0], sB[0]);
  __syncthreads();

  for (int kg = 0; kg < ngroups; ++kg) {
    const int cur = kg & 1;
    if (kg + 1 < ngroups) load_stage(p, r0, r_end, e, n0, kg + 1, st);
#pragma unroll
    for (int i = 0; i < 2; ++i)
#pragma unroll
      for (int j = 0; j < 4; ++j)
#pragma unroll
        for (int k = 0; k < 4; ++k) part[i][j][k] = 0.f;
#pragma unroll
    for (int kk = 0; kk < BK; kk += 16) {
      uint32_t af[2][4], bf[2][4];
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        const int row = wm * 32 + i * 16 + (lane & 15);
        ldmatrix_x4(af[i], sA[cur] + row * LDS + kk + (lane >> 4) * 8);
      }
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        // two n-tiles of 8 per ldmatrix.x4: matrices (n 0-7,k 0-7),(n 0-7,k 8-15),(n 8-15,...)
        const int nrow = wn * 32 + j * 16 + (lane & 7) + ((lane >> 4) << 3);
        const int kof = ((lane >> 3) & 1) * 8;
        ldmatrix_x4(bf[j], sB[cur] + nrow * LDS + kk + kof);
      }
#pragma unroll
      for (int i = 0; i < 2; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j)
          mma16816(part[i][j], af[i], bf[j >> 1][(j & 1) * 2], bf[j >> 1][(j & 1) * 2 + 1]);
    }
    // promotion: acc += s[g, n] * part
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int n = n0 + wn * 32 + j * 8 + 2 * t;
      const size_t sidx = ((size_t)e * p.N) * (p.K / BK) + kg;
      const float s0 = bf16_bits_to_f32(__ldg(p.ws + sidx + (size_t)min(n, p.N - 1) * (p.K / BK)));
      const float s1 = bf16_bits_to_f32(__ldg(p.ws + sidx + (size_t)min(n + 1, p.N - 1) * (p.K / BK)));
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        acc[i][j][0] = __fmaf_rn(part[i][j][0], s0, acc[i][j][0]);
        acc[i][j][1] = __fmaf_rn(part[i][j][1], s1, acc[i][j][1]);
        acc[i][j][2] = __fmaf_rn(part[i][j][2], s0, acc[i][j][2]);
        acc[i][j][3] = __fmaf_rn(part[i][j][3], s1, acc[i][j][3]);
      }
    }
    if (kg + 1 < ngroups) {
      store_stage(st, sA[cur ^ 1], sB[cur ^ 1]);
    }
    __syncthreads();
  }

  // ---- epilogue: per-row activation scale, bf16 store ------------------------
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const int ra = r0 + wm * 32 + i * 16 + g, rb = ra + 8;
    const float sa = ra < r_end ? __ldg(p.a_s + ra) : 0.f;
    const float sb = rb < r_end ? __ldg(p.a_s + rb) : 0.f;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int n = n0 + wn * 32 + j * 8 + 2 * t;
      if (n >= p.N) continue;
      if (ra < r_end) {
        const uint32_t v = uint32_t(f32_to_bf16_bits(acc[i][j][0] * sa)) |
                           (uint32_t(f32_to_bf16_bits(acc[i][j][1] * sa)) << 16);
        *reinterpret_cast<uint32_t*>(p.y + (size_t)ra * p.N + n) = v;
      }
      if (rb < r_end) {
        const uint32_t v = uint32_t(f32_to_bf16_bits(acc[i][j][2] * sb)) |
                           (uint32_t(f32_to_bf16_bits(acc[i][j][3] * sb)) << 16);
        *reinterpret_cast<uint32_t*>(p.y + (size_t)rb * p.N + n) = v;
      }
    }
  }
}

// The general path for shapes outside the tiled kernels' (g == 128,
// K % 128 == 0, N % 16 == 0): one thread per output y[r, n].  The row's
// expert is found by binary search in expert_off; each group's partial sum of
// the exact products e4m3(a) * q accumulates in fp32 in k order, the group
// scale is applied to it in fp32, the row scale to the total, then one bf16
// rounding -- the tiled kernels' arithmetic, without their tiling.  It is
// there for odd widths and group sizes, not for speed.
__global__ void moe_w4a8_any_kernel(const MoeArgs p, int g, int r0) {
  const int n = blockIdx.x * blockDim.x + threadIdx.x, r = r0 + (int)blockIdx.y;
  if (n >= p.N || r < __ldg(p.off) || r >= __ldg(p.off + p.E)) return;
  int lo = 0, hi = p.E;                               // off[lo] <= r < off[hi]
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (__ldg(p.off + mid) <= r) lo = mid; else hi = mid;
  }
  const size_t wrow = (size_t)lo * p.N + n;
  const uint8_t* wq = p.wq + wrow * (p.K / 2);
  const uint16_t* ws = p.ws + wrow * (p.K / g);
  const uint8_t* a = p.a + (size_t)r * p.K;
  float acc = 0.f;
  for (int k0 = 0; k0 < p.K; k0 += g) {
    float part = 0.f;
    for (int k = k0; k < k0 + g; ++k) {
      const uint32_t b = __ldg(wq + k / 2), u = (k & 1) ? b >> 4 : b & 15u;
      part = fmaf(e4m3_to_f32(__ldg(a + k)), (float)(u >= 8u ? (int)u - 16 : (int)u), part);
    }
    acc = fmaf(bf16_bits_to_f32(__ldg(ws + k0 / g)), part, acc);
  }
  p.y[(size_t)r * p.N + n] = f32_to_bf16_bits(acc * __ldg(p.a_s + r));
}

}  // namespace
}  // namespace qg

namespace qg {
qg_status moe_w4a8_e4m3_f16(const uint8_t* a_e4m3, const float* a_s, const int32_t* expert_off, const uint8_t* w_q,
                            const uint16_t* w_s, uint16_t* y, int R, int E, int N, int K, cudaStream_t st);
// rows from which the tcgen05 kernel (256-row tiles, codes converted to fp16
// in shared memory) takes over from the 64-row mma.sync tiles
constexpr int kTcMinRows = 256;
}  // namespace qg

extern "C" qg_status qgemm_w4a8_grouped(const uint8_t* a_e4m3, const float* a_s, const int32_t* expert_off,
                                        const uint8_t* w_q, const uint16_t* w_s, int g, uint16_t* y, int R,
                                        int E, int N, int K, qg_stream_t stream) {
  QG_REQUIRE(a_e4m3 && a_s && expert_off && w_q && w_s && y, QG_ERR_INVALID_ARG,
             "qgemm_w4a8_grouped: NULL pointer");
  QG_REQUIRE(R >= 0 && E >= 1 && N > 0 && K > 0, QG_ERR_INVALID_ARG, "qgemm_w4a8_grouped: bad sizes");
  QG_REQUIRE(g >= 32 && (g & (g - 1)) == 0 && K % g == 0 && K % 32 == 0 && N % 8 == 0,
             QG_ERR_UNSUPPORTED_SHAPE,
             "qgemm_w4a8_grouped: need g a power of two >= 32 dividing K, K %% 32 == 0, N %% 8 == 0");
  QG_REQUIRE(qg::aligned16(a_e4m3) && qg::aligned16(w_q) && qg::aligned16(y) && qg::aligned16(w_s),
             QG_ERR_MISALIGNED, "qgemm_w4a8_grouped: misaligned pointer");
  if (R == 0) return QG_OK;
  if (!(g == 128 && K % 128 == 0 && N % 16 == 0)) {
    const qg::MoeArgs p{a_e4m3, a_s, expert_off, w_q, w_s, y, R, E, N, K};
    for (int r0 = 0; r0 < R; r0 += 65535) {           // the grid's y extent is at most 65535 rows
      qg::moe_w4a8_any_kernel<<<dim3((N + 127) / 128, std::min(65535, R - r0)), 128, 0,
                                reinterpret_cast<cudaStream_t>(stream)>>>(p, g, r0);
      const qg_status r = qg::check_launch("qgemm_w4a8_grouped");
      if (r != QG_OK) return r;
    }
    return QG_OK;
  }
  if (R >= qg::kTcMinRows)
    return qg::moe_w4a8_e4m3_f16(a_e4m3, a_s, expert_off, w_q, w_s, y, R, E, N, K,
                                 reinterpret_cast<cudaStream_t>(stream));
  qg::MoeArgs p{a_e4m3, a_s, expert_off, w_q, w_s, y, R, E, N, K};
  const size_t smem = (size_t)(2 * qg::BM + 2 * qg::BN) * qg::LDS * 2;
  if (!qg::ensure_smem(qg::moe_w4a8_kernel, (int)smem))
    return qg::set_error(QG_ERR_CUDA, "qgemm_w4a8_grouped: cannot set shared memory size");
  dim3 grid((R + qg::BM - 1) / qg::BM + E, (N + qg::BN - 1) / qg::BN);
  qg::moe_w4a8_kernel<<<grid, qg::kThreadsMoe, smem, reinterpret_cast<cudaStream_t>(stream)>>>(p);
  return qg::check_launch("qgemm_w4a8_grouped");
}
