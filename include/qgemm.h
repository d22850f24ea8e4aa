/*
 * qgemm.h -- C ABI of the GB300 (sm_103a) quantized-weight GEMM/GEMV library.
 *
 * The problem is stated the way the pages state it: a packed weight buffer,
 * a scale buffer, a group/block size, an activation pointer and M/N/K
 * ("Numerics: FP32 to INT4, and why bf16 won", the block-scaled Triton GEMM
 * and the dequantization kernel excerpt; "Production-Ready W4A8", section
 * "High-Performance W4A8 GEMM Kernel").
 *
 * Conventions shared by every entry point
 * ----------------------------------------
 *  - Every data pointer is a DEVICE pointer owned by the caller.  Buffers are
 *    contiguous and row-major; base addresses must be 16-byte aligned (the
 *    vLLM MXFP4 fix PR added .contiguous() for exactly this class of bug).
 *  - bf16 tensors are passed as uint16_t bit patterns.
 *  - W is [N][K] (output channel major, K contiguous); X is [M][K]; Y is [M][N].
 *  - Packed 4-bit codes hold two elements per byte along K, the even k in the
 *    low nibble.  INT4 nibbles are two's complement in [-8, 7]; E2M1 nibbles
 *    are sign-magnitude (bit 3 = sign).
 *  - All work is enqueued on the caller's stream; the library never allocates,
 *    frees or synchronizes (except qg_check_device_error, which syncs).
 *  - Every call returns a qg_status and never aborts; qg_last_error_string()
 *    gives a message for the last failing call on the calling thread.
 *  - Results are deterministic: the same inputs give the same output bits.
 *  - Arithmetic: dequantized weights are formed in registers exactly as the
 *    canonical dequantization below; products accumulate in fp32; the output
 *    is rounded to bf16 once (round to nearest even) at the store.
 */
#ifndef QGEMM_H
#define QGEMM_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define QG_API __attribute__((visibility("default")))
#else
#define QG_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* Same object as cudaStream_t; NULL is the legacy default stream. */
typedef struct CUstream_st* qg_stream_t;

typedef enum qg_status {
  QG_OK = 0,
  QG_ERR_INVALID_ARG = 1,        /* NULL pointer, bad enum value, negative size */
  QG_ERR_UNSUPPORTED_SHAPE = 2,  /* sizes outside the documented rules */
  QG_ERR_MISALIGNED = 3,         /* a pointer is not 16-byte aligned */
  QG_ERR_CUDA = 4,               /* a CUDA runtime call or kernel launch failed */
  QG_ERR_TIMEOUT = 5             /* a device-side wait hit its iteration cap */
} qg_status;

/* scale formats of qgemm_fp4a16 */
enum { QG_SCALE_E8M0 = 0, QG_SCALE_E4M3 = 1 };
/* weight formats of qg_dequant_weights */
enum { QG_FMT_INT4 = 0, QG_FMT_FP8 = 1, QG_FMT_MXFP4 = 2, QG_FMT_NVFP4 = 3 };

/* ------------------------------------------------------------------------ *
 * Weight-only GEMM/GEMV (W x A16): Y = X . dequant(W)^T, fp32 accumulate.
 * M <= 16 runs the HBM-streaming decode kernel; larger M the prefill kernel.
 * Shape rules: M >= 0 (M = 0 launches nothing), N >= 1, N % 8 == 0,
 * K % 32 == 0 and K % g == 0.  The decode and prefill kernels walk K in
 * 128-element segments; a K that is not a multiple of 128 runs instead on a
 * general kernel (one thread per output, the same canonical weights, fp32
 * accumulation in k order, the same epilogue), correct at any such shape
 * but not tuned: it is for odd layer widths, not for the hot path.
 * Stream overlap: the decode kernel (M <= 16) is launched with programmatic
 * dependent launch.  It may start while kernels enqueued before it on the
 * stream are still running or have not yet made their writes visible, and it
 * reads its weights and scales (and the NVFP4 global scale) right away; only
 * X is read after it has waited for the previous kernel to complete.  A decode
 * kernel also lets the kernel after it start early, so in a chain of decode
 * calls the early reads can reach back past several kernels.  Rule for
 * callers: the weight, scale and global-scale buffers of a decode call must
 * not be written by any kernel that is still queued or running when the call
 * is enqueued.  Write them (weight quantizers, casts, copies by kernels), then
 * synchronise the stream or device -- or have the host wait for an event
 * recorded after the writes -- before the first decode call that reads them.
 * Weights written once at load time satisfy this.  X may be the Y of the
 * call just before (the wait covers it).
 * ------------------------------------------------------------------------ */

/* INT4 weights with one bf16 scale per group of g along K.
 * Canonical weight: bf16_RNE(q * s) (one rounding of the exact product): the
 * W4A16 baseline of Production-Ready W4A8 ("High-Performance W4A8 GEMM
 * Kernel") turns the INT4 weights into BF16 on the CUDA cores and multiplies
 * in BF16; symmetric affine map with zero-point 0 ("Numerics", integer
 * formats paragraph).
 *   w_q [N][K/2]  packed INT4        w_s [N][K/g] bf16
 *   x   [M][K]    bf16               y   [M][N]   bf16 (written)
 *   g a power of two >= 32 (32, 64, 128, 256, ...), K % g == 0.          */
QG_API qg_status qgemm_w4a16(const uint8_t* w_q, const uint16_t* w_s, int g,
                      const uint16_t* x, uint16_t* y, int M, int N, int K,
                      qg_stream_t stream);

/* W4A16 with asymmetric INT4: unsigned 4-bit codes and one zero point per
 * group ("Numerics": x = s (q - z), z an integer, z != 0 asymmetric; the
 * dequant line (iweights - zeros) * scales).  y[m,n] = sum_k x[m,k] *
 * bf16_RNE((q[n,k] - z[n,k/g]) * s[n,k/g]), fp32 accumulation, one bf16
 * rounding.  Same kernels as qgemm_w4a16 (GEMV for M <= 16, tcgen05 above).
 *   w_q [N][K/2] unsigned nibbles (even k low)   w_s [N][K/g] bf16
 *   w_z [N][K/g] uint8 zero points in [0, 15]    x [M][K] bf16  y [M][N] bf16
 * Rules as qgemm_w4a16 (g a power of two >= 32 dividing K, K % 32 == 0,
 * N % 8 == 0); w_z needs no alignment.                                      */
QG_API qg_status qgemm_w4a16_zp(const uint8_t* w_q, const uint16_t* w_s, const uint8_t* w_z, int g,
                         const uint16_t* x, uint16_t* y, int M, int N, int K,
                         qg_stream_t stream);

/* FP8 E4M3 weights with one fp32 scale per output channel.
 * y[m,n] = w_cs[n] * sum_k x[m,k] * e4m3(w[n,k]); the E4M3 -> bf16 decode is
 * exact: every E4M3 (and E2M1) value has an exact 16-bit float form
 * ("Your 3090 Isn't Missing Anything...", section 4.1).
 *   w_e4m3 [N][K] u8    w_cs [N] fp32                                      */
QG_API qg_status qgemm_w8a16(const uint8_t* w_e4m3, const float* w_cs,
                      const uint16_t* x, uint16_t* y, int M, int N, int K,
                      qg_stream_t stream);

/* W8A8 with the activation quantization inside the GEMV prologue (the
 * in-kernel act quant of an FP8 GEMV, FreeToken PR #805's list of native
 * E4M3 casts; the quantizer is quant_act_fp8_block's, 1 x 128 blocks):
 * y[m,n] = w_cs[n] * sum_b s[m,b] * sum_{k in b} e4m3(a[m,k]) * e4m3(w[n,k])
 * with (a, s) = the E4M3 block quantization of x (s = absmax/448, IEEE
 * division, RNE satfinite), fp32 accumulation, one bf16 rounding.
 *   w_e4m3 [N][K] u8   w_cs [N] fp32   x [M][K] bf16   y [M][N] bf16.
 * K % 128 == 0, N % 8 == 0; the decode GEMV (M is processed 16 rows at a time). */
QG_API qg_status qgemm_w8a8(const uint8_t* w_e4m3, const float* w_cs, const uint16_t* x,
                     uint16_t* y, int M, int N, int K, qg_stream_t stream);

/* FP4 E2M1 weights with block scales.
 *  scale_fmt QG_SCALE_E8M0: MXFP4, g == 32, w_bs [N][K/32] E8M0 codes,
 *     canonical weight e2m1 * 2^(c-127) (exact); global_scale must be NULL.
 *     ("Numerics", "MXFP4 and the block-scaled family": block of 32, bare
 *     power-of-two scale.)
 *  scale_fmt QG_SCALE_E4M3: NVFP4, g == 16, w_bs [N][K/16] E4M3 codes,
 *     canonical weight e2m1 * e4m3(sb) (exact); global_scale is a DEVICE
 *     pointer to one fp32 applied to the accumulated row (each 16-value
 *     E2M1 block and its E4M3 scale become BF16 before the MMA: 3090 article
 *     section 2.1).
 *   w_e2m1 [N][K/2] packed E2M1                                            */
QG_API qg_status qgemm_fp4a16(const uint8_t* w_e2m1, const uint8_t* w_bs, int scale_fmt,
                       int g, const float* global_scale, const uint16_t* x,
                       uint16_t* y, int M, int N, int K, qg_stream_t stream);

/* W4A4 with MXFP4 on both operands (the MXFP4 W4A4 MoE GEMM of vLLM PR
 * #43557; activations from quant_act_mxfp4 with g = 32, weights MXFP4):
 * y[m,n] = sum_k (e2m1(a[m,k]) * 2^(sa[m,k/32]-127)) * (e2m1(w[n,k]) *
 * 2^(sw[n,k/32]-127)), fp32 accumulation, one bf16 rounding.  Every product is
 * exact in fp32, so the result is the exact-product sum up to the order of
 * the fp32 additions.
 * For M > 16 with K % 256 == 0 and both scale arrays 8-byte aligned the
 * product runs on the block-scaled FP4 tensor cores (tcgen05 kind::mxf4 with
 * the E8M0 scales applied inside the MMA; the FP4 tensor rate of the 3090
 * article, section 5) and a_work is not touched.  Otherwise the activations
 * are expanded exactly to bf16 into a_work and multiplied on the bf16 path of
 * qgemm_fp4a16.  a_work is caller-owned scratch; its contents afterwards are
 * unspecified.
 *   w_e2m1 [N][K/2]  w_e8m0 [N][K/32]  a_e2m1 [M][K/2]  a_e8m0 [M][K/32]
 *   a_work [M][K] bf16 (scratch)  y [M][N] bf16.  Rules as qgemm_fp4a16.     */
QG_API qg_status qgemm_w4a4_mxfp4(const uint8_t* w_e2m1, const uint8_t* w_e8m0,
                           const uint8_t* a_e2m1, const uint8_t* a_e8m0,
                           uint16_t* a_work, uint16_t* y, int M, int N, int K,
                           qg_stream_t stream);

/* qgemm_w4a4_mxfp4 with the activations' block size as an argument: g_act =
 * 32 (exactly qgemm_w4a4_mxfp4) or 16 -- the block size of the fixed MXFP4
 * W4A4 MoE kernel in vLLM PR #43557 and of the configured MXFP4 activation
 * quantizer -- with a_e8m0 [M][K/g_act]:
 * y[m,n] = sum_k (e2m1(a[m,k]) * 2^(sa[m,k/g_act]-127)) * (e2m1(w[n,k]) *
 * 2^(sw[n,k/32]-127)), fp32 accumulation, one bf16 rounding.
 * For M > 16 with K % 256 == 0 and both scale arrays 8-byte aligned, g_act =
 * 16 runs on the block-scaled tensor cores with four scale factors per 64-k
 * step (tcgen05 kind::mxf4nvf4, scale_vec::4X, E8M0: each 32-element weight
 * code stands for two 16-element blocks); otherwise the activations are
 * expanded exactly to bf16 into a_work as for qgemm_w4a4_mxfp4.  Rules as
 * qgemm_w4a4_mxfp4; any other g_act returns QG_ERR_UNSUPPORTED_SHAPE.       */
QG_API qg_status qgemm_w4a4_mxfp4_g(const uint8_t* w_e2m1, const uint8_t* w_e8m0,
                             const uint8_t* a_e2m1, const uint8_t* a_e8m0, int g_act,
                             uint16_t* a_work, uint16_t* y, int M, int N, int K,
                             qg_stream_t stream);

/* qgemm_w4a4_mxfp4 for callers that cannot allocate device memory; the pages
 * have no counterpart of this entry point.  Plugin-style host interfaces that
 * hand an op only its inputs and outputs, and runtimes that committed all
 * device memory to their own pool (where cudaMalloc would fail, and where
 * cudaMalloc/cudaFree could synchronise the device mid-loop), have no way to
 * pass the a_work buffer.  Here the bf16 expansion of the activations goes to
 * a fixed 16 MiB array compiled into the library (every GPU that loads the
 * library holds it until the process exits), so the call allocates nothing:
 * no cudaMalloc, no cudaFree, no allocating library routine.
 *   Arguments and result as qgemm_w4a4_mxfp4, without a_work.
 *   Limit: M * K <= 8388608 (16 MiB of bf16); larger sizes return
 *   QG_ERR_UNSUPPORTED_SHAPE and launch nothing.
 *   Set-up: the first call made with a given device current looks up the
 *   array's device address (cudaGetSymbolAddress) and caches it; make that
 *   first call before any stream capture.  A failed lookup returns QG_ERR_CUDA.
 *   Sharing: every call on a device uses the same array, and it keeps the last
 *   call's contents.  Nothing needs clearing (each call writes all the
 *   elements it reads), but calls whose kernels overlap on the GPU -- e.g. on
 *   two streams without an event between them -- race on the array and give
 *   wrong results.  Calls on one stream are ordered and safe.                */
QG_API qg_status qgemm_w4a4_mxfp4_noalloc(const uint8_t* w_e2m1, const uint8_t* w_e8m0,
                                   const uint8_t* a_e2m1, const uint8_t* a_e8m0,
                                   uint16_t* y, int M, int N, int K, qg_stream_t stream);

/* ------------------------------------------------------------------------ *
 * Online activation quantizers.  Rules: M >= 1, K % g == 0, K % 8 == 0.
 * ------------------------------------------------------------------------ */

/* MXFP4 per block of g in {16, 32}: vecMax = max|x|; scale code from the
 * exponent-first 0.75-threshold rule (bits(vecMax) + (1<<21)) & 0xFF800000,
 * biased exponent - 2, clamped at 0; element code E2M1_RNE_satfinite(
 * x * 2^(127-se)) (vLLM PR #43557, "Fix: Exponent-First with 0.75-Threshold
 * Rounding").
 *   x [M][K] bf16 -> q [M][K/2] packed E2M1, s_e8m0 [M][K/g] E8M0 codes.    */
QG_API qg_status quant_act_mxfp4(const uint16_t* x, uint8_t* q, uint8_t* s_e8m0, int g,
                          int M, int K, qg_stream_t stream);

/* FP8 E4M3 per 1 x g block (g == K gives per-token): s = amax/448 in fp32
 * (all-zero block: s = 1), q = E4M3_RNE_satfinite(x / s) with IEEE fp32
 * division and a single rounding ("Numerics", fp8 linear walk-through;
 * FreeToken PR #805).  g % 8 == 0.
 *   x [M][K] bf16 -> q [M][K] E4M3 codes, s [M][K/g] fp32.                  */
QG_API qg_status quant_act_fp8_block(const uint16_t* x, uint8_t* q, float* s, int g,
                              int M, int K, qg_stream_t stream);

/* ------------------------------------------------------------------------ *
 * W4A8 grouped (MoE) GEMM.
 * Rows of A are grouped by expert: rows expert_off[e] .. expert_off[e+1]-1
 * use expert e.  y[r,n] = a_s[r] * sum_k e4m3(a[r,k]) * q_e[n,k] * s_e[n,k/g]
 * with the group scale applied in fp32 per K-group (INT4 x FP8 activations,
 * per-token x group scales: Production-Ready W4A8).
 *   a_e4m3 [R][K] E4M3   a_s [R] fp32   expert_off [E+1] int32 (DEVICE,
 *   non-decreasing, expert_off[0] == 0, expert_off[E] == R)
 *   w_q [E][N][K/2] packed INT4   w_s [E][N][K/g] bf16   y [R][N] bf16.
 * Rules: g a power of two >= 32, K % g == 0, K % 32 == 0, N % 8 == 0,
 * R >= 0, E >= 1.  g == 128 with K % 128 == 0 and N % 16 == 0 (the W4A8
 * configuration) runs on the tiled kernels (from 256 rows tcgen05 with the
 * codes converted to fp16 in shared memory, bit-identical to
 * qgemm_w4a8_grouped_f16act);
 * every other shape on a general kernel with the same arithmetic (per-group
 * fp32 partial sums, scaled in fp32), correct but not tuned.                */
QG_API qg_status qgemm_w4a8_grouped(const uint8_t* a_e4m3, const float* a_s,
                             const int32_t* expert_off, const uint8_t* w_q,
                             const uint16_t* w_s, int g, uint16_t* y, int R,
                             int E, int N, int K, qg_stream_t stream);

/* The same W4A8 grouped GEMM (exact bf16 group scales, identical result) for
 * activations handed over as fp16: a_f16[r,k] = the value of the E4M3 code
 * a_e4m3[r,k], exactly (every E4M3 value is an fp16; qg_e4m3_to_f16 makes the
 * copy, or a producer writes it directly).  With the activations in HBM as
 * fp16 they reach the tensor cores by TMA with no restaging in the kernel
 * (one CTA per SM, tcgen05 kind::f16), for one more read of R*K*2 bytes.
 *   a_f16 [R][K] fp16; w_e [E*N] int8 row shifts from qg_w4a8_row_shifts
 *   (or NULL); the other arguments as qgemm_w4a8_grouped.
 * Rules: g == 128, K % 128 == 0, N % 16 == 0, R >= 0, E >= 1.               */
QG_API qg_status qgemm_w4a8_grouped_f16act(const uint16_t* a_f16, const float* a_s,
                                    const int32_t* expert_off, const uint8_t* w_q,
                                    const uint16_t* w_s, const int8_t* w_e, int g, uint16_t* y,
                                    int R, int E, int N, int K, qg_stream_t stream);

/* Load-time companion of qgemm_w4a8_grouped_f16act: each weight row's power
 * of two e (the row's largest |scale| times 2^e lies in [2^11, 2^12), which
 * keeps every fp16 product q * s * 2^e exact and in range), so the GEMM need
 * not scan the row's scales on every tile.  Pass the result as w_e, or NULL
 * to have the GEMM compute it.
 *   w_s [rows][G] bf16 -> w_e [rows] int8 (rows = E*N, G = K/128).          */
QG_API qg_status qg_w4a8_row_shifts(const uint16_t* w_s, int8_t* w_e, int rows, int G,
                             qg_stream_t stream);

/* E4M3 codes -> their values as fp16 (exact; NaN codes give fp16 NaN).
 *   q [n] u8 (8-byte aligned) -> out [n] fp16 (16-byte aligned).  n % 8 == 0. */
QG_API qg_status qg_e4m3_to_f16(const uint8_t* q, uint16_t* out, long long n,
                         qg_stream_t stream);

/* W4A8 grouped GEMM with FP8 group scales and an FP8 x FP8 matmul
 * (Production-Ready W4A8, "Accurate W4A8 Kernel": the group scales are
 * quantized to FP8 per output channel, pre-scaled by 1/8 with the channel
 * scale times 8, and each weight becomes E4M3(q * s8) -- the page's per-scale
 * lookup table -- so the tensor cores run E4M3 x E4M3 with fp32 accumulation
 * and the per-token and per-channel scales are applied in the epilogue):
 *   y[r,n] = bf16( a_s[r] * cs8_e[n] * sum_k e4m3(a[r,k]) * E4M3(q_e[n,k] * s8_e[n,k/128]) )
 * One extra E4M3 rounding per weight against qgemm_w4a8_grouped.
 *   a_e4m3, a_s, expert_off, w_q, y as qgemm_w4a8_grouped;
 *   w_s8 [K/128][E*N] E4M3 codes, group-major (qg_w4a8_fp8_scales with
 *   rows = E*N), w_cs8 [E][N] fp32.
 * Rules: K % 128 == 0, N % 16 == 0, R >= 0, E >= 1.                          */
QG_API qg_status qgemm_w4a8_grouped_fp8s(const uint8_t* a_e4m3, const float* a_s,
                                  const int32_t* expert_off, const uint8_t* w_q,
                                  const uint8_t* w_s8, const float* w_cs8, uint16_t* y,
                                  int R, int E, int N, int K, qg_stream_t stream);

/* The group scales of qgemm_w4a8_grouped_fp8s from an INT4 checkpoint's bf16
 * group scales (same page): per row, cs = max|s| / 448 in fp32 (zero row: 1),
 * code = E4M3_RNE_satfinite(s / cs) (IEEE division) -- the activation
 * quantizer applied to the row of scales -- then s8 = E4M3(decode(code) / 8)
 * and cs8 = 8 * cs.
 *   w_s [rows][G] bf16 -> w_s8 [G][rows] E4M3 codes (group-major: the
 *   GEMM's warps then read 32 consecutive channels' scales at once),
 *   w_cs8 [rows] fp32.                                                      */
QG_API qg_status qg_w4a8_fp8_scales(const uint16_t* w_s, uint8_t* w_s8, float* w_cs8,
                             int rows, int G, qg_stream_t stream);

/* ------------------------------------------------------------------------ *
 * Load-time weight quantizers (fp32 weights -> the formats above).
 * ------------------------------------------------------------------------ */

/* INT4 round-to-nearest, s = bf16_RNE(absmax/7) per group (fp32 division),
 * q = clamp(rint(w/s), -8, 7); an all-zero group (or a scale that rounds to
 * zero) gets s = 1, q = 0 ("Numerics": symmetric scale from a live amax;
 * the page asks for an explicit all-zero-group rule and names s = 1).
 * K % g == 0, g % 8 == 0.                                                    */
QG_API qg_status qg_quantize_weights_int4(const float* w, uint8_t* w_q, uint16_t* w_s, int g,
                                   int N, int K, qg_stream_t stream);
/* Asymmetric INT4 with zero points, one per group of g (the reading of
 * "Numerics" for a quantizer the pages do not print): lo/hi = group min/max,
 * s = bf16_RNE((hi - lo) / 15) in fp32 (flat group or s rounding to 0: s = 1),
 * z = clamp(rint(-lo / s), 0, 15), q = clamp(rint(w / s) + z, 0, 15) with IEEE
 * fp32 divisions.  w [N][K] fp32 -> w_q [N][K/2] unsigned nibbles, w_s [N][K/g]
 * bf16, w_z [N][K/g] uint8.  g a power of two in [8, 256] dividing K.       */
QG_API qg_status qg_quantize_weights_int4_zp(const float* w, uint8_t* w_q, uint16_t* w_s,
                                      uint8_t* w_z, int g, int N, int K, qg_stream_t stream);
/* FP8 E4M3 per output channel: cs = absmax/448 (zero row: 1), code =
 * E4M3_RNE_satfinite(w / cs).  K % 8 == 0.                                  */
QG_API qg_status qg_quantize_weights_fp8(const float* w, uint8_t* w_e4m3, float* w_cs,
                                  int N, int K, qg_stream_t stream);
/* MXFP4 weights: the quant_act_mxfp4 rule on fp32 rows, g == 32.            */
QG_API qg_status qg_quantize_weights_mxfp4(const float* w, uint8_t* w_e2m1, uint8_t* w_e8m0,
                                    int g, int N, int K, qg_stream_t stream);
/* NVFP4 weights: gs = amax(W)/(448*6) (zero W: 1), sb = E4M3_RNE_sat(
 * amax_block / (6*gs)), code = E2M1_RNE_sat(w / (e4m3(sb)*gs)); sb == 0 gives
 * zero codes.  Elements are divided by the dequantized block scale (vLLM PR
 * #43557 review).  global_scale is a DEVICE fp32 written by the call.
 * K % 16 == 0.                                                              */
QG_API qg_status qg_quantize_weights_nvfp4(const float* w, uint8_t* w_e2m1, uint8_t* w_e4m3,
                                    float* global_scale, int N, int K, qg_stream_t stream);

/* ------------------------------------------------------------------------ *
 * MoE harness kernels (outside the GEMM, used between the two projections).
 * ------------------------------------------------------------------------ */

/* rows[r] <- src[route_rows[r]] for E4M3 codes and their per-row scale.
 *   src_q [T][K] u8, src_s [T] fp32, route_rows [R] int32 (DEVICE)
 *   dst_q [R][K] u8, dst_s [R] fp32.  K % 16 == 0.                          */
QG_API qg_status qg_moe_gather_fp8(const uint8_t* src_q, const float* src_s,
                            const int32_t* route_rows, uint8_t* dst_q, float* dst_s,
                            int R, int T, int K, qg_stream_t stream);
/* qg_moe_gather_fp8 writing the gathered codes' fp16 values (exact) instead
 * of the codes, for qgemm_w4a8_grouped_f16act.  dst_f16 [R][K] fp16.       */
QG_API qg_status qg_moe_gather_fp8_f16(const uint8_t* src_q, const float* src_s,
                                const int32_t* route_rows, uint16_t* dst_f16, float* dst_s,
                                int R, int T, int K, qg_stream_t stream);
/* h = SiLU(gate) * up in fp32 from the bf16 projection output [R][2I] (gate
 * columns first), then the per-row FP8 quantizer of quant_act_fp8_block
 * (block = I: s = amax/448, codes E4M3_RNE_satfinite(h / s) with IEEE
 * division).  h = (gate * up) / (1 + exp(-gate)) with the exact bf16 product,
 * CUDA's accurate expf, the sum 1 + e kept in two floats and one remainder
 * correction of the quotient, so h is within a few fp32 ulps of the exact
 * value (about half an ulp where expf's error does not reach it): a code can
 * differ from the correctly rounded h's code only where h / s lies that close
 * to an E4M3 rounding boundary.
 *   gate_up [R][2I] bf16 -> q [R][I] E4M3, s [R] fp32.  I % 8 == 0.          */
QG_API qg_status qg_swiglu_quant_fp8(const uint16_t* gate_up, uint8_t* q, float* s,
                              int R, int I, qg_stream_t stream);
/* qg_swiglu_quant_fp8 writing the codes' fp16 values (exact) instead of the
 * codes, for qgemm_w4a8_grouped_f16act.  q_f16 [R][I] fp16.                */
QG_API qg_status qg_swiglu_quant_fp8_f16(const uint16_t* gate_up, uint16_t* q_f16, float* s,
                                  int R, int I, qg_stream_t stream);
/* out[t] = bf16( sum_j weight[t,j] * down[row_of[t,j]] ), j < topk, fp32 sum.
 *   down [R][H] bf16, row_of [T][topk] int32, weight [T][topk] fp32 (DEVICE)
 *   out [T][H] bf16.  H % 8 == 0.                                           */
QG_API qg_status qg_moe_combine(const uint16_t* down, const int32_t* row_of,
                         const float* weight, uint16_t* out, int T, int topk,
                         int R, int H, qg_stream_t stream);

/* ------------------------------------------------------------------------ *
 * Test and diagnostics entry points.
 * ------------------------------------------------------------------------ */

/* Canonical dequantized weights as bf16 [N][K], through the same in-register
 * decode the GEMM kernels use (epilogue scales excluded: FP8 channel scale,
 * NVFP4 global scale).  scales: INT4 -> bf16 [N][K/g]; FP8 -> ignored (may be
 * NULL); MXFP4 -> E8M0 [N][K/32]; NVFP4 -> E4M3 [N][K/16].  K % 128 == 0.    */
QG_API qg_status qg_dequant_weights(int fmt, const uint8_t* w, const void* scales, int g,
                             uint16_t* w_out, int N, int K, qg_stream_t stream);
/* Test-only: the canonical asymmetric INT4 dequant bf16_RNE((q - z) * s) of a
 * whole matrix, with the decode routine of qgemm_w4a16_zp.  Arguments as
 * qgemm_w4a16_zp; w_out [N][K] bf16.  K % 128 == 0.                         */
QG_API qg_status qg_dequant_weights_int4_zp(const uint8_t* w_q, const uint16_t* w_s,
                                     const uint8_t* w_z, int g, uint16_t* w_out, int N, int K,
                                     qg_stream_t stream);

/* Synchronizes the stream, then reads and clears this device's error word.
 * Returns QG_ERR_TIMEOUT if a kernel gave up on a wait, QG_ERR_CUDA on an
 * asynchronous CUDA error, QG_OK otherwise.                                  */
QG_API qg_status qg_check_device_error(qg_stream_t stream);

/* Message for the last failing call on the calling thread ("" if none).     */
QG_API const char* qg_last_error_string(void);

/* Iteration cap of every device-side spin wait (0 restores the default).
 * Intended for tests that exercise the timeout path.                        */
QG_API void qg_set_wait_limit(uint32_t iterations);

/* Measurement aid, not part of the method: a plain streaming read of `bytes`
 * bytes at p (16-byte non-allocating loads, grid-stride over 8 CTAs per SM),
 * the rate one launch of that size reaches on this GPU -- the ceiling a
 * single decode launch of the same bytes is compared with.  p 16-byte
 * aligned, bytes a positive multiple of 16, sink one 4-byte device word that
 * the kernel may write.                                                      */
QG_API qg_status qg_stream_read(const void* p, long long bytes, unsigned int* sink,
                         qg_stream_t stream);

/* Failure-path self-test; the method has no counterpart.  Launches one CTA
 * whose thread waits on an mbarrier that nothing arrives at, giving up after
 * `polls` bounded polls (each suspends for at most about 1 us).  The kernel
 * records a timeout in the device error word and returns -- it never traps --
 * so the next qg_check_device_error reports QG_ERR_TIMEOUT and the context
 * stays usable.  polls must be in 1 .. 1<<20 (else QG_ERR_INVALID_ARG).      */
QG_API qg_status qg_selftest_wait_timeout(uint32_t polls, qg_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* QGEMM_H */
