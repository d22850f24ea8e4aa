"""GPU parity of the tcgen05 prefill GEMM (M > 16) against the fp64 oracle: INT4
with group scales, and the FP8 per-channel, MXFP4 and NVFP4 weight formats."""

import numpy as np
import pytest
import torch

from numerics_packed_int4_gb300 import inputs
from oracle import formats as OF
from oracle import gemm as OG
from oracle import quant as OQ
from tests.gpu_util import check_gemm, dev, empty, host

pytestmark = pytest.mark.gpu


def run(qg, x, q, s, M, N, K, g=128):
    y = empty((M, N), torch.int16)
    qg.qgemm_w4a16(dev(q), dev(s), g, dev(x), y, M, N, K)
    qg.qg_check_device_error()
    return OF.bf16_decode(host(y))


@pytest.mark.parametrize("M,N,K", [(256, 128, 128), (17, 128, 256), (300, 264, 512), (512, 384, 1024),
                                   (1024, 1000, 640), (257, 4096, 4096)])
def test_prefill_small(qg, M, N, K):
    w = inputs.weights_f32(N, K, seed=M + N)
    x = inputs.activations_bf16(M, K, seed=K + 7, outlier_frac=0.01, outlier_scale=50.0)
    q, s = OQ.quant_int4_rtn(w, 128)
    y = run(qg, x, q, s, M, N, K)
    ref = OF.bf16_decode(OG.to_bf16(OG.qgemm_w4a16(x, q, s, 128)))
    check_gemm(y, ref, "prefill M=%d N=%d K=%d" % (M, N, K))


@pytest.mark.parametrize("M,N,K", [(2000, 2600, 128), (1800, 3000, 384), (4100, 1200, 512)])
def test_prefill_multi_tile_per_cta(qg, M, N, K):
    """More tiles than SMs, so each persistent CTA computes several tiles and
    overlaps one tile's epilogue with the next; K = 128 and 384 give 2 and 6
    k-slabs per tile (fewer than the 8 dequant slots); ragged M and N."""
    w = inputs.weights_f32(N, K, seed=M + 3 * N)
    x = inputs.activations_bf16(M, K, seed=K + 11, outlier_frac=0.01, outlier_scale=50.0)
    q, s = OQ.quant_int4_rtn(w, 128)
    y = run(qg, x, q, s, M, N, K)
    ref = OF.bf16_decode(OG.to_bf16(OG.qgemm_w4a16(x, q, s, 128)))
    check_gemm(y, ref, "prefill M=%d N=%d K=%d" % (M, N, K))


@pytest.mark.parametrize("g", [32, 64, 256])
def test_prefill_group_sizes(qg, g):
    M, N, K = 256, 256, 512
    w = inputs.weights_f32(N, K, seed=g)
    x = inputs.activations_bf16(M, K, seed=g + 1)
    q, s = OQ.quant_int4_rtn(w, g)
    y = run(qg, x, q, s, M, N, K, g)
    ref = OF.bf16_decode(OG.to_bf16(OG.qgemm_w4a16(x, q, s, g)))
    check_gemm(y, ref, "prefill g=%d" % g)


@pytest.mark.parametrize("N,K", [(4096, 4096), (14336, 4096), (4096, 14336)])
def test_prefill_config_sampled(qg, N, K):
    """The prefill workload at full size (M = 8192, 1 % outlier channels x50);
    parity on a seeded sample of 256 rows, every output finite."""
    M = 8192
    w = inputs.weights_f32(N, K, seed=300 + N // 1024 + K // 1024)
    x = inputs.activations_bf16(M, K, seed=400 + K, outlier_frac=0.01, outlier_scale=50.0)
    q, s = OQ.quant_int4_rtn(w, 128)
    y = run(qg, x, q, s, M, N, K)
    assert np.all(np.isfinite(y))
    rows = np.sort(np.random.Generator(np.random.PCG64(5)).choice(M, 256, replace=False))
    ref = OF.bf16_decode(OG.to_bf16(OG.qgemm_w4a16(x[rows], q, s, 128)))
    check_gemm(y[rows], ref, "prefill config N=%d K=%d" % (N, K))


def test_prefill_deterministic(qg):
    M, N, K = 512, 512, 1024
    w = inputs.weights_f32(N, K, seed=1)
    x = inputs.activations_bf16(M, K, seed=2)
    q, s = OQ.quant_int4_rtn(w, 128)
    assert np.array_equal(run(qg, x, q, s, M, N, K), run(qg, x, q, s, M, N, K))


# ---- the other weight formats on the same tcgen05 kernel (M > 16) ----
from tests.test_gemv_gpu import quantized, reference as wo_reference, run_gpu  # noqa: E402

OTHER_FORMATS = ["fp8", "mxfp4", "nvfp4"]


@pytest.mark.parametrize("fmt", OTHER_FORMATS)
@pytest.mark.parametrize("M,N,K", [(17, 128, 128), (300, 264, 512), (1024, 1000, 640), (2000, 2600, 384),
                                   (4100, 1200, 256)])
def test_prefill_formats(qg, fmt, M, N, K):
    """FP8 per-channel, MXFP4 and NVFP4 weights: single-tile, ragged, and
    more tiles than SMs (several tiles per persistent CTA)."""
    Wd = quantized(fmt, N, K, seed=M + N)
    x = inputs.activations_bf16(M, K, seed=K + 13, outlier_frac=0.01, outlier_scale=50.0)
    y = run_gpu(qg, fmt, Wd, x, M, N, K)
    ref, _ = wo_reference(Wd, x)
    check_gemm(y, ref, "%s prefill M=%d N=%d K=%d" % (fmt, M, N, K))


@pytest.mark.parametrize("fmt", OTHER_FORMATS)
def test_prefill_formats_config_sampled(qg, fmt):
    """M = 8192, N = 14336, K = 4096: parity on a seeded sample of 128 rows,
    every output finite."""
    M, N, K = 8192, 14336, 4096
    Wd = quantized(fmt, N, K, seed=500)
    x = inputs.activations_bf16(M, K, seed=501, outlier_frac=0.01, outlier_scale=50.0)
    y = run_gpu(qg, fmt, Wd, x, M, N, K)
    assert np.all(np.isfinite(y))
    rows = np.sort(np.random.Generator(np.random.PCG64(7)).choice(M, 128, replace=False))
    ref, _ = wo_reference(Wd, x, rows)
    check_gemm(y[rows], ref, "%s prefill config sample" % fmt)


@pytest.mark.parametrize("fmt", OTHER_FORMATS)
def test_prefill_formats_deterministic(qg, fmt):
    M, N, K = 600, 512, 1024
    Wd = quantized(fmt, N, K, seed=9)
    x = inputs.activations_bf16(M, K, seed=10)
    assert np.array_equal(run_gpu(qg, fmt, Wd, x, M, N, K), run_gpu(qg, fmt, Wd, x, M, N, K))


@pytest.mark.parametrize("M", [40, 600])
def test_prefill_mxfp4_block_scales_across_the_code_range(qg, M):
    """MXFP4 rows whose block codes exceed 128 (the dequant warp holding them
    takes the two-multiply decode for the slab) next to rows of small codes
    (the folded single multiply): both give the canonical weights."""
    N, K = 384, 1024
    r = np.random.Generator(np.random.PCG64(M + 90))
    w = inputs.weights_f32(N, K, seed=M + 91)
    row_exp = r.integers(-60, 1, N).astype(np.float32)
    row_exp[:32] = 40.0                      # one dequant warp's 32 rows: every code > 128
    row_exp[200] = 20.0                      # one row of another warp
    w = (w * np.exp2(row_exp)[:, None]).astype(np.float32)
    q, se = OQ.quant_mxfp4_weights(w)
    Wd = dict(q=q, s=se, deq=OG.dequant_mxfp4(q, se), epi=None)
    x = inputs.activations_bf16(M, K, seed=M + 92)
    y = run_gpu(qg, "mxfp4", Wd, x, M, N, K)
    ref, _ = wo_reference(Wd, x)
    unit = np.exp2(-row_exp)[None, :]
    check_gemm(y * unit, ref * unit, "mxfp4 prefill scale range M=%d" % M)


@pytest.mark.parametrize("M", [40, 600])
def test_prefill_nvfp4_every_finite_block_scale_code(qg, M):
    """NVFP4 with block scales over every finite E4M3 code: the folded decode
    (weights times 2^-9, the row times 2^9 with the global scale) against the
    canonical product."""
    N, K = 256, 2048
    r = np.random.Generator(np.random.PCG64(M + 93))
    q = r.integers(0, 256, (N, K // 2)).astype(np.uint8)
    sb = r.integers(0, 0x7F, (N, K // 16)).astype(np.uint8)
    sb[0, :0x7F] = np.arange(0x7F, dtype=np.uint8)
    gs = np.float32(1.5)
    Wd = dict(q=q, s=sb, gs=gs, deq=OG.dequant_nvfp4(q, sb), epi=np.full(N, float(gs)))
    x = inputs.activations_bf16(M, K, seed=M + 94)
    y = run_gpu(qg, "nvfp4", Wd, x, M, N, K)
    ref, _ = wo_reference(Wd, x)
    check_gemm(y, ref, "nvfp4 prefill all scale codes M=%d" % M)
