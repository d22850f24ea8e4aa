"""GPU parity of the W4A4 MXFP4 path (vLLM PR #43557's W4A4 GEMM): the
activation quantizer's codes and the GEMM against the fp64 oracle, which
quantizes the same bf16 activations by the exponent-first 0.75-threshold rule
and multiplies the exact values.  For M > 16 with K a multiple of 256 the
product runs on the block-scaled FP4 tensor cores (scales applied inside the
MMA, the output written by TMA tile stores; with 16-element activation
blocks, through qgemm_w4a4_mxfp4_g, four scale factors per MMA); otherwise the activations are expanded
exactly to bf16 in the work buffer, which is then checked too."""

import numpy as np
import pytest
import torch

from numerics_packed_int4_gb300 import inputs
from oracle import formats as OF
from oracle import gemm as OG
from oracle import quant as OQ
from tests.gpu_util import check_gemm, dev, empty, host

pytestmark = pytest.mark.gpu


def run(qg, x, wq, wse, M, N, K, g=32):
    """Quantize x with blocks of g and multiply: g = 32 through qgemm_w4a4_mxfp4,
    g = 16 through qgemm_w4a4_mxfp4_g."""
    aq = empty((M, K // 2), torch.uint8)
    ase = empty((M, K // g), torch.uint8)
    work = empty((M, K), torch.int16)
    y = empty((M, N), torch.int16)
    dx = dev(x)
    qg.quant_act_mxfp4(dx, aq, ase, g, M, K)
    if g == 32:
        qg.qgemm_w4a4_mxfp4(dev(wq), dev(wse), aq, ase, work, y, M, N, K)
    else:
        qg.qgemm_w4a4_mxfp4_g(dev(wq), dev(wse), aq, ase, g, work, y, M, N, K)
    qg.qg_check_device_error()
    return host(aq), host(ase), host(work), OF.bf16_decode(host(y))


def weights(N, K, seed):
    return OQ.quant_mxfp4_weights(inputs.weights_f32(N, K, seed=seed))


def expanded(aq, ase, g=32):
    v = OF.e2m1_decode(OQ.unpack_nibbles(aq))
    v = (v.reshape(v.shape[0], -1, g) * OF.e8m0_decode(ase)[..., None]).reshape(v.shape)
    return OF.bf16_encode(v.astype(np.float32))


def block_scaled(M, K):
    """The cases qgemm_w4a4_mxfp4 runs on the block-scaled FP4 tensor cores
    (the test's scale arrays are fresh allocations, 8-byte aligned)."""
    return M > 16 and K % 256 == 0


@pytest.mark.parametrize("M,N,K", [(1, 1024, 1024), (5, 264, 384), (16, 512, 2048), (17, 128, 256),
                                   (300, 264, 512), (2000, 2600, 384), (129, 136, 256), (128, 128, 1280),
                                   (1000, 1032, 2048), (4096, 384, 768)])
@pytest.mark.parametrize("g", [32, 16])
def test_w4a4(qg, M, N, K, g):
    x = inputs.activations_bf16(M, K, seed=M + K, outlier_frac=0.01, outlier_scale=50.0)
    wq, wse = weights(N, K, seed=N + 3)
    gaq, gase, work, y = run(qg, x, wq, wse, M, N, K, g)
    y64, aq, ase = OG.w4a4_mxfp4_f64(x, wq, wse, g_act=g)
    np.testing.assert_array_equal(gaq, aq)
    np.testing.assert_array_equal(gase, ase)
    if not block_scaled(M, K):
        np.testing.assert_array_equal(work.view(np.uint16), expanded(aq, ase, g))
    check_gemm(y, OF.bf16_decode(OG.to_bf16(y64)), "w4a4 g=%d M=%d N=%d K=%d" % (g, M, N, K))


@pytest.mark.parametrize("g", [32, 16])
@pytest.mark.parametrize("band", ["low", "high"])
def test_w4a4_extreme_block_scales(qg, band, g):
    """Activation blocks near the bottom of the E8M0 range (scale codes down
    to 0, elements 2^-128 and 2^-127 that are subnormal in bf16) against
    weights scaled up by 2^110, and blocks near the top against ordinary
    weights, plus all-zero rows and blocks: the expansion must stay exact and
    the products normal."""
    M, N, K = 24, 256, 256
    xf = OF.bf16_decode(inputs.activations_bf16(M, K, seed=9)).astype(np.float32)
    wf = inputs.weights_f32(N, K, seed=10)
    if band == "low":
        xf[:8] *= np.float32(2.0 ** -126)
        xf[8:12] *= np.float32(2.0 ** -120)
        wf = wf * np.float32(2.0 ** 110)
    else:
        xf[:8] *= np.float32(2.0 ** 100)
    xf[12] = 0.0
    xf[13, :32] = 0.0
    x = OF.bf16_encode(xf)
    wq, wse = OQ.quant_mxfp4_weights(wf)
    gaq, gase, work, y = run(qg, x, wq, wse, M, N, K, g)
    y64, aq, ase = OG.w4a4_mxfp4_f64(x, wq, wse, g_act=g)
    np.testing.assert_array_equal(gaq, aq)
    np.testing.assert_array_equal(gase, ase)
    if band == "low":
        assert ase[:8].min() == 0
    if not block_scaled(M, K):
        np.testing.assert_array_equal(work.view(np.uint16), expanded(aq, ase, g))
    ref = OF.bf16_decode(OG.to_bf16(y64))
    for rows in (slice(0, 8), slice(8, 12), slice(12, M)):      # each magnitude band on its own
        check_gemm(y[rows], ref[rows], "w4a4 %s rows %s" % (band, rows))


@pytest.mark.parametrize("g", [32, 16])
def test_w4a4_config_sampled(qg, g):
    """M = 8192, N = 14336, K = 4096: parity on a seeded sample of 96 rows."""
    M, N, K = 8192, 14336, 4096
    x = inputs.activations_bf16(M, K, seed=71, outlier_frac=0.01, outlier_scale=50.0)
    wq, wse = weights(N, K, seed=72)
    _, _, _, y = run(qg, x, wq, wse, M, N, K, g)
    assert np.all(np.isfinite(y))
    rows = np.sort(np.random.Generator(np.random.PCG64(11)).choice(M, 96, replace=False))
    y64, _, _ = OG.w4a4_mxfp4_f64(x[rows], wq, wse, g_act=g)
    check_gemm(y[rows], OF.bf16_decode(OG.to_bf16(y64)), "w4a4 g=%d config sample" % g)


def test_w4a4_block_scaled_matches_the_expansion_path(qg):
    """The block-scaled product (M = 64, K = 1024) against the bf16-expansion
    product of the same codes (taken with M = 16 slices, which always expand):
    both sum the same exact products in fp32, so they agree to within the
    bf16 output rounding."""
    M, N, K = 64, 512, 1024
    x = inputs.activations_bf16(M, K, seed=41, outlier_frac=0.01, outlier_scale=50.0)
    wq, wse = weights(N, K, seed=42)
    _, _, _, y = run(qg, x, wq, wse, M, N, K)
    parts = [run(qg, x[i:i + 16], wq, wse, 16, N, K)[3] for i in range(0, M, 16)]
    check_gemm(y, np.concatenate(parts), "block-scaled vs expansion")

