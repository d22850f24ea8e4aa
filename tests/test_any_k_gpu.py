"""Dense entries at K a multiple of 32 but not of 128: the shapes the fast
kernels' 128-k segments do not cover run on the general kernel (one thread
per output, the canonical dequantized weights, fp32 accumulation).  Each
format is compared with its oracle GEMM (the canonical dequant, fp64 sums,
one bf16 rounding), at decode and prefill row counts; W4A4 through both
activation block sizes, with its exact bf16 expansion checked as well."""

import numpy as np
import pytest
import torch

from numerics_packed_int4_gb300 import inputs
from oracle import formats as OF
from oracle import gemm as OG
from oracle import quant as OQ
from tests.gpu_util import check_gemm, dev, empty, host

pytestmark = pytest.mark.gpu

SHAPES = [(1, 136, 96), (5, 264, 1056), (17, 128, 160), (300, 264, 1056)]


def _x(M, K, seed):
    return inputs.activations_bf16(M, K, seed=seed, outlier_frac=0.01, outlier_scale=50.0)


def _out(M, N):
    return empty((M, N), torch.int16)


K_G64 = {96: 192, 1056: 1088, 160: 320}      # multiples of 64 that are not multiples of 128


@pytest.mark.parametrize("M,N,K", SHAPES)
@pytest.mark.parametrize("g", [32, 64])
def test_w4a16_any_k(qg, M, N, K, g):
    if g == 64:
        K = K_G64[K]
    x = _x(M, K, seed=K + M)
    q, s = OQ.quant_int4_rtn(inputs.weights_f32(N, K, seed=N), g)
    y = _out(M, N)
    qg.qgemm_w4a16(dev(q), dev(s), g, dev(x), y, M, N, K)
    qg.qg_check_device_error()
    ref = OF.bf16_decode(OG.to_bf16(OG.qgemm_w4a16(x, q, s, g)))
    check_gemm(OF.bf16_decode(host(y)), ref, "w4a16 g=%d M=%d N=%d K=%d" % (g, M, N, K))


@pytest.mark.parametrize("M,N,K", SHAPES)
def test_w4a16_zp_any_k(qg, M, N, K):
    g = 32
    x = _x(M, K, seed=K + M + 1)
    q, s, z = OQ.quant_int4_zp(inputs.weights_f32(N, K, seed=N + 1), g)
    y = _out(M, N)
    qg.qgemm_w4a16_zp(dev(q), dev(s), dev(z), g, dev(x), y, M, N, K)
    qg.qg_check_device_error()
    ref = OF.bf16_decode(OG.to_bf16(OG.gemm_bf16_f64(x, OG.dequant_int4_zp(q, s, z, g), None)))
    check_gemm(OF.bf16_decode(host(y)), ref, "w4a16_zp M=%d N=%d K=%d" % (M, N, K))


@pytest.mark.parametrize("M,N,K", SHAPES)
def test_w8a16_any_k(qg, M, N, K):
    x = _x(M, K, seed=K + M + 2)
    codes, cs = OQ.quant_fp8_channel(inputs.weights_f32(N, K, seed=N + 2))
    y = _out(M, N)
    qg.qgemm_w8a16(dev(codes), dev(np.asarray(cs, np.float32)), dev(x), y, M, N, K)
    qg.qg_check_device_error()
    ref = OF.bf16_decode(OG.to_bf16(OG.qgemm_w8a16(x, codes, cs)))
    check_gemm(OF.bf16_decode(host(y)), ref, "w8a16 M=%d N=%d K=%d" % (M, N, K))


@pytest.mark.parametrize("M,N,K", SHAPES)
@pytest.mark.parametrize("fmt", ["mxfp4", "nvfp4"])
def test_fp4a16_any_k(qg, M, N, K, fmt):
    x = _x(M, K, seed=K + M + 3)
    w = inputs.weights_f32(N, K, seed=N + 3)
    y = _out(M, N)
    if fmt == "mxfp4":
        q, se = OQ.quant_mxfp4_weights(w)
        qg.qgemm_fp4a16(dev(q), dev(se), qg.QG_SCALE_E8M0, 32, None, dev(x), y, M, N, K)
        ref = OG.qgemm_mxfp4a16(x, q, se)
    else:
        q, sb, gs = OQ.quant_nvfp4(w)
        gsd = dev(np.asarray([gs], np.float32))
        qg.qgemm_fp4a16(dev(q), dev(sb), qg.QG_SCALE_E4M3, 16, gsd, dev(x), y, M, N, K)
        ref = OG.qgemm_nvfp4a16(x, q, sb, gs)
    qg.qg_check_device_error()
    check_gemm(OF.bf16_decode(host(y)), OF.bf16_decode(OG.to_bf16(ref)), "%s M=%d N=%d K=%d" % (fmt, M, N, K))


@pytest.mark.parametrize("M,N,K", SHAPES)
@pytest.mark.parametrize("g", [32, 16])
def test_w4a4_any_k(qg, M, N, K, g):
    x = _x(M, K, seed=K + M + 4)
    wq, wse = OQ.quant_mxfp4_weights(inputs.weights_f32(N, K, seed=N + 4))
    aq = empty((M, K // 2), torch.uint8)
    ase = empty((M, K // g), torch.uint8)
    work = empty((M, K), torch.int16)
    y = _out(M, N)
    qg.quant_act_mxfp4(dev(x), aq, ase, g, M, K)
    qg.qgemm_w4a4_mxfp4_g(dev(wq), dev(wse), aq, ase, g, work, y, M, N, K)
    qg.qg_check_device_error()
    y64, raq, rase = OG.w4a4_mxfp4_f64(x, wq, wse, g_act=g)
    np.testing.assert_array_equal(host(aq), raq)
    np.testing.assert_array_equal(host(ase), rase)
    v = OF.e2m1_decode(OQ.unpack_nibbles(raq))
    v = (v.reshape(M, -1, g) * OF.e8m0_decode(rase)[..., None]).reshape(M, K)
    np.testing.assert_array_equal(host(work).view(np.uint16), OF.bf16_encode(v.astype(np.float32)))
    check_gemm(OF.bf16_decode(host(y)), OF.bf16_decode(OG.to_bf16(y64)), "w4a4 g=%d M=%d N=%d K=%d" % (g, M, N, K))


@pytest.mark.parametrize("sizes,N,K,g", [([5, 0, 70, 129], 264, 1056, 32), ([1], 136, 96, 32),
                                         ([0, 0, 3], 128, 192, 64), ([300, 0, 700], 200, 512, 128),
                                         ([64, 64], 256, 512, 64), ([40, 1], 128, 1024, 256)])
def test_w4a8_grouped_any_shape(qg, sizes, N, K, g):
    """The grouped call outside the tiled kernels' shapes (g != 128, K % 128
    != 0 or N % 16 != 0): empty and uneven experts, against the oracle."""
    E = len(sizes)
    off = np.concatenate([[0], np.cumsum(sizes)]).astype(np.int32)
    R = int(off[-1])
    x = inputs.activations_bf16(R, K, seed=R + K + 5)
    a8, a_s = OQ.quant_fp8_block(x, K)
    qs, ss = zip(*(OQ.quant_int4_rtn(inputs.weights_f32(N, K, seed=70 + e), g) for e in range(E)))
    wq, ws = np.stack(qs), np.stack(ss)
    y = _out(R, N)
    qg.qgemm_w4a8_grouped(dev(a8), dev(a_s[:, 0]), dev(off), dev(wq), dev(ws), g, y, R, E, N, K)
    qg.qg_check_device_error()
    ref = OF.bf16_decode(OG.to_bf16(OG.w4a8_grouped_f64(a8, a_s[:, 0], off, wq, ws, g)))
    check_gemm(OF.bf16_decode(host(y)), ref, "grouped %s N=%d K=%d g=%d" % (sizes, N, K, g))
