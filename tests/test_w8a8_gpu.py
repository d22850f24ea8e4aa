"""GPU parity of the W8A8 GEMV with the activation quantization in its
prologue: FP8 per-channel weights, activations quantized per 1 x 128 block by
the quant_act_fp8_block rule inside the kernel; against the fp64 oracle on
the oracle's own quantization of the same activations."""

import numpy as np
import pytest
import torch

from numerics_packed_int4_gb300 import inputs
from oracle import formats as OF
from oracle import gemm as OG
from oracle import quant as OQ
from tests.gpu_util import check_gemm, dev, empty, host

pytestmark = pytest.mark.gpu


def run(qg, q, cs, x, M, N, K):
    y = empty((M, N), torch.int16)
    qg.qgemm_w8a8(dev(q), dev(cs), dev(x), y, M, N, K)
    qg.qg_check_device_error()
    return OF.bf16_decode(host(y))


def reference(q, cs, x):
    a, s = OQ.quant_fp8_block(x, 128)
    return OF.bf16_decode(OG.to_bf16(OG.w8a8_f64(a, s, q, cs, 128)))


@pytest.mark.parametrize("M,N,K", [(1, 1024, 1024), (1, 4096, 4096), (4, 4096, 14336), (16, 264, 1280),
                                   (9, 136, 384), (20, 512, 2048), (1, 14336, 4096)])
def test_w8a8_gemv(qg, M, N, K):
    w = inputs.weights_f32(N, K, seed=N + K)
    q, cs = OQ.quant_fp8_channel(w)
    x = inputs.activations_bf16(M, K, seed=M + K, outlier_frac=0.01, outlier_scale=30.0)
    check_gemm(run(qg, q, cs, x, M, N, K), reference(q, cs, x), "w8a8 M=%d N=%d K=%d" % (M, N, K))


def test_w8a8_zero_and_tiny_blocks(qg):
    """An all-zero activation block (scale 1, codes 0), a block of subnormal
    range values and one dominated by a single outlier."""
    M, N, K = 3, 256, 512
    w = inputs.weights_f32(N, K, seed=3)
    q, cs = OQ.quant_fp8_channel(w)
    xf = OF.bf16_decode(inputs.activations_bf16(M, K, seed=4)).astype(np.float32)
    xf[0, :128] = 0.0
    xf[1, 128:256] *= np.float32(2.0 ** -20)
    xf[2, 256] = 1.0e4
    x = OF.bf16_encode(xf)
    check_gemm(run(qg, q, cs, x, M, N, K), reference(q, cs, x), "w8a8 edge blocks")


def test_w8a8_close_to_w8a16(qg):
    """Quantizing the activations to E4M3 per block costs a few 1e-2 relative
    error against the bf16-activation product, no more."""
    M, N, K = 2, 1024, 4096
    w = inputs.weights_f32(N, K, seed=8)
    q, cs = OQ.quant_fp8_channel(w)
    x = inputs.activations_bf16(M, K, seed=9)
    y = run(qg, q, cs, x, M, N, K)
    exact = OG.gemm_bf16_f64(x, OG.dequant_fp8(q), cs.astype(np.float64))
    err = float(np.linalg.norm(y - exact) / np.linalg.norm(exact))
    assert 1e-3 < err < 5e-2, err
