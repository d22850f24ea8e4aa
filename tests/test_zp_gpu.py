"""GPU parity of asymmetric INT4 (one zero point per group; "Numerics":
x = s (q - z)): the load-time quantizer and the canonical dequant bit-exact
against the oracle, the GEMV (M <= 16) and tcgen05 prefill (M > 16) paths
within the GEMM tolerance, and the z = 8 special case equal to the symmetric
path bit for bit."""

import numpy as np
import pytest
import torch

from numerics_packed_int4_gb300 import inputs
from oracle import formats as OF
from oracle import gemm as OG
from oracle import quant as OQ
from tests.gpu_util import check_gemm, dev, empty, host

pytestmark = pytest.mark.gpu


def zp_weights(N, K, g, seed, shift=0.01):
    """Seeded weights with a per-row offset, so the groups are not centred on
    zero (what the zero point is for), quantized by the oracle."""
    w = inputs.weights_f32(N, K, seed=seed)
    w = (w + np.float32(shift) * np.sin(np.arange(N, dtype=np.float32))[:, None]).astype(np.float32)
    q, s, z = OQ.quant_int4_zp(w, g)
    return w, q, s, z


def gpu_quant(qg, w, g):
    N, K = w.shape
    q = empty((N, K // 2), torch.uint8)
    s = empty((N, K // g), torch.int16)
    z = empty((N, K // g), torch.uint8)
    qg.qg_quantize_weights_int4_zp(dev(w), q, s, z, g, N, K)
    qg.qg_check_device_error()
    return host(q), host(s), host(z)


@pytest.mark.parametrize("N,K,g", [(64, 256, 32), (96, 512, 64), (200, 1024, 128), (8, 256, 8), (16, 512, 256)])
def test_quantizer_bit_exact(qg, N, K, g):
    w, q, s, z = zp_weights(N, K, g, seed=N + K + g)
    w[0, :g] = 0.0                                   # all-zero group
    w[1, :g] = 0.375                                 # flat nonzero group
    w[2, :g] = np.abs(w[2, :g]) + 0.01               # all positive: z clamps to 0
    w[3, :g] = -np.abs(w[3, :g]) - 0.01              # all negative: z clamps to 15
    q, s, z = OQ.quant_int4_zp(w, g)
    gq, gs, gz = gpu_quant(qg, w, g)
    np.testing.assert_array_equal(gq, q)
    np.testing.assert_array_equal(gs, s)
    np.testing.assert_array_equal(gz, z)


@pytest.mark.parametrize("g", [32, 64, 128])
def test_dequant_bit_exact(qg, g):
    N, K = 136, 1152
    _, q, s, z = zp_weights(N, K, g, seed=g)
    out = empty((N, K), torch.int16)
    qg.qg_dequant_weights_int4_zp(dev(q), dev(s), dev(z), g, out, N, K)
    qg.qg_check_device_error()
    np.testing.assert_array_equal(host(out), OG.dequant_int4_zp(q, s, z, g))


def run(qg, x, q, s, z, g, M, N, K):
    y = empty((M, N), torch.int16)
    qg.qgemm_w4a16_zp(dev(q), dev(s), dev(z), g, dev(x), y, M, N, K)
    qg.qg_check_device_error()
    return OF.bf16_decode(host(y))


def reference(x, q, s, z, g, rows=None):
    xs = x if rows is None else x[rows]
    return OF.bf16_decode(OG.to_bf16(OG.gemm_bf16_f64(xs, OG.dequant_int4_zp(q, s, z, g), None)))


@pytest.mark.parametrize("M,N,K,g", [(1, 1024, 1024, 64), (1, 136, 384, 128), (4, 4096, 512, 32),
                                     (16, 264, 1280, 64), (11, 512, 640, 128)])
def test_gemv(qg, M, N, K, g):
    _, q, s, z = zp_weights(N, K, g, seed=N + M)
    x = inputs.activations_bf16(M, K, seed=K + M)
    check_gemm(run(qg, x, q, s, z, g, M, N, K), reference(x, q, s, z, g), "zp gemv M=%d N=%d K=%d g=%d" % (M, N, K, g))


@pytest.mark.parametrize("M,N,K,g", [(17, 128, 256, 64), (300, 264, 512, 64), (1024, 1000, 640, 128),
                                     (2000, 2600, 384, 64), (513, 384, 1024, 32)])
def test_prefill(qg, M, N, K, g):
    _, q, s, z = zp_weights(N, K, g, seed=M + N + 1)
    x = inputs.activations_bf16(M, K, seed=K + 5, outlier_frac=0.01, outlier_scale=50.0)
    check_gemm(run(qg, x, q, s, z, g, M, N, K), reference(x, q, s, z, g),
               "zp prefill M=%d N=%d K=%d g=%d" % (M, N, K, g))


def test_prefill_config_sampled(qg):
    """M = 8192, N = 14336, K = 4096, g = 64: parity on seeded sampled rows."""
    M, N, K, g = 8192, 14336, 4096, 64
    _, q, s, z = zp_weights(N, K, g, seed=77)
    x = inputs.activations_bf16(M, K, seed=78, outlier_frac=0.01, outlier_scale=50.0)
    y = run(qg, x, q, s, z, g, M, N, K)
    assert np.all(np.isfinite(y))
    rows = np.sort(np.random.Generator(np.random.PCG64(5)).choice(M, size=48, replace=False))
    check_gemm(y[rows], reference(x, q, s, z, g, rows), "zp prefill config sample")


@pytest.mark.parametrize("M", [1, 8, 600])
def test_zero_point_8_is_the_symmetric_path(qg, M):
    """u = q + 8 with z = 8 everywhere is the symmetric format: both GPU
    paths (GEMV for M <= 16, tcgen05 above) must give identical bits."""
    N, K, g = 384, 1024, 128
    w = inputs.weights_f32(N, K, seed=M + 99)
    qs, s = OQ.quant_int4_rtn(w, g)
    u = OQ.pack_nibbles((OF.int4_decode(OQ.unpack_nibbles(qs)) + 8).astype(np.uint8))
    z = np.full((N, K // g), 8, np.uint8)
    x = inputs.activations_bf16(M, K, seed=M + 100)
    y_sym = empty((M, N), torch.int16)
    qg.qgemm_w4a16(dev(qs), dev(s), g, dev(x), y_sym, M, N, K)
    y_zp = empty((M, N), torch.int16)
    qg.qgemm_w4a16_zp(dev(u), dev(s), dev(z), g, dev(x), y_zp, M, N, K)
    qg.qg_check_device_error()
    np.testing.assert_array_equal(host(y_zp), host(y_sym))
