"""GPU parity of the load-time weight quantizers and of the in-register decode
(through the test-only qg_dequant_weights export) -- bit exact."""

import numpy as np
import pytest
import torch

from numerics_packed_int4_gb300 import inputs, qgemm as Q
from oracle import gemm as OG
from oracle import quant as OQ
from tests.gpu_util import dev, empty, host

pytestmark = pytest.mark.gpu

SHAPES = [(256, 1024), (136, 384), (4096, 4096)]


@pytest.mark.parametrize("N,K", SHAPES)
def test_quantize_int4(qg, N, K):
    w = inputs.weights_f32(N, K, seed=N + K)
    w[1, :128] = 0
    q, s = empty((N, K // 2), torch.uint8), empty((N, K // 128), torch.int16)
    qg.qg_quantize_weights_int4(dev(w), q, s, 128, N, K)
    torch.cuda.synchronize()
    rq, rs = OQ.quant_int4_rtn(w, 128)
    assert np.array_equal(host(s), rs) and np.array_equal(host(q), rq)


@pytest.mark.parametrize("N,K", SHAPES)
def test_quantize_fp8_channel(qg, N, K):
    w = inputs.weights_f32(N, K, seed=N + K + 1)
    w[2] = 0
    q, cs = empty((N, K), torch.uint8), empty((N,), torch.float32)
    qg.qg_quantize_weights_fp8(dev(w), q, cs, N, K)
    torch.cuda.synchronize()
    rq, rcs = OQ.quant_fp8_channel(w)
    assert np.array_equal(host(cs), rcs) and np.array_equal(host(q), rq)


@pytest.mark.parametrize("N,K", SHAPES)
def test_quantize_mxfp4(qg, N, K):
    w = inputs.weights_f32(N, K, seed=N + K + 2)
    q, s = empty((N, K // 2), torch.uint8), empty((N, K // 32), torch.uint8)
    qg.qg_quantize_weights_mxfp4(dev(w), q, s, 32, N, K)
    torch.cuda.synchronize()
    rq, rs = OQ.quant_mxfp4_weights(w)
    assert np.array_equal(host(s), rs) and np.array_equal(host(q), rq)


@pytest.mark.parametrize("N,K", SHAPES)
def test_quantize_nvfp4(qg, N, K):
    w = inputs.weights_f32(N, K, seed=N + K + 3)
    w[3, 16:32] = 0
    q, sb = empty((N, K // 2), torch.uint8), empty((N, K // 16), torch.uint8)
    gs = empty((1,), torch.float32)
    qg.qg_quantize_weights_nvfp4(dev(w), q, sb, gs, N, K)
    torch.cuda.synchronize()
    rq, rsb, rgs = OQ.quant_nvfp4(w)
    assert host(gs)[0] == rgs
    assert np.array_equal(host(sb), rsb) and np.array_equal(host(q), rq)


def test_quantize_nvfp4_all_zero(qg):
    w = np.zeros((16, 256), np.float32)
    q, sb, gs = empty((16, 128), torch.uint8), empty((16, 16), torch.uint8), empty((1,), torch.float32)
    qg.qg_quantize_weights_nvfp4(dev(w), q, sb, gs, 16, 256)
    torch.cuda.synchronize()
    assert host(gs)[0] == 1.0 and not host(q).any() and not host(sb).any()


# ---- decode: every code, extreme scales ---------------------------------------

def _dequant(qg, fmt, w, scales, g, N, K):
    out = empty((N, K), torch.int16)
    qg.qg_dequant_weights(fmt, dev(w), None if scales is None else dev(scales), g, out, N, K)
    torch.cuda.synchronize()
    return host(out)


def test_dequant_int4_every_code_and_scale_range(qg):
    N, K, g = 64, 512, 128
    r = np.random.Generator(np.random.PCG64(31))
    codes = np.tile(np.arange(16, dtype=np.uint8), N * K // 16).reshape(N, K)
    codes = np.take_along_axis(codes, r.permuted(np.tile(np.arange(K), (N, 1)), axis=1), axis=1)
    packed = OQ.pack_nibbles(codes)
    # scales over the whole positive and negative bf16 range, incl. subnormals
    s = r.integers(0, 0x7F80, (N, K // g)).astype(np.uint16)
    s[::3] |= 0x8000
    got = _dequant(qg, Q.QG_FMT_INT4, packed, s, g, N, K)
    ref = OG.dequant_int4(packed, s, g)
    assert np.array_equal(got, ref), "%d mismatches" % int(np.sum(got != ref))


def test_dequant_fp8_every_code(qg):
    N, K = 32, 512
    codes = np.tile(np.arange(256, dtype=np.uint8), N * K // 256).reshape(N, K)
    ok = (codes & 0x7F) != 0x7F
    got = _dequant(qg, Q.QG_FMT_FP8, codes, None, 0, N, K)
    ref = OG.dequant_fp8(codes)
    assert np.array_equal(got[ok], ref[ok])


def test_dequant_mxfp4_every_code_and_scale(qg):
    N, K = 64, 1024
    r = np.random.Generator(np.random.PCG64(32))
    codes = r.integers(0, 16, (N, K)).astype(np.uint8)
    packed = OQ.pack_nibbles(codes)
    se = r.integers(0, 253, (N, K // 32)).astype(np.uint8)
    se[0, :] = np.arange(K // 32)           # the low end, including the subnormal code 0
    got = _dequant(qg, Q.QG_FMT_MXFP4, packed, se, 32, N, K)
    ref = OG.dequant_mxfp4(packed, se)
    assert np.array_equal(got, ref), "%d mismatches" % int(np.sum(got != ref))


def test_dequant_nvfp4_every_code_and_scale(qg):
    N, K = 64, 1024
    r = np.random.Generator(np.random.PCG64(33))
    codes = r.integers(0, 16, (N, K)).astype(np.uint8)
    packed = OQ.pack_nibbles(codes)
    sb = r.integers(0, 0x7F, (N, K // 16)).astype(np.uint8)     # every finite non-negative E4M3
    sb[0, :] = np.arange(K // 16)
    got = _dequant(qg, Q.QG_FMT_NVFP4, packed, sb, 16, N, K)
    ref = OG.dequant_nvfp4(packed, sb)
    assert np.array_equal(got, ref), "%d mismatches" % int(np.sum(got != ref))
