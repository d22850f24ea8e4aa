"""GPU parity of the online activation quantizers and the fp32 casts (bit exact)."""

import numpy as np
import pytest
import torch

from numerics_packed_int4_gb300 import inputs
from oracle import formats as OF
from oracle import quant as OQ
from tests.gpu_util import dev, empty, host

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def qact():
    """The quantizer workload: 4096 x 7168 bf16 with outliers and injected edges."""
    return inputs.quantizer_activations_bf16(4096, 7168, seed=0)


def run_fp8(qg, x, g):
    M, K = x.shape
    q, s = empty((M, K), torch.uint8), empty((M, K // g), torch.float32)
    qg.quant_act_fp8_block(dev(x), q, s, g, M, K)
    torch.cuda.synchronize()
    return host(q), host(s)


def run_mxfp4(qg, x, g):
    M, K = x.shape
    q, s = empty((M, K // 2), torch.uint8), empty((M, K // g), torch.uint8)
    qg.quant_act_mxfp4(dev(x), q, s, g, M, K)
    torch.cuda.synchronize()
    return host(q), host(s)


def test_fp8_block128_full_workload_bit_exact(qg, qact):
    q, s = run_fp8(qg, qact, 128)
    rq, rs = OQ.quant_fp8_block(qact, 128)
    assert np.array_equal(s, rs), "scales differ in %d blocks" % int(np.sum(s != rs))
    assert np.array_equal(q, rq), "codes differ in %d of %d bytes" % (int(np.sum(q != rq)), q.size)


def test_fp8_per_token_bit_exact(qg, qact):
    x = qact[:512]
    q, s = run_fp8(qg, x, 7168)
    rq, rs = OQ.quant_fp8_block(x, 7168)
    assert np.array_equal(s, rs) and np.array_equal(q, rq)


@pytest.mark.parametrize("g", [16, 32])
def test_mxfp4_full_workload_bit_exact(qg, qact, g):
    q, s = run_mxfp4(qg, qact, g)
    rq, rs = OQ.quant_mxfp4(qact, g)
    assert np.array_equal(s, rs), "scale codes differ in %d blocks" % int(np.sum(s != rs))
    assert np.array_equal(q, rq), "codes differ in %d of %d bytes" % (int(np.sum(q != rq)), q.size)


@pytest.mark.parametrize("M,K,g", [(1, 128, 128), (3, 384, 64), (7, 256, 32), (5, 1024, 256),
                                   (2, 1536, 1536), (9, 640, 8)])
def test_fp8_small_and_ragged(qg, M, K, g):
    x = inputs.activations_bf16(M, K, seed=M * 1000 + K)
    x[0, :g] = 0                                 # an all-zero block: scale 1
    q, s = run_fp8(qg, x, g)
    rq, rs = OQ.quant_fp8_block(x, g)
    assert np.array_equal(s, rs) and np.array_equal(q, rq)


def test_mxfp4_edge_blocks(qg):
    x = np.zeros((4, 64), np.float32)
    x[1, :16] = -0.0
    x[2, :16] = np.float32(2.0 ** -130)           # bf16 subnormal block maximum
    x[3, :16] = np.array([1.75 * 2 ** 120] + [0.3] * 15, np.float32)
    x[3, 16:32] = np.array([1.625] + [-1.625 * 0.25 * 3.5] * 15, np.float32)
    xb = inputs.f32_to_bf16_bits(x)
    q, s = run_mxfp4(qg, xb, 16)
    rq, rs = OQ.quant_mxfp4(xb, 16)
    assert np.array_equal(s, rs) and np.array_equal(q, rq)


def _e4m3_sweep_f32():
    g = OF.E4M3_GRID
    mids = ((g[:-1] + g[1:]) / 2).astype(np.float32)
    r = np.random.Generator(np.random.PCG64(21))
    parts = [g.astype(np.float32), mids, np.nextafter(mids, np.float32(np.inf)),
             np.nextafter(mids, np.float32(-np.inf)), r.uniform(0, 448, 3_000_000).astype(np.float32),
             r.uniform(0, 2.0 ** -6, 1_000_000).astype(np.float32), np.float32([200.04, 0.0005, 0.001])]
    x = np.concatenate(parts)
    return np.concatenate([x, -x])


def test_e4m3_cast_sweep_matches_oracle_and_torch(qg):
    """fp32 -> E4M3 through the per-channel weight quantizer with every row
    anchored at 448 (channel scale exactly 1): the FreeToken PR #805 sweep."""
    x = _e4m3_sweep_f32()
    K = 1024
    rows = -(-x.size // (K - 1))
    w = np.zeros((rows, K), np.float32)
    w[:, 0] = 448.0
    flat = w[:, 1:].reshape(-1)
    flat[:x.size] = x
    w[:, 1:] = flat.reshape(rows, K - 1)
    q, cs = empty((rows, K), torch.uint8), empty((rows,), torch.float32)
    dw = dev(w)
    qg.qg_quantize_weights_fp8(dw, q, cs, rows, K)
    torch.cuda.synchronize()
    assert np.all(host(cs) == 1.0)
    got = host(q)[:, 1:].reshape(-1)[:x.size]
    assert np.array_equal(got, OF.e4m3_encode(x))
    t = torch.from_numpy(x).cuda().to(torch.float8_e4m3fn).view(torch.uint8).cpu().numpy()
    assert np.array_equal(got, t)                   # CUDA's own cast as a third opinion
    assert OF.e4m3_decode(got[x.size // 2 - 3]) == 208.0   # 200.04 -> 208


def test_e2m1_cast_sweep_matches_oracle(qg):
    """fp32 -> E2M1 through the MXFP4 weight quantizer with every 32-block
    anchored at 6.0 (scale code 127, i.e. scale 1)."""
    g = OF.E2M1_GRID
    mids = ((g[:-1] + g[1:]) / 2).astype(np.float32)
    r = np.random.Generator(np.random.PCG64(22))
    x = np.concatenate([g.astype(np.float32), mids, np.nextafter(mids, np.float32(9)),
                        np.nextafter(mids, np.float32(-9)), r.uniform(-6, 6, 200000).astype(np.float32)])
    x = np.concatenate([x, -x])
    nb = -(-x.size // 31)
    w = np.zeros((nb, 32), np.float32)
    w[:, 0] = 6.0
    flat = w[:, 1:].reshape(-1)
    flat[:x.size] = x
    w[:, 1:] = flat.reshape(nb, 31)
    rows = -(-nb // 32)
    wp = np.zeros((rows * 32, 32), np.float32)
    wp[:nb] = w
    wp[nb:, 0] = 6.0
    wp = wp.reshape(rows, 1024)
    q, s = empty((rows, 512), torch.uint8), empty((rows, 32), torch.uint8)
    qg.qg_quantize_weights_mxfp4(dev(wp), q, s, 32, rows, 1024)
    torch.cuda.synchronize()
    assert np.all(host(s) == 127)
    codes = OQ.unpack_nibbles(host(q)).reshape(rows * 32, 32)[:nb, 1:].reshape(-1)[:x.size]
    assert np.array_equal(codes, OF.e2m1_encode(x))
