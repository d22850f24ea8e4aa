"""GPU parity of the W4A8 path with FP8 group scales (Production-Ready W4A8,
"Accurate W4A8 Kernel"): the scale preparation bit-exact against the oracle,
and the FP8 x FP8 grouped GEMM against the oracle's exact products of the
same E4M3 operands."""

import numpy as np
import pytest
import torch

from numerics_packed_int4_gb300 import inputs
from oracle import formats as OF
from oracle import gemm as OG
from oracle import quant as OQ
from tests.gpu_util import check_gemm, config_expert_weights, dev, empty, host

pytestmark = pytest.mark.gpu


def gpu_scales(qg, s_bits):
    """The GPU scale preparation; its group-major [G][rows] codes come back
    transposed to the oracle's [rows][G]."""
    rows, G = s_bits.shape
    s8 = empty((G, max(rows, 1)), torch.uint8)
    cs8 = empty((max(rows, 1),), torch.float32)
    qg.qg_w4a8_fp8_scales(dev(s_bits), s8, cs8, rows, G)
    qg.qg_check_device_error()
    return np.ascontiguousarray(host(s8)[:, :rows].T), host(cs8)[:rows]


@pytest.mark.parametrize("rows,G", [(1, 1), (7, 32), (300, 32), (129, 5), (64, 112), (33, 257)])
def test_fp8_scales_bit_exact(qg, rows, G):
    K = 128 * G
    _, s = OQ.quant_int4_rtn(inputs.weights_f32(rows, K, seed=rows + G), 128)
    s8, cs8 = gpu_scales(qg, s)
    r8, rcs8 = OQ.fp8_group_scales(s)
    np.testing.assert_array_equal(s8, r8)
    np.testing.assert_array_equal(cs8.view(np.uint32), rcs8.view(np.uint32))


def test_fp8_scales_edge_rows(qg):
    """A zero row (cs = 1), a row whose small scales fall to E4M3 subnormals or
    zero after the 1/8, a row of equal scales, and one with a single nonzero."""
    f = np.zeros((4, 40), np.float32)
    f[1] = np.geomspace(1.0, 2.0 ** -24, 40)
    f[2] = 0.037
    f[3, 17] = 3.0e-3
    s = OF.bf16_encode(f)
    s8, cs8 = gpu_scales(qg, s)
    r8, rcs8 = OQ.fp8_group_scales(s)
    np.testing.assert_array_equal(s8, r8)
    np.testing.assert_array_equal(cs8.view(np.uint32), rcs8.view(np.uint32))
    assert cs8[0] == 8.0 and np.all(s8[0] == 0)


def expert_weights(E, N, K, seed):
    qs, ss = [], []
    for e in range(E):
        q, s = OQ.quant_int4_rtn(inputs.weights_f32(N, K, seed=seed + e), 128)
        qs.append(q)
        ss.append(s)
    return np.stack(qs), np.stack(ss)


def oracle_operands(wq, ws):
    """E4M3 weights E4M3(q * s8) and channel scales, per expert, from the oracle."""
    w8, cs8 = [], []
    for e in range(wq.shape[0]):
        s8, c = OQ.fp8_group_scales(ws[e])
        w8.append(OQ.fp8_lut_weights(wq[e], s8, 128))
        cs8.append(c)
    return np.stack(w8), np.stack(cs8)


def grouped_fp8s(qg, a8, a_s, off, wq, ws, N, K):
    """The GPU path end to end: scale preparation, then the grouped GEMM."""
    R, E = a8.shape[0], wq.shape[0]
    G = K // 128
    s8 = empty((G, E * N), torch.uint8)
    cs8 = empty((E * N,), torch.float32)
    qg.qg_w4a8_fp8_scales(dev(ws.reshape(E * N, G)), s8, cs8, E * N, G)
    y = empty((max(R, 1), N), torch.int16)
    qg.qgemm_w4a8_grouped_fp8s(dev(a8) if R else empty((1, K), torch.uint8), dev(a_s) if R else
                               empty((1,), torch.float32), dev(off.astype(np.int32)), dev(wq), s8, cs8,
                               y, R, E, N, K)
    qg.qg_check_device_error()
    return OF.bf16_decode(host(y))[:R]


def reference(a8, a_s, off, wq, ws):
    w8, cs8 = oracle_operands(wq, ws)
    return OF.bf16_decode(OG.to_bf16(OG.w4a8_fp8s_grouped_f64(a8, a_s, off, w8, cs8)))


@pytest.mark.parametrize("sizes,N,K", [([5, 0, 70, 129], 256, 512), ([1], 128, 128), ([0, 0, 3], 144, 384),
                                       ([300, 0, 700, 50, 1000], 384, 512), ([512], 272, 1024),
                                       ([0, 513, 0, 255, 257], 128, 384), ([2048, 2048], 1024, 2048)])
def test_grouped_fp8s(qg, sizes, N, K):
    """Uneven and empty experts, partial row tiles (256 rows), a partial channel
    tile (128 channels), more k-slabs than the 8 weight slots and fewer."""
    E = len(sizes)
    off = np.concatenate([[0], np.cumsum(sizes)]).astype(np.int32)
    R = int(off[-1])
    x = inputs.activations_bf16(max(R, 1), K, seed=R + K + 7)[:R]
    a8, a_s = OQ.quant_fp8_block(x, K)
    wq, ws = expert_weights(E, N, K, seed=120)
    y = grouped_fp8s(qg, a8, a_s[:, 0], off, wq, ws, N, K)
    if R:
        check_gemm(y, reference(a8, a_s[:, 0], off, wq, ws), "fp8s %s" % sizes)


@pytest.mark.parametrize("sizes,N,K", [([700, 900, 1000], 2048, 384), ([2000, 0, 600], 2560, 1024),
                                       ([4100], 1200, 512), ([33, 1500, 7, 1100], 1664, 128)])
def test_grouped_fp8s_several_tiles_per_cta(qg, sizes, N, K):
    """More tiles than SMs, so the persistent CTAs walk several tiles across
    expert boundaries; K from one slab to more than the 8 weight slots."""
    E = len(sizes)
    off = np.concatenate([[0], np.cumsum(sizes)]).astype(np.int32)
    R = int(off[-1])
    x = inputs.activations_bf16(R, K, seed=R + K + 11)
    a8, a_s = OQ.quant_fp8_block(x, K)
    wq, ws = expert_weights(E, N, K, seed=140)
    y = grouped_fp8s(qg, a8, a_s[:, 0], off, wq, ws, N, K)
    check_gemm(y, reference(a8, a_s[:, 0], off, wq, ws), "fp8s multi-tile %s" % sizes)


def test_grouped_fp8s_all_empty(qg):
    """Every expert empty but R = 0: nothing launched, nothing written."""
    off = np.zeros(4, np.int32)
    wq, ws = expert_weights(3, 128, 256, seed=5)
    y = grouped_fp8s(qg, np.zeros((0, 256), np.uint8), np.zeros(0, np.float32), off, wq, ws, 128, 256)
    assert y.shape == (0, 128)


def test_grouped_fp8s_config_size_sampled(qg):
    """T=4096 top-2 over E=8: R=8192 rows, gate/up N=2*14336, K=4096; parity on
    a seeded sample of 24 rows per expert and 512 channels."""
    T, E, H, I = 4096, 8, 4096, 14336
    rt = inputs.moe_routing(T, E, 2, seed=9)
    off = rt["expert_off"]
    x = inputs.activations_bf16(T, H, seed=10)
    a8, a_s = OQ.quant_fp8_block(x, H)
    rows = rt["route_rows"]
    a8r, asr = a8[rows], a_s[rows, 0]
    wq, ws = config_expert_weights(E, 2 * I, H, 60)
    y = grouped_fp8s(qg, a8r, asr, off, wq, ws, 2 * I, H)
    assert np.all(np.isfinite(y))
    r = np.random.Generator(np.random.PCG64(4))
    pick = np.concatenate([r.choice(np.arange(off[e], off[e + 1]), size=min(24, off[e + 1] - off[e]),
                                    replace=False) for e in range(E)])
    pick.sort()
    cols = np.sort(r.choice(2 * I, size=512, replace=False))
    sub_off = np.searchsorted(pick, off).astype(np.int32)
    ref = reference(a8r[pick], asr[pick], sub_off, wq[:, cols], ws[:, cols])
    check_gemm(y[pick][:, cols], ref, "fp8s config sample")


def test_fp8s_close_to_bf16_scale_path(qg):
    """The extra E4M3 rounding per weight keeps the result within a few 1e-2
    (relative Frobenius) of the W4A8 path that applies the bf16 group scales
    exactly -- the accuracy the page reports for the recipe."""
    sizes, N, K = [200, 312], 256, 1024
    off = np.concatenate([[0], np.cumsum(sizes)]).astype(np.int32)
    R = int(off[-1])
    x = inputs.activations_bf16(R, K, seed=77)
    a8, a_s = OQ.quant_fp8_block(x, K)
    wq, ws = expert_weights(2, N, K, seed=130)
    y = grouped_fp8s(qg, a8, a_s[:, 0], off, wq, ws, N, K)
    exact = OG.w4a8_grouped_f64(a8, a_s[:, 0], off, wq, ws, 128)
    err = float(np.linalg.norm(y - exact) / np.linalg.norm(exact))
    assert 1e-3 < err < 5e-2, err
