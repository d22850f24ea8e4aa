"""GPU parity of the W4A8 grouped GEMM and of the MoE layer built from it."""

import numpy as np
import pytest
import torch

from numerics_packed_int4_gb300 import inputs
from oracle import formats as OF
from oracle import gemm as OG
from oracle import quant as OQ
from tests.gpu_util import check_gemm, dev, empty, host

pytestmark = pytest.mark.gpu


def expert_weights(E, N, K, seed):
    qs, ss = [], []
    for e in range(E):
        q, s = OQ.quant_int4_rtn(inputs.weights_f32(N, K, seed=seed + e), 128)
        qs.append(q)
        ss.append(s)
    return np.stack(qs), np.stack(ss)


def grouped(qg, a8, a_s, off, wq, ws, N, K):
    R, E = a8.shape[0], wq.shape[0]
    y = empty((max(R, 1), N), torch.int16)
    qg.qgemm_w4a8_grouped(dev(a8), dev(a_s), dev(off.astype(np.int32)), dev(wq), dev(ws), 128, y,
                          R, E, N, K)
    qg.qg_check_device_error()
    return OF.bf16_decode(host(y))[:R]


@pytest.mark.parametrize("sizes,N,K", [([5, 0, 70, 129], 256, 512), ([1], 128, 128),
                                       ([0, 0, 3], 144, 384), ([64, 64], 512, 1024)])
def test_grouped_small(qg, sizes, N, K):
    E = len(sizes)
    off = np.concatenate([[0], np.cumsum(sizes)]).astype(np.int32)
    R = int(off[-1])
    x = inputs.activations_bf16(max(R, 1), K, seed=R + K)[:R]
    a8, a_s = OQ.quant_fp8_block(x, K)
    wq, ws = expert_weights(E, N, K, seed=50)
    y = grouped(qg, a8, a_s[:, 0], off, wq, ws, N, K)
    ref = OF.bf16_decode(OG.to_bf16(OG.w4a8_grouped_f64(a8, a_s[:, 0], off, wq, ws, 128)))
    if R:
        check_gemm(y, ref, "grouped %s" % sizes)


@pytest.mark.parametrize("sizes,N,K", [([300, 0, 700, 50, 1000], 384, 512), ([512], 272, 1024),
                                       ([0, 513, 0, 255, 257], 128, 384), ([2048, 2048], 1024, 2048)])
def test_grouped_tensor_core_path(qg, sizes, N, K):
    """R >= 512 takes the tcgen05 kernel: uneven experts, empty experts, partial
    row tiles and a partial channel tile."""
    E = len(sizes)
    off = np.concatenate([[0], np.cumsum(sizes)]).astype(np.int32)
    R = int(off[-1])
    x = inputs.activations_bf16(R, K, seed=R + K + 1)
    a8, a_s = OQ.quant_fp8_block(x, K)
    wq, ws = expert_weights(E, N, K, seed=90)
    y = grouped(qg, a8, a_s[:, 0], off, wq, ws, N, K)
    ref = OF.bf16_decode(OG.to_bf16(OG.w4a8_grouped_f64(a8, a_s[:, 0], off, wq, ws, 128)))
    check_gemm(y, ref, "grouped tc %s" % sizes)


def test_grouped_config_size_sampled(qg):
    """T=4096 top-2 over E=8: R=8192 rows, gate/up N=2*14336, K=4096; parity on
    a seeded sample of 24 rows per expert (full output is checked for
    finiteness)."""
    T, E, H, I = 4096, 8, 4096, 14336
    rt = inputs.moe_routing(T, E, 2, seed=9)
    off = rt["expert_off"]
    x = inputs.activations_bf16(T, H, seed=10)
    a8, a_s = OQ.quant_fp8_block(x, H)
    rows = rt["route_rows"]
    a8r, asr = a8[rows], a_s[rows, 0]
    wq, ws = expert_weights(E, 2 * I, H, seed=60)
    y = grouped(qg, a8r, asr, off, wq, ws, 2 * I, H)
    assert np.all(np.isfinite(y))
    r = np.random.Generator(np.random.PCG64(3))
    pick = np.concatenate([r.choice(np.arange(off[e], off[e + 1]), size=min(24, off[e + 1] - off[e]),
                                    replace=False) for e in range(E)])
    pick.sort()
    cols = np.sort(r.choice(2 * I, size=512, replace=False))
    # the oracle on the sampled rows (each keeps its expert) and columns
    sub_off = np.searchsorted(pick, off).astype(np.int32)
    ref = OF.bf16_decode(OG.to_bf16(
        OG.w4a8_grouped_f64(a8r[pick], asr[pick], sub_off, wq[:, cols], ws[:, cols], 128)))
    check_gemm(y[pick][:, cols], ref, "grouped config sample")


def test_moe_layer_small(qg):
    """Full layer: per-token FP8 quant, gather, grouped gate/up, SwiGLU + FP8
    requant, grouped down, weighted combine -- against the oracle layer."""
    T, E, H, I, topk = 96, 4, 256, 384, 2
    rt = inputs.moe_routing(T, E, topk, seed=13)
    off, rows, wts = rt["expert_off"], rt["route_rows"], rt["route_weight"]
    R = int(off[-1])
    x = inputs.activations_bf16(T, H, seed=14)
    w1 = expert_weights(E, 2 * I, H, seed=70)
    w2 = expert_weights(E, H, I, seed=80)

    xq, xs = empty((T, H), torch.uint8), empty((T,), torch.float32)
    qg.quant_act_fp8_block(dev(x), xq, xs, H, T, H)
    d_rows = dev(rows)
    aq, as_ = empty((R, H), torch.uint8), empty((R,), torch.float32)
    qg.qg_moe_gather_fp8(xq, xs, d_rows, aq, as_, R, T, H)
    gu = empty((R, 2 * I), torch.int16)
    d_off = dev(off)
    qg.qgemm_w4a8_grouped(aq, as_, d_off, dev(w1[0]), dev(w1[1]), 128, gu, R, E, 2 * I, H)
    hq, hs = empty((R, I), torch.uint8), empty((R,), torch.float32)
    qg.qg_swiglu_quant_fp8(gu, hq, hs, R, I)
    down = empty((R, H), torch.int16)
    qg.qgemm_w4a8_grouped(hq, hs, d_off, dev(w2[0]), dev(w2[1]), 128, down, R, E, H, I)
    # combine: per token, its rows in expert order
    row_of = np.full((T, topk), -1, np.int32)
    wt = np.zeros((T, topk), np.float32)
    fill = np.zeros(T, np.int64)
    for r_, t_ in enumerate(rows):
        row_of[t_, fill[t_]] = r_
        wt[t_, fill[t_]] = wts[r_]
        fill[t_] += 1
    out = empty((T, H), torch.int16)
    qg.qg_moe_combine(down, dev(row_of), dev(wt), out, T, topk, R, H)
    qg.qg_check_device_error()

    down_ref, gu_ref = OG.moe_layer(x, rows, off, w1, w2, 128, I)
    out_ref = OG.moe_combine(down_ref, rows, wts, T)
    check_gemm(OF.bf16_decode(host(gu)), OF.bf16_decode(gu_ref), "gate/up")
    check_gemm(OF.bf16_decode(host(out)), OF.bf16_decode(out_ref), "moe out")


@pytest.mark.parametrize("R,I", [(1, 8), (37, 384), (300, 1408), (64, 14336)])
def test_swiglu_quant_vs_oracle(qg, R, I):
    """SwiGLU + per-row FP8 requantization against the oracle's fp64 SwiGLU
    (rounded once to fp32) and FP8 quantizer.  The kernel evaluates SiLU with
    the fast exponential and division, so h carries a few fp32 ulps of error:
    a code may differ by one E4M3 step where h / s lies within those ulps of a
    rounding midpoint, the row scale by a few ulps, and nothing more."""
    gu = OF.bf16_encode((inputs.activations_bf16(R, 2 * I, seed=R + I).astype(np.uint32) << 16)
                        .view(np.float32) * np.float32(3.0))
    hq, hs = empty((R, I), torch.uint8), empty((R,), torch.float32)
    qg.qg_swiglu_quant_fp8(dev(gu), hq, hs, R, I)
    qg.qg_check_device_error()
    ref_q, ref_s = OQ.quant_fp8_block(OG.swiglu_f32(gu, I), I)
    q, s = host(hq), host(hs)
    assert np.allclose(s, ref_s[:, 0], rtol=4 * 2.0 ** -23, atol=0)
    # compare by E4M3 grid position: sign-magnitude code -> ordinal
    ordv = lambda c: np.where(c & 0x80, -(c.astype(np.int32) & 0x7F), c.astype(np.int32) & 0x7F)
    d = np.abs(ordv(q) - ordv(ref_q))
    assert d.max() <= 1, d.max()
    assert np.mean(d != 0) < 1e-3, np.mean(d != 0)

