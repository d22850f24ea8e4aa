"""GPU parity of the W4A8 grouped GEMM and of the MoE layer built from it."""

import numpy as np
import pytest
import torch

from numerics_packed_int4_gb300 import inputs
from oracle import formats as OF
from oracle import gemm as OG
from oracle import quant as OQ
from tests.gpu_util import check_gemm, config_expert_weights, dev, empty, host

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
    """Larger R: uneven experts, empty experts, partial row tiles and a partial
    channel tile, with many tiles per expert."""
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
    wq, ws = config_expert_weights(E, 2 * I, H, 60)
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


# Error budget of the kernel's h = (g * u) / (1 + expf(-g)) against the
# oracle's fp64 SiLU rounded once to fp32: g * u is exact, expf is within 2
# ulps (CUDA's documented bound), the add and the division round once each, so
# h is within 3 * 2^-23 relative of the exact value; with the oracle's half
# ulp, EPS_H = 2^-21 covers both sides with margin.
EPS_H = 2.0 ** -21


def _e4m3_midpoints():
    v = np.unique(np.abs(OF.e4m3_decode(np.arange(256, dtype=np.uint8))))
    v = v[np.isfinite(v)]
    return (v[:-1] + v[1:]) / 2.0                 # 0 .. 448 in steps; nothing above 448 is a boundary


def check_swiglu_codes(q, s, gu, I):
    """Row scales within EPS_H relative plus one ulp of the oracle's; codes
    identical wherever the oracle's h / s lies farther than the combined
    relative error from every E4M3 rounding boundary, at most one step apart
    elsewhere.  Returns (fraction of elements near a boundary, max scale ulps)."""
    h = OG.swiglu_f32(gu, I)
    ref_q, ref_s = OQ.quant_fp8_block(h, I)
    ref_s = ref_s[:, 0].astype(np.float64)
    ulp = np.spacing(ref_s.astype(np.float32)).astype(np.float64)
    ds = np.abs(s.astype(np.float64) - ref_s)
    assert np.all(ds <= EPS_H * ref_s + ulp), (ds / ulp).max()
    t = np.abs(h.astype(np.float64) / ref_s[:, None])
    delta = 2 * EPS_H + 4 * 2.0 ** -24           # h and s errors plus the quotient's rounding
    mid = _e4m3_midpoints()
    near = np.searchsorted(mid, t * (1 + delta), side="right") != np.searchsorted(mid, t * (1 - delta),
                                                                                 side="left")
    ordv = lambda c: np.where(c & 0x80, -(c.astype(np.int32) & 0x7F), c.astype(np.int32) & 0x7F)
    d = np.abs(ordv(q) - ordv(ref_q))
    assert np.all(d[~near] == 0), int(np.count_nonzero(d[~near]))
    assert d.max() <= 1, d.max()
    return float(np.mean(near)), float((ds / ulp).max())


def _swiglu_inputs(R, I, scale=3.0):
    return OF.bf16_encode((inputs.activations_bf16(R, 2 * I, seed=R + I).astype(np.uint32) << 16)
                          .view(np.float32) * np.float32(scale))


@pytest.mark.parametrize("R,I", [(1, 8), (37, 384), (300, 1408), (64, 14336)])
def test_swiglu_quant_vs_oracle(qg, R, I):
    """SwiGLU + per-row FP8 requantization against the oracle's fp64 SwiGLU
    (rounded once to fp32) and its FP8 quantizer (IEEE h / s, one E4M3
    rounding).  The kernel's h carries the few-ulp error of expf: codes must
    match exactly except where h / s lies within that error of an E4M3
    rounding boundary."""
    gu = _swiglu_inputs(R, I)
    hq, hs = empty((R, I), torch.uint8), empty((R,), torch.float32)
    qg.qg_swiglu_quant_fp8(dev(gu), hq, hs, R, I)
    qg.qg_check_device_error()
    near, _ = check_swiglu_codes(host(hq), host(hs), gu, I)
    assert near < 1e-3, near


@pytest.mark.parametrize("R,I", [(5, 136), (64, 14336)])
def test_swiglu_quant_f16_values_vs_oracle(qg, R, I):
    """The fp16-value output of the same kernel: each value must be exactly the
    E4M3 value of the code the E4M3-output kernel writes, and pass the same
    comparison with the oracle."""
    gu = _swiglu_inputs(R, I, scale=5.0)
    d_gu = dev(gu)
    hq, hs = empty((R, I), torch.uint8), empty((R,), torch.float32)
    qg.qg_swiglu_quant_fp8(d_gu, hq, hs, R, I)
    hv, hs2 = empty((R, I), torch.int16), empty((R,), torch.float32)
    qg.qg_swiglu_quant_fp8_f16(d_gu, hv, hs2, R, I)
    qg.qg_check_device_error()
    q = host(hq)
    np.testing.assert_array_equal(host(hs2), host(hs))
    vals = OF.fp16_decode(host(hv).view(np.uint16))
    np.testing.assert_array_equal(vals, OF.e4m3_decode(q))
    check_swiglu_codes(q, host(hs), gu, I)


@pytest.mark.parametrize("entry", ["grouped", "f16act", "fp8s"])
@pytest.mark.parametrize("R", [200, 640])
def test_malformed_expert_offsets_stay_inside_the_buffers(qg, entry, R):
    """expert_off comes from device memory and is not validated on the host:
    a last offset past R (R + 64) and a decreasing entry must still keep every
    access inside A and y.  y is the head of a larger allocation whose tail
    holds a sentinel; the tail must be untouched, and with only the last
    offset too large the rows are those of the clamped offsets."""
    E, N, K = 3, 256, 512
    x = inputs.activations_bf16(R, K, seed=R + 5)
    a8, a_s = OQ.quant_fp8_block(x, K)
    wq, ws = expert_weights(E, N, K, seed=33)
    d_a8, d_as, d_wq, d_ws = dev(a8), dev(a_s[:, 0].copy()), dev(wq), dev(ws)
    d_s8 = d_cs8 = d_a16 = None
    if entry == "fp8s":
        d_s8 = empty((K // 128, E * N), torch.uint8)
        d_cs8 = empty((E * N,), torch.float32)
        qg.qg_w4a8_fp8_scales(d_ws, d_s8, d_cs8, E * N, K // 128)
    if entry == "f16act":
        d_a16 = empty((R, K), torch.int16)
        qg.qg_e4m3_to_f16(d_a8, d_a16, R * K)
    sentinel = -12345
    cases = {"past_end": np.array([0, R // 3, R // 2, R + 64], np.int32),
             "decreasing": np.array([0, (2 * R) // 3, R // 4, R + 64], np.int32)}
    for name, off in cases.items():
        buf = torch.full((R + 96, N), sentinel, dtype=torch.int16, device="cuda")
        y = buf[:R]
        d_off = dev(off)
        if entry == "grouped":
            qg.qgemm_w4a8_grouped(d_a8, d_as, d_off, d_wq, d_ws, 128, y, R, E, N, K)
        elif entry == "f16act":
            qg.qgemm_w4a8_grouped_f16act(d_a16, d_as, d_off, d_wq, d_ws, None, 128, y, R, E, N, K)
        else:
            qg.qgemm_w4a8_grouped_fp8s(d_a8, d_as, d_off, d_wq, d_s8, d_cs8, y, R, E, N, K)
        qg.qg_check_device_error()
        tail = host(buf[R:]).view(np.int16)
        assert np.all(tail == sentinel), "%s %s: rows past R written" % (entry, name)
        if name == "past_end" and entry != "fp8s":
            clamped = np.minimum(off, R).astype(np.int32)
            ref = OF.bf16_decode(OG.to_bf16(OG.w4a8_grouped_f64(a8, a_s[:, 0], clamped, wq, ws, 128)))
            check_gemm(OF.bf16_decode(host(y)), ref, "%s clamped offsets" % entry)


def test_grouped_long_k_config_size_repeatable(qg):
    """The down projection of the config layer (R = 8192 rows over E = 8
    experts, N = 4096, K = 14336 -- 112 scale groups) three times over: the
    outputs must be bit-identical run to run (the kernel is deterministic, so
    any difference is a race) and match the oracle on sampled rows."""
    T, E, H, I = 4096, 8, 4096, 14336
    rt = inputs.moe_routing(T, E, 2, seed=9)
    off = rt["expert_off"]
    R = int(off[-1])
    h = inputs.activations_bf16(R, I, seed=31)
    a8, a_s = OQ.quant_fp8_block(h, I)
    wq, ws = config_expert_weights(E, H, I, 61)
    d_a8, d_as, d_off, d_wq, d_ws = dev(a8), dev(a_s[:, 0].copy()), dev(off), dev(wq), dev(ws)
    outs = []
    for _ in range(3):
        y = torch.zeros((R, H), dtype=torch.int16, device="cuda")
        qg.qgemm_w4a8_grouped(d_a8, d_as, d_off, d_wq, d_ws, 128, y, R, E, H, I)
        qg.qg_check_device_error()
        outs.append(host(y))
    assert np.array_equal(outs[0], outs[1]) and np.array_equal(outs[1], outs[2]), "nondeterministic output"
    r = np.random.Generator(np.random.PCG64(8))
    pick = np.sort(np.concatenate([r.choice(np.arange(off[e], off[e + 1]), size=6, replace=False)
                                   for e in range(E)]))
    sub_off = np.searchsorted(pick, off).astype(np.int32)
    ref = OF.bf16_decode(OG.to_bf16(OG.w4a8_grouped_f64(a8[pick], a_s[pick, 0], sub_off, wq, ws, 128)))
    check_gemm(OF.bf16_decode(outs[0][pick]), ref, "grouped K=14336 sampled rows")
