"""GPU parity of the W4A8 grouped GEMM fed with fp16 copies of the E4M3
activations (exact re-encoding): the copy itself bit-exact over every code,
and the GEMM against the same fp64 oracle as the E4M3-input entry point."""

import numpy as np
import pytest
import torch

from numerics_packed_int4_gb300 import inputs
from oracle import formats as OF
from oracle import gemm as OG
from oracle import quant as OQ
from tests.gpu_util import check_gemm, config_expert_weights, dev, empty, host

pytestmark = pytest.mark.gpu


def test_e4m3_to_f16_every_code(qg):
    codes = np.tile(np.arange(256, dtype=np.uint8), 4)
    out = empty((codes.size,), torch.int16)
    qg.qg_e4m3_to_f16(dev(codes), out, codes.size)
    qg.qg_check_device_error()
    got = host(out).view(np.float16).astype(np.float64)
    want = OF.e4m3_decode(codes)
    nan = np.isnan(want)
    assert np.all(np.isnan(got[nan]))
    np.testing.assert_array_equal(got[~nan], want[~nan])
    assert np.array_equal(np.signbit(got[~nan]), np.signbit(want[~nan]))   # signed zero kept


def expert_weights(E, N, K, seed):
    qs, ss = [], []
    for e in range(E):
        q, s = OQ.quant_int4_rtn(inputs.weights_f32(N, K, seed=seed + e), 128)
        qs.append(q)
        ss.append(s)
    return np.stack(qs), np.stack(ss)


def grouped_f16(qg, a8, a_s, off, wq, ws, N, K, shifts=True):
    """E4M3 codes -> fp16 copy on the GPU, then the grouped GEMM (with the
    row shifts prepared by qg_w4a8_row_shifts, or computed in the kernel)."""
    R, E = a8.shape[0], wq.shape[0]
    y = empty((max(R, 1), N), torch.int16)
    a16 = empty((max(R, 1), K), torch.int16)
    if R:
        qg.qg_e4m3_to_f16(dev(a8), a16, R * K)
    dws = dev(ws)
    we = None
    if shifts:
        we = empty((E * N,), torch.int8)
        qg.qg_w4a8_row_shifts(dws, we, E * N, K // 128)
    qg.qgemm_w4a8_grouped_f16act(a16, dev(a_s) if R else empty((1,), torch.float32),
                                 dev(off.astype(np.int32)), dev(wq), dws, we, 128, y, R, E, N, K)
    qg.qg_check_device_error()
    return OF.bf16_decode(host(y))[:R]


@pytest.mark.parametrize("sizes,N,K", [([5, 0, 70, 129], 256, 512), ([1], 128, 128), ([0, 0, 3], 144, 384),
                                       ([300, 0, 700, 50, 1000], 384, 512), ([512], 272, 1024),
                                       ([0, 513, 0, 255, 257], 128, 384), ([2048, 2048], 1024, 2048)])
def test_grouped_f16act(qg, sizes, N, K):
    E = len(sizes)
    off = np.concatenate([[0], np.cumsum(sizes)]).astype(np.int32)
    R = int(off[-1])
    x = inputs.activations_bf16(max(R, 1), K, seed=R + K + 3)[:R]
    a8, a_s = OQ.quant_fp8_block(x, K)
    wq, ws = expert_weights(E, N, K, seed=150)
    y = grouped_f16(qg, a8, a_s[:, 0], off, wq, ws, N, K)
    if R:
        ref = OF.bf16_decode(OG.to_bf16(OG.w4a8_grouped_f64(a8, a_s[:, 0], off, wq, ws, 128)))
        check_gemm(y, ref, "f16act %s" % sizes)


@pytest.mark.parametrize("sizes,N,K", [([700, 900, 1000], 2048, 384), ([2000, 0, 600], 2560, 1024),
                                       ([4100], 1200, 512), ([33, 1500, 7, 1100], 1664, 128)])
def test_grouped_f16act_several_tiles_per_cta(qg, sizes, N, K):
    E = len(sizes)
    off = np.concatenate([[0], np.cumsum(sizes)]).astype(np.int32)
    R = int(off[-1])
    x = inputs.activations_bf16(R, K, seed=R + K + 13)
    a8, a_s = OQ.quant_fp8_block(x, K)
    wq, ws = expert_weights(E, N, K, seed=160)
    y = grouped_f16(qg, a8, a_s[:, 0], off, wq, ws, N, K)
    ref = OF.bf16_decode(OG.to_bf16(OG.w4a8_grouped_f64(a8, a_s[:, 0], off, wq, ws, 128)))
    check_gemm(y, ref, "f16act multi-tile %s" % sizes)


def test_row_shifts_given_or_computed_give_the_same_bits(qg):
    """The load-time row shifts are the ones the kernel would compute: both
    modes produce identical outputs, including a row whose scales span a wide
    range and an all-zero expert row."""
    sizes, N, K = [300, 700], 256, 1024
    E = len(sizes)
    off = np.concatenate([[0], np.cumsum(sizes)]).astype(np.int32)
    R = int(off[-1])
    x = inputs.activations_bf16(R, K, seed=93)
    a8, a_s = OQ.quant_fp8_block(x, K)
    w = np.stack([inputs.weights_f32(N, K, seed=180 + e) for e in range(E)])
    w[0, 5] *= np.float32(2.0 ** -12)
    w[1, 7] = 0.0
    qs, ss = zip(*[OQ.quant_int4_rtn(w[e], 128) for e in range(E)])
    wq, ws = np.stack(qs), np.stack(ss)
    y1 = grouped_f16(qg, a8, a_s[:, 0], off, wq, ws, N, K, shifts=True)
    y0 = grouped_f16(qg, a8, a_s[:, 0], off, wq, ws, N, K, shifts=False)
    np.testing.assert_array_equal(OF.bf16_encode(y1), OF.bf16_encode(y0))


@pytest.mark.parametrize("sizes", [[600, 424], [0, 300, 5, 700], [100, 50]])
def test_grouped_f16act_matches_e4m3_entry(qg, sizes):
    """From 256 rows the E4M3 entry runs the same tcgen05 kernel, converting
    the codes to fp16 in shared memory: its output is bit-identical to the
    fp16-copy entry's.  Below 256 rows (the mma.sync kernel) both compute the
    same exact products in fp32 and agree to within the order of the fp32
    accumulation."""
    N, K = 512, 1024
    E = len(sizes)
    off = np.concatenate([[0], np.cumsum(sizes)]).astype(np.int32)
    R = int(off[-1])
    x = inputs.activations_bf16(R, K, seed=91)
    a8, a_s = OQ.quant_fp8_block(x, K)
    wq, ws = expert_weights(E, N, K, seed=170)
    y16 = grouped_f16(qg, a8, a_s[:, 0], off, wq, ws, N, K)
    y8 = empty((R, N), torch.int16)
    qg.qgemm_w4a8_grouped(dev(a8), dev(a_s[:, 0]), dev(off), dev(wq), dev(ws), 128, y8, R, E, N, K)
    qg.qg_check_device_error()
    y8 = OF.bf16_decode(host(y8))
    if R >= 256:
        np.testing.assert_array_equal(OF.bf16_encode(y8), OF.bf16_encode(y16))
    else:
        assert np.max(np.abs(y16 - y8)) <= 2.0 ** -7 * np.max(np.abs(y8))


def test_grouped_f16act_config_size_sampled(qg):
    """T=4096 top-2 over E=8: R=8192 rows, gate/up N=2*14336, K=4096."""
    T, E, H, I = 4096, 8, 4096, 14336
    rt = inputs.moe_routing(T, E, 2, seed=9)
    off = rt["expert_off"]
    x = inputs.activations_bf16(T, H, seed=10)
    a8, a_s = OQ.quant_fp8_block(x, H)
    rows = rt["route_rows"]
    a8r, asr = a8[rows], a_s[rows, 0]
    wq, ws = config_expert_weights(E, 2 * I, H, 60)
    y = grouped_f16(qg, a8r, asr, off, wq, ws, 2 * I, H)
    assert np.all(np.isfinite(y))
    r = np.random.Generator(np.random.PCG64(6))
    pick = np.concatenate([r.choice(np.arange(off[e], off[e + 1]), size=min(24, off[e + 1] - off[e]),
                                    replace=False) for e in range(E)])
    pick.sort()
    cols = np.sort(r.choice(2 * I, size=512, replace=False))
    sub_off = np.searchsorted(pick, off).astype(np.int32)
    ref = OF.bf16_decode(OG.to_bf16(
        OG.w4a8_grouped_f64(a8r[pick], asr[pick], sub_off, wq[:, cols], ws[:, cols], 128)))
    check_gemm(y[pick][:, cols], ref, "f16act config sample")


def test_gather_and_swiglu_f16_outputs_are_the_codes_values(qg):
    """The fp16-output harness kernels write exactly the fp16 values of the
    codes (and the same row scales) that their E4M3-output forms write."""
    T, R, K, I = 50, 97, 1024, 1408
    r = np.random.Generator(np.random.PCG64(7))
    x = inputs.activations_bf16(T, K, seed=31)
    xq, xs = empty((T, K), torch.uint8), empty((T,), torch.float32)
    qg.quant_act_fp8_block(dev(x), xq, xs, K, T, K)
    rows = dev(r.integers(0, T, R).astype(np.int32))
    aq, as8 = empty((R, K), torch.uint8), empty((R,), torch.float32)
    a16, as16 = empty((R, K), torch.int16), empty((R,), torch.float32)
    qg.qg_moe_gather_fp8(xq, xs, rows, aq, as8, R, T, K)
    qg.qg_moe_gather_fp8_f16(xq, xs, rows, a16, as16, R, T, K)
    ref16 = empty((R, K), torch.int16)
    qg.qg_e4m3_to_f16(aq, ref16, R * K)
    gu = OF.bf16_encode((inputs.activations_bf16(R, 2 * I, seed=32).astype(np.uint32) << 16)
                        .view(np.float32) * np.float32(2.0))
    hq, hs = empty((R, I), torch.uint8), empty((R,), torch.float32)
    h16, hs16 = empty((R, I), torch.int16), empty((R,), torch.float32)
    qg.qg_swiglu_quant_fp8(dev(gu), hq, hs, R, I)
    qg.qg_swiglu_quant_fp8_f16(dev(gu), h16, hs16, R, I)
    href16 = empty((R, I), torch.int16)
    qg.qg_e4m3_to_f16(hq, href16, R * I)
    qg.qg_check_device_error()
    np.testing.assert_array_equal(host(a16), host(ref16))
    np.testing.assert_array_equal(host(as16), host(as8))
    np.testing.assert_array_equal(host(h16), host(href16))
    np.testing.assert_array_equal(host(hs16), host(hs))


def test_moe_layer_small_f16(qg):
    """Full layer on the fp16-activation path: per-token FP8 quant, gather to
    fp16, grouped gate/up, SwiGLU + FP8 requant to fp16, grouped down,
    weighted combine -- against the oracle layer."""
    T, E, H, I, topk = 96, 4, 256, 384, 2
    rt = inputs.moe_routing(T, E, topk, seed=13)
    off, rows, wts = rt["expert_off"], rt["route_rows"], rt["route_weight"]
    R = int(off[-1])
    x = inputs.activations_bf16(T, H, seed=14)
    w1 = expert_weights(E, 2 * I, H, seed=70)
    w2 = expert_weights(E, H, I, seed=80)
    xq, xs = empty((T, H), torch.uint8), empty((T,), torch.float32)
    qg.quant_act_fp8_block(dev(x), xq, xs, H, T, H)
    a16, as_ = empty((R, H), torch.int16), empty((R,), torch.float32)
    qg.qg_moe_gather_fp8_f16(xq, xs, dev(rows), a16, as_, R, T, H)
    gu = empty((R, 2 * I), torch.int16)
    d_off = dev(off)
    qg.qgemm_w4a8_grouped_f16act(a16, as_, d_off, dev(w1[0]), dev(w1[1]), None, 128, gu, R, E, 2 * I, H)
    h16, hs = empty((R, I), torch.int16), empty((R,), torch.float32)
    qg.qg_swiglu_quant_fp8_f16(gu, h16, hs, R, I)
    down = empty((R, H), torch.int16)
    qg.qgemm_w4a8_grouped_f16act(h16, hs, d_off, dev(w2[0]), dev(w2[1]), None, 128, down, R, E, H, I)
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
