"""GPU parity of the weight-only GEMM/GEMV entry points against the fp64 oracle.

Tolerance (the path's contract): relative Frobenius <= 2e-3 and max |err| <=
1e-2 * max |ref| against the oracle's bf16 output.  Inputs are the seeded
synthetic workloads quantized by the oracle's own weight quantizers.
"""

import functools

import numpy as np
import pytest
import torch

from numerics_packed_int4_gb300 import inputs, qgemm as Q
from oracle import formats as OF
from oracle import gemm as OG
from oracle import quant as OQ
from tests.gpu_util import check_gemm, dev, empty, host

pytestmark = pytest.mark.gpu

FORMATS = ["int4", "fp8", "mxfp4", "nvfp4"]


@functools.lru_cache(maxsize=16)
def quantized(fmt, N, K, seed):
    """Oracle-quantized weights for one format, plus its canonical dequant."""
    w = inputs.weights_f32(N, K, seed=seed)
    if fmt == "int4":
        q, s = OQ.quant_int4_rtn(w, 128)
        return dict(q=q, s=s, deq=OG.dequant_int4(q, s, 128), epi=None)
    if fmt == "fp8":
        q, cs = OQ.quant_fp8_channel(w)
        return dict(q=q, s=cs, deq=OG.dequant_fp8(q), epi=cs.astype(np.float64))
    if fmt == "mxfp4":
        q, se = OQ.quant_mxfp4_weights(w)
        return dict(q=q, s=se, deq=OG.dequant_mxfp4(q, se), epi=None)
    q, sb, gs = OQ.quant_nvfp4(w)
    return dict(q=q, s=sb, gs=gs, deq=OG.dequant_nvfp4(q, sb), epi=np.full(N, float(gs)))


def run_gpu(qg, fmt, Wd, x, M, N, K):
    y = empty((M, N), torch.int16)
    dq, ds, dx = dev(Wd["q"]), dev(Wd["s"]), dev(x)
    if fmt == "int4":
        qg.qgemm_w4a16(dq, ds, 128, dx, y, M, N, K)
    elif fmt == "fp8":
        qg.qgemm_w8a16(dq, ds, dx, y, M, N, K)
    elif fmt == "mxfp4":
        qg.qgemm_fp4a16(dq, ds, Q.QG_SCALE_E8M0, 32, None, dx, y, M, N, K)
    else:
        gs = dev(np.array([Wd["gs"]], np.float32))
        qg.qgemm_fp4a16(dq, ds, Q.QG_SCALE_E4M3, 16, gs, dx, y, M, N, K)
    qg.qg_check_device_error()
    return OF.bf16_decode(host(y))


def reference(Wd, x, rows=None):
    xs = x if rows is None else x[rows]
    y64 = OG.gemm_bf16_f64(xs, Wd["deq"], Wd["epi"])
    return OF.bf16_decode(OG.to_bf16(y64)), y64


@pytest.mark.parametrize("fmt", FORMATS)
@pytest.mark.parametrize("M,N,K", [(1, 1024, 1024), (1, 1000, 384), (3, 136, 1280), (8, 512, 2048),
                                   (9, 256, 896), (16, 392, 512), (17, 264, 256), (40, 128, 640)])
def test_small_shapes(qg, fmt, M, N, K):
    Wd = quantized(fmt, N, K, seed=11)
    x = inputs.activations_bf16(M, K, seed=12 + M)
    y = run_gpu(qg, fmt, Wd, x, M, N, K)
    ref, y64 = reference(Wd, x)
    check_gemm(y, ref, "%s M=%d N=%d K=%d" % (fmt, M, N, K))


@pytest.mark.parametrize("fmt", FORMATS)
@pytest.mark.parametrize("N,K", [(4096, 4096), (14336, 4096), (4096, 14336)])
def test_decode_sweep_config(qg, fmt, N, K):
    """The decode sweep at full size: M in {1, 4, 16}, full parity (the oracle
    handles M <= 16 at these sizes in seconds)."""
    Wd = quantized(fmt, N, K, seed=100 + N // 1024 + K // 1024)
    for M in (1, 4, 16):
        x = inputs.activations_bf16(M, K, seed=200 + M)
        y = run_gpu(qg, fmt, Wd, x, M, N, K)
        ref, _ = reference(Wd, x)
        check_gemm(y, ref, "%s M=%d N=%d K=%d" % (fmt, M, N, K))


def test_gemv_is_deterministic(qg):
    Wd = quantized("int4", 4096, 4096, seed=5)
    x = inputs.activations_bf16(4, 4096, seed=6)
    a = run_gpu(qg, "int4", Wd, x, 4, 4096, 4096)
    b = run_gpu(qg, "int4", Wd, x, 4, 4096, 4096)
    assert np.array_equal(a, b)


def test_zero_rows_and_zero_m(qg):
    N, K = 256, 512
    Wd = quantized("int4", N, K, seed=7)
    x = np.zeros((2, K), np.uint16)
    y = run_gpu(qg, "int4", Wd, x, 2, N, K)
    assert np.all(y == 0)
    y0 = empty((1, N), torch.int16)
    qg.qgemm_w4a16(dev(Wd["q"]), dev(Wd["s"]), 128, dev(x), y0, 0, N, K)   # M = 0 is a no-op


def test_chained_gemvs_wait_for_the_previous_output(qg):
    """Layer chain on one stream, no host sync: y1 = W1.x, y2 = W2.y1, y3 = W3.y2
    (the decode kernels overlap their weight streaming with the previous
    kernel, so each must still read the previous kernel's finished output)."""
    N = K = 4096
    Ws = [quantized(f, N, K, seed=40 + i) for i, f in enumerate(["int4", "fp8", "nvfp4"])]
    x = inputs.activations_bf16(1, K, seed=41)
    d = [dev(x)] + [empty((1, N), torch.int16) for _ in range(3)]
    dq = [(dev(W["q"]), dev(W["s"])) for W in Ws]
    gs = dev(np.array([Ws[2]["gs"]], np.float32))
    for rep in range(3):
        qg.qgemm_w4a16(dq[0][0], dq[0][1], 128, d[0], d[1], 1, N, K)
        qg.qgemm_w8a16(dq[1][0], dq[1][1], d[1], d[2], 1, N, K)
        qg.qgemm_fp4a16(dq[2][0], dq[2][1], Q.QG_SCALE_E4M3, 16, gs, d[2], d[3], 1, N, K)
    qg.qg_check_device_error()
    ref = x
    for W, fmt in zip(Ws, ["int4", "fp8", "nvfp4"]):
        ref = OG.to_bf16(OG.gemm_bf16_f64(ref, W["deq"], W["epi"]))
    y = OF.bf16_decode(host(d[3]))
    check_gemm(y, OF.bf16_decode(ref), "chained")


@pytest.mark.parametrize("M", [1, 5, 16])
def test_mxfp4_block_scales_across_the_code_range(qg, M):
    """MXFP4 rows whose block scales span the E8M0 range: codes above 128
    (magnitudes of 12 and more) take the decode with two multiplies for the
    warp that holds them, the others the folded single multiply; both must
    give the canonical weights."""
    N, K = 256, 1024
    r = np.random.Generator(np.random.PCG64(M + 70))
    w = inputs.weights_f32(N, K, seed=M + 71)
    row_exp = r.integers(-60, 1, N).astype(np.float32)
    row_exp[:16] = 40.0                      # the first warp's rows: every code > 128
    row_exp[40] = 20.0                       # one row in another warp
    w = (w * np.exp2(row_exp)[:, None]).astype(np.float32)
    q, se = OQ.quant_mxfp4_weights(w)
    assert (se > 128).any() and (se <= 128).any()
    Wd = dict(q=q, s=se, deq=OG.dequant_mxfp4(q, se), epi=None)
    x = inputs.activations_bf16(M, K, seed=M + 72)
    y = run_gpu(qg, "mxfp4", Wd, x, M, N, K)
    ref, _ = reference(Wd, x)
    unit = np.exp2(-row_exp)[None, :]        # every row back to unit order (exact)
    check_gemm(y * unit, ref * unit, "mxfp4 scale range M=%d" % M)


@pytest.mark.parametrize("M", [1, 16])
def test_nvfp4_every_finite_block_scale_code(qg, M):
    """NVFP4 block scales over every finite E4M3 code (subnormals and 448
    included) and random E2M1 codes: the folded decode (factor 2^117 times
    the scale, the row multiplied by 2^9 at the end) must give the product of
    the canonical weights."""
    N, K = 128, 2048
    r = np.random.Generator(np.random.PCG64(80 + M))
    q = r.integers(0, 256, (N, K // 2)).astype(np.uint8)
    sb = r.integers(0, 0x7F, (N, K // 16)).astype(np.uint8)      # 0x00 .. 0x7E, all finite
    sb[0, :0x7F] = np.arange(0x7F, dtype=np.uint8)
    gs = np.float32(0.75)
    Wd = dict(q=q, s=sb, gs=gs, deq=OG.dequant_nvfp4(q, sb), epi=np.full(N, float(gs)))
    x = inputs.activations_bf16(M, K, seed=81 + M)
    y = run_gpu(qg, "nvfp4", Wd, x, M, N, K)
    ref, _ = reference(Wd, x)
    check_gemm(y, ref, "nvfp4 all scale codes M=%d" % M)


def test_stream_read_measurement_aid(qg):
    """The bench's read-ceiling probe runs on any 16-byte multiple, leaves no
    device error and writes its sink only on the one sentinel value."""
    buf = torch.arange(1 << 20, dtype=torch.int32, device="cuda")
    sink = torch.zeros(1, dtype=torch.int32, device="cuda")
    for nbytes in (16, 4096, 4 << 20):
        qg.qg_stream_read(buf, nbytes, sink)
    qg.qg_check_device_error()
    assert int(sink.item()) == 0


@pytest.mark.parametrize("fmt", FORMATS)
def test_decode_large_n_sampled_rows(qg, fmt):
    """N = 65536, K = 4096 (well past one wave of CTAs) at M = 1 and 16:
    seeded random codes and scales of each format (no quantizer needed at
    this size), parity on a seeded sample of 256 output channels, every
    output finite."""
    N, K = 65536, 4096
    r = np.random.Generator(np.random.PCG64(123))
    if fmt == "fp8":
        q = r.integers(0, 0x7F, (N, K)).astype(np.uint8) | (r.integers(0, 2, (N, K)) << 7).astype(np.uint8)
        q[(q & 0x7F) == 0x7F] = 0x30                                  # no NaN codes
    else:
        q = r.integers(0, 256, (N, K // 2)).astype(np.uint8)
    if fmt == "int4":
        s = OF.bf16_encode((r.uniform(0.5, 2.0, (N, K // 128)) * 0.003).astype(np.float32))
    elif fmt == "fp8":
        s = (r.uniform(0.5, 2.0, N) * 0.001).astype(np.float32)
    elif fmt == "mxfp4":
        s = r.integers(117, 124, (N, K // 32)).astype(np.uint8)
    else:
        s = r.integers(0x20, 0x50, (N, K // 16)).astype(np.uint8)
    cols = np.sort(r.choice(N, 256, replace=False))
    if fmt == "int4":
        Wd = dict(q=q, s=s, deq=OG.dequant_int4(q[cols], s[cols], 128), epi=None)
    elif fmt == "fp8":
        Wd = dict(q=q, s=s, deq=OG.dequant_fp8(q[cols]), epi=s[cols].astype(np.float64))
    elif fmt == "mxfp4":
        Wd = dict(q=q, s=s, deq=OG.dequant_mxfp4(q[cols], s[cols]), epi=None)
    else:
        gs = np.float32(0.01)
        Wd = dict(q=q, s=s, gs=gs, deq=OG.dequant_nvfp4(q[cols], s[cols]), epi=np.full(len(cols), float(gs)))
    for M in (1, 16):
        x = inputs.activations_bf16(M, K, seed=125 + M)
        y = run_gpu(qg, fmt, Wd, x, M, N, K)
        assert np.all(np.isfinite(y))
        ref, _ = reference(Wd, x)
        check_gemm(y[:, cols], ref, "%s large N M=%d" % (fmt, M))
