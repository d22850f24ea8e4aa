"""Host-side checks of the C ABI (no GPU): the library builds and loads, every
symbol declared in include/qgemm.h is exported and bound, and argument
validation fails cleanly before any CUDA call."""

import ctypes
import os
import re

import numpy as np
import pytest

from tests.conftest import ROOT

HEADER = os.path.join(ROOT, "include", "qgemm.h")


def header_symbols():
    src = open(HEADER).read()
    return re.findall(r"QG_API\s+(?:const\s+char\s*\*|qg_status|void)\s+(\w+)\s*\(", src)


@pytest.fixture(scope="module")
def lib():
    from numerics_packed_int4_gb300 import _build, qgemm
    if not os.path.exists(qgemm.LIB_PATH):
        _build.build()
    return qgemm.load()


def test_header_declares_the_six_path_entry_points():
    names = set(header_symbols())
    for n in ("qgemm_w4a16", "qgemm_w8a16", "qgemm_fp4a16", "quant_act_mxfp4",
              "quant_act_fp8_block", "qgemm_w4a8_grouped"):
        assert n in names


def test_library_exports_every_header_symbol(lib):
    for name in header_symbols():
        assert hasattr(lib, name), name


def test_binding_covers_every_header_symbol():
    from numerics_packed_int4_gb300 import qgemm
    bound = set(qgemm.SIGNATURES) | {"qg_last_error_string", "qg_set_wait_limit"}
    assert bound == set(header_symbols())
    for name in qgemm.SIGNATURES:
        if name != "qg_check_device_error":
            assert callable(getattr(qgemm, name))


P = ctypes.c_void_p
FAKE = P(0x10000)            # aligned, never dereferenced: validation fails first
FAKE_MIS = P(0x10001)


def _rc(lib, name, *args):
    return getattr(lib, name)(*args, P(0))


def test_null_pointers_are_invalid_args(lib):
    assert _rc(lib, "qgemm_w4a16", None, FAKE, 128, FAKE, FAKE, 1, 128, 128) == 1
    assert _rc(lib, "qgemm_w8a16", FAKE, None, FAKE, FAKE, 1, 128, 128) == 1
    assert _rc(lib, "quant_act_fp8_block", FAKE, None, FAKE, 128, 1, 128) == 1
    assert _rc(lib, "qgemm_w4a8_grouped", None, FAKE, FAKE, FAKE, FAKE, 128, FAKE, 1, 1, 16, 128) == 1
    assert "NULL" in lib.qg_last_error_string().decode()


def test_shape_rules(lib):
    assert _rc(lib, "qgemm_w4a16", FAKE, FAKE, 128, FAKE, FAKE, 1, 128, 100) == 2    # K % 32
    assert _rc(lib, "qgemm_w4a16", FAKE, FAKE, 128, FAKE, FAKE, 1, 128, 160) == 2    # K % g
    assert _rc(lib, "qgemm_w8a16", FAKE, FAKE, FAKE, FAKE, 1, 128, 112) == 2         # K % 32
    assert _rc(lib, "qgemm_w8a8", FAKE, FAKE, FAKE, FAKE, 1, 128, 160) == 2          # K % 128 (1 x 128 blocks)
    assert _rc(lib, "qgemm_w4a16", FAKE, FAKE, 48, FAKE, FAKE, 1, 128, 384) == 2     # g % 32
    assert _rc(lib, "qgemm_w8a16", FAKE, FAKE, FAKE, FAKE, 1, 12, 128) == 2          # N % 8
    assert _rc(lib, "qgemm_fp4a16", FAKE, FAKE, 0, 16, None, FAKE, FAKE, 1, 128, 128) == 2
    assert _rc(lib, "qgemm_fp4a16", FAKE, FAKE, 1, 16, None, FAKE, FAKE, 1, 128, 128) == 1
    assert _rc(lib, "qgemm_fp4a16", FAKE, FAKE, 7, 16, FAKE, FAKE, FAKE, 1, 128, 128) == 1
    assert _rc(lib, "quant_act_mxfp4", FAKE, FAKE, FAKE, 8, 1, 128) == 2
    assert _rc(lib, "quant_act_fp8_block", FAKE, FAKE, FAKE, 12, 1, 96) == 2
    assert _rc(lib, "qgemm_w4a8_grouped", FAKE, FAKE, FAKE, FAKE, FAKE, 48, FAKE, 1, 1, 16, 384) == 2  # g
    assert _rc(lib, "qgemm_w4a8_grouped", FAKE, FAKE, FAKE, FAKE, FAKE, 32, FAKE, 1, 1, 12, 128) == 2  # N % 8
    assert _rc(lib, "qgemm_w4a8_grouped", FAKE, FAKE, FAKE, FAKE, FAKE, 128, FAKE, 1, 1, 16, 160) == 2  # K % g
    assert _rc(lib, "qgemm_w4a8_grouped", FAKE, FAKE, FAKE, FAKE, FAKE, 64, FAKE, 0, 1, 8, 96) == 2  # K % g
    assert _rc(lib, "qg_dequant_weights", 9, FAKE, FAKE, 128, FAKE, 8, 128) == 1


def test_misaligned_pointers(lib):
    assert _rc(lib, "qgemm_w4a16", FAKE_MIS, FAKE, 128, FAKE, FAKE, 1, 128, 128) == 3
    assert _rc(lib, "quant_act_fp8_block", FAKE, FAKE_MIS, FAKE, 128, 1, 128) == 3


def test_validation_of_the_widened_entry_points(lib):
    """The entry points beyond the six of the path reject bad arguments
    before touching the GPU."""
    # asymmetric INT4
    assert _rc(lib, "qgemm_w4a16_zp", FAKE, FAKE, None, 64, FAKE, FAKE, 1, 128, 128) == 1
    assert _rc(lib, "qgemm_w4a16_zp", FAKE, FAKE, FAKE, 48, FAKE, FAKE, 1, 128, 384) == 2
    assert _rc(lib, "qg_quantize_weights_int4_zp", FAKE, FAKE, FAKE, FAKE, 12, 8, 96) == 2
    assert _rc(lib, "qg_dequant_weights_int4_zp", FAKE, FAKE, FAKE, 16, FAKE, 8, 128) == 2
    # W8A8 GEMV
    assert _rc(lib, "qgemm_w8a8", FAKE, None, FAKE, FAKE, 1, 128, 128) == 1
    assert _rc(lib, "qgemm_w8a8", FAKE, FAKE, FAKE, FAKE, 1, 12, 128) == 2
    assert _rc(lib, "qgemm_w8a8", FAKE, FAKE, FAKE_MIS, FAKE, 1, 128, 128) == 3
    # W4A8 on fp16 activation copies, and its harness kernels
    assert _rc(lib, "qgemm_w4a8_grouped_f16act", None, FAKE, FAKE, FAKE, FAKE, None, 128, FAKE, 1, 1, 16, 128) == 1
    assert _rc(lib, "qgemm_w4a8_grouped_f16act", FAKE, FAKE, FAKE, FAKE, FAKE, None, 64, FAKE, 1, 1, 16, 128) == 2
    assert _rc(lib, "qgemm_w4a8_grouped_f16act", FAKE, FAKE, FAKE, FAKE, FAKE, None, 128, FAKE, 1, 1, 24, 128) == 2
    assert _rc(lib, "qgemm_w4a8_grouped_f16act", FAKE_MIS, FAKE, FAKE, FAKE, FAKE, None, 128, FAKE, 1, 1, 16, 128) == 3
    assert _rc(lib, "qg_w4a8_row_shifts", FAKE, None, 4, 8) == 1
    assert _rc(lib, "qg_e4m3_to_f16", FAKE, FAKE, 12) == 2
    assert _rc(lib, "qg_e4m3_to_f16", FAKE, FAKE_MIS, 16) == 3
    assert _rc(lib, "qg_moe_gather_fp8_f16", FAKE, FAKE, FAKE, FAKE, FAKE, 4, 4, 24) == 2
    assert _rc(lib, "qg_swiglu_quant_fp8_f16", FAKE, FAKE, FAKE, 4, 12) == 2
    # W4A8 with FP8 group scales
    assert _rc(lib, "qgemm_w4a8_grouped_fp8s", FAKE, FAKE, FAKE, FAKE, None, FAKE, FAKE, 1, 1, 16, 128) == 1
    assert _rc(lib, "qgemm_w4a8_grouped_fp8s", FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 1, 1, 16, 96) == 2
    assert _rc(lib, "qg_w4a8_fp8_scales", FAKE, FAKE, None, 4, 8) == 1
    assert _rc(lib, "qg_w4a8_fp8_scales", FAKE, FAKE, FAKE, 4, 0) == 1


def test_wait_limit_setter_is_callable(lib):
    lib.qg_set_wait_limit(5)
    lib.qg_set_wait_limit(0)


def test_input_generators_are_deterministic():
    from numerics_packed_int4_gb300 import inputs
    a = inputs.activations_bf16(4, 256, seed=3, outlier_frac=0.01, outlier_scale=50)
    b = inputs.activations_bf16(4, 256, seed=3, outlier_frac=0.01, outlier_scale=50)
    assert a.dtype == np.uint16 and np.array_equal(a, b)
    w = inputs.weights_f32(8, 64, seed=1)
    assert w.dtype == np.float32 and abs(float(w.std()) - 0.02) < 0.005
    r = inputs.moe_routing(64, 8, 2, seed=4)
    assert r["expert_off"][-1] == 128 and np.all(np.diff(r["expert_off"]) >= 0)
    assert np.all(r["route_weight"] > 0)


def test_quantizer_workload_injects_edges():
    from numerics_packed_int4_gb300 import inputs
    x = inputs.quantizer_activations_bf16(16, 1024, seed=0)
    v = (x.astype(np.uint32) << 16).view(np.float32)
    anchors = np.abs(v[0, ::128][::3])
    assert np.all(np.log2(anchors / 448.0) == np.round(np.log2(anchors / 448.0)))


def test_w4a4_argument_validation(lib):
    # (w_e2m1, w_e8m0, a_e2m1, a_e8m0, a_work, y, M, N, K, stream)
    assert _rc(lib, "qgemm_w4a4_mxfp4", FAKE, FAKE, None, FAKE, FAKE, FAKE, 1, 128, 128) == 1
    assert _rc(lib, "qgemm_w4a4_mxfp4", FAKE, None, FAKE, FAKE, FAKE, FAKE, 1, 128, 128) == 1
    assert _rc(lib, "qgemm_w4a4_mxfp4", FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 1, 12, 128) == 2     # N % 8
    assert _rc(lib, "qgemm_w4a4_mxfp4", FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 1, 128, 80) == 2     # K % 32
    assert _rc(lib, "qgemm_w4a4_mxfp4", FAKE, FAKE, FAKE_MIS, FAKE, FAKE, FAKE, 1, 128, 128) == 3
    assert _rc(lib, "qgemm_w4a4_mxfp4", FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 0, 128, 128) == 0    # M = 0


def test_stream_read_argument_validation(lib):
    # (p, bytes, sink, stream)
    assert _rc(lib, "qg_stream_read", None, 1024, FAKE) == 1
    assert _rc(lib, "qg_stream_read", FAKE, 1024, None) == 1
    assert _rc(lib, "qg_stream_read", FAKE, 1000, FAKE) == 2
    assert _rc(lib, "qg_stream_read", FAKE, 0, FAKE) == 2
    assert _rc(lib, "qg_stream_read", FAKE_MIS, 1024, FAKE) == 3


def _bf16_round(x):
    """float64 -> nearest bf16 value (ties to even), as float64."""
    from oracle import formats as F
    return F.bf16_decode(F.bf16_encode(np.asarray(x, np.float32)))


def test_folded_fp4_decode_is_exact_for_every_code():
    """The decode kernels form an E2M1 weight with one bf16 multiply of its
    bit pattern (value x 2^-126, the 0.5 code a bf16 subnormal) by a folded
    factor: NVFP4 2^117 x e4m3(sb), MXFP4 2^(c-1) for E8M0 codes c <= 128.
    Emulated here with IEEE arithmetic over every E2M1 code and every finite
    scale code: the one rounding never changes the value, so the NVFP4 weight
    is exactly 2^-9 times the canonical one and the MXFP4 weight is exact."""
    from oracle import formats as F
    e2m1 = F.e2m1_decode(np.arange(16)).astype(np.float64)
    raw = e2m1 * 2.0 ** -126                               # the bit pattern's value
    assert np.array_equal(_bf16_round(raw), raw)           # representable (subnormal for 0.5)
    sb = np.array([c for c in range(256) if (c & 0x7F) != 0x7F])
    e4m3 = F.e4m3_decode(sb).astype(np.float64)
    fold = _bf16_round(e4m3 * 2.0 ** 117)
    assert np.array_equal(fold, e4m3 * 2.0 ** 117)          # the factor is exact
    assert np.all(np.abs(fold[fold != 0]) >= 2.0 ** -126)  # and normal
    prod = _bf16_round(raw[:, None] * fold[None, :])
    assert np.array_equal(prod, e2m1[:, None] * e4m3[None, :] * 2.0 ** -9)
    c = np.arange(0, 129)
    f = _bf16_round(2.0 ** (c - 1.0))
    assert np.array_equal(f, 2.0 ** (c - 1.0))
    prod = _bf16_round(raw[:, None] * f[None, :])
    assert np.array_equal(prod, e2m1[:, None] * 2.0 ** (c[None, :] - 127.0))


def test_binding_argument_counts_match_the_header():
    """Every ctypes signature in the binding has as many arguments as the
    prototype in include/qgemm.h (a dropped or extra argument would shift
    every pointer after it)."""
    from numerics_packed_int4_gb300 import qgemm
    src = re.sub(r"/\*.*?\*/", "", open(HEADER).read(), flags=re.S)
    protos = dict(re.findall(r"QG_API\s+(?:const\s+char\s*\*|qg_status|void)\s+(\w+)\s*\(([^)]*)\)", src))
    def ctype_of(param):
        p = param.strip()
        if "*" in p or p.startswith("qg_stream_t"):
            return ctypes.c_void_p
        if p.startswith("long long"):
            return ctypes.c_longlong
        if p.startswith("uint32_t"):
            return ctypes.c_uint32
        if p.startswith("int "):
            return ctypes.c_int
        raise AssertionError("unexpected parameter type: " + p)

    for name, argtypes in qgemm.SIGNATURES.items():
        params = [p for p in protos[name].split(",") if p.strip() and p.strip() != "void"]
        assert len(params) == len(argtypes), (name, len(params), len(argtypes))
        for prm, at in zip(params, argtypes):
            assert ctype_of(prm) == at, (name, prm, at)


def test_w4a4_noalloc_argument_validation(lib):
    # (w_e2m1, w_e8m0, a_e2m1, a_e8m0, y, M, N, K, stream): sizes are checked
    # before the work array is touched, so none of these needs a GPU
    assert _rc(lib, "qgemm_w4a4_mxfp4_noalloc", FAKE, FAKE, FAKE, FAKE, FAKE, -1, 128, 128) == 1
    assert _rc(lib, "qgemm_w4a4_mxfp4_noalloc", FAKE, FAKE, FAKE, FAKE, FAKE, 1, 128, 0) == 1
    assert _rc(lib, "qgemm_w4a4_mxfp4_noalloc", FAKE, FAKE, FAKE, FAKE, FAKE, 4097, 128, 2048) == 2
    assert "static work area" in lib.qg_last_error_string().decode()


def test_w4a4_g_argument_validation(lib):
    # (w_e2m1, w_e8m0, a_e2m1, a_e8m0, g_act, a_work, y, M, N, K, stream)
    for g in (8, 24, 64):
        assert _rc(lib, "qgemm_w4a4_mxfp4_g", FAKE, FAKE, FAKE, FAKE, g, FAKE, FAKE, 1, 128, 128) == 2
    assert "g_act" in lib.qg_last_error_string().decode()
    assert _rc(lib, "qgemm_w4a4_mxfp4_g", FAKE, FAKE, None, FAKE, 16, FAKE, FAKE, 1, 128, 128) == 1
    assert _rc(lib, "qgemm_w4a4_mxfp4_g", FAKE, FAKE, FAKE, FAKE, 16, FAKE, FAKE, 1, 12, 128) == 2   # N % 8
    assert _rc(lib, "qgemm_w4a4_mxfp4_g", FAKE, FAKE, FAKE_MIS, FAKE, 16, FAKE, FAKE, 1, 128, 128) == 3
    assert _rc(lib, "qgemm_w4a4_mxfp4_g", FAKE, FAKE, FAKE, FAKE, 16, FAKE, FAKE, 0, 128, 128) == 0  # M = 0
