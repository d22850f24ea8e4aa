"""ctypes binding of libqgemm.so (include/qgemm.h), argument marshalling only.

Each function takes torch CUDA tensors (or ``None`` where the C ABI allows a
NULL pointer), passes their device pointers and the current torch stream to
the C entry point of the same name, and raises ``QgemmError`` on a non-zero
status.  No computation happens here.  The library must have been built
(``numerics_packed_int4_gb300._build.build()``); if it is missing, ``load``
raises -- there is no fallback.
"""

import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libqgemm.so")

STATUS = {0: "QG_OK", 1: "QG_ERR_INVALID_ARG", 2: "QG_ERR_UNSUPPORTED_SHAPE", 3: "QG_ERR_MISALIGNED",
          4: "QG_ERR_CUDA", 5: "QG_ERR_TIMEOUT"}
QG_SCALE_E8M0, QG_SCALE_E4M3 = 0, 1
QG_FMT_INT4, QG_FMT_FP8, QG_FMT_MXFP4, QG_FMT_NVFP4 = 0, 1, 2, 3

P, I, U32, I64 = ctypes.c_void_p, ctypes.c_int, ctypes.c_uint32, ctypes.c_longlong

# name -> argument types (every data pointer and the stream are void*)
SIGNATURES = {
    "qgemm_w4a16": [P, P, I, P, P, I, I, I, P],
    "qgemm_w8a16": [P, P, P, P, I, I, I, P],
    "qgemm_w8a8": [P, P, P, P, I, I, I, P],
    "qgemm_fp4a16": [P, P, I, I, P, P, P, I, I, I, P],
    "qgemm_w4a4_mxfp4": [P, P, P, P, P, P, I, I, I, P],
    "qgemm_w4a4_mxfp4_noalloc": [P, P, P, P, P, I, I, I, P],
    "qgemm_w4a4_mxfp4_g": [P, P, P, P, I, P, P, I, I, I, P],
    "qg_stream_read": [P, I64, P, P],
    "quant_act_mxfp4": [P, P, P, I, I, I, P],
    "quant_act_fp8_block": [P, P, P, I, I, I, P],
    "qgemm_w4a8_grouped": [P, P, P, P, P, I, P, I, I, I, I, P],
    "qgemm_w4a8_grouped_fp8s": [P, P, P, P, P, P, P, I, I, I, I, P],
    "qg_w4a8_fp8_scales": [P, P, P, I, I, P],
    "qgemm_w4a16_zp": [P, P, P, I, P, P, I, I, I, P],
    "qgemm_w4a8_grouped_f16act": [P, P, P, P, P, P, I, P, I, I, I, I, P],
    "qg_w4a8_row_shifts": [P, P, I, I, P],
    "qg_e4m3_to_f16": [P, P, I64, P],
    "qg_moe_gather_fp8_f16": [P, P, P, P, P, I, I, I, P],
    "qg_swiglu_quant_fp8_f16": [P, P, P, I, I, P],
    "qg_quantize_weights_int4_zp": [P, P, P, P, I, I, I, P],
    "qg_dequant_weights_int4_zp": [P, P, P, I, P, I, I, P],
    "qg_quantize_weights_int4": [P, P, P, I, I, I, P],
    "qg_quantize_weights_fp8": [P, P, P, I, I, P],
    "qg_quantize_weights_mxfp4": [P, P, P, I, I, I, P],
    "qg_quantize_weights_nvfp4": [P, P, P, P, I, I, P],
    "qg_moe_gather_fp8": [P, P, P, P, P, I, I, I, P],
    "qg_swiglu_quant_fp8": [P, P, P, I, I, P],
    "qg_moe_combine": [P, P, P, P, I, I, I, I, P],
    "qg_dequant_weights": [I, P, P, I, P, I, I, P],
    "qg_check_device_error": [P],
    "qg_selftest_wait_timeout": [U32, P],
}

_lib = None


class QgemmError(RuntimeError):
    def __init__(self, name, status, msg):
        super().__init__("%s -> %s: %s" % (name, STATUS.get(status, status), msg))
        self.status = status


def load(path=None):
    """Load the shared library once; raise if it is not built."""
    global _lib
    if _lib is not None:
        return _lib
    path = path or LIB_PATH
    if not os.path.exists(path):
        raise OSError("libqgemm.so is not built (%s); run __graft_entry__.build()" % path)
    lib = ctypes.CDLL(path)
    for name, argtypes in SIGNATURES.items():
        f = getattr(lib, name)
        f.argtypes = argtypes
        f.restype = ctypes.c_int
    lib.qg_last_error_string.argtypes = []
    lib.qg_last_error_string.restype = ctypes.c_char_p
    lib.qg_set_wait_limit.argtypes = [U32]
    lib.qg_set_wait_limit.restype = None
    _lib = lib
    return lib


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is not None:
        return ctypes.c_void_p(stream)
    import torch
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def _call(name, *args, stream=None):
    lib = load()
    st = getattr(lib, name)(*args, _stream(stream))
    if st != 0:
        raise QgemmError(name, st, lib.qg_last_error_string().decode())
    return st


def call_raw(name, *args):
    """Call an entry point with already-marshalled ctypes arguments (tests)."""
    lib = load()
    return getattr(lib, name)(*args)


def last_error_string():
    return load().qg_last_error_string().decode()


# ---- entry points ---------------------------------------------------------------

def qgemm_w4a16(w_q, w_s, g, x, y, M, N, K, stream=None):
    return _call("qgemm_w4a16", _ptr(w_q), _ptr(w_s), g, _ptr(x), _ptr(y), M, N, K, stream=stream)


def qgemm_w8a16(w_e4m3, w_cs, x, y, M, N, K, stream=None):
    return _call("qgemm_w8a16", _ptr(w_e4m3), _ptr(w_cs), _ptr(x), _ptr(y), M, N, K, stream=stream)


def qgemm_w8a8(w_e4m3, w_cs, x, y, M, N, K, stream=None):
    return _call("qgemm_w8a8", _ptr(w_e4m3), _ptr(w_cs), _ptr(x), _ptr(y), M, N, K, stream=stream)


def qgemm_fp4a16(w_e2m1, w_bs, scale_fmt, g, global_scale, x, y, M, N, K, stream=None):
    return _call("qgemm_fp4a16", _ptr(w_e2m1), _ptr(w_bs), scale_fmt, g, _ptr(global_scale),
                 _ptr(x), _ptr(y), M, N, K, stream=stream)


def qg_stream_read(p, nbytes, sink, stream=None):
    return _call("qg_stream_read", _ptr(p), nbytes, _ptr(sink), stream=stream)


def qgemm_w4a4_mxfp4(w_e2m1, w_e8m0, a_e2m1, a_e8m0, a_work, y, M, N, K, stream=None):
    return _call("qgemm_w4a4_mxfp4", _ptr(w_e2m1), _ptr(w_e8m0), _ptr(a_e2m1), _ptr(a_e8m0), _ptr(a_work),
                 _ptr(y), M, N, K, stream=stream)


def qgemm_w4a4_mxfp4_g(w_e2m1, w_e8m0, a_e2m1, a_e8m0, g_act, a_work, y, M, N, K, stream=None):
    return _call("qgemm_w4a4_mxfp4_g", _ptr(w_e2m1), _ptr(w_e8m0), _ptr(a_e2m1), _ptr(a_e8m0), g_act,
                 _ptr(a_work), _ptr(y), M, N, K, stream=stream)


def qgemm_w4a4_mxfp4_noalloc(w_e2m1, w_e8m0, a_e2m1, a_e8m0, y, M, N, K, stream=None):
    return _call("qgemm_w4a4_mxfp4_noalloc", _ptr(w_e2m1), _ptr(w_e8m0), _ptr(a_e2m1), _ptr(a_e8m0),
                 _ptr(y), M, N, K, stream=stream)


def quant_act_mxfp4(x, q, s_e8m0, g, M, K, stream=None):
    return _call("quant_act_mxfp4", _ptr(x), _ptr(q), _ptr(s_e8m0), g, M, K, stream=stream)


def quant_act_fp8_block(x, q, s, g, M, K, stream=None):
    return _call("quant_act_fp8_block", _ptr(x), _ptr(q), _ptr(s), g, M, K, stream=stream)


def qgemm_w4a8_grouped(a_e4m3, a_s, expert_off, w_q, w_s, g, y, R, E, N, K, stream=None):
    return _call("qgemm_w4a8_grouped", _ptr(a_e4m3), _ptr(a_s), _ptr(expert_off), _ptr(w_q),
                 _ptr(w_s), g, _ptr(y), R, E, N, K, stream=stream)


def qgemm_w4a8_grouped_fp8s(a_e4m3, a_s, expert_off, w_q, w_s8, w_cs8, y, R, E, N, K, stream=None):
    return _call("qgemm_w4a8_grouped_fp8s", _ptr(a_e4m3), _ptr(a_s), _ptr(expert_off), _ptr(w_q),
                 _ptr(w_s8), _ptr(w_cs8), _ptr(y), R, E, N, K, stream=stream)


def qg_w4a8_fp8_scales(w_s, w_s8, w_cs8, rows, G, stream=None):
    return _call("qg_w4a8_fp8_scales", _ptr(w_s), _ptr(w_s8), _ptr(w_cs8), rows, G, stream=stream)


def qgemm_w4a8_grouped_f16act(a_f16, a_s, expert_off, w_q, w_s, w_e, g, y, R, E, N, K, stream=None):
    return _call("qgemm_w4a8_grouped_f16act", _ptr(a_f16), _ptr(a_s), _ptr(expert_off), _ptr(w_q),
                 _ptr(w_s), _ptr(w_e), g, _ptr(y), R, E, N, K, stream=stream)


def qg_w4a8_row_shifts(w_s, w_e, rows, G, stream=None):
    return _call("qg_w4a8_row_shifts", _ptr(w_s), _ptr(w_e), rows, G, stream=stream)


def qg_moe_gather_fp8_f16(src_q, src_s, route_rows, dst_f16, dst_s, R, T, K, stream=None):
    return _call("qg_moe_gather_fp8_f16", _ptr(src_q), _ptr(src_s), _ptr(route_rows), _ptr(dst_f16),
                 _ptr(dst_s), R, T, K, stream=stream)


def qg_swiglu_quant_fp8_f16(gate_up, q_f16, s, R, I, stream=None):
    return _call("qg_swiglu_quant_fp8_f16", _ptr(gate_up), _ptr(q_f16), _ptr(s), R, I, stream=stream)


def qg_e4m3_to_f16(q, out, n, stream=None):
    return _call("qg_e4m3_to_f16", _ptr(q), _ptr(out), int(n), stream=stream)


def qgemm_w4a16_zp(w_q, w_s, w_z, g, x, y, M, N, K, stream=None):
    return _call("qgemm_w4a16_zp", _ptr(w_q), _ptr(w_s), _ptr(w_z), g, _ptr(x), _ptr(y), M, N, K,
                 stream=stream)


def qg_quantize_weights_int4_zp(w, w_q, w_s, w_z, g, N, K, stream=None):
    return _call("qg_quantize_weights_int4_zp", _ptr(w), _ptr(w_q), _ptr(w_s), _ptr(w_z), g, N, K,
                 stream=stream)


def qg_dequant_weights_int4_zp(w_q, w_s, w_z, g, w_out, N, K, stream=None):
    return _call("qg_dequant_weights_int4_zp", _ptr(w_q), _ptr(w_s), _ptr(w_z), g, _ptr(w_out), N, K,
                 stream=stream)


def qg_quantize_weights_int4(w, w_q, w_s, g, N, K, stream=None):
    return _call("qg_quantize_weights_int4", _ptr(w), _ptr(w_q), _ptr(w_s), g, N, K, stream=stream)


def qg_quantize_weights_fp8(w, w_e4m3, w_cs, N, K, stream=None):
    return _call("qg_quantize_weights_fp8", _ptr(w), _ptr(w_e4m3), _ptr(w_cs), N, K, stream=stream)


def qg_quantize_weights_mxfp4(w, w_e2m1, w_e8m0, g, N, K, stream=None):
    return _call("qg_quantize_weights_mxfp4", _ptr(w), _ptr(w_e2m1), _ptr(w_e8m0), g, N, K, stream=stream)


def qg_quantize_weights_nvfp4(w, w_e2m1, w_e4m3, global_scale, N, K, stream=None):
    return _call("qg_quantize_weights_nvfp4", _ptr(w), _ptr(w_e2m1), _ptr(w_e4m3), _ptr(global_scale),
                 N, K, stream=stream)


def qg_moe_gather_fp8(src_q, src_s, route_rows, dst_q, dst_s, R, T, K, stream=None):
    return _call("qg_moe_gather_fp8", _ptr(src_q), _ptr(src_s), _ptr(route_rows), _ptr(dst_q),
                 _ptr(dst_s), R, T, K, stream=stream)


def qg_swiglu_quant_fp8(gate_up, q, s, R, I_, stream=None):
    return _call("qg_swiglu_quant_fp8", _ptr(gate_up), _ptr(q), _ptr(s), R, I_, stream=stream)


def qg_moe_combine(down, row_of, weight, out, T, topk, R, H, stream=None):
    return _call("qg_moe_combine", _ptr(down), _ptr(row_of), _ptr(weight), _ptr(out), T, topk, R, H,
                 stream=stream)


def qg_dequant_weights(fmt, w, scales, g, w_out, N, K, stream=None):
    return _call("qg_dequant_weights", fmt, _ptr(w), _ptr(scales), g, _ptr(w_out), N, K, stream=stream)


def qg_check_device_error(stream=None):
    return _call("qg_check_device_error", stream=stream)


def qg_selftest_wait_timeout(polls, stream=None):
    return _call("qg_selftest_wait_timeout", int(polls), stream=stream)


def qg_set_wait_limit(iterations):
    load().qg_set_wait_limit(int(iterations))
