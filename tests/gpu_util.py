"""Host<->device helpers for the GPU parity tests (no arithmetic of the method)."""

import functools

import numpy as np
import torch


def dev(a):
    """numpy array -> contiguous CUDA tensor with the same bytes (uint16 via int16)."""
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        a = a.view(np.int16)
    return torch.from_numpy(a).cuda()


def host(t, dtype=None):
    """CUDA tensor -> numpy array; bf16 bit tensors (int16) come back as uint16."""
    a = t.detach().cpu().numpy()
    if a.dtype == np.int16:
        a = a.view(np.uint16)
    return a if dtype is None else a.view(dtype)


def empty(shape, dtype):
    return torch.empty(shape, dtype=dtype, device="cuda")


def rel_fro(y, ref):
    y = np.asarray(y, np.float64)
    ref = np.asarray(ref, np.float64)
    return float(np.linalg.norm(y - ref) / max(np.linalg.norm(ref), 1e-300))


def check_gemm(y, ref, tag=""):
    """The spec bar: relative Frobenius <= 2e-3 and max |err| <= 1e-2 max |ref|."""
    fro = rel_fro(y, ref)
    mx = float(np.max(np.abs(np.asarray(y, np.float64) - ref))) if ref.size else 0.0
    bound = 1e-2 * float(np.max(np.abs(ref))) if ref.size else 0.0
    assert np.all(np.isfinite(y)), "%s: non-finite output" % tag
    assert fro <= 2e-3, "%s: rel Frobenius %.3e > 2e-3" % (tag, fro)
    assert mx <= bound, "%s: max abs err %.3e > %.3e" % (tag, mx, bound)
    return fro


@functools.lru_cache(maxsize=2)
def config_expert_weights(E, N, K, seed):
    """INT4 g128 expert weights [E][N][K/2] and bf16 scales [E][N][K/128] from
    N(0, 0.02) weights (the oracle's RTN quantizer), generated once per
    process: the config-size MoE tests of several files share them (callers
    must not modify the arrays)."""
    from numerics_packed_int4_gb300 import inputs
    from oracle import quant as OQ
    qs, ss = [], []
    for e in range(E):
        q, s = OQ.quant_int4_rtn(inputs.weights_f32(N, K, seed=seed + e), 128)
        qs.append(q)
        ss.append(s)
    return np.stack(qs), np.stack(ss)
