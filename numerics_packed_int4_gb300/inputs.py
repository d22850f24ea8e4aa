"""Seeded synthetic inputs shared by the tests, the bench and the oracle.

This module holds no quantization, dequantization or product arithmetic: it
only draws random numbers and arranges them into the shapes, value
distributions and injected edge values of the workloads.  It imports numpy
and torch (CPU) only, never the CUDA library and never the oracle.

Distributions (all seeded, numpy PCG64):
* weights: fp32 N(0, 0.02)
* activations: N(0, 1) rounded to bf16 (torch's CPU cast), optionally with a
  fraction of K-channels multiplied by an outlier factor (x50 for the prefill
  workload, x100 on 0.5 % of channels for the quantizer workload)
* quantizer workload: additionally injected E4M3 midpoints/ties/subnormals in
  1x128 blocks anchored so the block scale is a power of two, and 16-element
  blocks whose maximum has significand 1.75 / 1.7421875 / 1.625 / 1.5 with
  elements at E2M1 midpoints of the block scale
* MoE routing: N(0, 1) logits, top-2 experts by logit (ties to the lower
  index), combine weights softmax(logits) of the chosen experts (not
  renormalized), rows grouped by expert in token order
"""

import numpy as np
import torch


def rng(seed):
    return np.random.Generator(np.random.PCG64(seed))


def f32_to_bf16_bits(x):
    """bf16 bit patterns (uint16) of float32 data, via torch's CPU cast."""
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16).copy()


def weights_f32(N, K, seed, std=0.02):
    return (rng(seed).standard_normal((N, K), dtype=np.float32) * np.float32(std)).astype(np.float32)


def activations_bf16(M, K, seed, outlier_frac=0.0, outlier_scale=1.0):
    r = rng(seed)
    x = r.standard_normal((M, K), dtype=np.float32)
    n_out = int(round(outlier_frac * K))
    if n_out:
        ch = r.permutation(K)[:n_out]
        x[:, ch] *= np.float32(outlier_scale)
    return f32_to_bf16_bits(x)


def _e4m3_positive_values():
    """Every positive finite E4M3 value (subnormals m*2**-9, normals up to 448)."""
    sub = [m * 2.0 ** -9 for m in range(1, 8)]
    nor = [2.0 ** (e - 7) * (1 + m / 8) for e in range(1, 16) for m in range(8)
           if not (e == 15 and m == 7)]
    return np.array(sub + nor)


def quantizer_activations_bf16(M, K, seed, outlier_frac=0.005, outlier_scale=100.0):
    """The quantizer workload: N(0,1) with outlier channels plus injected edges.

    Every 8th row carries injected 1x128 blocks: element 0 is the anchor
    448 * 2**j (so the FP8 block scale is exactly 2**j), the other 127 are
    E4M3 midpoints (ties) times 2**j, or one bf16 ulp either side, or
    subnormal-range values.  Every 8th row (offset 4) carries injected 16-blocks
    whose max has significand 1.75 / 1.7421875 / 1.625 / 1.5 and whose other
    elements sit at E2M1 midpoints times a power of two.
    """
    r = rng(seed)
    x = r.standard_normal((M, K), dtype=np.float32)
    n_out = int(round(outlier_frac * K))
    if n_out:
        ch = r.permutation(K)[:n_out]
        x[:, ch] *= np.float32(outlier_scale)
    vals = _e4m3_positive_values()
    mids = (vals[:-1] + vals[1:]) / 2.0
    mids = np.concatenate([[vals[0] / 2.0], mids])          # includes the 2**-10 tie
    for row in range(0, M, 8):
        for blk in range(0, K // 128, 3):
            j = int(r.integers(-6, 4))
            base = np.float32(2.0 ** j)
            pick = r.choice(mids, size=127) * base
            kind = r.integers(0, 4, size=127)
            bits = f32_to_bf16_bits(pick.astype(np.float32)).astype(np.int32)
            bits = np.where(kind == 1, bits + 1, np.where(kind == 2, bits - 1, bits))
            sign = np.where(r.integers(0, 2, size=127) == 1, 0x8000, 0)
            vals_blk = ((bits & 0x7FFF) | sign).astype(np.uint16)
            x[row, blk * 128] = np.float32(448.0) * base * (1 if r.integers(0, 2) else -1)
            x[row, blk * 128 + 1: blk * 128 + 128] = (
                vals_blk.astype(np.uint32) << 16).view(np.float32)
    e2m1_mids = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0])
    sig = np.array([1.75, 1.7421875, 1.625, 1.5])
    for row in range(4, M, 8):
        for blk in range(0, K // 16, 5):
            k = int(r.integers(-8, 8))
            vmax = np.float32(sig[int(r.integers(0, 4))] * 2.0 ** k)
            # block scale under the 0.75-threshold rule is 2**(k-2) or 2**(k-1);
            # place elements at E2M1 midpoints of both candidates
            scl = 2.0 ** (k - 2 + int(r.integers(0, 2)))
            el = r.choice(e2m1_mids, size=15) * scl
            el = np.minimum(el, float(vmax))
            sgn = np.where(r.integers(0, 2, size=15) == 1, -1.0, 1.0)
            x[row, blk * 16] = vmax
            x[row, blk * 16 + 1: blk * 16 + 16] = (el * sgn).astype(np.float32)
    return f32_to_bf16_bits(x)


def moe_routing(T, E, topk, seed):
    """Top-k routing from N(0,1) logits; rows grouped by expert in token order.

    Returns dict(route_rows [R] int32 source token per row, route_weight [R]
    float32 softmax probability, expert_off [E+1] int32, logits [T, E]).
    """
    logits = rng(seed).standard_normal((T, E), dtype=np.float32)
    lg = logits.astype(np.float64)
    p = np.exp(lg - lg.max(axis=1, keepdims=True))
    p /= p.sum(axis=1, keepdims=True)
    order = np.argsort(-lg, axis=1, kind="stable")[:, :topk]       # ties -> lower index
    rows, weights, off = [], [], [0]
    for e in range(E):
        toks = np.nonzero((order == e).any(axis=1))[0]
        rows.append(toks)
        weights.append(p[toks, e])
        off.append(off[-1] + len(toks))
    return dict(route_rows=np.concatenate(rows).astype(np.int32),
                route_weight=np.concatenate(weights).astype(np.float32),
                expert_off=np.array(off, dtype=np.int32),
                logits=logits)
