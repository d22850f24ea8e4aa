"""Benchmark of the quantized-weight GEMM/GEMV hot path on GB300.

One step = one pass over every row of the hot path at its workload size:
  decode sweep   W x A16 GEMV, M in {1, 4, 16} x (N,K) in {4096^2, 14336x4096,
                 4096x14336} x {INT4-g128, FP8-channel, MXFP4, NVFP4}
  prefill        W4A16 GEMM, M = 8192, same three (N, K), INT4 g128
  quantizers     4096 x 7168 bf16 -> FP8 E4M3 per 1x128, MXFP4 (E8M0 per 16)
  MoE            W4A8 layer, T = 4096, hidden 4096, inter 14336, E = 8, top-2
                 (E4M3 activations handed to the GEMMs as exact fp16 copies)
  MoE, FP8 scales  the same layer on the FP8-group-scale recipe (E4M3 x E4M3
                 tensor-core GEMMs; roofline against the FP8 dense peak)
  MoE, E4M3 entry  the same layer through qgemm_w4a8_grouped (E4M3 activations
                 handed over as codes, converted to fp16 inside the GEMM, exact
                 bf16 group scales; fp16 tensor cores, roofline against bf16)
  zero points    asymmetric INT4 (zero point per group of 64): M = 1 GEMVs and
                 M = 8192 prefill over the same three (N, K)
  W8A8 GEMV      FP8 weights, activations quantized per 1 x 128 block inside the
                 GEMV prologue: M = 1 over the same three (N, K)
  prefill, other weights  M = 8192 over the same three (N, K) with FP8
                 per-channel, MXFP4 and NVFP4 weights
  W4A4           MXFP4 activations (quantized in the step) x MXFP4 weights on
                 the block-scaled FP4 tensor cores, M = 8192 over the three (N, K)
Each row is one CUDA graph (the MoE rows five, so that their grouped GEMMs --
the step's dominant kernel -- are timed on their own); CUDA events between
the graphs time every row inside the timed region.  Measured beside the step,
outside the timed region: the M = 1 row's single-launch read ceiling (a plain
streaming read of the same 12 weight matrices, one launch each), the dense
FP8 rate of this GPU (the FP8 rows' roofline denominator; three times it, the
nominal FP4/FP8 ratio, for the FP4 row), the library's block-scaled FP4 GEMM
(a comparator for the W4A4 row), a bf16 dense GEMM (cuBLAS) on the prefill's
own data, the 1 x 1024 x 1024 GEMV as latency, the
pinned host link, and the oracle on the host cores.  The first output line
holds every row in full; the last is the contract line.  The headline value is the metric's first quantity:
effective HBM GB/s of the M = 1 GEMVs (algorithmic bytes / time); the
M = 8192 TFLOP/s is reported beside it.  Inputs are seeded synthetic data
(weights N(0, 0.02), activations N(0, 1)), resident in HBM before timing; the
step's working set is far larger than L2, and every weight matrix is read
once per step.

--impl reference times the CPU oracle on a bounded sample of the same
workload (there is no other implementation to run).
"""

import argparse
import json
import os
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "M=1 effective HBM GB/s (% of peak); M=8192 TFLOP/s (% of bf16 dense peak)"
SHAPES = [(4096, 4096), (14336, 4096), (4096, 14336)]
FORMATS = ["int4", "fp8", "mxfp4", "nvfp4"]
ZP_G = 64                                   # group size of the zero-point rows
BYTES_PER_PARAM = {"int4": 0.5 + 2 / 128, "fp8": 1.0, "mxfp4": 0.5 + 1 / 32, "nvfp4": 0.5 + 1 / 16}


# DRAM traffic (dram__bytes_read.sum + dram__bytes_write.sum) of one launch
# of each row's main kernel, from one ncu capture, with the launch it was taken
# on and that launch's algorithmic bytes.  The summaries and the commands are
# under profiles/.  An entry goes back to None whenever its kernel changes.
PROFILED_TRAFFIC = {
    "decode_m1": {"bytes": 30.32e6, "launch": "gemv_kernel<0, 1, 1> INT4 M=1 N=14336 K=4096",
                  "algorithmic_bytes": 30.30e6, "profile": "profiles/gemv_int4_m1_n14336_k4096.md"},
    "prefill": {"bytes": 309.86e6, "launch": "w4a16_tc_kernel<0> M=8192 N=14336 K=4096",
                "algorithmic_bytes": 332.3e6, "profile": "profiles/prefill_w4a16_tc_m8192_n14336_k4096.md"},
    "moe": {"bytes": 985.5e6, "launch": "moe_f16_kernel<false> gate/up R=8192 N=28672 K=4096",
            "algorithmic_bytes": 1021.4e6, "profile": "profiles/moe_w4a8_f16act_t4096_e8.md"},
    "moe_fp8s": {"bytes": 940.19e6, "launch": "moe_fp8s_kernel gate/up R=8192 N=28672 K=4096",
                 "algorithmic_bytes": 981.4e6, "profile": "profiles/moe_fp8s_t4096_e8.md"},
    "moe_e4m3": {"bytes": 949.82e6, "launch": "moe_f16_kernel<true> gate/up R=8192 N=28672 K=4096",
                 "algorithmic_bytes": 987.8e6, "profile": "profiles/moe_w4a8_e4m3_f16conv_t4096_e8.md"},
    "prefill_w4a4": {"bytes": 246.08e6, "launch": "w4a4_bs_kernel<true, false> M=8192 N=14336 K=4096",
                     "algorithmic_bytes": 283.9e6, "profile": "profiles/w4a4_bs_m8192.md"},
}


# the main kernel of rows timed in parts
MAIN_KERNEL = {"moe": "moe_f16_kernel<false> (gate/up + down launches)",
               "moe_fp8s": "moe_fp8s_kernel (gate/up + down launches)",
               "moe_e4m3": "moe_f16_kernel<true> (gate/up + down launches)"}
MOE_ROWS = ("moe", "moe_fp8s", "moe_e4m3")
FP8_ROWS = ("moe_fp8s",)                     # FP8 tensor-core contractions: roofline against the FP8 peak
FP4_ROWS = ("prefill_w4a4",)                  # block-scaled FP4 contractions: 3 x the FP8 peak (nominal 13.5 / 4.5)


def gemv_bytes(fmt, M, N, K):
    """Algorithmic bytes: weights + scales, activations in, outputs out."""
    b = N * K * BYTES_PER_PARAM[fmt] + 2 * M * K + 2 * M * N
    if fmt == "fp8":
        b += 4 * N
    if fmt == "nvfp4":
        b += 4
    return b


def traffic_of(row):
    t = PROFILED_TRAFFIC.get(row)
    return None if t is None else t["bytes"]


def traffic_info(row):
    t = PROFILED_TRAFFIC.get(row)
    if t is None:
        return {}
    return {"traffic_launch": t["launch"], "traffic_algorithmic_bytes": t["algorithmic_bytes"],
            "traffic_profile": t["profile"]}


def load_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        pk = dict(hbm=float(p["hbm_gbs"]), bf16=float(p["bf16_tflops"]),
                  bf16_sus=float(p.get("bf16_tflops_sustained", p["bf16_tflops"])), src="measured")
    except Exception:
        pk = dict(hbm=6800.0, bf16=1900.0, bf16_sus=1700.0, src="fallback")
    # dense FP8: the measured bf16 peak x the nominal fp8/bf16 ratio (4.5 / 2.25)
    pk["fp8"] = 2.0 * pk["bf16"]
    return pk


# ----------------------------------------------------------------------------
# distributed plumbing (replicas only: the path has no exchange step)
# ----------------------------------------------------------------------------

def dist_env():
    return int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1)), \
        int(os.environ.get("LOCAL_RANK", 0))


def dist_init(world, backend):
    import torch.distributed as dist
    if world > 1 and not dist.is_initialized():
        dist.init_process_group(backend=backend)


def dist_barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def dist_max(v, world, device="cpu"):
    """Max of a float over ranks (timing: the slowest replica sets the time)."""
    if world == 1:
        return float(v)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(v)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate(per_rank_units, elapsed_s_max):
    """Whole-job throughput: units processed by all ranks / slowest rank's time."""
    return float(per_rank_units) / float(elapsed_s_max)


# ----------------------------------------------------------------------------
# clocks during the timed region
# ----------------------------------------------------------------------------

class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "20"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            threading.Thread(target=self._read, daemon=True).start()
        except Exception:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.perf_counter(), line.strip()))

    def wait_ready(self, timeout=3.0):
        """Block until the sampler has produced its first line (it takes a
        moment to start), so that samples cover the timed region."""
        t0 = time.perf_counter()
        while self.proc is not None and not self.lines and time.perf_counter() - t0 < timeout:
            time.sleep(0.01)

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self, t0=None, t1=None):
        """Median SM clock and the throttle reasons seen between t0 and t1
        (perf_counter seconds; the timed region), all samples if not given."""
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        lines = [ln for t, ln in self.lines if t0 is None or (t0 <= t <= t1 + 0.025)]
        for ln in lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 8:
                continue
            try:
                sm.append(float(f[0]))
                mx = float(f[1])
            except ValueError:
                continue
            for n, v in zip(names, f[4:8]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": float(np.median(sm)), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


# ----------------------------------------------------------------------------
# the workload on the device
# ----------------------------------------------------------------------------

class Workload:
    def __init__(self, torch, qg, dev, rows):
        self.t, self.qg, self.dev = torch, qg, dev
        self.rows = rows
        self.launches = {}          # segment -> kernel launches per replay
        self.bytes = {}             # segment -> algorithmic bytes per replay
        self.flops = {}
        self.detail = {}
        self._build()

    def _randn(self, shape, seed, std=1.0):
        g = self.t.Generator(device=self.dev)
        g.manual_seed(seed)
        return self.t.randn(shape, generator=g, device=self.dev, dtype=self.t.float32) * std

    def _bf16(self, x):
        return x.to(self.t.bfloat16).view(self.t.int16).contiguous()

    def _weights(self, fmt, w):
        t, qg = self.t, self.qg
        N, K = w.shape
        if fmt == "int4":
            q = t.empty((N, K // 2), dtype=t.uint8, device=self.dev)
            s = t.empty((N, K // 128), dtype=t.int16, device=self.dev)
            qg.qg_quantize_weights_int4(w, q, s, 128, N, K)
            return dict(q=q, s=s)
        if fmt == "fp8":
            q = t.empty((N, K), dtype=t.uint8, device=self.dev)
            s = t.empty((N,), dtype=t.float32, device=self.dev)
            qg.qg_quantize_weights_fp8(w, q, s, N, K)
            return dict(q=q, s=s)
        if fmt == "mxfp4":
            q = t.empty((N, K // 2), dtype=t.uint8, device=self.dev)
            s = t.empty((N, K // 32), dtype=t.uint8, device=self.dev)
            qg.qg_quantize_weights_mxfp4(w, q, s, 32, N, K)
            return dict(q=q, s=s)
        q = t.empty((N, K // 2), dtype=t.uint8, device=self.dev)
        s = t.empty((N, K // 16), dtype=t.uint8, device=self.dev)
        gs = t.empty((1,), dtype=t.float32, device=self.dev)
        qg.qg_quantize_weights_nvfp4(w, q, s, gs, N, K)
        return dict(q=q, s=s, gs=gs)

    def _weights_zp(self, w):
        t = self.t
        N, K = w.shape
        d = dict(q=t.empty((N, K // 2), dtype=t.uint8, device=self.dev),
                 s=t.empty((N, K // ZP_G), dtype=t.int16, device=self.dev),
                 z=t.empty((N, K // ZP_G), dtype=t.uint8, device=self.dev))
        self.qg.qg_quantize_weights_int4_zp(w, d["q"], d["s"], d["z"], ZP_G, N, K)
        return d

    def gemv(self, fmt, W, x, y, M, N, K):
        qg = self.qg
        if fmt == "int4":
            qg.qgemm_w4a16(W["q"], W["s"], 128, x, y, M, N, K)
        elif fmt == "fp8":
            qg.qgemm_w8a16(W["q"], W["s"], x, y, M, N, K)
        elif fmt == "mxfp4":
            qg.qgemm_fp4a16(W["q"], W["s"], qg.QG_SCALE_E8M0, 32, None, x, y, M, N, K)
        else:
            qg.qgemm_fp4a16(W["q"], W["s"], qg.QG_SCALE_E4M3, 16, W["gs"], x, y, M, N, K)

    def _build(self):
        t = self.t
        from numerics_packed_int4_gb300 import inputs
        self.W = {}
        prefill_rows = [r for r in self.rows if r.startswith("prefill")]
        if any(r.startswith("decode") for r in self.rows) or prefill_rows:
            for i, (N, K) in enumerate(SHAPES):
                w = self._randn((N, K), seed=1000 + i, std=0.02)
                for fmt in FORMATS:
                    if (fmt != "int4" and not any(r.startswith("decode") for r in self.rows)
                            and "prefill_" + fmt not in self.rows
                            and not (fmt == "mxfp4" and "prefill_w4a4" in self.rows)):
                        continue
                    self.W[(fmt, N, K)] = self._weights(fmt, w)
                if "decode_zp" in self.rows or "prefill_zp" in self.rows:
                    self.W[("int4zp", N, K)] = self._weights_zp(w)
                del w
        self.X, self.Y = {}, {}
        for M in (1, 4, 16):
            for K in sorted({k for _, k in SHAPES}):
                self.X[(M, K)] = self._bf16(self._randn((M, K), seed=2000 + M * 7 + K))
            for N in sorted({n for n, _ in SHAPES}):
                self.Y[(M, N)] = t.empty((M, N), dtype=t.int16, device=self.dev)
        if prefill_rows:
            self.XP = {}
            for K in sorted({k for _, k in SHAPES}):
                x = self._randn((8192, K), seed=3000 + K)
                g = np.random.Generator(np.random.PCG64(3001 + K))
                ch = t.from_numpy(g.permutation(K)[: K // 100]).to(self.dev)
                x[:, ch] *= 50.0                               # 1 % outlier channels x50
                self.XP[K] = self._bf16(x)
            self.YP = {N: t.empty((8192, N), dtype=t.int16, device=self.dev) for N, _ in SHAPES}
        if "prefill_w4a4" in self.rows:                     # MXFP4 activation codes, scales, bf16 expansion
            ks = sorted({k for _, k in SHAPES})
            self.A4 = {K: t.empty((8192, K // 2), dtype=t.uint8, device=self.dev) for K in ks}
            self.A4s = {K: t.empty((8192, K // 32), dtype=t.uint8, device=self.dev) for K in ks}
            self.A4w = {K: t.empty((8192, K), dtype=t.int16, device=self.dev) for K in ks}
        if "quant" in self.rows:
            xq = inputs.quantizer_activations_bf16(4096, 7168, seed=0)
            self.XQ = t.from_numpy(xq.view(np.int16)).to(self.dev)
            self.QF = t.empty((4096, 7168), dtype=t.uint8, device=self.dev)
            self.QFs = t.empty((4096, 56), dtype=t.float32, device=self.dev)
            self.QM = t.empty((4096, 3584), dtype=t.uint8, device=self.dev)
            self.QMs = t.empty((4096, 448), dtype=t.uint8, device=self.dev)
        if any(r in self.rows for r in MOE_ROWS):
            self._build_moe(inputs)

    def _build_moe(self, inputs):
        t, dev = self.t, self.dev
        T, E, H, I, topk = 4096, 8, 4096, 14336, 2
        rt = inputs.moe_routing(T, E, topk, seed=9)
        R = int(rt["expert_off"][-1])
        self.moe = dict(T=T, E=E, H=H, I=I, topk=topk, R=R)
        row_of = np.full((T, topk), -1, np.int32)
        wt = np.zeros((T, topk), np.float32)
        fill = np.zeros(T, np.int64)
        for r, tok in enumerate(rt["route_rows"]):
            row_of[tok, fill[tok]] = r
            wt[tok, fill[tok]] = rt["route_weight"][r]
            fill[tok] += 1
        m = self.moe
        m["off"] = t.from_numpy(rt["expert_off"]).to(dev)
        m["rows"] = t.from_numpy(rt["route_rows"]).to(dev)
        m["row_of"] = t.from_numpy(row_of).to(dev)
        m["wt"] = t.from_numpy(wt).to(dev)
        m["x"] = self._bf16(self._randn((T, H), seed=4000))
        w1q = t.empty((E, 2 * I, H // 2), dtype=t.uint8, device=dev)
        w1s = t.empty((E, 2 * I, H // 128), dtype=t.int16, device=dev)
        w2q = t.empty((E, H, I // 2), dtype=t.uint8, device=dev)
        w2s = t.empty((E, H, I // 128), dtype=t.int16, device=dev)
        for e in range(E):
            w = self._randn((2 * I, H), seed=5000 + e, std=0.02)
            self.qg.qg_quantize_weights_int4(w, w1q[e], w1s[e], 128, 2 * I, H)
            w = self._randn((H, I), seed=6000 + e, std=0.02)
            self.qg.qg_quantize_weights_int4(w, w2q[e], w2s[e], 128, H, I)
            del w
        m.update(w1q=w1q, w1s=w1s, w2q=w2q, w2s=w2s)
        m["w1e"] = t.empty((E * 2 * I,), dtype=t.int8, device=dev)    # load-time row shifts
        m["w2e"] = t.empty((E * H,), dtype=t.int8, device=dev)
        self.qg.qg_w4a8_row_shifts(w1s, m["w1e"], E * 2 * I, H // 128)
        self.qg.qg_w4a8_row_shifts(w2s, m["w2e"], E * H, I // 128)
        if "moe_fp8s" in self.rows:                       # load-time scale preparation
            m["w1s8"] = t.empty((H // 128, E * 2 * I), dtype=t.uint8, device=dev)      # group-major
            m["w1cs8"] = t.empty((E, 2 * I), dtype=t.float32, device=dev)
            m["w2s8"] = t.empty((I // 128, E * H), dtype=t.uint8, device=dev)
            m["w2cs8"] = t.empty((E, H), dtype=t.float32, device=dev)
            self.qg.qg_w4a8_fp8_scales(w1s, m["w1s8"], m["w1cs8"], E * 2 * I, H // 128)
            self.qg.qg_w4a8_fp8_scales(w2s, m["w2s8"], m["w2cs8"], E * H, I // 128)
        m["xq"] = t.empty((T, H), dtype=t.uint8, device=dev)
        m["xs"] = t.empty((T,), dtype=t.float32, device=dev)
        m["aq"] = t.empty((R, H), dtype=t.uint8, device=dev)
        m["aq16"] = t.empty((R, H), dtype=t.int16, device=dev)      # fp16 copy of the E4M3 codes
        m["hq16"] = t.empty((R, I), dtype=t.int16, device=dev)
        m["as"] = t.empty((R,), dtype=t.float32, device=dev)
        m["gu"] = t.empty((R, 2 * I), dtype=t.int16, device=dev)
        m["hq"] = t.empty((R, I), dtype=t.uint8, device=dev)
        m["hs"] = t.empty((R,), dtype=t.float32, device=dev)
        m["down"] = t.empty((R, H), dtype=t.int16, device=dev)
        m["out"] = t.empty((T, H), dtype=t.int16, device=dev)

    # ---- segments -----------------------------------------------------------
    def run_segment(self, name):
        qg = self.qg
        if name.startswith("decode_m"):
            M = int(name[len("decode_m"):])
            for fmt in FORMATS:
                for N, K in SHAPES:
                    self.gemv(fmt, self.W[(fmt, N, K)], self.X[(M, K)], self.Y[(M, N)], M, N, K)
        elif name == "prefill":
            for N, K in SHAPES:
                W = self.W[("int4", N, K)]
                qg.qgemm_w4a16(W["q"], W["s"], 128, self.XP[K], self.YP[N], 8192, N, K)
        elif name == "prefill_w4a4":
            for N, K in SHAPES:                             # MXFP4 activations x MXFP4 weights
                qg.quant_act_mxfp4(self.XP[K], self.A4[K], self.A4s[K], 32, 8192, K)
                qg.qgemm_w4a4_mxfp4(self.W[("mxfp4", N, K)]["q"], self.W[("mxfp4", N, K)]["s"], self.A4[K],
                                    self.A4s[K], self.A4w[K], self.YP[N], 8192, N, K)
        elif name.startswith("prefill_") and name[len("prefill_"):] in FORMATS:
            fmt = name[len("prefill_"):]                    # FP8 / MXFP4 / NVFP4 weights, same kernel
            for N, K in SHAPES:
                self.gemv(fmt, self.W[(fmt, N, K)], self.XP[K], self.YP[N], 8192, N, K)
        elif name == "decode_w8a8":
            for N, K in SHAPES:
                W = self.W[("fp8", N, K)]
                qg.qgemm_w8a8(W["q"], W["s"], self.X[(1, K)], self.Y[(1, N)], 1, N, K)
        elif name == "decode_zp":
            for N, K in SHAPES:
                W = self.W[("int4zp", N, K)]
                qg.qgemm_w4a16_zp(W["q"], W["s"], W["z"], ZP_G, self.X[(1, K)], self.Y[(1, N)], 1, N, K)
        elif name == "prefill_zp":
            for N, K in SHAPES:
                W = self.W[("int4zp", N, K)]
                qg.qgemm_w4a16_zp(W["q"], W["s"], W["z"], ZP_G, self.XP[K], self.YP[N], 8192, N, K)
        elif name == "quant":
            qg.quant_act_fp8_block(self.XQ, self.QF, self.QFs, 128, 4096, 7168)
            qg.quant_act_mxfp4(self.XQ, self.QM, self.QMs, 16, 4096, 7168)
        elif name in MOE_ROWS:
            for _, fn, _ in self.parts(name):
                fn()

    # The MoE layer in its five launches groups; the two grouped GEMMs are the
    # layer's main kernel, timed on their own inside the step.
    def parts(self, name):
        qg = self.qg
        if name not in MOE_ROWS:
            return [(name, lambda: self.run_segment(name), False)]
        m = self.moe
        T, E, H, I, R, topk = m["T"], m["E"], m["H"], m["I"], m["R"], m["topk"]
        if name == "moe":
            def pre():
                qg.quant_act_fp8_block(m["x"], m["xq"], m["xs"], H, T, H)
                qg.qg_moe_gather_fp8_f16(m["xq"], m["xs"], m["rows"], m["aq16"], m["as"], R, T, H)

            def gemm1():
                qg.qgemm_w4a8_grouped_f16act(m["aq16"], m["as"], m["off"], m["w1q"], m["w1s"], m["w1e"], 128,
                                             m["gu"], R, E, 2 * I, H)

            def mid():
                qg.qg_swiglu_quant_fp8_f16(m["gu"], m["hq16"], m["hs"], R, I)

            def gemm2():
                qg.qgemm_w4a8_grouped_f16act(m["hq16"], m["hs"], m["off"], m["w2q"], m["w2s"], m["w2e"], 128,
                                             m["down"], R, E, H, I)
        elif name == "moe_e4m3":            # the E4M3-input entry with exact bf16 group scales
            def pre():
                qg.quant_act_fp8_block(m["x"], m["xq"], m["xs"], H, T, H)
                qg.qg_moe_gather_fp8(m["xq"], m["xs"], m["rows"], m["aq"], m["as"], R, T, H)

            def gemm1():
                qg.qgemm_w4a8_grouped(m["aq"], m["as"], m["off"], m["w1q"], m["w1s"], 128, m["gu"], R, E, 2 * I, H)

            def mid():
                qg.qg_swiglu_quant_fp8(m["gu"], m["hq"], m["hs"], R, I)

            def gemm2():
                qg.qgemm_w4a8_grouped(m["hq"], m["hs"], m["off"], m["w2q"], m["w2s"], 128, m["down"], R, E, H, I)
        else:
            def pre():
                qg.quant_act_fp8_block(m["x"], m["xq"], m["xs"], H, T, H)
                qg.qg_moe_gather_fp8(m["xq"], m["xs"], m["rows"], m["aq"], m["as"], R, T, H)

            def gemm1():
                qg.qgemm_w4a8_grouped_fp8s(m["aq"], m["as"], m["off"], m["w1q"], m["w1s8"], m["w1cs8"], m["gu"],
                                           R, E, 2 * I, H)

            def mid():
                qg.qg_swiglu_quant_fp8(m["gu"], m["hq"], m["hs"], R, I)

            def gemm2():
                qg.qgemm_w4a8_grouped_fp8s(m["hq"], m["hs"], m["off"], m["w2q"], m["w2s8"], m["w2cs8"], m["down"],
                                           R, E, H, I)

        def post():
            qg.qg_moe_combine(m["down"], m["row_of"], m["wt"], m["out"], T, topk, R, H)

        return [("pre", pre, False), ("gemm1", gemm1, True), ("mid", mid, False), ("gemm2", gemm2, True),
                ("post", post, False)]

    def accounting(self):
        for M in (1, 4, 16):
            name = "decode_m%d" % M
            if name in self.rows:
                self.bytes[name] = sum(gemv_bytes(f, M, N, K) for f in FORMATS for N, K in SHAPES)
                self.launches[name] = None
        if "prefill" in self.rows:
            self.flops["prefill"] = sum(2.0 * 8192 * N * K for N, K in SHAPES)
        for r in ("prefill_zp", "prefill_fp8", "prefill_mxfp4", "prefill_nvfp4", "prefill_w4a4"):
            if r in self.rows:
                self.flops[r] = sum(2.0 * 8192 * N * K for N, K in SHAPES)
        if "decode_w8a8" in self.rows:
            self.bytes["decode_w8a8"] = sum(N * K + 4 * N + 2 * K + 2 * N for N, K in SHAPES)
            self.launches["decode_w8a8"] = None
        if "decode_zp" in self.rows:
            self.bytes["decode_zp"] = sum(N * K * (0.5 + 3.0 / ZP_G) + 2 * K + 2 * N for N, K in SHAPES)
            self.launches["decode_zp"] = None
        if "quant" in self.rows:
            M, K = 4096, 7168
            self.bytes["quant"] = M * K * (2 + 1) + M * K // 128 * 4 + M * K * 2 + M * K // 2 + M * K // 16
        for r in MOE_ROWS:
            if r in self.rows:
                m = self.moe
                self.flops[r] = 2.0 * m["R"] * (2 * m["I"] * m["H"] + m["H"] * m["I"])


def count_launches(torch, fn):
    """Kernel launches of one segment: count them with the profiler once."""
    from torch.profiler import ProfilerActivity, profile
    with profile(activities=[ProfilerActivity.CUDA]) as prof:
        fn()
        torch.cuda.synchronize()
    n = 0
    for ev in prof.events():
        if ev.device_type.name == "CUDA" and "memcpy" not in ev.name.lower() and "memset" not in ev.name.lower():
            n += 1
    return n


# ----------------------------------------------------------------------------
# CPU oracle timing (the reference arm and cpu_baseline)
# ----------------------------------------------------------------------------

def oracle_gemv_sample(seconds_budget=15.0, max_items=None):
    """Time the oracle on M=1 GEMVs of the decode workload (a bounded sample).

    Returns (GB/s in the metric's unit, seconds, description)."""
    from numerics_packed_int4_gb300 import inputs
    from oracle import gemm as OG
    from oracle import quant as OQ
    done_bytes, spent, items = 0.0, 0.0, []
    plan = [(f, N, K) for N, K in SHAPES for f in FORMATS]
    for i, (fmt, N, K) in enumerate(plan):
        if spent > seconds_budget or (max_items and i >= max_items):
            break
        w = inputs.weights_f32(N, K, seed=1000 + i)
        x = inputs.activations_bf16(1, K, seed=2000 + K)
        t0 = time.perf_counter()
        if fmt == "int4":
            q, s = OQ.quant_int4_rtn(w, 128)
            t0 = time.perf_counter()
            OG.to_bf16(OG.qgemm_w4a16(x, q, s, 128))
        elif fmt == "fp8":
            q, cs = OQ.quant_fp8_channel(w)
            t0 = time.perf_counter()
            OG.to_bf16(OG.qgemm_w8a16(x, q, cs))
        elif fmt == "mxfp4":
            q, se = OQ.quant_mxfp4_weights(w)
            t0 = time.perf_counter()
            OG.to_bf16(OG.qgemm_mxfp4a16(x, q, se))
        else:
            q, sb, gs = OQ.quant_nvfp4(w)
            t0 = time.perf_counter()
            OG.to_bf16(OG.qgemm_nvfp4a16(x, q, sb, gs))
        dt = time.perf_counter() - t0
        spent += dt
        done_bytes += gemv_bytes(fmt, 1, N, K)
        items.append("%s %dx%d" % (fmt, N, K))
    return done_bytes / spent / 1e9, spent, ", ".join(items)


def oracle_other_rows():
    """The oracle beside the other rows, on the host cores: both activation
    quantizers at full size (4096 x 7168), and 256-row samples of the M=8192
    prefill (INT4, 14336 x 4096) and of the MoE layer (256 rows of one expert:
    gate/up, SwiGLU + requant, down), the latter two reported as the rate of
    the sample (extrapolated linearly to the full row count).  Returns
    {row: {"value", "unit", "seconds", "sample"}}."""
    from numerics_packed_int4_gb300 import inputs
    from oracle import gemm as OG
    from oracle import quant as OQ
    out = {}
    M, K = 4096, 7168
    x = inputs.quantizer_activations_bf16(M, K, seed=0)
    t0 = time.perf_counter()
    OQ.quant_fp8_block(x, 128)
    t1 = time.perf_counter()
    OQ.quant_mxfp4(x, 16)
    t2 = time.perf_counter()
    fp8_bytes = M * K * 3 + M * K // 128 * 4
    mx_bytes = M * K * 2 + M * K // 2 + M * K // 16
    out["quant"] = {"value": (fp8_bytes + mx_bytes) / (t2 - t0) / 1e9, "unit": "GB/s", "seconds": t2 - t0,
                    "sample": "full size: FP8 1x128 %.1f s, MXFP4 g16 %.1f s" % (t1 - t0, t2 - t1)}
    N, K = 14336, 4096
    q, sc = OQ.quant_int4_rtn(inputs.weights_f32(N, K, seed=1001), 128)
    xa = inputs.activations_bf16(256, K, seed=3001, outlier_frac=0.01, outlier_scale=50.0)
    t0 = time.perf_counter()
    OG.to_bf16(OG.qgemm_w4a16(xa, q, sc, 128))
    dt = time.perf_counter() - t0
    out["prefill"] = {"value": 2.0 * 256 * N * K / dt / 1e12, "unit": "TFLOP/s", "seconds": dt,
                      "sample": "256 of 8192 rows, INT4 14336x4096 (dequant + fp64 product); "
                                "extrapolated linearly"}
    H, I = 4096, 14336
    w1 = OQ.quant_int4_rtn(inputs.weights_f32(2 * I, H, seed=5000), 128)
    w2 = OQ.quant_int4_rtn(inputs.weights_f32(H, I, seed=6000), 128)
    xm = inputs.activations_bf16(256, H, seed=4000)
    w1 = (w1[0][None], w1[1][None])
    w2 = (w2[0][None], w2[1][None])
    t0 = time.perf_counter()
    OG.moe_layer(xm, np.arange(256), np.array([0, 256], np.int32), w1, w2, 128, I)
    dt = time.perf_counter() - t0
    out["moe"] = {"value": 2.0 * 256 * (2 * I * H + H * I) / dt / 1e12, "unit": "TFLOP/s", "seconds": dt,
                  "sample": "256 of 8192 rows, one expert (gate/up, SwiGLU + FP8 requant, down); "
                            "extrapolated linearly"}
    return out


def cpu_cores():
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count() or 1


# ----------------------------------------------------------------------------
# arms
# ----------------------------------------------------------------------------

def bench_config(rows, world):
    """The workload of the bench line (shared by both arms)."""
    return {"workload": "decode sweep M in {1,4,16} x {4096^2, 14336x4096, 4096x14336} x "
                        "{INT4-g128, FP8-channel, MXFP4, NVFP4} + prefill M=8192 (W4A16; FP8, MXFP4, NVFP4 weights) + "
                        "act quantizers 4096x7168 + W4A8 MoE T=4096 E=8 top-2 (bf16 group scales on fp16 copies; "
                        "FP8 group scales; E4M3 entry) + asymmetric INT4 g64 M=1 and M=8192 + W8A8 GEMV M=1",
            "rows": rows, "l2": "inputs larger than L2: every weight matrix read once per step; "
                                "step working set > 1 GB vs 129 MB L2",
            "parallelism": "replicas" if world > 1 else "single"}


def run_reference(args):
    rank, world, _ = dist_env()
    if world > 1:
        dist_init(world, "gloo")
        if rank != 0:
            dist_barrier(world)
            return 0
    vals = []
    for _ in range(args.warmup):
        oracle_gemv_sample(max_items=1)
    t0 = time.perf_counter()
    desc = ""
    for _ in range(args.steps):
        v, _, desc = oracle_gemv_sample(max_items=1)
        vals.append(v)
    el = time.perf_counter() - t0
    value = float(np.mean(vals))
    line = {
        "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": args.gpus, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": 1e3 * el / max(args.steps, 1), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "impl": "reference",
        "config": bench_config(args.rows.split(","), world),
        "cpu_baseline": {"value": value, "unit": "GB/s", "cores": cpu_cores(), "kind": "oracle",
                         "sample": "each step one M=1 GEMV of the decode sweep through the oracle "
                                   "(dequantization + fp64 product): %s; value = its effective GB/s" % desc},
        "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    if world > 1:
        dist_barrier(world)
    return 0


def run_ours(args):
    import torch
    rank, world, local = dist_env()
    if world > 1:
        dist_init(world, "nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    from numerics_packed_int4_gb300 import qgemm as qg
    qg.load()
    peaks = load_peaks()

    rows = args.rows.split(",")
    wl = Workload(torch, qg, dev, rows)
    wl.accounting()
    torch.cuda.synchronize()

    # eager warm-up of every segment (sets kernel attributes), then capture graphs
    for r in rows:
        wl.run_segment(r)
    qg.qg_check_device_error()
    count_launches(torch, lambda: wl.run_segment(rows[0]))      # first profiler session warms CUPTI
    for r in rows:
        wl.launches[r] = count_launches(torch, lambda r=r: wl.run_segment(r))
    graphs = {}                                # row -> [(part, graph, is_main_kernel)]
    cap = torch.cuda.Stream(device=dev)
    for r in rows:
        graphs[r] = []
        for part, fn, main in wl.parts(r):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=cap):
                fn()
            graphs[r].append((part, g, main))
    torch.cuda.synchronize()

    stream = torch.cuda.current_stream(dev)
    for _ in range(args.warmup):
        for r in rows:
            for _, g, _ in graphs[r]:
                g.replay()
    qg.qg_check_device_error()

    ev = {r: [] for r in rows}
    dist_barrier(world)
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        clk.wait_ready()
        start = torch.cuda.Event(enable_timing=True)
        end = torch.cuda.Event(enable_timing=True)
        t_wall = time.perf_counter()
        t_region0 = t_wall
        start.record(stream)
        for _ in range(args.steps):
            for r in rows:
                marks = [torch.cuda.Event(enable_timing=True)]
                marks[0].record(stream)
                for _, g, _ in graphs[r]:
                    g.replay()
                    marks.append(torch.cuda.Event(enable_timing=True))
                    marks[-1].record(stream)
                ev[r].append(marks)
        end.record(stream)
        torch.cuda.synchronize()
        t_region1 = time.perf_counter()
        t_wall = t_region1 - t_wall
        time.sleep(0.03)                       # let the sampler deliver the region's last line
    dist_barrier(world)
    qg.qg_check_device_error()
    total_ms = dist_max(start.elapsed_time(end), world, dev)
    seg_ms = {r: sum(m[0].elapsed_time(m[-1]) for m in ev[r]) / args.steps for r in rows}
    seg_ms_max = {r: dist_max(seg_ms[r], world, dev) for r in rows}
    # the main kernel's own launches inside rows timed in parts (the MoE GEMMs)
    kern_ms = {}
    for r in rows:
        idx = [i for i, (_, _, main) in enumerate(graphs[r]) if main]
        if idx and len(graphs[r]) > 1:
            t = sum(sum(m[i].elapsed_time(m[i + 1]) for i in idx) for m in ev[r]) / args.steps
            kern_ms[r] = (dist_max(t, world, dev), len(idx))

    # ---- measurements beside the step (not part of it) --------------------------
    fp8_meas = measure_fp8_peak(torch, dev) if any(r in FP8_ROWS + FP4_ROWS for r in rows) else None
    if fp8_meas is not None:
        peaks["fp8"], peaks["fp8_src"] = fp8_meas, "measured in this run (torch._scaled_mm E4M3 8192^3, best of 10)"
    else:
        peaks["fp8_src"] = "measured bf16 x 2 (nominal fp8/bf16 ratio)"
    side = {}
    fp4_lib = measure_fp4_cublas(torch, dev) if any(r in FP4_ROWS for r in rows) else None
    if fp4_lib is not None:
        side["fp4_library"] = {"TFLOP/s": fp4_lib,
                               "what": "torch._scaled_mm E2M1 x E2M1, E4M3 scales per 16, 8192^3, best of 10"}
    if "prefill" in rows:
        side["prefill_vs_bf16"] = bf16_comparator(torch, qg, wl, dev)
    side["gemv_1x1024x1024"] = gemv_1k_latency(torch, qg, dev)

    # ---- per-row throughput and rooflines ----------------------------------------
    row_out = {}
    for r in rows:
        ms = seg_ms_max[r]
        if r in wl.bytes:
            gbs = wl.bytes[r] / (ms * 1e-3) / 1e9
            row_out[r] = {"ms": ms, "GB/s": gbs, "launches": wl.launches[r],
                          "roofline": {"bound": "hbm", "achieved": gbs, "peak": peaks["hbm"], "unit": "GB/s",
                                       "frac": gbs / peaks["hbm"],
                                       "traffic": traffic_of(r), **traffic_info(r)}}
        else:
            tf = wl.flops[r] / (ms * 1e-3) / 1e12
            fp8 = r in FP8_ROWS
            peak = 3.0 * peaks["fp8"] if r in FP4_ROWS else (peaks["fp8"] if fp8 else peaks["bf16"])
            row_out[r] = {"ms": ms, "TFLOP/s": tf, "launches": wl.launches[r],
                          "roofline": {"bound": "tensor", "achieved": tf, "peak": peak, "unit": "TFLOP/s",
                                       "frac": tf / peak, "traffic": traffic_of(r), **traffic_info(r)}}
            if fp8:
                row_out[r]["roofline"]["peak_kind"] = "fp8 dense: " + peaks["fp8_src"]
            if r in FP4_ROWS:
                row_out[r]["roofline"]["peak_kind"] = ("fp4 dense: 3 x the fp8 peak, the nominal 13.5 / 4.5 ratio ("
                                                       + peaks["fp8_src"] + ")")
                if fp4_lib is not None:
                    row_out[r]["vs_fp4_library"] = tf / fp4_lib
            if r in kern_ms:
                kms, nl = kern_ms[r]
                ktf = wl.flops[r] / (kms * 1e-3) / 1e12
                row_out[r]["kernel"] = {
                    "name": MAIN_KERNEL[r], "launches": nl, "ms": kms,
                    "roofline": {"bound": "tensor", "achieved": ktf, "peak": peak, "unit": "TFLOP/s",
                                 "frac": ktf / peak, "traffic": traffic_of(r), **traffic_info(r)}}
    dominant = max(rows, key=lambda r: kern_ms[r][0] if r in kern_ms else seg_ms_max[r])
    value = aggregate(world * wl.bytes.get("decode_m1", 0.0), seg_ms_max.get("decode_m1", 1.0) * 1e-3) / 1e9

    e2e = e2e_decode_m1(torch, qg, wl, dev, steps=max(2, min(args.steps, 5))) if "decode_m1" in rows else None
    if e2e is not None:
        e2e["host_link"] = h2d_link(torch, dev)
    if "decode_m1" in rows:
        rc = read_ceiling(torch, qg, wl, dev)
        rc["gemv_row_over_read_time"] = seg_ms_max["decode_m1"] / rc["ms"]
        row_out["decode_m1"]["single_launch_read"] = rc
    clocks = clk.summary(t_region0, t_region1)
    launches_per_step = sum((wl.launches[r] or 0) for r in rows)

    if rank != 0:
        return 0
    cpu = None
    if not args.no_cpu_baseline and world == 1:
        v, spent, desc = oracle_gemv_sample(seconds_budget=args.cpu_seconds)
        other = {} if args.cpu_seconds <= 0 else oracle_other_rows()
        cpu = {"value": v, "unit": "GB/s", "cores": cpu_cores(), "kind": "oracle",
               "sample": "M=1 GEMVs (oracle dequant + fp64 product), %d matrices, %.1f s; other rows below"
                         % (len(desc.split(", ")), spent),
               "rows": {k: {"value": o["value"], "unit": o["unit"], "s": round(o["seconds"], 1)}
                        for k, o in other.items()}}
        side["cpu_baseline_detail"] = {"decode_m1": desc, **{k: o["sample"] for k, o in other.items()}}

    # line 1: every row in full, the side measurements and the peaks used
    detail = {"detail": "per-row results of the step below", "rows": row_out, "side": side,
              "peaks": peaks, "wall_s": t_wall}
    print(json.dumps(detail), flush=True)

    # line 2: the contract line, kept short
    summary = {}
    for r, o in row_out.items():
        ach = o.get("GB/s", o.get("TFLOP/s"))
        summary[r] = [round(o["ms"], 4), round(ach, 1), round(o["roofline"]["frac"], 3)]
    line = {
        "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": total_ms / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded: weights N(0,0.02), activations N(0,1))",
        "config": bench_config(rows, world),
        "secondary": None,
        "roofline": (dict(row_out[dominant]["kernel"]["roofline"], kernel=row_out[dominant]["kernel"]["name"],
                          row=dominant) if "kernel" in row_out[dominant]
                     else dict(row_out[dominant]["roofline"], kernel=dominant)),
        "rows": {"columns": ["ms", "GB/s or TFLOP/s", "frac of measured peak"], **summary},
        "clocks": clocks, "gpu_launches": launches_per_step * args.steps, "e2e": e2e,
    }
    if "decode_m1" in row_out:
        rc = row_out["decode_m1"]["single_launch_read"]
        line["roofline_value"] = {"kernel": "decode_m1 (12 GEMVs)", "achieved": value, "peak": peaks["hbm"],
                                  "frac": value / peaks["hbm"], "single_launch_read_GB/s": rc["GB/s"],
                                  "frac_of_single_launch_read": value / rc["GB/s"]}
    if "prefill" in row_out:
        p = row_out["prefill"]
        line["secondary"] = {"metric": "M=8192 TFLOP/s", "value": p["TFLOP/s"], "unit": "TFLOP/s",
                             "frac_of_bf16_peak": p["TFLOP/s"] / peaks["bf16"],
                             "frac_of_bf16_sustained": p["TFLOP/s"] / peaks["bf16_sus"]}
        if "prefill_vs_bf16" in side:
            c = side["prefill_vs_bf16"]
            line["secondary"]["bf16_dense_same_data_TFLOP/s"] = c["bf16_TFLOP/s"]
            line["secondary"]["w4a16_over_bf16_speed"] = c["w4a16_over_bf16_speed"]
    g1 = side["gemv_1x1024x1024"]
    line["gemv_1x1024x1024"] = {"us": g1["graph_us_per_launch"], "GB/s": g1["graph_GB/s"],
                                "single_call_us": g1["single_call_us_median"]}
    line["peaks"] = {"hbm": peaks["hbm"], "bf16": peaks["bf16"], "fp8": peaks["fp8"], "src": peaks["src"]}
    if "fp4_library" in side:
        line["peaks"]["fp4_library"] = side["fp4_library"]["TFLOP/s"]
    if cpu is not None:
        line["cpu_baseline"] = cpu
    print(json.dumps(line), flush=True)
    return 0


def read_ceiling(torch, qg, wl, dev, reps=5):
    """A plain streaming read of each of the decode row's 12 packed weight
    matrices, one launch each, in the row's order and under the same L2
    conditions: what one launch of that many bytes reaches on this GPU.
    Measured outside the timed step (it is not part of the path)."""
    bufs = [wl.W[(f, N, K)]["q"] for f in FORMATS for N, K in SHAPES]
    nbytes = sum(b.numel() * b.element_size() for b in bufs)
    sink = torch.zeros(1, dtype=torch.int32, device=dev)

    def seg():
        for b in bufs:
            qg.qg_stream_read(b, b.numel() * b.element_size(), sink)

    seg()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=torch.cuda.Stream(device=dev)):
        seg()
    for _ in range(3):
        g.replay()
    ts = []
    stream = torch.cuda.current_stream(dev)
    for _ in range(reps):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        g.replay()
        b.record(stream)
        torch.cuda.synchronize()
        ts.append(a.elapsed_time(b))
    ms = sorted(ts)[len(ts) // 2]
    qg.qg_check_device_error()
    return {"what": "qg_stream_read of each decode weight matrix, one launch each", "bytes": nbytes,
            "launches": len(bufs), "ms": ms, "GB/s": nbytes / (ms * 1e-3) / 1e9}


def _time_graph(torch, dev, fn, reps=10, warm=3):
    """Capture fn in a CUDA graph and return (median, best) replay times in ms."""
    fn()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=torch.cuda.Stream(device=dev)):
        fn()
    for _ in range(warm):
        g.replay()
    stream = torch.cuda.current_stream(dev)
    ts = []
    for _ in range(reps):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        g.replay()
        b.record(stream)
        torch.cuda.synchronize()
        ts.append(a.elapsed_time(b))
    return sorted(ts)[len(ts) // 2], min(ts)


def measure_fp8_peak(torch, dev, n=8192, reps=10):
    """Dense E4M3 x E4M3 (fp32 accumulate, bf16 out) rate of this GPU through
    the vendor library (torch._scaled_mm, 8192^3, best of `reps`): the
    denominator of the FP8 tensor-core rows, measured in the same run.  A
    measurement of the library, not part of the path.  None if unavailable."""
    try:
        a = (torch.randn((n, n), device=dev) * 0.5).to(torch.float8_e4m3fn)
        b = (torch.randn((n, n), device=dev) * 0.5).to(torch.float8_e4m3fn).t()     # column-major
        one = torch.ones((), device=dev, dtype=torch.float32)
        out = torch.empty((n, n), device=dev, dtype=torch.bfloat16)

        def f():
            torch._scaled_mm(a, b, scale_a=one, scale_b=one, out_dtype=torch.bfloat16, out=out)

        _, best = _time_graph(torch, dev, f, reps=reps)
        del a, b, out
        return 2.0 * n ** 3 / (best * 1e-3) / 1e12
    except Exception:
        return None


def measure_fp4_cublas(torch, dev, n=8192, reps=10):
    """The vendor library's block-scaled FP4 GEMM on this GPU: torch._scaled_mm
    with E2M1 operands and E4M3 scales per 16 elements (the FP4 form this
    PyTorch exposes), 8192^3, best of `reps`.  Reported beside the W4A4 row as a
    comparator (the row's roofline uses the nominal FP4/FP8 ratio on the
    measured FP8 peak).  A measurement of the library, not part of the path.
    None if unavailable."""
    try:
        a = torch.randint(0, 256, (n, n // 2), dtype=torch.uint8, device=dev).view(torch.float4_e2m1fn_x2)
        b = torch.randint(0, 256, (n, n // 2), dtype=torch.uint8, device=dev).view(torch.float4_e2m1fn_x2)
        ns = ((n + 127) // 128 * 128) * ((n // 16 + 3) // 4 * 4)
        sa = torch.full((ns,), 0x38, dtype=torch.uint8, device=dev).view(torch.float8_e4m3fn)   # 1.0
        sb = torch.full((ns,), 0x38, dtype=torch.uint8, device=dev).view(torch.float8_e4m3fn)
        out = torch.empty((n, n), device=dev, dtype=torch.bfloat16)

        def f():
            torch._scaled_mm(a, b.t(), sa, sb, out_dtype=torch.bfloat16, out=out)

        _, best = _time_graph(torch, dev, f, reps=reps)
        del a, b, out
        return 2.0 * n ** 3 / (best * 1e-3) / 1e12
    except Exception:
        return None


def bf16_comparator(torch, qg, wl, dev, reps=10):
    """The prefill config's comparison: a bf16 dense GEMM (torch.matmul,
    cuBLAS) on the same data -- the same outlier activations times the
    canonical dequantized INT4 weights -- over the three (N, K), against the
    W4A16 prefill on the same inputs.  Reports both times, the ratio, and how
    far apart the two outputs are (relative Frobenius).  Outside the timed step."""
    Wd, out = {}, {}
    for N, K in SHAPES:
        W = wl.W[("int4", N, K)]
        wd = torch.empty((N, K), dtype=torch.int16, device=dev)
        qg.qg_dequant_weights(qg.QG_FMT_INT4, W["q"], W["s"], 128, wd, N, K)
        Wd[(N, K)] = wd.view(torch.bfloat16)
        out[N] = torch.empty((8192, N), dtype=torch.bfloat16, device=dev)
    qg.qg_check_device_error()

    def dense():
        for N, K in SHAPES:
            torch.matmul(wl.XP[K].view(torch.bfloat16), Wd[(N, K)].t(), out=out[N])

    def ours():
        for N, K in SHAPES:
            W = wl.W[("int4", N, K)]
            qg.qgemm_w4a16(W["q"], W["s"], 128, wl.XP[K], wl.YP[N], 8192, N, K)

    flops = sum(2.0 * 8192 * N * K for N, K in SHAPES)
    d_ms, d_best = _time_graph(torch, dev, dense, reps=reps)
    o_ms, o_best = _time_graph(torch, dev, ours, reps=reps)
    ours()
    torch.cuda.synchronize()
    diff = []
    for N, _ in SHAPES:
        y = wl.YP[N].view(torch.bfloat16).float()
        r = out[N].float()
        diff.append(float(torch.linalg.vector_norm(y - r) / torch.linalg.vector_norm(r)))
    qg.qg_check_device_error()
    return {"what": "torch.matmul bf16 (cuBLAS) on the dequantized INT4 weights and the same outlier "
                    "activations, M=8192 over the three (N,K)",
            "bf16_ms": d_ms, "bf16_TFLOP/s": flops / (d_ms * 1e-3) / 1e12,
            "w4a16_ms": o_ms, "w4a16_TFLOP/s": flops / (o_ms * 1e-3) / 1e12,
            "w4a16_over_bf16_speed": d_ms / o_ms, "rel_fro_vs_bf16": max(diff)}


def gemv_1k_latency(torch, qg, dev, copies=512, calls=200):
    """The 1 x 1024 x 1024 W4A16 GEMV (INT4 g128): launch-bound at 0.54 MB,
    so it is reported as latency plus effective GB/s.  (a) a CUDA graph of one
    GEMV per weight copy, `copies` copies (277 MB, more than L2) so every
    launch streams its weights from HBM: time per launch; (b) single calls
    through the C ABI from Python, each timed with events on the stream."""
    N = K = 1024
    g = torch.Generator(device=dev)
    g.manual_seed(7000)
    w = torch.randn((copies * N, K), generator=g, device=dev) * 0.02
    q = torch.empty((copies * N, K // 2), dtype=torch.uint8, device=dev)
    s = torch.empty((copies * N, K // 128), dtype=torch.int16, device=dev)
    qg.qg_quantize_weights_int4(w, q, s, 128, copies * N, K)
    del w
    x = torch.randn((1, K), generator=g, device=dev).to(torch.bfloat16).view(torch.int16)
    y = torch.empty((1, N), dtype=torch.int16, device=dev)
    torch.cuda.synchronize()
    nbytes = gemv_bytes("int4", 1, N, K)

    def sweep():
        for i in range(copies):
            qg.qgemm_w4a16(q[i * N:(i + 1) * N], s[i * N:(i + 1) * N], 128, x, y, 1, N, K)

    ms, _ = _time_graph(torch, dev, sweep, reps=5)
    per = ms / copies
    stream = torch.cuda.current_stream(dev)
    single = []
    for c in range(calls):
        i = (c * 97) % copies
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        qg.qgemm_w4a16(q[i * N:(i + 1) * N], s[i * N:(i + 1) * N], 128, x, y, 1, N, K)
        b.record(stream)
        torch.cuda.synchronize()
        single.append(a.elapsed_time(b))
    single.sort()
    qg.qg_check_device_error()
    return {"what": "W4A16 GEMV M=1 N=1024 K=1024 INT4 g128", "bytes": nbytes,
            "graph_us_per_launch": per * 1e3, "graph_GB/s": nbytes / (per * 1e-3) / 1e9,
            "single_call_us_median": single[len(single) // 2] * 1e3,
            "single_call_GB/s": nbytes / (single[len(single) // 2] * 1e-3) / 1e9,
            "weight_copies": copies}


def h2d_link(torch, dev, nbytes=1 << 30, reps=5):
    """One pinned host-to-device copy of 1 GiB (a single cudaMemcpyAsync),
    best of `reps`: the host link's rate, the ceiling of the end-to-end figure."""
    h = torch.empty((nbytes,), dtype=torch.uint8).pin_memory()
    d = torch.empty((nbytes,), dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    ts = []
    for _ in range(reps + 1):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        d.copy_(h, non_blocking=True)
        b.record(stream)
        torch.cuda.synchronize()
        ts.append(a.elapsed_time(b))
    best = min(ts[1:])
    del h, d
    return {"bytes": nbytes, "ms": best, "GB/s": nbytes / (best * 1e-3) / 1e9}


def e2e_decode_m1(torch, qg, wl, dev, steps):
    """M=1 GB/s through the C ABI with host buffers: every step copies each
    GEMV's weights, scales and activation from pinned host memory (on a side
    stream, overlapping the GEMVs), runs the 12 GEMVs and copies the outputs
    back.  The host link (~160-200 GB/s measured for pinned copies) bounds it."""
    host = {}
    h2d = 0
    for fmt in FORMATS:
        for N, K in SHAPES:
            W = wl.W[(fmt, N, K)]
            hw = {k: v.cpu().pin_memory() for k, v in W.items()}
            dw = {k: torch.empty_like(v) for k, v in W.items()}
            host[(fmt, N, K)] = (hw, dw)
            h2d += sum(v.numel() * v.element_size() for v in hw.values())
    hx = {K: wl.X[(1, K)].cpu().pin_memory() for _, K in SHAPES}
    h2d += len(FORMATS) * sum(hx[K].numel() * 2 for _, K in SHAPES)   # one activation copy per GEMV
    hy = {N: torch.empty((1, N), dtype=torch.int16).pin_memory() for N, _ in SHAPES}
    d2h = len(FORMATS) * sum(hy[N].numel() * 2 for N, _ in SHAPES)
    dx = {(fmt, K): torch.empty_like(wl.X[(1, K)]) for fmt in FORMATS for _, K in SHAPES}
    stream = torch.cuda.current_stream(dev)
    copy_stream = torch.cuda.Stream(dev)
    keys = [(fmt, N, K) for fmt in FORMATS for N, K in SHAPES]
    copied = {k: torch.cuda.Event() for k in keys}
    consumed = {k: torch.cuda.Event() for k in keys}
    started = torch.cuda.Event()

    def one(first):
        # host->device copies on a side stream, each GEMV waiting only for its
        # own inputs, so the copy of the next GEMV's weights overlaps this one
        started.record(stream)
        copy_stream.wait_event(started)
        for k in keys:
            fmt, N, K = k
            hw, dw = host[k]
            with torch.cuda.stream(copy_stream):
                if not first:
                    copy_stream.wait_event(consumed[k])   # the previous step's GEMV has read them
                for name in hw:
                    dw[name].copy_(hw[name], non_blocking=True)
                dx[(fmt, K)].copy_(hx[K], non_blocking=True)
                copied[k].record(copy_stream)
        for k in keys:
            fmt, N, K = k
            hw, dw = host[k]
            stream.wait_event(copied[k])
            wl.gemv(fmt, dw, dx[(fmt, K)], wl.Y[(1, N)], 1, N, K)
            consumed[k].record(stream)
            hy[N].copy_(wl.Y[(1, N)], non_blocking=True)

    one(True)
    torch.cuda.synchronize()
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for _ in range(steps):
        one(False)
    b.record(stream)
    torch.cuda.synchronize()
    ms = a.elapsed_time(b) / steps
    return {"value": wl.bytes["decode_m1"] / (ms * 1e-3) / 1e9, "unit": "GB/s",
            "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h), "ms_per_step": ms}


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--rows", default="decode_m1,decode_m4,decode_m16,prefill,quant,moe,moe_fp8s,moe_e4m3,"
                                      "decode_zp,prefill_zp,decode_w8a8,prefill_fp8,prefill_mxfp4,prefill_nvfp4,"
                                      "prefill_w4a4",
                    help="segments to time")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    args = ap.parse_args(argv)
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
