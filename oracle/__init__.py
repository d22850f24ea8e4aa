"""Plain CPU oracle for the quantized-weight GEMM/GEMV path.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path may import, call or
execute anything in this package: only ``tests/``, ``__graft_entry__.smoke()``
and the ``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` use it.
It shares no code, constants or helpers with the CUDA library, and it does not
import the ``numerics_packed_int4_gb300`` package.

Every function is written to be checked by eye against the pages it cites:

* "Numerics: FP32 to INT4, and why bf16 won" (mlinterviewnotes.com, section
  0.5) -- float layouts, max-finite values, fp32 accumulation, scale policy,
  granularity, the MXFP4 block-scaled family, the FP8 activation path.
* vLLM PR #43557 "Fix the E8M0 scale computation in the MXFP4 (W4A4) MOE
  CUTLASS kernel" -- the exponent-first 0.75-threshold E8M0 rule.
* FreeToken PR #805 (fp32 -> e4m3 cast on sm_89) -- round-once RNE satfinite.
* "Your 3090 Isn't Missing Anything for FP8/NVFP4 Weight-Only Inference" --
  dequantize to bf16 in registers, bf16 MMA, fp32 accumulate.
* "Production-Ready W4A8: vLLM Integration and Quality Recovery Techniques
  Explained" (Cohere) -- INT4 weights x FP8 activations, per-token x group
  scales.

Precision rules: floating-point steps that the method performs in fp32 are
done in numpy float32 (IEEE, correctly rounded, no flush-to-zero); every
rounding to a narrow format is done from the exact value by an explicit
round-to-nearest-even onto that format's grid; matrix products are fp64.

Parity status per function is stated in each module header.  Functions whose
only pins are invariants (no page value fixes them) say "parity unpinned".
"""

from . import formats, quant, gemm  # noqa: F401
