"""GB300 (sm_103a) mixed-precision quantized-weight GEMM/GEMV library.

The compute lives in ``libqgemm.so`` (CUDA, built from ``csrc/``) behind the
C ABI declared in ``include/qgemm.h``.  ``qgemm`` is the thin ctypes binding
(argument marshalling only); ``inputs`` draws the seeded synthetic workloads.
Importing this package has no side effects: the library is loaded on first
use and a missing or unloadable library raises, never falls back.
"""
