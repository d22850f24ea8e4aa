"""The allocation-free W4A4 entry point against the ordinary one.

qgemm_w4a4_mxfp4_noalloc serves callers that cannot allocate device memory
(an op behind a plugin interface that receives only its input and output
buffers, or a runtime whose memory is all committed to its own pool): instead
of a caller-supplied work buffer it expands the activations into a fixed array
compiled into the library.  Its output must match qgemm_w4a4_mxfp4 with a
freshly allocated work buffer, on two calls in a row -- the second call
reuses the array the first one left filled, with different sizes and data.

This file is named so that pytest collects it last; it also passes alone in a
fresh process (the first call there performs the array's one-time address
lookup).
"""

import numpy as np
import pytest
import torch

from numerics_packed_int4_gb300 import inputs
from numerics_packed_int4_gb300.qgemm import QgemmError
from oracle import formats as OF
from oracle import quant as OQ
from tests.gpu_util import check_gemm, dev, empty, host

pytestmark = pytest.mark.gpu


def _case(qg, M, N, K, seed):
    x = inputs.activations_bf16(M, K, seed=seed, outlier_frac=0.01, outlier_scale=50.0)
    wq, wse = OQ.quant_mxfp4_weights(inputs.weights_f32(N, K, seed=seed + 1))
    aq = empty((M, K // 2), torch.uint8)
    ase = empty((M, K // 32), torch.uint8)
    qg.quant_act_mxfp4(dev(x), aq, ase, 32, M, K)
    return dev(wq), dev(wse), aq, ase


def _both(qg, M, N, K, seed):
    dwq, dwse, aq, ase = _case(qg, M, N, K, seed)
    work = empty((M, K), torch.int16)
    y_ref = empty((M, N), torch.int16)
    qg.qgemm_w4a4_mxfp4(dwq, dwse, aq, ase, work, y_ref, M, N, K)
    y = torch.full((M, N), -1, dtype=torch.int16, device="cuda")
    qg.qgemm_w4a4_mxfp4_noalloc(dwq, dwse, aq, ase, y, M, N, K)
    qg.qg_check_device_error()
    return OF.bf16_decode(host(y)), OF.bf16_decode(host(y_ref))


def test_noalloc_matches_the_work_buffer_entry_on_two_calls():
    from numerics_packed_int4_gb300 import qgemm as qg
    qg.load()
    # call 1: the tensor-core path (M > 16), several tiles and a ragged edge
    y1, r1 = _both(qg, 300, 264, 1024, seed=5)
    check_gemm(y1, r1, "noalloc call 1 (M=300)")
    # call 2: the decode path on a smaller problem, the array still holding call 1's data
    y2, r2 = _both(qg, 7, 512, 2048, seed=9)
    check_gemm(y2, r2, "noalloc call 2 (M=7)")


def test_noalloc_rejects_sizes_beyond_its_array():
    from numerics_packed_int4_gb300 import qgemm as qg
    qg.load()
    M, N, K = 4097, 128, 2048                      # M*K just above 8388608 elements
    t = empty((16,), torch.uint8)
    with pytest.raises(QgemmError) as e:
        qg.qgemm_w4a4_mxfp4_noalloc(t, t, t, t, t, M, N, K)
    assert e.value.status == 2 and "static work area" in str(e.value)
