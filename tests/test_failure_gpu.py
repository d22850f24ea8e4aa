"""Failure path on the GPU without a fault: a bounded device wait that nothing
satisfies gives up, the timeout is reported through the device error word,
and the context keeps computing correct results afterwards."""

import numpy as np
import pytest
import torch

from numerics_packed_int4_gb300 import inputs, qgemm as Q
from oracle import formats as OF
from oracle import gemm as OG
from oracle import quant as OQ
from tests.gpu_util import check_gemm, dev, empty, host

pytestmark = pytest.mark.gpu


def _small_gemv(qg):
    N, K = 256, 512
    w = inputs.weights_f32(N, K, seed=21)
    q, s = OQ.quant_int4_rtn(w, 128)
    x = inputs.activations_bf16(1, K, seed=22)
    y = empty((1, N), torch.int16)
    qg.qgemm_w4a16(dev(q), dev(s), 128, dev(x), y, 1, N, K)
    qg.qg_check_device_error()
    ref = OF.bf16_decode(OG.to_bf16(OG.gemm_bf16_f64(x, OG.dequant_int4(q, s, 128), None)))
    check_gemm(OF.bf16_decode(host(y)), ref, "after timeout")


def test_wait_timeout_is_reported_and_cleared(qg):
    qg.qg_check_device_error()                     # start from a clean error word
    qg.qg_selftest_wait_timeout(2000)
    with pytest.raises(Q.QgemmError) as ei:
        qg.qg_check_device_error()
    assert ei.value.status == 5                    # QG_ERR_TIMEOUT
    qg.qg_check_device_error()                     # reading it cleared it
    _small_gemv(qg)                                # and the context still computes


def test_repeated_timeouts(qg):
    for _ in range(3):
        qg.qg_selftest_wait_timeout(500)
        with pytest.raises(Q.QgemmError):
            qg.qg_check_device_error()
    _small_gemv(qg)


@pytest.mark.parametrize("polls", [0, (1 << 20) + 1])
def test_selftest_rejects_bad_poll_counts(qg, polls):
    with pytest.raises(Q.QgemmError) as ei:
        qg.qg_selftest_wait_timeout(polls)
    assert ei.value.status == 1                    # QG_ERR_INVALID_ARG
