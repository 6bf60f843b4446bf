"""Failure detection on the GPU without a fault: a bounded wait that runs out.

qz_selftest_bounded_wait launches one CTA that waits on an mbarrier nothing ever
completes, with the bounded wait every GEMM kernel uses but a short poll limit.
The wait must give up, record QZ_ERR_TIMEOUT in the device error word and let the
kernel return: the host then reads QZ_ERR_TIMEOUT once (the read clears it), and
the context stays usable for ordinary work afterwards.
"""
import numpy as np
import pytest
import torch

import oracle
import synthetic as syn
from gpu_util import assert_same_bytes, dev_bf16, host

pytestmark = pytest.mark.gpu

QZ_OK, QZ_ERR_INVALID_ARG, QZ_ERR_TIMEOUT = 0, 1, 6


@pytest.fixture(scope="module")
def qz():
    import bit_quantized_linear_quantizers_gb300 as q
    return q


def test_bounded_wait_runs_out_and_context_survives(qz):
    assert qz.qz_device_error() == QZ_OK                  # nothing pending before
    for polls in (1, 1000):
        qz.qz_selftest_bounded_wait(polls)
        torch.cuda.synchronize()                          # the kernel returned by itself
        assert qz.qz_device_error() == QZ_ERR_TIMEOUT
        assert qz.qz_device_error() == QZ_OK              # the read cleared the word
    # the context still runs ordinary work correctly
    a = syn.to_bf16_bits(np.random.default_rng(5).standard_normal((32, 256)).astype(np.float32))
    c, s, _ = qz.qz_quantize_fp8(dev_bf16(a), qz.FP8_GROUP_1x128)
    rc, rs, _ = oracle.quant_fp8(a, oracle.FP8_GROUP_1x128, want_deq=False)
    assert_same_bytes(host(c), rc, "codes after the timeout")
    assert_same_bytes(host(s), rs, "scales after the timeout")
    assert qz.qz_device_error() == QZ_OK


def test_bounded_wait_rejects_out_of_range_limits(qz):
    for polls in (0, (1 << 20) + 1):
        assert qz.lib.qz_selftest_bounded_wait(polls, None) == QZ_ERR_INVALID_ARG
