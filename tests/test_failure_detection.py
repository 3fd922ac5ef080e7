"""Failure detection on the GPU without a fault: a pipeline wait that nothing completes gives
up after its time limit, the kernel records BSFP8_ERR_DEVICE_TIMEOUT in the device error word
and returns, and the context stays usable (a GEMM right after it is correct).  Invalid
expert offsets and ids are covered in the parity test files."""
import time

import numpy as np
import pytest

import gen
import oracle
from helpers import parity_report

pytestmark = pytest.mark.gpu


def test_bounded_wait_reports_timeout_and_context_survives():
    import torch
    import block_scaled_fp8_persistent_gb300 as bsfp8
    assert bsfp8.bsfp8_get_device_error() == 0
    t0 = time.perf_counter()
    bsfp8.bsfp8_check_wait_timeout(20_000_000)  # 20 ms
    assert bsfp8.bsfp8_get_device_error() == 7   # BSFP8_ERR_DEVICE_TIMEOUT
    assert time.perf_counter() - t0 >= 0.015     # it did wait out the limit
    assert bsfp8.bsfp8_get_device_error() == 0   # read clears
    from gpu_util import DeviceProblem
    p = gen.blockwise_problem([70, 0, 58], 256, 512, seed=50)
    d = DeviceProblem(p)
    d.run()
    got = d.c_bits()
    assert bsfp8.bsfp8_get_device_error() == 0
    ref, T = oracle.problem_reference(p)
    bad, ratio, _ = parity_report(got, ref, T)
    assert bad == 0
    torch.cuda.synchronize()
