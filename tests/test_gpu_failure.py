"""Failure detection on the GPU without a fault: every device-side wait in
the library is bounded; one that runs out records WQMM_ERR_TIMEOUT in the
device error word (read and cleared by wqmm_device_status) and the kernel
returns.  Here a diagnostic kernel waits on a barrier that nothing completes,
through the same bounded-wait helper the kernels use."""

import time

import numpy as np
import pytest

import fp8_weight_only_nvfp4_gb300 as wq
import oracle
import workloads as wl
from gpu_util import assert_within_tolerance, run_fp4

pytestmark = pytest.mark.gpu

WQMM_ERR_TIMEOUT = 5


def test_bounded_wait_reports_timeout_and_context_survives():
    L = wq.lib()
    assert wq.device_status() == 0
    t0 = time.monotonic()
    assert L.wqmm_selftest_wait_timeout(None) == 0
    assert wq.device_status() == WQMM_ERR_TIMEOUT
    waited = time.monotonic() - t0
    assert 1.5 < waited < 60, waited           # the limit is 2 s of device time
    assert wq.device_status() == 0             # cleared by the read
    # The context is intact: the next calls run and are correct.
    p = wl.parity_small()
    Yr, S = oracle.fp4_matmul(p.A, p.B_packed, p.weight_scale, p.weight_scale_2, p.bias, p.M,
                              p.N, p.K, p.block_size, p.dtype)
    assert_within_tolerance(run_fp4(p), Yr, S, p.dtype, "after a timeout")
    q = wl.make_fp4(64, 256, 512, 16, oracle.BF16, seed=2, bias_sigma=0.05)
    Yq, Sq = oracle.fp4_matmul(q.A, q.B_packed, q.weight_scale, q.weight_scale_2, q.bias, q.M,
                               q.N, q.K, q.block_size, q.dtype)
    assert_within_tolerance(run_fp4(q), Yq, Sq, q.dtype, "GEMM after a timeout")
    assert wq.device_status() == 0
