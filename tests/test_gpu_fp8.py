"""FP8 E4M3 weight-only matmul parity (secondary format)."""

import numpy as np
import pytest

import oracle
import workloads as wl
from gpu_util import assert_within_tolerance, run_fp8

pytestmark = pytest.mark.gpu


def _ref(p):
    return oracle.fp8_matmul(p.A, p.B, p.b_scale, p.bias, p.M, p.N, p.K, p.block_size, p.dtype)


@pytest.mark.parametrize("M", [1, 4, 8])
def test_fp8_gemv_5120(M):
    p = wl.fp8_problem(M)
    assert_within_tolerance(run_fp8(p), *_ref(p), p.dtype, f"fp8 M={M}")


@pytest.mark.parametrize("M", [1, 4, 8, 24])
def test_fp8_tail_k5000(M):
    """K = 5000, bs = 128: S = 40, the last block is 8 wide and uses column 39."""
    p = wl.fp8_problem(M, N=5120, K=5000, bias_sigma=0.02)
    assert_within_tolerance(run_fp8(p), *_ref(p), p.dtype, f"fp8 tail M={M}")


@pytest.mark.parametrize("dtype", [oracle.BF16, oracle.FP16])
@pytest.mark.parametrize("M,N,K,bs", [(3, 40, 1000, 128), (8, 17, 48, 16), (2, 64, 4096, 64),
                                      (5, 33, 130, 32),
                                      # block scale applied per 128-k window after the MMAs:
                                      # partial last window, and blocks spanning two windows
                                      (4, 96, 4064, 128), (7, 130, 1056, 128), (6, 72, 2048, 256),
                                      (1, 64, 8192, 512)])
def test_fp8_shapes(M, N, K, bs, dtype):
    p = wl.make_fp8(M, N, K, bs, dtype, seed=K, bias_sigma=0.1)
    assert_within_tolerance(run_fp8(p), *_ref(p), dtype, f"fp8 {M}x{N}x{K}")
