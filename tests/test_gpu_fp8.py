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


def _with_scales(p, b_scale):
    return wl.Fp8Problem(p.M, p.N, p.K, p.block_size, p.dtype, p.A, p.B,
                         np.ascontiguousarray(b_scale, dtype=np.float32), p.bias)


@pytest.mark.parametrize("dtype", [oracle.FP16, oracle.BF16])
@pytest.mark.parametrize("M,bs", [(4, 16), (4, 64), (4, 128), (24, 128), (64, 16), (64, 128),
                                  (200, 64)])
@pytest.mark.parametrize("lo,hi,a_sigma", [(150.0, 250.0, 1e-3), (1e-7, 1e-6, 1.0)],
                         ids=["b_scale_150_250", "b_scale_1e-7_1e-6"])
def test_fp8_block_scale_range(M, bs, dtype, lo, hi, a_sigma):
    """FP32 block scales far outside the configs' U[0.001, 0.02] ("MatMulBlock
    QuantizedFp8Weight - CUDA Operator Documentation" §2: b_scale is FP32).
    With FP16 activations 448 * b_scale overflows a 16-bit operand above
    b_scale ~ 146 and tiny products become FP16 subnormals: every path (decode
    GEMV, tcgen05 GEMM, both block-size regimes) must stay within the bound."""
    p = wl.make_fp8(M, 96, 1024, bs, dtype, seed=M + bs, scale_lo=lo, scale_hi=hi,
                    bias_sigma=0.01, a_sigma=a_sigma)
    Yr, S = _ref(p)
    assert np.isfinite(Yr).all()
    assert_within_tolerance(run_fp8(p), Yr, S, dtype, f"fp8 b_scale [{lo}, {hi}] M={M} bs={bs}")


@pytest.mark.parametrize("dtype", [oracle.FP16, oracle.BF16])
@pytest.mark.parametrize("M", [4, 64])
def test_fp8_block_scales_spanning_six_decades_in_a_row(M, dtype):
    """Log-uniform block scales over [1e-3, 1e3] inside every weight row: the
    GEMM's per-row power-of-two normalisation keeps the largest block of a row
    in range while the smallest lose only what the bound allows."""
    p = wl.make_fp8(M, 128, 2048, 128, dtype, seed=7 + M, bias_sigma=0.01, a_sigma=1e-3)
    r = np.random.Generator(np.random.PCG64(11))
    b = np.exp(r.uniform(np.log(1e-3), np.log(1e3), size=p.b_scale.shape))
    q = _with_scales(p, b)
    Yr, S = _ref(q)
    assert_within_tolerance(run_fp8(q), Yr, S, dtype, f"fp8 six decades M={M}")
