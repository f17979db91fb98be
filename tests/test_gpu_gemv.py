"""Decode GEMV (M <= 8) parity against the oracle: every output element
within |Y - Y_ref| <= 8e-3*S + 1e-3 (BF16) or 2e-3*S + 1e-4 (FP16), with
S = sum_k |A * B_dq|; plus the invariants the pages name (one-hot lane
ownership probe, K-permutation, row independence)."""

import numpy as np
import pytest
import torch

import fp8_weight_only_nvfp4_gb300 as wq
import oracle
import workloads as wl
from gpu_util import (act_to_dev, assert_within_tolerance, bits_of, f64_of, fp4_dev, run_fp4,
                      DEV)

pytestmark = pytest.mark.gpu


def _ref(p):
    return oracle.fp4_matmul(p.A, p.B_packed, p.weight_scale, p.weight_scale_2, p.bias, p.M, p.N,
                             p.K, p.block_size, p.dtype)


def test_parity_small_config():
    """NVFP4 M=1, N=256, K=512, bs=16, FP16, bias (the small parity workload)."""
    p = wl.parity_small()
    Y = run_fp4(p)
    Yr, S = _ref(p)
    assert_within_tolerance(Y, Yr, S, p.dtype, "parity_small")


@pytest.mark.parametrize("M", [1, 2, 3, 4, 5, 8])
def test_decode_gemv_5120(M):
    p = wl.decode_gemv(M=M)
    Y = run_fp4(p)
    Yr, S = _ref(p)
    assert_within_tolerance(Y, Yr, S, p.dtype, f"decode M={M}")


@pytest.mark.parametrize("M", [4, 5])
def test_repeated_runs_bit_identical(M):
    """The K split across a CTA cluster adds its partial sums in a fixed
    order, so repeated runs (fresh device buffers each time, which changes
    the timing of the shared-memory ring) must agree to the bit and stay
    within tolerance.  Catches a stage of the ring being refilled while its
    operands are still being read."""
    p = wl.decode_gemv(M=M)
    Yr, S = _ref(p)
    first = None
    for _ in range(10):
        Y = run_fp4(p)
        b = bits_of(Y)
        if first is None:
            first = b
            assert_within_tolerance(Y, Yr, S, p.dtype, f"repeat M={M}")
        else:
            assert np.array_equal(b, first), f"{int((b != first).sum())} elements changed"


@pytest.mark.parametrize("dtype", [oracle.BF16, oracle.FP16])
@pytest.mark.parametrize("M,N,K,bs", [
    (1, 17, 32, 16), (3, 33, 96, 32), (8, 100, 1000, 16), (5, 257, 128, 16), (2, 16, 40, 16),
    (7, 31, 4130, 16), (4, 64, 2, 16), (6, 48, 5136, 48), (1, 1, 16, 16), (8, 129, 1056, 32),
])
def test_shapes(M, N, K, bs, dtype):
    p = wl.make_fp4(M, N, K, bs, dtype, seed=M + N + K, bias_sigma=0.1)
    Y = run_fp4(p)
    Yr, S = _ref(p)
    assert_within_tolerance(Y, Yr, S, dtype, f"M={M} N={N} K={K} bs={bs}")


def test_lm_head_full():
    """NVFP4 lm_head GEMV, M=4, N=152064, K=5120, every output."""
    p = wl.lm_head()
    Y = run_fp4(p)
    Yr, S = _ref(p)
    assert_within_tolerance(Y, Yr, S, p.dtype, "lm_head")


def test_fp16_error_level():
    """FP16 activations: max relative error of order 1e-4
    (FP4 page §4 reports 2.4e-4 .. 3.5e-4 against an fp64 reference)."""
    p = wl.make_fp4(4, 2048, 4096, 16, oracle.FP16, seed=3)
    Y = run_fp4(p)
    Yr, S = _ref(p)
    rel = np.abs(f64_of(Y) - Yr) / np.maximum(np.abs(Yr), 1e-3 * S)
    assert np.max(rel) < 2e-3
    assert np.median(rel) < 5e-4


def test_one_hot_probe():
    """A = e_k in row m: Y[m, n] = B_dq[n, k] for every (m, n, k), bit-exact
    (weight_scale_2 = 1 and no bias, so every folded weight is exact in FP16):
    pins which lane supplies which weight column, activation row and k-slot."""
    M, N, K, bs = 8, 48, 256, 16
    p = wl.make_fp4(M, N, K, bs, oracle.FP16, seed=5, ws2=1.0)
    d = fp4_dev(p)
    W = oracle.fp4_dequantize_f64(p.B_packed, p.weight_scale, 1.0, N, K, bs)
    for k in range(K):
        A = np.zeros((M, K))
        for m in range(M):
            A[m, (k + 37 * m) % K] = 1.0
        d["A"] = act_to_dev(wl.act_bits(A, p.dtype), p.dtype)
        Y = f64_of(run_fp4(p, d))
        for m in range(M):
            assert np.array_equal(Y[m], W[:, (k + 37 * m) % K]), (k, m)


def test_rows_independent_of_M():
    """Each row's result is bit-identical whether it is computed alone or with
    the other rows of an M = 8 batch (FP4 page §4: per-row order is fixed)."""
    p8 = wl.make_fp4(8, 640, 2048, 16, oracle.BF16, seed=9, bias_sigma=0.1)
    d = fp4_dev(p8)
    Y8 = bits_of(run_fp4(p8, d))
    for m in range(8):
        d1 = dict(d)
        d1["A"] = d["A"][m:m + 1].contiguous()
        p1 = wl.Fp4Problem(1, p8.N, p8.K, 16, p8.dtype, p8.A[m:m + 1], p8.B_packed,
                           p8.weight_scale, p8.weight_scale_2, p8.bias)
        Y1 = bits_of(run_fp4(p1, d1))
        assert np.array_equal(Y1[0], Y8[m])


def test_k_permutation_within_tolerance():
    """Permuting whole scale blocks of K on A, B and the scales gives a result
    within tolerance of the unpermuted oracle (K is a reduction axis)."""
    M, N, K, bs = 4, 96, 1024, 16
    p = wl.make_fp4(M, N, K, bs, oracle.BF16, seed=13)
    perm = np.random.Generator(np.random.PCG64(1)).permutation(K // bs)
    kperm = (perm[:, None] * bs + np.arange(bs)[None, :]).ravel()
    q = wl.Fp4Problem(M, N, K, bs, p.dtype, p.A[:, kperm],
                      p.B_packed[:, (kperm[0::2] // 2)], p.weight_scale[:, perm],
                      p.weight_scale_2, None)
    Yr, S = _ref(p)
    assert_within_tolerance(run_fp4(q), Yr, S, p.dtype, "permuted")


def test_k_zero_writes_bias():
    p = wl.make_fp4(3, 40, 0, 16, oracle.BF16, seed=1, bias_sigma=1.0)
    d = fp4_dev(p)
    Y = run_fp4(p, d)
    assert np.array_equal(bits_of(Y), np.tile(p.bias, (3, 1)))


def test_no_bias_and_out_argument():
    p = wl.make_fp4(2, 64, 256, 16, oracle.BF16, seed=4)
    d = fp4_dev(p)
    out = torch.full((2, 64), float("nan"), dtype=torch.bfloat16, device=DEV)
    wq.fp4_weight_matmul(d["A"], d["B"], d["ws"], d["ws2"], None, out=out)
    torch.cuda.synchronize()
    Yr, S = _ref(p)
    assert_within_tolerance(out, Yr, S, p.dtype, "out=")


def test_leading_dims():
    p = wl.make_fp4(6, 32, 64, 16, oracle.BF16, seed=2)
    d = fp4_dev(p)
    A3 = d["A"].view(2, 3, 64)
    Y = wq.fp4_weight_matmul(A3, d["B"], d["ws"], d["ws2"])
    torch.cuda.synchronize()
    assert Y.shape == (2, 3, 32)
    Yr, S = _ref(p)
    assert_within_tolerance(Y.view(6, 32), Yr, S, p.dtype, "3-D A")


def _with_activation(p, A):
    return wl.Fp4Problem(p.M, p.N, p.K, p.block_size, p.dtype, wl.act_bits(A, p.dtype),
                         p.B_packed, p.weight_scale, p.weight_scale_2, p.bias)


def test_bf16_activation_dynamic_range_fallback():
    """BF16 activations with extreme dynamic range inside one 256-k step
    (1e30 next to 1e-10), a step entirely below 2^-111 and an all-zero row
    stay within tolerance: every folded weight is exact in BF16 and the
    products accumulate in FP32, so no activation range is special."""
    M, N, K = 4, 256, 2048
    p = wl.make_fp4(M, N, K, 16, oracle.BF16, seed=31, bias_sigma=0.1)
    r = np.random.Generator(np.random.PCG64(5))
    A = r.standard_normal((M, K))
    A[1, 300] = 1e30      # step 1 of row 1: huge and ...
    A[1, 301] = 1e-10     # ... tiny in the same 256-k step
    A[2, 1024:1280] *= 1e-35  # step 4 of row 2: everything below 2^-111
    A[3, :] = 0.0             # an all-zero row
    q = _with_activation(p, A)
    Yr, S = _ref(q)
    assert_within_tolerance(run_fp4(q), Yr, S, q.dtype, "dynamic range")


def test_bf16_activation_wide_but_exact_range():
    """Activations spread over 2^-30 .. 2^2 (32 binades) inside one step stay
    within tolerance."""
    M, N, K = 2, 128, 512
    p = wl.make_fp4(M, N, K, 16, oracle.BF16, seed=32)
    r = np.random.Generator(np.random.PCG64(6))
    A = r.standard_normal((M, K)) * np.exp2(r.integers(-30, 2, size=(M, K)))
    q = _with_activation(p, A)
    Yr, S = _ref(q)
    assert_within_tolerance(run_fp4(q), Yr, S, q.dtype, "wide exact range")


# --- 8 < M <= 32: the TMA decode GEMV with up to four 8-row activation tiles ---

@pytest.mark.parametrize("dtype", [oracle.BF16, oracle.FP16])
@pytest.mark.parametrize("M", [9, 12, 16, 17, 24, 31, 32])
def test_mid_m_decode_gemv(M, dtype):
    p = wl.make_fp4(M, 320, 1024, 16, dtype, seed=100 + M, bias_sigma=0.1)
    Y = run_fp4(p)
    Yr, S = _ref(p)
    assert_within_tolerance(Y, Yr, S, dtype, f"mid M={M}")


def test_mid_m_5120():
    """M=16, N=K=5120 (split-K across a cluster), every output."""
    p = wl.make_fp4(16, 5120, 5120, 16, oracle.BF16, seed=77)
    Y = run_fp4(p)
    Yr, S = _ref(p)
    assert_within_tolerance(Y, Yr, S, p.dtype, "M=16 N=K=5120")


def test_one_hot_probe_mid_m():
    """One-hot activations for M=24 (three activation tiles): Y[m, n] =
    B_dq[n, k] bit-exact, pinning which lane and tile supply each row."""
    M, N, K, bs = 24, 48, 256, 16
    p = wl.make_fp4(M, N, K, bs, oracle.FP16, seed=6, ws2=1.0)
    d = fp4_dev(p)
    W = oracle.fp4_dequantize_f64(p.B_packed, p.weight_scale, 1.0, N, K, bs)
    for k in range(0, K, 5):
        A = np.zeros((M, K))
        for m in range(M):
            A[m, (k + 37 * m) % K] = 1.0
        d["A"] = act_to_dev(wl.act_bits(A, p.dtype), p.dtype)
        Y = f64_of(run_fp4(p, d))
        for m in range(M):
            assert np.array_equal(Y[m], W[:, (k + 37 * m) % K]), (k, m)


def test_rows_independent_mid_m():
    """Each row of an M=32 batch is bit-identical to the same row computed
    alone (each activation tile accumulates in its own registers)."""
    p32 = wl.make_fp4(32, 384, 2048, 16, oracle.BF16, seed=19, bias_sigma=0.1)
    d = fp4_dev(p32)
    Y32 = bits_of(run_fp4(p32, d))
    for m in (0, 7, 8, 15, 16, 23, 24, 31):
        d1 = dict(d)
        d1["A"] = d["A"][m:m + 1].contiguous()
        p1 = wl.Fp4Problem(1, p32.N, p32.K, 16, p32.dtype, p32.A[m:m + 1], p32.B_packed,
                           p32.weight_scale, p32.weight_scale_2, p32.bias)
        Y1 = bits_of(run_fp4(p1, d1))
        assert np.array_equal(Y1[0], Y32[m]), m
