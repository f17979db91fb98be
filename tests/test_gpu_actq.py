"""NVFP4 activation quantization (FP4 page §6, step 1 of the native FP4 x FP4
path) on the GPU against the oracle: packed codes, E4M3 scales and the
quantize-dequantize output bit for bit, and the activation-and-weight FP4
matmul (quantize-dequantize, then the weight-only matmul) against an FP4 x
FP4 reference built from the oracle's codes and scales."""

import numpy as np
import pytest
import torch

import fp8_weight_only_nvfp4_gb300 as wq
import oracle
import workloads as wl
from gpu_util import DEV, act_to_dev, assert_within_tolerance, bits_of, fp4_dev

pytestmark = pytest.mark.gpu


def _quantize(A_bits, dtype):
    A = act_to_dev(A_bits, dtype)
    pc, sc = wq.fp4_quantize_activation(A)
    q = wq.fp4_quantize_dequantize_activation(A)
    torch.cuda.synchronize()
    return pc.cpu().numpy(), sc.cpu().numpy(), bits_of(q)


@pytest.mark.parametrize("dtype", [oracle.BF16, oracle.FP16])
@pytest.mark.parametrize("M,K", [(1, 16), (3, 40), (7, 1000), (16, 5120), (5, 36), (2, 2)])
@pytest.mark.parametrize("sigma", [1.0, 1e-2, 1e3])
def test_quantize_bit_exact(M, K, sigma, dtype):
    """Random activations: 1e-2 reaches subnormal E4M3 scales, 1e3 (BF16)
    saturates scales at 448; K = 40 / 1000 end in a partial block, K = 36
    gives rows that are not 16-byte aligned (element-wise path)."""
    if dtype == oracle.FP16 and sigma == 1e3:
        sigma = 3e3  # still finite in FP16, amax / 6 above 448
    r = np.random.Generator(np.random.PCG64(M * 1000 + K))
    A = wl.act_bits(r.normal(0, sigma, (M, K)), dtype)
    pc, sc, q = _quantize(A, dtype)
    opc, osc = oracle.nvfp4_quantize_activation(A, dtype)
    assert np.array_equal(sc, osc), f"{int((sc != osc).sum())} scales differ"
    assert np.array_equal(pc, opc), f"{int((pc != opc).sum())} code bytes differ"
    oq = oracle.nvfp4_qdq_activation(A, dtype)
    assert np.array_equal(q, oq), f"{int((q != oq).sum())} values differ"


@pytest.mark.parametrize("dtype", [oracle.BF16, oracle.FP16])
def test_golden_blocks(dtype):
    """The hand-computed blocks of tests/golden/nvfp4_activation.txt (every
    E2M1 tie, signed zeros, a scale that underflows to zero)."""
    import test_oracle_pins as pins
    for name, c in pins._nvfp4_golden_cases().items():
        A = wl.act_bits(np.array([c["x"]]), dtype)
        pc, sc, q = _quantize(A, dtype)
        assert sc.tolist() == [[c["scale"]]], name
        assert pc.tolist() == [c["packed"]], name
        assert np.array_equal(q, wl.act_bits(np.array([c["qdq"]]), dtype)), name


def test_prefill_activation_full():
    """The 8K-token prefill activation (M = 8192, K = 5120, BF16), every code,
    scale and value."""
    A = wl.gen_activation(8192, 5120, oracle.BF16, 3)
    pc, sc, q = _quantize(A, oracle.BF16)
    opc, osc = oracle.nvfp4_quantize_activation(A, oracle.BF16)
    assert np.array_equal(sc, osc) and np.array_equal(pc, opc)
    assert np.array_equal(q, oracle.nvfp4_qdq_activation(A, oracle.BF16))


def test_leading_dims_and_out_arguments():
    A = act_to_dev(wl.gen_activation(6, 64, oracle.BF16, 9), oracle.BF16).view(2, 3, 64)
    pc, sc = wq.fp4_quantize_activation(A)
    assert pc.shape == (2, 3, 32) and sc.shape == (2, 3, 4)
    out = torch.empty_like(A)
    q = wq.fp4_quantize_dequantize_activation(A, out=out)
    torch.cuda.synchronize()
    assert q.data_ptr() == out.data_ptr()
    opc, osc = oracle.nvfp4_quantize_activation(wl.gen_activation(6, 64, oracle.BF16, 9),
                                                oracle.BF16)
    assert np.array_equal(pc.cpu().numpy().reshape(6, 32), opc)
    assert np.array_equal(sc.cpu().numpy().reshape(6, 4), osc)


def _fp4x4_reference(A, p):
    """FP4 x FP4 product in float64 from the oracle's activation codes and
    scales: sum_k e2m1(qa) e4m3(sa) * B_dq + bias, and the magnitude sum."""
    codes, scales = oracle.nvfp4_quantize_activation(A, p.dtype)
    table = np.array([oracle.e2m1_value(c) for c in range(16)])
    e4 = np.array([oracle.e4m3_value(b) for b in range(256)])
    M, K = A.shape
    qa = np.empty((M, K), dtype=np.int64)
    qa[:, 0::2] = codes & 0xF
    qa[:, 1::2] = codes >> 4
    Ad = table[qa] * np.repeat(e4[scales], 16, axis=1)[:, :K]
    W = oracle.fp4_dequantize_f64(p.B_packed, p.weight_scale, p.weight_scale_2, p.N, p.K,
                                  p.block_size)
    Y = Ad @ W.T
    if p.bias is not None:
        Y = Y + np.array([oracle.act_to_double(int(b), p.dtype) for b in p.bias])
    return Y, np.abs(Ad) @ np.abs(W).T


@pytest.mark.parametrize("M", [4, 64, 300])
def test_w4a4_two_call_matmul(M):
    """fp4_weight_matmul of the quantize-dequantize output (decode GEMV for
    M = 4, tcgen05 GEMM for M = 64 / 300) within the matmul bound of the
    FP4 x FP4 reference."""
    N, K = 640, 2048
    p = wl.make_fp4(M, N, K, 16, oracle.BF16, seed=M, bias_sigma=0.02)
    d = fp4_dev(p)
    d["A"] = wq.fp4_quantize_dequantize_activation(d["A"])
    Y = wq.fp4_weight_matmul(d["A"], d["B"], d["ws"], d["ws2"], d["bias"], block_size=16)
    torch.cuda.synchronize()
    assert wq.device_status() == 0
    Yr, S = _fp4x4_reference(p.A, p)
    assert_within_tolerance(Y, Yr, S, p.dtype, f"W4A4 M={M}")
    # The two references agree: the oracle's weight-only matmul of its own
    # quantize-dequantize output is the same FP4 x FP4 sum.
    Yo, So = oracle.fp4_matmul(oracle.nvfp4_qdq_activation(p.A, p.dtype), p.B_packed,
                               p.weight_scale, p.weight_scale_2, p.bias, M, N, K, 16, p.dtype)
    assert np.allclose(Yo, Yr, rtol=0, atol=1e-9 * (1 + So.max()))
