"""W8A8 activation path of the FP8 operator ("MatMulBlockQuantizedFp8Weight -
CUDA Operator Documentation" §6): A_deq = fp8_e4m3(A / a_scale) * a_scale.

The quantize-dequantize decides a code per element, so it is compared bit for
bit with the oracle; the matmul that consumes A_deq is held to the usual
accuracy bound against the oracle's FP8 matmul of the oracle's A_deq."""

import numpy as np
import pytest
import torch

import fp8_weight_only_nvfp4_gb300 as wq
import oracle
import workloads as wl
from gpu_util import DEV, act_to_dev, assert_within_tolerance, bits_of, fp8_dev

pytestmark = pytest.mark.gpu

DTYPES = [oracle.BF16, oracle.FP16]


def _scale_dev(a_scale):
    return torch.tensor([a_scale], dtype=torch.float32, device=DEV)


def _qdq_gpu(bits, a_scale, dtype):
    out = wq.fp8_quantize_dequantize_activation(act_to_dev(bits, dtype), _scale_dev(a_scale))
    torch.cuda.synchronize()
    assert wq.device_status() == 0
    return bits_of(out).reshape(bits.shape)


def _e4m3_midpoints():
    """Every midpoint between adjacent non-negative E4M3FN values (ties)."""
    vals = [oracle.e4m3_value(c) for c in range(0x7F)]
    return np.array([(a + b) / 2 for a, b in zip(vals[:-1], vals[1:])], dtype=np.float64)


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("a_scale", [1.0, 0.0371, 2.0 ** -5, 3.7])
def test_qdq_random_bit_exact(dtype, a_scale):
    bits = wl.gen_activation(97, 333, dtype, seed=11, sigma=40.0 * a_scale)
    got = _qdq_gpu(bits, a_scale, dtype)
    ref = oracle.fp8_qdq_activation(bits, a_scale, dtype)
    np.testing.assert_array_equal(got, ref)


@pytest.mark.parametrize("dtype", DTYPES)
def test_qdq_ties_saturation_specials(dtype):
    """a_scale = 2^-5 makes A / a_scale exact, so every tie between two E4M3
    codes reaches the rounding step as a tie (ties go to the even code); values
    past 448 saturate; zeros keep their sign; infinities saturate."""
    s = 2.0 ** -5
    mids = _e4m3_midpoints() * s
    big = np.array([448.0, 464.0, 480.0, 1000.0, 30000.0]) * s
    vals = np.concatenate([mids, -mids, big, -big, [0.0, -0.0, np.inf, -np.inf]])
    bits = wl.act_bits(vals, dtype)
    got = _qdq_gpu(bits, s, dtype)
    ref = oracle.fp8_qdq_activation(bits, s, dtype)
    np.testing.assert_array_equal(got, ref)
    # Spot facts that do not come from the oracle: saturation gives 448 * s.
    back = oracle.act_to_double(int(got[len(mids) * 2 + 3]), dtype)
    assert back == 448.0 * s


@pytest.mark.parametrize("dtype", DTYPES)
def test_qdq_nan_stays_nan(dtype):
    bits = wl.act_bits(np.array([np.nan, -np.nan, 1.0]), dtype)
    got = _qdq_gpu(bits, 0.5, dtype)
    assert np.isnan(oracle.act_to_double(int(got[0]), dtype))
    assert np.isnan(oracle.act_to_double(int(got[1]), dtype))
    assert oracle.act_to_double(int(got[2]), dtype) == 1.0


@pytest.mark.parametrize("count", [1, 7, 8, 9, 4096 + 3])
def test_qdq_ragged_counts(count):
    dtype = oracle.BF16
    bits = wl.gen_activation(1, count, dtype, seed=count, sigma=3.0)
    got = _qdq_gpu(bits, 0.25, dtype)
    np.testing.assert_array_equal(got, oracle.fp8_qdq_activation(bits, 0.25, dtype))


def _w8a8_ref(p, a_scale):
    Aq = oracle.fp8_qdq_activation(p.A, a_scale, p.dtype)
    return oracle.fp8_matmul(Aq, p.B, p.b_scale, p.bias, p.M, p.N, p.K, p.block_size, p.dtype)


def _w8a8_gpu(p, a_scale):
    d = fp8_dev(p)
    Y = wq.fp8_weight_matmul_w8a8(d["A"], _scale_dev(a_scale), d["B"], d["s"], d["bias"],
                                  block_size=p.block_size)
    torch.cuda.synchronize()
    assert wq.device_status() == 0
    return Y


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("M,N,K,bs", [(1, 256, 1024, 128), (4, 130, 2048, 128),
                                      (8, 64, 4096, 256), (13, 40, 512, 64),
                                      (20, 17, 1000, 128),   # K % 32 != 0: general GEMV
                                      (3, 33, 130, 32)])
def test_w8a8_matmul_shapes(M, N, K, bs, dtype):
    a_scale = 0.0213
    p = wl.make_fp8(M, N, K, bs, dtype, seed=N + K, bias_sigma=0.1)
    assert_within_tolerance(_w8a8_gpu(p, a_scale), *_w8a8_ref(p, a_scale), dtype,
                            f"w8a8 {M}x{N}x{K}")


@pytest.mark.parametrize("M", [1, 4])
def test_w8a8_matmul_5120(M):
    p = wl.fp8_problem(M)
    a_scale = 0.01   # A ~ N(0, 1): codes up to about 450, a few saturate
    assert_within_tolerance(_w8a8_gpu(p, a_scale), *_w8a8_ref(p, a_scale), p.dtype,
                            f"w8a8 5120 M={M}")


def test_w8a8_equals_two_call_route():
    """The fused path and quantize-then-fp8_weight_matmul consume the same A_deq;
    at M <= 8 both run the same GEMV, so the outputs agree bit for bit."""
    p = wl.make_fp8(6, 256, 2048, 128, oracle.BF16, seed=5, bias_sigma=0.1)
    a_scale = 0.05
    d = fp8_dev(p)
    Y1 = wq.fp8_weight_matmul_w8a8(d["A"], _scale_dev(a_scale), d["B"], d["s"], d["bias"],
                                   block_size=128)
    Aq = wq.fp8_quantize_dequantize_activation(d["A"], _scale_dev(a_scale))
    Y2 = wq.fp8_weight_matmul(Aq, d["B"], d["s"], d["bias"], block_size=128)
    torch.cuda.synchronize()
    assert wq.device_status() == 0
    assert torch.equal(Y1.view(torch.int16), Y2.view(torch.int16))


def test_w8a8_k0_fills_bias():
    dtype = oracle.BF16
    bias = wl.gen_bias(24, dtype, 0.5, seed=3)
    A = torch.empty(3, 0, dtype=torch.bfloat16, device=DEV)
    B = torch.empty(24, 0, dtype=torch.uint8, device=DEV)
    s = torch.empty(24, 0, dtype=torch.float32, device=DEV)
    Y = wq.fp8_weight_matmul_w8a8(A, _scale_dev(1.0), B, s, act_to_dev(bias, dtype))
    torch.cuda.synchronize()
    np.testing.assert_array_equal(bits_of(Y), np.broadcast_to(bias, (3, 24)))


# ---------------------------------------------------------------------------
# Prefill-sized M with a caller-owned workspace (fp8_weight_matmul_w8a8_ws)
# ---------------------------------------------------------------------------

def _ws_gpu(d, a_scale, M, K, block_size, extra=0):
    ws = torch.empty(wq.fp8_w8a8_workspace_bytes(M, K) + extra, dtype=torch.uint8, device=DEV)
    Y = wq.fp8_weight_matmul_w8a8_ws(d["A"], _scale_dev(a_scale), d["B"], d["s"], ws, d["bias"],
                                     block_size=block_size)
    torch.cuda.synchronize()
    assert wq.device_status() == 0
    return Y, ws


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("M,N,K,bs", [(9, 384, 512, 128), (64, 256, 1024, 128),
                                      (300, 384, 640, 64), (40, 17, 1000, 128)])
def test_w8a8_ws_against_oracle(M, N, K, bs, dtype):
    """Above 8 rows A_deq goes through the workspace into the FP8 GEMM (or the
    general GEMV for odd shapes); the product is held to the matmul bound
    against the oracle's FP8 matmul of the oracle's A_deq."""
    a_scale = 0.0213
    p = wl.make_fp8(M, N, K, bs, dtype, seed=M + N + K, bias_sigma=0.1)
    Y, _ = _ws_gpu(fp8_dev(p), a_scale, M, K, bs)
    assert_within_tolerance(Y, *_w8a8_ref(p, a_scale), dtype, f"w8a8 ws {M}x{N}x{K}")


@pytest.mark.parametrize("M", [9, 256, 1000])
def test_w8a8_ws_equals_two_call_route(M):
    """The workspace path is quantize-dequantize followed by fp8_weight_matmul:
    bit-identical to those two calls, and the workspace holds A_deq."""
    p = wl.make_fp8(M, 512, 1024, 128, oracle.BF16, seed=M, bias_sigma=0.1)
    a_scale = 0.05
    d = fp8_dev(p)
    Y1, ws = _ws_gpu(d, a_scale, M, 1024, 128)
    Aq = wq.fp8_quantize_dequantize_activation(d["A"], _scale_dev(a_scale))
    Y2 = wq.fp8_weight_matmul(Aq, d["B"], d["s"], d["bias"], block_size=128)
    torch.cuda.synchronize()
    assert torch.equal(Y1.view(torch.int16), Y2.view(torch.int16))
    assert torch.equal(ws.view(torch.int16).view(M, 1024), Aq.view(torch.int16))


def test_w8a8_ws_small_m_is_the_fused_gemv():
    """Up to 8 rows the workspace is not used: same output as
    fp8_weight_matmul_w8a8, bit for bit, and the workspace untouched."""
    p = wl.make_fp8(6, 256, 2048, 128, oracle.BF16, seed=7, bias_sigma=0.1)
    d = fp8_dev(p)
    Y1 = wq.fp8_weight_matmul_w8a8(d["A"], _scale_dev(0.05), d["B"], d["s"], d["bias"],
                                   block_size=128)
    ws = torch.full((64,), 0x5A, dtype=torch.uint8, device=DEV)
    Y2 = wq.fp8_weight_matmul_w8a8_ws(d["A"], _scale_dev(0.05), d["B"], d["s"], ws, d["bias"],
                                      block_size=128)
    torch.cuda.synchronize()
    assert torch.equal(Y1.view(torch.int16), Y2.view(torch.int16))
    assert bool((ws == 0x5A).all())


def test_w8a8_ws_prefill_sampled():
    """The FP8 prefill shape (M = 8192, N = 17408, K = 5120, bs = 128) through the
    workspace path: bit-identical to the two-call route, and 4096 sampled
    outputs within the bound of the oracle's FP8 matmul of the oracle's A_deq."""
    p = wl.fp8_problem(8192, N=17408, K=5120, bias_sigma=0.02)
    a_scale = 0.01
    d = fp8_dev(p)
    Y, _ = _ws_gpu(d, a_scale, p.M, p.K, p.block_size)
    Aq = wq.fp8_quantize_dequantize_activation(d["A"], _scale_dev(a_scale))
    Y2 = wq.fp8_weight_matmul(Aq, d["B"], d["s"], d["bias"], block_size=p.block_size)
    torch.cuda.synchronize()
    assert wq.device_status() == 0
    assert torch.equal(Y.view(torch.int16), Y2.view(torch.int16))
    rng = np.random.default_rng(17)
    ms = rng.integers(0, p.M, 4096)
    ns = rng.integers(0, p.N, 4096)
    Aq_h = oracle.fp8_qdq_activation(p.A[ms], a_scale, p.dtype)
    yref, sabs = oracle.fp8_matmul_sampled(Aq_h, p.B, p.b_scale, p.bias, p.K, p.block_size,
                                           p.dtype, np.arange(4096), ns)
    got = bits_of(Y).reshape(p.M, p.N)[ms, ns]
    Yg = torch.from_numpy(got.astype(np.uint16).view(np.int16)).view(torch.bfloat16)
    assert_within_tolerance(Yg, yref, sabs, p.dtype, "w8a8 ws prefill sampled")
