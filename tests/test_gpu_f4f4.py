"""NVFP4 x NVFP4 block-scaled tensor-core GEMM (fp4_fp4_matmul) against the
oracle.

The FP4 page §6 defines the product from NVFP4 codes and block scales of
both operands.  Its reference here is the oracle alone: every
e2m1(code) * e4m3(scale) has at most 6 significant bits and lies in the
FP16/BF16 range, so oracle.fp4_dequantize(codes, scales, 1.0) is the exact
dequantized activation, and oracle.fp4_matmul of it is the FP4 x FP4 sum in
float64.  Structured inputs with power-of-two values give outputs that are
exact in the output type, compared bit for bit against closed forms: they pin
which scale the tensor core applies to which row and 16-element block."""

import numpy as np
import pytest
import torch

import fp8_weight_only_nvfp4_gb300 as wq
import oracle
import workloads as wl
from gpu_util import DEV, act_to_dev, assert_within_tolerance, bits_of, f32_to_dev, f64_of, u8_to_dev

pytestmark = pytest.mark.gpu

DTYPES = [oracle.BF16, oracle.FP16]
ONE_CODES = 0x22          # two E2M1 codes of 1.0
E4M3_ONE = 0x38           # 1.0


def _tdt(dtype):
    return torch.bfloat16 if dtype == oracle.BF16 else torch.float16


def _run(Ac, As, w, M, bias=True):
    """fp4_fp4_matmul on host arrays: activation codes/scales, weight problem."""
    Y = wq.fp4_fp4_matmul(u8_to_dev(Ac), u8_to_dev(As), u8_to_dev(w.B_packed),
                          u8_to_dev(w.weight_scale),
                          f32_to_dev(np.array([w.weight_scale_2], dtype=np.float32)),
                          act_to_dev(w.bias, w.dtype) if (bias and w.bias is not None) else None,
                          dtype=_tdt(w.dtype))
    torch.cuda.synchronize()
    assert wq.device_status() == 0
    assert tuple(Y.shape) == (M, w.N)
    return Y


def _reference(Ac, As, w, M):
    Ad = oracle.fp4_dequantize(Ac, As, 1.0, M, w.K, 16, w.dtype)
    return oracle.fp4_matmul(Ad, w.B_packed, w.weight_scale, w.weight_scale_2, w.bias, M, w.N,
                             w.K, 16, w.dtype)


def _activation(M, K, dtype, seed, log_uniform=False):
    """Random activation codes (uniform nibbles) and E4M3 block scales."""
    a = wl.make_fp4(1, M, K, 16, dtype, seed=seed, log_uniform=log_uniform,
                    scale_lo=2.0 ** -6 if log_uniform else 2.0 ** -4)
    return a.B_packed, a.weight_scale


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("M,N,K", [(1, 128, 256), (200, 384, 512), (300, 200, 1024),
                                   (513, 100, 2048), (256, 256, 5120), (64, 1000, 768)])
def test_f4f4_against_oracle(M, N, K, dtype):
    """Ragged token tiles (M % 256), ragged weight tiles (N % 128), direct
    stores (N % 8 != 0) and several K; random codes and scales of both
    operands, bias."""
    w = wl.make_fp4(1, N, K, 16, dtype, seed=M + N + K, bias_sigma=0.1)
    Ac, As = _activation(M, K, dtype, seed=7 * M + K, log_uniform=(M % 2 == 1))
    Yr, S = _reference(Ac, As, w, M)
    assert_within_tolerance(_run(Ac, As, w, M), Yr, S, dtype, f"f4f4 {M}x{N}x{K}")


def _structured(M, N, K, dtype, a_scale, w_scale, a_codes=None, w_codes=None):
    """Operands with all codes 1.0 unless given; scales from the callables
    a_scale(m, b) / w_scale(n, b) (E4M3 bytes); weight_scale_2 = 1, no bias."""
    S = K // 16
    Ac = np.full((M, K // 2), ONE_CODES, np.uint8) if a_codes is None else a_codes
    Bp = np.full((N, K // 2), ONE_CODES, np.uint8) if w_codes is None else w_codes
    As = np.array([[a_scale(m, b) for b in range(S)] for m in range(M)], dtype=np.uint8)
    Ws = np.array([[w_scale(n, b) for b in range(S)] for n in range(N)], dtype=np.uint8)
    w = wl.Fp4Problem(M=M, N=N, K=K, block_size=16, dtype=dtype, A=None, B_packed=Bp,
                      weight_scale=Ws, weight_scale_2=1.0, bias=None)
    return Ac, As, w


def _e4m3_pow2(e):
    """E4M3FN byte of 2^e for -6 <= e <= 8."""
    return (e + 7) << 3


def _exact_bits(values, dtype):
    return wl.act_bits(np.asarray(values, dtype=np.float32), dtype)


@pytest.mark.parametrize("dtype", DTYPES)
def test_f4f4_weight_scale_lanes(dtype):
    """Weight row n has one nonzero block scale, 2^(n % 8 - 4), at block
    (7 n) % S: Y[m, n] = 16 * 2^(n % 8 - 4) for every token, exactly.  A
    wrong row-to-lane or chunk-to-column mapping of the weight scales gives a
    different power of two or zero."""
    M, N, K = 40, 384, 1024
    S = K // 16
    Ac, As, w = _structured(M, N, K, dtype, lambda m, b: E4M3_ONE,
                            lambda n, b: _e4m3_pow2(n % 8 - 4) if b == (7 * n) % S else 0)
    Y = _run(Ac, As, w, M)
    want = np.broadcast_to(16.0 * 2.0 ** (np.arange(N) % 8 - 4), (M, N))
    np.testing.assert_array_equal(bits_of(Y), _exact_bits(want, dtype))


@pytest.mark.parametrize("dtype", DTYPES)
def test_f4f4_token_scale_lanes(dtype):
    """Token row m has one nonzero block scale, 2^(m % 8 - 4), at block
    (5 m) % S: Y[m, n] = 16 * 2^(m % 8 - 4), exactly; 600 tokens cover the
    upper 128 rows of a 256-token tile and a ragged last tile."""
    M, N, K = 600, 128, 512
    S = K // 16
    Ac, As, w = _structured(M, N, K, dtype,
                            lambda m, b: _e4m3_pow2(m % 8 - 4) if b == (5 * m) % S else 0,
                            lambda n, b: E4M3_ONE)
    Y = _run(Ac, As, w, M)
    want = np.broadcast_to((16.0 * 2.0 ** (np.arange(M) % 8 - 4))[:, None], (M, N))
    np.testing.assert_array_equal(bits_of(Y), _exact_bits(want, dtype))


@pytest.mark.parametrize("dtype", DTYPES)
def test_f4f4_scale_meets_its_block(dtype):
    """Each block's scale multiplies that block's codes: weight row n has
    codes 1.0 only in block b(n) = n % S (zero codes elsewhere) and block
    scales 2^(b % 8 - 4) on every block; token m likewise has codes only in
    block c(m) = (3 m) % S with scales 2^(3 - b % 8).  Y[m, n] =
    16 * 2^(b % 8 - 4) * 2^(3 - b % 8) = 8 if b(n) == c(m), else 0."""
    M, N, K = 96, 256, 512
    S = K // 16

    def one_block(rows, blk):
        c = np.zeros((rows, K // 2), np.uint8)
        for r in range(rows):
            b = blk(r)
            c[r, 8 * b: 8 * b + 8] = ONE_CODES
        return c
    Ac, As, w = _structured(M, N, K, dtype,
                            lambda m, b: _e4m3_pow2(3 - b % 8), lambda n, b: _e4m3_pow2(b % 8 - 4),
                            a_codes=one_block(M, lambda m: (3 * m) % S),
                            w_codes=one_block(N, lambda n: n % S))
    Y = _run(Ac, As, w, M)
    want = np.where((np.arange(N)[None, :] % S) == ((3 * np.arange(M))[:, None] % S), 8.0, 0.0)
    np.testing.assert_array_equal(bits_of(Y), _exact_bits(want, dtype))


def test_f4f4_quantized_activation_full_size_sampled():
    """The native FP4 x FP4 prefill: a BF16 activation M = 8192, K = 5120
    quantized to NVFP4 (the oracle's codes and scales), the gate/up weight
    N = 17408 with bias; 4096 random outputs plus 4 full rows and 4 full
    columns against the oracle's weight-only matmul of the oracle's
    quantize-dequantize activation (the same FP4 x FP4 sum)."""
    p = wl.prefill("gate_up")
    codes, scales = oracle.nvfp4_quantize_activation(p.A, p.dtype)
    Y = f64_of(_run(codes, scales, p, p.M)).reshape(p.M, p.N)
    Ad = oracle.nvfp4_qdq_activation(p.A, p.dtype)
    r = np.random.Generator(np.random.PCG64(3))
    ms = [r.integers(0, p.M, 4096)]
    ns = [r.integers(0, p.N, 4096)]
    for m in r.integers(0, p.M, 4):
        ms.append(np.full(p.N, m))
        ns.append(np.arange(p.N))
    for n in r.integers(0, p.N, 4):
        ms.append(np.arange(p.M))
        ns.append(np.full(p.M, n))
    ms = np.concatenate(ms).astype(np.int64)
    ns = np.concatenate(ns).astype(np.int64)
    Yr, S = oracle.fp4_matmul_sampled(Ad, p.B_packed, p.weight_scale, p.weight_scale_2, p.bias,
                                      p.K, 16, p.dtype, ms, ns)
    assert_within_tolerance(Y[ms, ns], Yr, S, p.dtype, "f4f4 prefill sampled")


def test_f4f4_gpu_quantizer_then_gemm():
    """fp4_quantize_activation followed by fp4_fp4_matmul, all on the GPU,
    within the bound of the oracle's FP4 x FP4 product of the same activation."""
    p = wl.make_fp4(300, 640, 2048, 16, oracle.BF16, seed=21, bias_sigma=0.02)
    A = act_to_dev(p.A, p.dtype)
    qc, qs = wq.fp4_quantize_activation(A)
    Y = wq.fp4_fp4_matmul(qc, qs, u8_to_dev(p.B_packed), u8_to_dev(p.weight_scale),
                          f32_to_dev(np.array([p.weight_scale_2], np.float32)),
                          act_to_dev(p.bias, p.dtype))
    torch.cuda.synchronize()
    assert wq.device_status() == 0
    Yr, S = oracle.fp4_matmul(oracle.nvfp4_qdq_activation(p.A, p.dtype), p.B_packed,
                              p.weight_scale, p.weight_scale_2, p.bias, p.M, p.N, p.K, 16,
                              p.dtype)
    assert_within_tolerance(Y, Yr, S, p.dtype, "quantize + f4f4")


def test_f4f4_k0_and_empty():
    bias = wl.gen_bias(24, oracle.BF16, 0.5, seed=3)
    z = torch.empty(3, 0, dtype=torch.uint8, device=DEV)
    Y = wq.fp4_fp4_matmul(z, torch.empty(3, 0, dtype=torch.uint8, device=DEV),
                          torch.empty(24, 0, dtype=torch.uint8, device=DEV),
                          torch.empty(24, 0, dtype=torch.uint8, device=DEV),
                          torch.ones(1, device=DEV), act_to_dev(bias, oracle.BF16))
    torch.cuda.synchronize()
    np.testing.assert_array_equal(bits_of(Y), np.broadcast_to(bias, (3, 24)))
    e = wq.fp4_fp4_matmul(torch.empty(0, 128, dtype=torch.uint8, device=DEV),
                          torch.empty(0, 16, dtype=torch.uint8, device=DEV),
                          torch.zeros(8, 128, dtype=torch.uint8, device=DEV),
                          torch.zeros(8, 16, dtype=torch.uint8, device=DEV),
                          torch.ones(1, device=DEV))
    assert tuple(e.shape) == (0, 8)


def test_f4f4_unsupported_k():
    """K not a multiple of 32 is refused (no launch)."""
    A = torch.zeros(4, 40, dtype=torch.uint8, device=DEV)
    with pytest.raises(wq.WqmmError):
        wq.fp4_fp4_matmul(A, torch.zeros(4, 5, dtype=torch.uint8, device=DEV),
                          torch.zeros(16, 40, dtype=torch.uint8, device=DEV),
                          torch.zeros(16, 5, dtype=torch.uint8, device=DEV),
                          torch.ones(1, device=DEV))


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("M,N,K", [(300, 200, 32), (257, 384, 96), (64, 1000, 480),
                                   (513, 129, 1056), (200, 300, 5152), (9, 100, 5024)])
def test_f4f4_k_not_multiple_of_256(M, N, K, dtype):
    """K % 256 != 0: the scale rows are read from global memory (4-byte loads
    when K % 64 == 0, byte loads otherwise) and the last stage is partial."""
    w = wl.make_fp4(1, N, K, 16, dtype, seed=M + N + K + 1, bias_sigma=0.1)
    Ac, As = _activation(M, K, dtype, seed=5 * M + K, log_uniform=(K % 64 != 0))
    Yr, S = _reference(Ac, As, w, M)
    assert_within_tolerance(_run(Ac, As, w, M), Yr, S, dtype, f"f4f4 {M}x{N}x{K}")


def test_f4f4_in_cuda_graph():
    """Activation quantization + FP4 x FP4 GEMM captured in one CUDA graph:
    replays equal the eager result bit for bit."""
    p = wl.make_fp4(600, 1000, 1024, 16, oracle.BF16, seed=41, bias_sigma=0.05)
    A = act_to_dev(p.A, p.dtype)
    B, Ws = u8_to_dev(p.B_packed), u8_to_dev(p.weight_scale)
    g2 = f32_to_dev(np.array([p.weight_scale_2], np.float32))
    bias = act_to_dev(p.bias, p.dtype)
    qc, qs = wq.fp4_quantize_activation(A)
    eager = wq.fp4_fp4_matmul(qc, qs, B, Ws, g2, bias)
    torch.cuda.synchronize()
    Y = torch.empty_like(eager)
    stream = torch.cuda.Stream()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        wq.fp4_quantize_activation(A, out_packed=qc, out_scale=qs, stream=stream)
        wq.fp4_fp4_matmul(qc, qs, B, Ws, g2, bias, out=Y, stream=stream)
        stream.synchronize()
        with torch.cuda.graph(graph, stream=stream):
            wq.fp4_quantize_activation(A, out_packed=qc, out_scale=qs, stream=stream)
            wq.fp4_fp4_matmul(qc, qs, B, Ws, g2, bias, out=Y, stream=stream)
    for _ in range(2):
        Y.fill_(float("nan"))
        graph.replay()
        stream.synchronize()
        assert wq.device_status() == 0
        assert torch.equal(Y.view(torch.int16), eager.view(torch.int16))


def test_f4f4_full_size_sampled_fp16():
    """FP4 x FP4 at M = 8192, N = 17408, K = 5120 with FP16 output and bias,
    random codes and log-uniform scales of both operands: 4096 sampled outputs
    against the oracle's sum."""
    M, N, K = 8192, 17408, 5120
    w = wl.make_fp4(1, N, K, 16, oracle.FP16, seed=8, bias_sigma=0.02)
    Ac, As = _activation(M, K, oracle.FP16, seed=9, log_uniform=True)
    Y = f64_of(_run(Ac, As, w, M)).reshape(M, N)
    Ad = oracle.fp4_dequantize(Ac, As, 1.0, M, K, 16, oracle.FP16)
    r = np.random.Generator(np.random.PCG64(10))
    ms = r.integers(0, M, 4096).astype(np.int64)
    ns = r.integers(0, N, 4096).astype(np.int64)
    Yr, S = oracle.fp4_matmul_sampled(Ad, w.B_packed, w.weight_scale, w.weight_scale_2, w.bias,
                                      K, 16, oracle.FP16, ms, ns)
    assert_within_tolerance(Y[ms, ns], Yr, S, oracle.FP16, "f4f4 full size fp16")
