"""Fused dequantize + tcgen05 GEMM (M > 8) parity against the oracle."""

import numpy as np
import pytest

import oracle
import workloads as wl
from gpu_util import act_to_dev, assert_within_tolerance, f64_of, fp4_dev, run_fp4, run_fp8

pytestmark = pytest.mark.gpu


def _ref(p):
    return oracle.fp4_matmul(p.A, p.B_packed, p.weight_scale, p.weight_scale_2, p.bias, p.M, p.N,
                             p.K, p.block_size, p.dtype)


@pytest.mark.parametrize("dtype", [oracle.BF16, oracle.FP16])
@pytest.mark.parametrize("M,N,K,bs", [
    (16, 128, 64, 16), (256, 128, 128, 16), (9, 1, 32, 16), (300, 200, 320, 16),
    (17, 129, 96, 32), (257, 255, 1024, 16), (512, 384, 2048, 64), (100, 64, 5120, 16),
])
def test_small_shapes(M, N, K, bs, dtype):
    p = wl.make_fp4(M, N, K, bs, dtype, seed=M * 3 + N + K, bias_sigma=0.05)
    assert_within_tolerance(run_fp4(p), *_ref(p), dtype, f"gemm {M}x{N}x{K} bs={bs}")


@pytest.mark.parametrize("M", [24, 64, 128, 256])
def test_one_hot_probe_gemm(M):
    """Bit-exact one-hot probe through the GEMM path (weight_scale_2 = 1, no
    bias): token m selects column k(m) of the weight; Y[m, n] = B_dq[n, k(m)].
    M = 24 / 64 / 128 / 256 run the 32 / 64 / 128 / 256-token tiles (K = 320
    keeps M = 24 off the decode GEMV)."""
    N, K, bs = 128, 320, 16
    p = wl.make_fp4(M, N, K, bs, oracle.BF16, seed=17, ws2=1.0)
    d = fp4_dev(p)
    W = oracle.fp4_dequantize_f64(p.B_packed, p.weight_scale, 1.0, N, K, bs)
    for shift in (0, 1, 101):
        ks = (np.arange(M) * 7 + shift) % K
        A = np.zeros((M, K))
        A[np.arange(M), ks] = 1.0
        d["A"] = act_to_dev(wl.act_bits(A, p.dtype), p.dtype)
        Y = f64_of(run_fp4(p, d))
        assert np.array_equal(Y, W[:, ks].T), shift


def _sampled_check(p, run, ref_sampled, seed=0, n_random=4096, full_rows=4, full_cols=4):
    Y = f64_of(run(p)).reshape(p.M, p.N)
    r = np.random.Generator(np.random.PCG64(seed))
    ms = [r.integers(0, p.M, n_random)]
    ns = [r.integers(0, p.N, n_random)]
    for m in r.integers(0, p.M, full_rows):
        ms.append(np.full(p.N, m))
        ns.append(np.arange(p.N))
    for n in r.integers(0, p.N, full_cols):
        ms.append(np.arange(p.M))
        ns.append(np.full(p.M, n))
    ms = np.concatenate(ms).astype(np.int64)
    ns = np.concatenate(ns).astype(np.int64)
    Yr, S = ref_sampled(p, ms, ns)
    return assert_within_tolerance(Y[ms, ns], Yr, S, p.dtype, "sampled")


def _fp4_sampled(p, ms, ns):
    return oracle.fp4_matmul_sampled(p.A, p.B_packed, p.weight_scale, p.weight_scale_2, p.bias,
                                     p.K, p.block_size, p.dtype, ms, ns)


@pytest.mark.parametrize("shape", ["gate_up", "down"])
def test_prefill_full_size_sampled(shape):
    """NVFP4 prefill M=8192: gate/up (N=17408, K=5120) and down (N=5120,
    K=17408), in the launch configuration the benchmark times; outputs checked
    at 4096 random positions plus 4 full rows and 4 full columns."""
    p = wl.prefill(shape)
    _sampled_check(p, run_fp4, _fp4_sampled)


def test_fp8_gemm_shapes():
    for (M, N, K, bs) in [(64, 128, 256, 128), (300, 257, 1024, 64), (16, 96, 5120, 128)]:
        p = wl.make_fp8(M, N, K, bs, oracle.BF16, seed=K, bias_sigma=0.02)
        Yr, S = oracle.fp8_matmul(p.A, p.B, p.b_scale, p.bias, M, N, K, bs, p.dtype)
        assert_within_tolerance(run_fp8(p), Yr, S, p.dtype, f"fp8 gemm {M}x{N}x{K}")


def test_fp8_prefill_sampled():
    """FP8 M=8192, N=17408, K=5120, bs=128."""
    p = wl.fp8_problem(8192, N=17408, K=5120, bias_sigma=0.02)

    def ref(p, ms, ns):
        return oracle.fp8_matmul_sampled(p.A, p.B, p.b_scale, p.bias, p.K, p.block_size,
                                         p.dtype, ms, ns)
    _sampled_check(p, run_fp8, ref)


def test_fp8_tail_prefill_sampled():
    """FP8 K=5000 (partial last block) at M=8192 takes the row-group GEMV path."""
    p = wl.fp8_problem(8192, N=5120, K=5000, bias_sigma=0.02)

    def ref(p, ms, ns):
        return oracle.fp8_matmul_sampled(p.A, p.B, p.b_scale, p.bias, p.K, p.block_size,
                                         p.dtype, ms, ns)
    _sampled_check(p, run_fp8, ref, n_random=2048, full_rows=2, full_cols=2)


# --- split-K: a thread-block cluster splits K, partial tiles reduce-scattered
# --- through distributed shared memory (used when the tiles fill < half the GPU)

@pytest.mark.parametrize("dtype", [oracle.BF16, oracle.FP16])
@pytest.mark.parametrize("M,N,K,bs", [
    (40, 384, 2048, 16),    # 3 tiles: 4 ranks
    (100, 640, 1600, 16),   # 5 tiles, 25 stages: 3 ranks of 9, 9, 7 stages
    (200, 128, 17408, 16),  # 1 tile, long K: 4 ranks
    (33, 256, 4096, 32),
])
def test_split_k_shapes(M, N, K, bs, dtype):
    p = wl.make_fp4(M, N, K, bs, dtype, seed=M + N + K, bias_sigma=0.05)
    assert_within_tolerance(run_fp4(p), *_ref(p), dtype, f"split-K {M}x{N}x{K}")


def test_split_k_5120_full():
    """M=64, N=K=5120 (40 tiles, 3 ranks): every output."""
    p = wl.make_fp4(64, 5120, 5120, 16, oracle.BF16, seed=64, bias_sigma=0.02)
    assert_within_tolerance(run_fp4(p), *_ref(p), p.dtype, "split-K 64x5120x5120")


def test_one_hot_probe_split_k():
    """One-hot probe through the split-K path (K=2048: 4 ranks), bit-exact:
    each token's single product lives in one rank's partial and crosses the
    reduce-scatter unchanged."""
    M, N, K, bs = 64, 128, 2048, 16
    p = wl.make_fp4(M, N, K, bs, oracle.FP16, seed=23, ws2=1.0)
    d = fp4_dev(p)
    W = oracle.fp4_dequantize_f64(p.B_packed, p.weight_scale, 1.0, N, K, bs)
    for shift in (0, 555, 1999):
        ks = (np.arange(M) * 31 + shift) % K
        A = np.zeros((M, K))
        A[np.arange(M), ks] = 1.0
        d["A"] = act_to_dev(wl.act_bits(A, p.dtype), p.dtype)
        Y = f64_of(run_fp4(p, d))
        assert np.array_equal(Y, W[:, ks].T), shift


def test_fp8_split_k():
    p = wl.make_fp8(48, 256, 4096, 128, oracle.BF16, seed=48, bias_sigma=0.05)
    Y = run_fp8(p)
    Yr, S = oracle.fp8_matmul(p.A, p.B, p.b_scale, p.bias, p.M, p.N, p.K, p.block_size, p.dtype)
    assert_within_tolerance(Y, Yr, S, p.dtype, "fp8 split-K")


# --- mid-range M: the token tile narrows to 32 / 64 / 128 (MMA N) so that a
# --- small batch does not pay for a 256-token tile of padding rows

@pytest.mark.parametrize("dtype", [oracle.BF16, oracle.FP16])
@pytest.mark.parametrize("M,N,K,bs", [
    (24, 256, 320, 16),     # 32-token tile (K % 256 != 0 keeps it off the GEMV)
    (32, 384, 640, 32),     # 32-token tile, bs 32
    (20, 256, 4160, 16),    # 32-token tile, split-K over 4 ranks (K % 256 != 0)
    (48, 200, 512, 16),     # 64-token tile, ragged N
    (64, 128, 1024, 16),    # 64-token tile, full
    (40, 640, 2048, 16),    # 64-token tile, split-K (5 tiles, 4 ranks)
    (65, 256, 256, 16),     # 128-token tile, one real row past the 64-token tile
    (128, 129, 768, 16),    # 128-token tile, full, ragged N
    (100, 1280, 1600, 16),  # 128-token tile, split-K (10 tiles, 3 ranks)
    (129, 64, 320, 16),     # back to the 256-token tile
])
def test_mid_m_tiles(M, N, K, bs, dtype):
    p = wl.make_fp4(M, N, K, bs, dtype, seed=M * 7 + N + K, bias_sigma=0.05)
    assert_within_tolerance(run_fp4(p), *_ref(p), dtype, f"mid-M {M}x{N}x{K} bs={bs}")


@pytest.mark.parametrize("M,N,K,bs", [(20, 256, 4096, 128), (33, 300, 1024, 64),
                                      (96, 257, 1024, 128), (128, 64, 5120, 128)])
def test_fp8_mid_m_tiles(M, N, K, bs):
    p = wl.make_fp8(M, N, K, bs, oracle.BF16, seed=M + K, bias_sigma=0.05)
    Yr, S = oracle.fp8_matmul(p.A, p.B, p.b_scale, p.bias, M, N, K, bs, p.dtype)
    assert_within_tolerance(run_fp8(p), Yr, S, p.dtype, f"fp8 mid-M {M}x{N}x{K}")


@pytest.mark.parametrize("M", [64, 128])
def test_mid_m_gate_up_sampled(M):
    """M = 64 / 128 tokens at the gate/up shape (N = 17408, K = 5120), as the
    benchmark times it: sampled outputs plus full rows and columns."""
    p = wl.make_fp4(M, 17408, 5120, 16, oracle.BF16, seed=M, bias_sigma=0.02)
    _sampled_check(p, run_fp4, _fp4_sampled, n_random=2048)


# --- two light CTAs per SM (narrow tiles whose count fills half the SMs) ---

@pytest.mark.parametrize("dtype", [oracle.BF16, oracle.FP16])
@pytest.mark.parametrize("M,N,K,bs", [
    (64, 12800, 1024, 16),    # 64-token tile, 100 tiles: K split over 2 ranks
    (100, 20485, 512, 16),    # 128-token tile, 161 tiles: no split, ragged N
    (32, 12800, 2080, 32),    # 32-token tile (K % 256 != 0), 100 tiles, split 2
    (28, 12800, 1024, 16),    # 25..32 rows of a many-tile weight: GEMM, not the GEMV
])
def test_light_ctas(M, N, K, bs, dtype):
    p = wl.make_fp4(M, N, K, bs, dtype, seed=M + N + K, bias_sigma=0.05)
    assert_within_tolerance(run_fp4(p), *_ref(p), dtype, f"light {M}x{N}x{K}")


def test_light_ctas_fp8():
    p = wl.make_fp8(64, 12800, 1024, 128, oracle.BF16, seed=3, bias_sigma=0.05)
    Yr, S = oracle.fp8_matmul(p.A, p.B, p.b_scale, p.bias, p.M, p.N, p.K, 128, p.dtype)
    assert_within_tolerance(run_fp8(p), Yr, S, p.dtype, "fp8 light")


def test_one_hot_probe_light_ctas():
    """Bit-exact one-hot probe through two light CTAs per SM with a K split
    (M = 64, N = 12800: 100 tiles, 2 ranks)."""
    M, N, K, bs = 64, 12800, 1024, 16
    p = wl.make_fp4(M, N, K, bs, oracle.FP16, seed=41, ws2=1.0)
    d = fp4_dev(p)
    W = oracle.fp4_dequantize_f64(p.B_packed, p.weight_scale, 1.0, N, K, bs)
    for shift in (0, 517):
        ks = (np.arange(M) * 13 + shift) % K
        A = np.zeros((M, K))
        A[np.arange(M), ks] = 1.0
        d["A"] = act_to_dev(wl.act_bits(A, p.dtype), p.dtype)
        Y = f64_of(run_fp4(p, d))
        assert np.array_equal(Y, W[:, ks].T), shift


@pytest.mark.parametrize("kind,M,N,K,bs", [
    ("fp4", 8192, 17408, 5120, 16),   # the prefill launch: full CTAs, 256-token tiles
    ("fp4", 64, 17408, 5120, 16),     # two light CTAs per SM, K split over 2
    ("fp4", 256, 640, 5120, 16),      # full CTAs, K split over 4
    ("fp8", 8192, 5120, 4096, 128),   # FP8 prefill
])
def test_gemm_repeated_runs_bit_identical(kind, M, N, K, bs):
    """Ten runs into fresh output buffers give the same bits: the stage ring
    hands every stage to the MMA only after its copies have landed and its
    operand is stored (a stage read early or overwritten late would show up
    as run-to-run differences)."""
    import torch
    if kind == "fp4":
        p = wl.make_fp4(8, N, K, bs, oracle.BF16, seed=N + K, bias_sigma=0.02)
        d = fp4_dev(p)
        d["A"] = torch.randn(M, K, device="cuda:0", dtype=torch.bfloat16)
        run = lambda: run_fp4(p, d)
    else:
        p = wl.make_fp8(8, N, K, bs, oracle.BF16, seed=N + K, bias_sigma=0.02)
        from gpu_util import fp8_dev
        d = fp8_dev(p)
        d["A"] = torch.randn(M, K, device="cuda:0", dtype=torch.bfloat16)
        run = lambda: run_fp8(p, d)
    first = run()
    assert torch.isfinite(first.float()).all()
    for _ in range(9):
        assert torch.equal(run(), first)


# ---------------------------------------------------------------------------
# Persistent prefill kernel: 256-token tiles, enough of them to fill the GPU
# without a K split (tiles * 2 > SMs); with more tiles than SMs some CTAs run
# several tiles in turn, the stage ring and parities running on across them.
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("dtype", [oracle.BF16, oracle.FP16])
@pytest.mark.parametrize("M,N,K,bs", [
    (1000, 5000, 640, 16),     # 4 x 40 = 160 tiles: ragged last token and row tiles
    (2048, 2560, 1024, 32),    # 8 x 20 = 160 tiles
    (700, 4096, 320, 16),      # 3 x 32 = 96 tiles: one per CTA
])
def test_persistent_prefill_tiles(M, N, K, bs, dtype):
    p = wl.make_fp4(M, N, K, bs, dtype, seed=M + N + K, bias_sigma=0.05)
    assert_within_tolerance(run_fp4(p), *_ref(p), dtype, f"persistent {M}x{N}x{K} bs={bs}")


@pytest.mark.parametrize("dtype", [oracle.BF16, oracle.FP16])
@pytest.mark.parametrize("K", [1024, 256])
def test_persistent_fp8_tiles(dtype, K):
    """FP8 weights through the persistent kernel (five decoder phases), 160
    tiles, FP16 included (row scale normalisation per tile); K = 256 gives
    four stages per tile, fewer than the decoder phases, so some decoder warps
    have no stage in a tile and run its epilogue all the same."""
    M, N, bs = 1000, 5000, 128
    # Block scales up to 200 (e4m3 * b_scale beyond the FP16 range) with small
    # activations, so that the outputs stay finite.
    p = wl.make_fp8(M, N, K, bs, dtype, seed=5, bias_sigma=0.05, scale_lo=1.0, scale_hi=200.0,
                    a_sigma=1e-3)
    Yr, S = oracle.fp8_matmul(p.A, p.B, p.b_scale, p.bias, M, N, K, bs, p.dtype)
    assert_within_tolerance(run_fp8(p), Yr, S, dtype, "persistent fp8")


def test_one_hot_probe_persistent():
    """Bit-exact one-hot probe through the persistent kernel: 160 tiles of 256
    tokens, token m selects column k(m); every CTA's second tile included."""
    M, N, K, bs = 1024, 5120, 320, 16
    p = wl.make_fp4(M, N, K, bs, oracle.BF16, seed=23, ws2=1.0)
    d = fp4_dev(p)
    W = oracle.fp4_dequantize_f64(p.B_packed, p.weight_scale, 1.0, N, K, bs)
    ks = (np.arange(M) * 13 + 5) % K
    A = np.zeros((M, K))
    A[np.arange(M), ks] = 1.0
    d["A"] = act_to_dev(wl.act_bits(A, p.dtype), p.dtype)
    Y = f64_of(run_fp4(p, d))
    assert np.array_equal(Y, W[:, ks].T)


def test_persistent_gemm_in_cuda_graph():
    """The persistent prefill GEMM captured in a CUDA graph: replays equal the
    eager result bit for bit (no host-side state between calls)."""
    import torch
    p = wl.make_fp4(1000, 5000, 640, 16, oracle.BF16, seed=31, bias_sigma=0.05)
    d = fp4_dev(p)
    import fp8_weight_only_nvfp4_gb300 as wq
    eager = run_fp4(p, d)
    Y = torch.empty_like(eager)
    stream = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        wq.fp4_weight_matmul(d["A"], d["B"], d["ws"], d["ws2"], d["bias"], 16, out=Y,
                             stream=stream)
        stream.synchronize()
        with torch.cuda.graph(g, stream=stream):
            wq.fp4_weight_matmul(d["A"], d["B"], d["ws"], d["ws2"], d["bias"], 16, out=Y,
                                 stream=stream)
    for _ in range(2):
        Y.fill_(float("nan"))
        g.replay()
        stream.synchronize()
        assert wq.device_status() == 0
        assert torch.equal(Y.view(torch.int16), eager.view(torch.int16))


@pytest.mark.parametrize("shape", ["gate_up", "down"])
def test_prefill_full_size_sampled_fp16(shape):
    """The NVFP4 prefill shapes at M = 8192 with FP16 activations and bias
    (persistent kernel, FP16 operands): 4096 random outputs plus 4 full rows
    and 4 full columns against the oracle."""
    N, K = (17408, 5120) if shape == "gate_up" else (5120, 17408)
    p = wl.make_fp4(8192, N, K, 16, oracle.FP16, seed=3, ws2=0.0125, bias_sigma=0.02)
    _sampled_check(p, run_fp4, _fp4_sampled, seed=5)


def test_fp8_prefill_sampled_fp16():
    """FP8 M = 8192, N = 17408, K = 5120, bs = 128 with FP16 activations and
    block scales up to 200 (each weight row's scales divided by a power of two
    in the decode and multiplied back in the epilogue), small activations so
    that the outputs stay finite."""
    p = wl.make_fp8(8192, 17408, 5120, 128, oracle.FP16, seed=4, scale_lo=0.5, scale_hi=200.0,
                    bias_sigma=0.02, a_sigma=1e-3)

    def ref(p, ms, ns):
        return oracle.fp8_matmul_sampled(p.A, p.B, p.b_scale, p.bias, p.K, p.block_size,
                                         p.dtype, ms, ns)
    _sampled_check(p, run_fp8, ref, seed=6)
