"""Pins for the CPU oracle: each check ties the oracle to something other than
itself -- values the pages state (tests/golden, with citations), library
routines (torch float8_e4m3fn decode, torch dtype casts, torch float64
matmul), closed forms and invariants.  A plausible mistake in the oracle (a
swapped nibble, a wrong scale index, a transposed operand, a dropped term, a
wrong rounding) fails at least one of these.
"""

import math
import os

import numpy as np
import pytest
import torch

import oracle
import workloads as wl

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden_lines(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return [ln.split() for ln in f if ln.strip() and not ln.startswith("#")]


def _e2m1_golden():
    return {int(c): float(v) for c, v in _golden_lines("e2m1_values.txt")}


def _torch_e4m3(byte_arr):
    t = torch.from_numpy(np.ascontiguousarray(byte_arr, dtype=np.uint8))
    return t.view(torch.float8_e4m3fn).to(torch.float64).numpy()


def _lib_fp4_dequant_f64(Bp, ws, ws2, N, K, bs):
    """Independent decode: golden E2M1 list + torch float8_e4m3fn decode."""
    table = np.array([_e2m1_golden()[c] for c in range(16)], dtype=np.float64)
    lo = Bp & 0xF
    hi = Bp >> 4
    codes = np.empty((N, K), dtype=np.int64)
    codes[:, 0::2] = lo
    codes[:, 1::2] = hi
    kidx = np.arange(K) // bs
    sc = _torch_e4m3(ws)[:, kidx]
    return table[codes] * sc * float(np.float32(ws2))


# ---------------------------------------------------------------------------
# Format primitives
# ---------------------------------------------------------------------------

def test_e2m1_table_matches_pages():
    gold = _e2m1_golden()
    for code in range(16):
        v = oracle.e2m1_value(code)
        assert v == gold[code], code
        # sign of zero matters: 0x8 is -0.0
        assert math.copysign(1.0, v) == math.copysign(1.0, gold[code]) or gold[code] != 0.0
    assert math.copysign(1.0, oracle.e2m1_value(8)) == -1.0
    assert math.copysign(1.0, oracle.e2m1_value(0)) == 1.0


def test_e4m3_table_matches_torch_all_bytes():
    ref = _torch_e4m3(np.arange(256, dtype=np.uint8))
    for b in range(256):
        v = oracle.e4m3_value(b)
        if math.isnan(ref[b]):
            assert math.isnan(v), b
        else:
            assert v == ref[b], (b, v, ref[b])
            assert math.copysign(1.0, v) == math.copysign(1.0, ref[b])


def test_format_extremes_from_pages():
    g = {k: float(v) for k, v in _golden_lines("format_extremes.txt")}
    e2m1 = [abs(oracle.e2m1_value(c)) for c in range(16)]
    e4m3 = [abs(oracle.e4m3_value(b)) for b in range(256)
            if not math.isnan(oracle.e4m3_value(b))]
    assert max(e2m1) == g["e2m1_max"]
    assert min(v for v in e2m1 if v > 0) == g["e2m1_min_nonzero"]
    assert max(e4m3) == g["e4m3_max"]
    assert min(v for v in e4m3 if v > 0) == g["e4m3_min_subnormal"]
    prods = [a * b for a in e2m1 for b in e4m3]
    assert max(prods) == g["fold_max"]
    assert min(p for p in prods if p > 0) == g["fold_min_nonzero"]


def test_fold_is_exact_in_fp16_and_bf16():
    """Every e2m1 * e4m3 product is representable in FP16 and BF16
    (FP4 page §4: at most 6 significant bits, range 2^-10 .. 2688)."""
    prods = np.array([oracle.e2m1_value(c) * oracle.e4m3_value(b)
                      for c in range(16) for b in range(256)
                      if not math.isnan(oracle.e4m3_value(b))], dtype=np.float64)
    for dt in (torch.float16, torch.bfloat16):
        back = torch.from_numpy(prods).to(dt).to(torch.float64).numpy()
        assert np.array_equal(back, prods)


def _rne_cases():
    r = np.random.Generator(np.random.PCG64(1234))
    bits = [r.integers(0, 2 ** 32, size=1 << 20, dtype=np.uint64).astype(np.uint32)]
    special = []
    # ties and neighbours around every binade, both signs, for both targets
    for e in range(0, 255):
        base = e << 23
        for low in (0x0000, 0x0001, 0x7FFF, 0x8000, 0x8001, 0xFFFF, 0x1000, 0x0FFF,
                    0x17FFF, 0x18000, 0x18001, 0x10000, 0x7FFFFF, 0x400000, 0x1FFF,
                    0x2000, 0x2001, 0x3000, 0x6000, 0xE000):
            special.append(base | (low & 0x7FFFFF))
    special += [0x7F800000, 0x7F800001, 0x7FC00000, 0x00000001, 0x00800000,
                0x477FE000, 0x477FEFFF, 0x477FF000, 0x477FF001, 0x47800000,
                0x33000000, 0x33000001, 0x32FFFFFF, 0x33800000, 0x387FC000,
                0x38800000, 0x387FE000, 0x7F7FFFFF, 0x7F7F8000]
    sp = np.array(special, dtype=np.uint32)
    bits.append(sp)
    bits.append(sp | np.uint32(0x80000000))
    return np.concatenate(bits)


@pytest.mark.parametrize("dtype", [oracle.BF16, oracle.FP16])
def test_rne_matches_torch_cast(dtype):
    bits = _rne_cases()
    f = bits.view(np.float32)
    ours = oracle.rne_f32_to_act(f, dtype)
    tdt = torch.bfloat16 if dtype == oracle.BF16 else torch.float16
    ref = torch.from_numpy(f.copy()).to(tdt).view(torch.int16).numpy().view(np.uint16)
    nan = np.isnan(f)
    assert np.array_equal(ours[~nan], ref[~nan])
    # NaN stays NaN (payload not compared)
    back = torch.from_numpy(ours[nan].view(np.int16).copy()).view(tdt).float().numpy()
    assert np.all(np.isnan(back))


def test_act_decode_matches_torch():
    for dtype, tdt in ((oracle.BF16, torch.bfloat16), (oracle.FP16, torch.float16)):
        r = np.random.Generator(np.random.PCG64(7))
        bits = r.integers(0, 65536, size=4096, dtype=np.uint32).astype(np.uint16)
        bits = np.concatenate([bits, np.array([0, 0x8000, 1, 0x3C00, 0x7BFF, 0x0400, 0x03FF,
                                               0x3F80, 0x7F7F], dtype=np.uint16)])
        ref = torch.from_numpy(bits.view(np.int16).copy()).view(tdt).to(torch.float64).numpy()
        for b, v in zip(bits, ref):
            o = oracle.act_to_double(int(b), dtype)
            if math.isnan(v):
                assert math.isnan(o)
            else:
                assert o == v


# ---------------------------------------------------------------------------
# Dequantize (bit-exact contract)
# ---------------------------------------------------------------------------

def test_hand_nibble_order_and_negative_byte():
    cases = {ln[0]: ln[1:] for ln in _golden_lines("hand_cases.txt")}
    for key in ("nibble_order", "negative_byte"):
        byte = int(cases[key][0], 16)
        want = [float(x) for x in cases[key][1:3]]
        Bp = np.array([[byte]], dtype=np.uint8)
        ws = np.array([[0x38]], dtype=np.uint8)  # 1.0
        out = oracle.fp4_dequantize_f64(Bp, ws, 1.0, 1, 2, 16)
        assert out[0].tolist() == want
        q = oracle.fp4_dequantize(Bp, ws, 1.0, 1, 2, 16, oracle.FP16)
        vals = [oracle.act_to_double(int(x), oracle.FP16) for x in q[0]]
        assert vals == want


@pytest.mark.parametrize("dtype", [oracle.BF16, oracle.FP16])
def test_dequant_all_bytes_against_torch_float32(dtype):
    """All 256 packed bytes x a spread of scale bytes x several weight_scale_2
    values, against torch float32 arithmetic on torch-decoded operands:
    (e2m1 * e4m3) * ws2 in float32, then a torch cast to the activation type."""
    scale_bytes = [0x00, 0x01, 0x07, 0x08, 0x18, 0x30, 0x38, 0x39, 0x3F, 0x48, 0x70,
                   0x7E, 0x80, 0xB8, 0xFE]
    N = len(scale_bytes)
    K = 512  # 256 bytes per row -> every packed byte once
    Bp = np.tile(np.arange(256, dtype=np.uint8), (N, 1))
    ws = np.array(scale_bytes, dtype=np.uint8).reshape(N, 1).repeat(K // 16, axis=1)
    tdt = torch.bfloat16 if dtype == oracle.BF16 else torch.float16
    table = torch.tensor([_e2m1_golden()[c] for c in range(16)], dtype=torch.float32)
    codes = np.empty((N, K), dtype=np.int64)
    codes[:, 0::2] = Bp & 0xF
    codes[:, 1::2] = Bp >> 4
    for ws2 in (1.0, 0.0125, 0.01, 3.0e-5, 1234.5, 7.0e-3):
        got = oracle.fp4_dequantize(Bp, ws, ws2, N, K, 16, dtype)
        e2 = table[torch.from_numpy(codes)]
        sc = torch.from_numpy(_torch_e4m3(ws)).float()[:, np.arange(K) // 16]
        t = (e2 * sc) * torch.tensor(ws2, dtype=torch.float32)
        ref = t.to(tdt).view(torch.int16).numpy().view(np.uint16)
        assert np.array_equal(got, ref), ws2


def test_dequant_negative_zero_code():
    Bp = np.array([[0x88, 0x08, 0x80]], dtype=np.uint8)
    ws = np.array([[0x38]], dtype=np.uint8)
    for dtype in (oracle.BF16, oracle.FP16):
        out = oracle.fp4_dequantize(Bp, ws, 0.5, 1, 6, 16, dtype)[0]
        sign = 0x8000
        assert [int(x) for x in out] == [sign, sign, sign, 0, 0, sign]


def test_partial_last_block_fp4():
    row = [ln for ln in _golden_lines("hand_cases.txt") if ln[0] == "partial_block_fp4"][0]
    K, bs, S, k0, k1, col = (int(x) for x in row[1:])
    assert wl.scale_cols(K, bs) == S
    Bp = np.full((1, K // 2), 0x22, dtype=np.uint8)  # all 1.0
    ws = np.full((1, S), 0x38, dtype=np.uint8)        # 1.0
    ws[0, col] = 0x40                                  # 2.0 in the last column only
    out = oracle.fp4_dequantize_f64(Bp, ws, 1.0, 1, K, bs)[0]
    assert np.all(out[k0:k1 + 1] == 2.0)
    assert np.all(out[:k0] == 1.0)


def test_partial_last_block_fp8():
    row = [ln for ln in _golden_lines("hand_cases.txt") if ln[0] == "partial_block_fp8"][0]
    K, bs, S, k0, k1, col = (int(x) for x in row[1:])
    assert wl.scale_cols(K, bs) == S
    B = np.full((1, K), 0x38, dtype=np.uint8)  # 1.0
    sc = np.ones((1, S), dtype=np.float32)
    sc[0, col] = 0.375
    out = oracle.fp8_dequantize_f64(B, sc, 1, K, bs)[0]
    assert np.all(out[k0:k1 + 1] == 0.375)
    assert np.all(out[:k0] == 1.0)
    q = oracle.fp8_dequantize(B, sc, 1, K, bs, oracle.BF16)[0]
    assert oracle.act_to_double(int(q[k1]), oracle.BF16) == 0.375


@pytest.mark.parametrize("dtype", [oracle.BF16, oracle.FP16])
def test_fp8_dequant_against_torch(dtype):
    p = wl.make_fp8(1, 64, 1000, 128, dtype, seed=3)
    got = oracle.fp8_dequantize(p.B, p.b_scale, 64, 1000, 128, dtype)
    w = torch.from_numpy(p.B).view(torch.float8_e4m3fn).float()
    sc = torch.from_numpy(p.b_scale)[:, np.arange(1000) // 128]
    tdt = torch.bfloat16 if dtype == oracle.BF16 else torch.float16
    ref = (w * sc).to(tdt).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(got, ref)


# ---------------------------------------------------------------------------
# Matmul reference
# ---------------------------------------------------------------------------

def _hand_matmul(byte, scale_byte, ws2, dtype):
    K = 16
    A = wl.act_bits(np.arange(1, 17, dtype=np.float64).reshape(1, K), dtype)
    Bp = np.full((1, K // 2), byte, dtype=np.uint8)
    ws = np.array([[scale_byte]], dtype=np.uint8)
    Y, S = oracle.fp4_matmul(A, Bp, ws, ws2, None, 1, 1, K, 16, dtype)
    return Y[0, 0], S[0, 0]


@pytest.mark.parametrize("dtype", [oracle.BF16, oracle.FP16])
def test_hand_sums(dtype):
    cases = {ln[0]: ln[1:] for ln in _golden_lines("hand_cases.txt")}
    y, s = _hand_matmul(0x22, 0x38, 1.0, dtype)
    assert y == float(cases["sum16"][0]) and s == 136.0
    y, s = _hand_matmul(0xF9, 0x40, 0.25, dtype)
    assert y == float(cases["mixed16"][0]) and s == 232.0


def test_matmul_matches_torch_float64_library():
    p = wl.make_fp4(5, 48, 320, 32, oracle.BF16, seed=11, bias_sigma=0.5)
    Y, S = oracle.fp4_matmul(p.A, p.B_packed, p.weight_scale, p.weight_scale_2, p.bias,
                             p.M, p.N, p.K, p.block_size, p.dtype)
    W = _lib_fp4_dequant_f64(p.B_packed, p.weight_scale, p.weight_scale_2, p.N, p.K,
                             p.block_size)
    A = torch.from_numpy(p.A.view(np.int16).copy()).view(torch.bfloat16).double().numpy()
    b = torch.from_numpy(p.bias.view(np.int16).copy()).view(torch.bfloat16).double().numpy()
    ref = torch.from_numpy(A) @ torch.from_numpy(W).T + torch.from_numpy(b)
    refS = torch.from_numpy(np.abs(A)) @ torch.from_numpy(np.abs(W)).T
    assert np.allclose(Y, ref.numpy(), rtol=1e-12, atol=1e-12 * refS.numpy().max())
    assert np.allclose(S, refS.numpy(), rtol=1e-12)


def test_fp8_matmul_matches_torch_float64_library():
    p = wl.make_fp8(3, 40, 1000, 128, oracle.FP16, seed=5, bias_sigma=0.1)
    Y, S = oracle.fp8_matmul(p.A, p.B, p.b_scale, p.bias, p.M, p.N, p.K, p.block_size,
                             p.dtype)
    W = (torch.from_numpy(p.B).view(torch.float8_e4m3fn).double()
         * torch.from_numpy(p.b_scale).double()[:, np.arange(p.K) // p.block_size])
    A = torch.from_numpy(p.A.view(np.int16).copy()).view(torch.float16).double()
    b = torch.from_numpy(p.bias.view(np.int16).copy()).view(torch.float16).double()
    ref = A @ W.T + b
    assert np.allclose(Y, ref.numpy(), rtol=1e-12, atol=1e-9)
    assert np.allclose(S, (A.abs() @ W.abs().T).numpy(), rtol=1e-12)


def test_one_hot_probe_every_position():
    """A = e_k for row m gives Y[m, n] = B_dq[n, k] + bias[n] for every n:
    pins operand orientation (no transpose) and the k/n indexing."""
    N, K, bs = 24, 64, 16
    p = wl.make_fp4(1, N, K, bs, oracle.FP16, seed=2, bias_sigma=0.25)
    W = _lib_fp4_dequant_f64(p.B_packed, p.weight_scale, p.weight_scale_2, N, K, bs)
    bias = torch.from_numpy(p.bias.view(np.int16).copy()).view(torch.float16).double().numpy()
    M = 3
    for k in range(K):
        A = np.zeros((M, K), dtype=np.float64)
        A[1, k] = 1.0
        Y, _ = oracle.fp4_matmul(wl.act_bits(A, oracle.FP16), p.B_packed, p.weight_scale,
                                 p.weight_scale_2, p.bias, M, N, K, bs, oracle.FP16)
        assert np.array_equal(Y[1], W[:, k] + bias)
        assert np.array_equal(Y[0], bias) and np.array_equal(Y[2], bias)


def test_k_permutation_invariance():
    """Permuting K identically on A and on the weight (whole scale blocks moved
    together, plus a permutation inside each block that keeps byte pairs)
    leaves the float64 reference unchanged (FP4 page §4: K is a reduction axis)."""
    M, N, K, bs = 3, 16, 128, 16
    p = wl.make_fp4(M, N, K, bs, oracle.BF16, seed=9)
    Y, S = oracle.fp4_matmul(p.A, p.B_packed, p.weight_scale, p.weight_scale_2, None,
                             M, N, K, bs, p.dtype)
    r = np.random.Generator(np.random.PCG64(4))
    nb = K // bs
    bperm = r.permutation(nb)
    inner = r.permutation(bs // 2)  # permutation of byte pairs inside a block
    kperm = np.concatenate([b * bs + np.stack([2 * inner, 2 * inner + 1], 1).ravel()
                            for b in bperm])
    bytes_perm = kperm[0::2] // 2
    A2 = p.A[:, kperm]
    B2 = p.B_packed[:, bytes_perm]
    ws2_ = p.weight_scale[:, bperm]
    Y2, S2 = oracle.fp4_matmul(A2, B2, ws2_, p.weight_scale_2, None, M, N, K, bs, p.dtype)
    assert np.allclose(Y2, Y, rtol=0, atol=1e-12 * S.max())
    assert np.allclose(S2, S, rtol=1e-12)


def test_sampled_equals_full():
    p = wl.make_fp4(6, 40, 96, 16, oracle.BF16, seed=8, bias_sigma=0.1)
    Y, S = oracle.fp4_matmul(p.A, p.B_packed, p.weight_scale, p.weight_scale_2, p.bias,
                             p.M, p.N, p.K, 16, p.dtype)
    ms = np.array([0, 5, 3, 2, 5], dtype=np.int64)
    ns = np.array([0, 39, 17, 1, 0], dtype=np.int64)
    y, s = oracle.fp4_matmul_sampled(p.A, p.B_packed, p.weight_scale, p.weight_scale_2,
                                     p.bias, p.K, 16, p.dtype, ms, ns)
    assert np.array_equal(y, Y[ms, ns]) and np.array_equal(s, S[ms, ns])
    q = wl.make_fp8(4, 20, 300, 128, oracle.FP16, seed=8)
    Y, S = oracle.fp8_matmul(q.A, q.B, q.b_scale, None, q.M, q.N, q.K, 128, q.dtype)
    y, s = oracle.fp8_matmul_sampled(q.A, q.B, q.b_scale, None, q.K, 128, q.dtype,
                                     ms % 4, ns % 20)
    assert np.array_equal(y, Y[ms % 4, ns % 20])


def test_threads_do_not_change_results():
    p = wl.make_fp4(2, 33, 64, 16, oracle.BF16, seed=1)
    a = oracle.fp4_matmul(p.A, p.B_packed, p.weight_scale, p.weight_scale_2, None,
                          2, 33, 64, 16, p.dtype, threads=1)
    b = oracle.fp4_matmul(p.A, p.B_packed, p.weight_scale, p.weight_scale_2, None,
                          2, 33, 64, 16, p.dtype, threads=5)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])
    d1 = oracle.fp4_dequantize(p.B_packed, p.weight_scale, 0.3, 33, 64, 16, 1, threads=1)
    d2 = oracle.fp4_dequantize(p.B_packed, p.weight_scale, 0.3, 33, 64, 16, 1, threads=7)
    assert np.array_equal(d1, d2)


def test_pins_catch_a_planted_nibble_swap():
    """A mistake planted on the CPU side (nibbles swapped in the input) must
    change the one-hot result: the pins above are sensitive to nibble order."""
    N, K = 4, 32
    p = wl.make_fp4(1, N, K, 16, oracle.FP16, seed=21)
    swapped = ((p.B_packed & 0xF) << 4) | (p.B_packed >> 4)
    assert not np.array_equal(swapped, p.B_packed)
    a = oracle.fp4_dequantize_f64(p.B_packed, p.weight_scale, 1.0, N, K, 16)
    b = oracle.fp4_dequantize_f64(swapped.astype(np.uint8), p.weight_scale, 1.0, N, K, 16)
    ref = _lib_fp4_dequant_f64(p.B_packed, p.weight_scale, 1.0, N, K, 16)
    assert np.array_equal(a, ref) and not np.array_equal(b, ref)


def test_tolerance_formula():
    S = np.array([0.0, 1.0, 100.0])
    assert np.allclose(oracle.tolerance(S, oracle.BF16), [1e-3, 9e-3, 0.801])
    assert np.allclose(oracle.tolerance(S, oracle.FP16), [1e-4, 2.1e-3, 0.2001])


# --- W8A8 activation path (FP8 page §6: A_deq = fp8_e4m3(A / a_scale) * a_scale) ---

def test_e4m3_encode_roundtrip_every_code():
    """Every finite E4M3FN value encodes back to its own code (+-0 keep their sign)."""
    for c in list(range(0x00, 0x7F)) + list(range(0x80, 0xFF)):
        v = np.float32(oracle.e4m3_value(c))
        assert oracle.e4m3_from_f32(v) == c, hex(c)


def test_e4m3_encode_ties_to_even_and_nearest():
    """Midpoints between neighbouring codes go to the even code; a hair off a
    midpoint goes to the nearer one (all 126 positive gaps, and negated)."""
    for c in range(0x00, 0x7E):
        lo, hi = oracle.e4m3_value(c), oracle.e4m3_value(c + 1)
        mid = np.float32((lo + hi) / 2)      # exact: one bit more than the codes
        assert float(mid) == (lo + hi) / 2
        even = c if c % 2 == 0 else c + 1
        assert oracle.e4m3_from_f32(mid) == even, hex(c)
        assert oracle.e4m3_from_f32(-mid) == 0x80 | even, hex(c)
        below = np.nextafter(mid, np.float32(-np.inf))
        above = np.nextafter(mid, np.float32(np.inf))
        assert oracle.e4m3_from_f32(below) == c, hex(c)
        assert oracle.e4m3_from_f32(above) == c + 1, hex(c)


def test_e4m3_encode_saturation_and_nan():
    for v in (448.0, 449.0, 464.0, 480.0, 1e30, np.inf):
        assert oracle.e4m3_from_f32(v) == 0x7E
        assert oracle.e4m3_from_f32(-v) == 0xFE
    assert oracle.e4m3_from_f32(np.nan) & 0x7F == 0x7F
    assert oracle.e4m3_from_f32(2.0 ** -10) == 0x00        # half the smallest subnormal: tie -> 0
    assert oracle.e4m3_from_f32(1.5 * 2.0 ** -10) == 0x01  # nearer to 2^-9


def test_e4m3_encode_matches_torch_in_range():
    """Library cross-check: torch's float32 -> float8_e4m3fn conversion (its
    own implementation, round to nearest even) agrees on in-range values."""
    torch = pytest.importorskip("torch")
    r = np.random.Generator(np.random.PCG64(12))
    v = np.concatenate([r.uniform(-448, 448, 20000), r.normal(0, 1, 20000),
                        r.normal(0, 1e-2, 5000)]).astype(np.float32)
    t = torch.from_numpy(v).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    o = np.array([oracle.e4m3_from_f32(x) for x in v], dtype=np.uint8)
    assert np.array_equal(t, o)


def test_fp8_qdq_activation_hand_cases():
    """Hand-computed W8A8 activation rounding (a_scale = 2): 6.5 / 2 = 3.25 is
    an E4M3 value; 6.75 / 2 = 3.375 is the midpoint of 3.25 and 3.5 and goes
    to the even mantissa 3.5 -> 7.0; 1000 / 2 saturates at 448 -> 896; 0 stays."""
    for dtype in (oracle.BF16, oracle.FP16):
        A = wl.act_bits(np.array([6.5, 6.75, -6.75, 1000.0, 0.0]), dtype)
        out = oracle.fp8_qdq_activation(A, 2.0, dtype)
        got = [oracle.act_to_double(int(b), dtype) for b in out]
        assert got == [6.5, 7.0, -7.0, 896.0, 0.0], (dtype, got)


# --- NVFP4 activation quantization (FP4 page §6, step 1 of the native path) ---

def _nvfp4_golden_cases():
    cases, cur = {}, None
    for ln in _golden_lines("nvfp4_activation.txt"):
        if ln[0] == "case":
            cur = cases.setdefault(ln[1], {})
        elif ln[0] in ("x", "qdq"):
            cur[ln[0]] = [float(v) for v in ln[1:]]
        elif ln[0] == "scale":
            cur["scale"] = int(ln[1], 16)
        elif ln[0] == "packed":
            cur["packed"] = [int(v, 16) for v in ln[1:]]
    return cases


@pytest.mark.parametrize("dtype", [oracle.BF16, oracle.FP16])
def test_nvfp4_activation_golden_blocks(dtype):
    for name, c in _nvfp4_golden_cases().items():
        A = wl.act_bits(np.array([c["x"]]), dtype)
        codes, scales = oracle.nvfp4_quantize_activation(A, dtype)
        assert scales.tolist() == [[c["scale"]]], name
        assert codes.tolist() == [c["packed"]], name
        q = oracle.nvfp4_qdq_activation(A, dtype)
        got = [oracle.act_to_double(int(b), dtype) for b in q[0]]
        assert got == c["qdq"], name
        # signs of zeros as listed
        assert [math.copysign(1, g) for g in got] == [math.copysign(1, v) for v in c["qdq"]], name


def test_e2m1_encode_roundtrip_every_code():
    """Every E2M1 value encodes back to its own code (-0.0 keeps its sign)."""
    table = _e2m1_golden()
    for c in range(16):
        assert oracle.e2m1_from_f32(np.float32(table[c])) == c or (c == 0 and table[c] == 0.0)
    assert oracle.e2m1_from_f32(np.float32(-0.0)) == 0x8


def test_e2m1_encode_ties_nearest_and_saturation():
    """Midpoints of neighbouring magnitudes go to the even code; a hair off
    goes to the nearer one; beyond 6 saturates; signs mirror."""
    table = _e2m1_golden()
    for c in range(7):
        lo, hi = table[c], table[c + 1]
        mid = np.float32((lo + hi) / 2)
        even = c if c % 2 == 0 else c + 1
        assert oracle.e2m1_from_f32(mid) == even, c
        assert oracle.e2m1_from_f32(-mid) == 0x8 | even, c
        assert oracle.e2m1_from_f32(np.nextafter(mid, np.float32(-1))) == c, c
        assert oracle.e2m1_from_f32(np.nextafter(mid, np.float32(10))) == c + 1, c
    for v in (6.0, 6.5, 7.0, 100.0, 1e30):
        assert oracle.e2m1_from_f32(v) == 7
        assert oracle.e2m1_from_f32(-v) == 15


@pytest.mark.parametrize("dtype", [oracle.BF16, oracle.FP16])
def test_nvfp4_activation_exact_grid_round_trip(dtype):
    """Blocks built from E2M1 values times 2^e with a +-6 entry (so amax/6 is
    exactly 2^e, an E4M3 value) quantize to exactly those codes and scales:
    pins the amax/6 rule, the division, the sign and the nibble order."""
    r = np.random.Generator(np.random.PCG64(31))
    table = np.array([_e2m1_golden()[c] for c in range(16)])
    M, K = 6, 64
    for e in (-6, -2, 0, 3, 6):
        codes = r.integers(0, 16, (M, K))
        codes[:, ::16] = r.choice([7, 15], (M, K // 16))  # every block reaches |6|
        x = table[codes] * 2.0 ** e
        A = wl.act_bits(x, dtype)
        pc, sc = oracle.nvfp4_quantize_activation(A, dtype)
        want_scale = oracle.e4m3_from_f32(2.0 ** e)
        assert (sc == want_scale).all(), e
        assert oracle.e4m3_value(want_scale) == 2.0 ** e
        assert np.array_equal(pc & 0xF, codes[:, 0::2]), e
        assert np.array_equal(pc >> 4, codes[:, 1::2]), e
        q = oracle.nvfp4_qdq_activation(A, dtype)
        assert np.array_equal(q, A), e  # the grid values come back unchanged


@pytest.mark.parametrize("dtype", [oracle.BF16, oracle.FP16])
def test_nvfp4_activation_error_bound_and_consistency(dtype):
    """Random activations (three magnitudes, the smallest one reaching
    subnormal E4M3 scales): an element within 6 scales is off by at most
    half the local E2M1 gap times the scale (gaps 0.5 below 2, 1 up to 4, 2
    up to 6); one beyond is exactly +-6 scales; with a normal E4M3 scale no
    element is beyond 6 * (1 + 2^-4) scales (amax / 6 rounds within 2^-4).
    qdq equals e2m1(code) * e4m3(scale) read back from the packed codes."""
    r = np.random.Generator(np.random.PCG64(5))
    M, K = 8, 400  # 25 blocks per row
    table = np.array([_e2m1_golden()[c] for c in range(16)])
    for sigma in (1.0, 30.0, 1e-2):
        A = wl.act_bits(r.normal(0, sigma, (M, K)), dtype)
        x = np.array([[oracle.act_to_double(int(b), dtype) for b in row] for row in A])
        pc, sc = oracle.nvfp4_quantize_activation(A, dtype)
        q = oracle.nvfp4_qdq_activation(A, dtype)
        qv = np.array([[oracle.act_to_double(int(b), dtype) for b in row] for row in q])
        sd = np.repeat(np.array([[oracle.e4m3_value(int(b)) for b in row] for row in sc]), 16,
                       axis=1)[:, :K]
        normal = np.repeat((sc & 0x78) != 0, 16, axis=1)[:, :K]
        u = np.abs(x) / sd
        inside = u <= 6.0
        half_gap = np.where(u < 2, 0.25, np.where(u < 4, 0.5, 1.0))
        assert np.all(np.abs(qv - x)[inside] <= (half_gap * sd)[inside]), sigma
        assert np.array_equal(qv[~inside], (np.sign(x) * 6 * sd)[~inside]), sigma
        assert np.all(u[normal] <= 6 * (1 + 2.0 ** -4)), sigma
        codes = np.empty((M, K), dtype=np.int64)
        codes[:, 0::2] = pc & 0xF
        codes[:, 1::2] = pc >> 4
        assert np.array_equal(qv, table[codes] * sd), sigma


def test_nvfp4_activation_partial_last_block():
    """K = 40: the last block has 8 elements and takes its amax over those
    only (a large value in the first block does not reach it)."""
    x = np.zeros((1, 40))
    x[0, :16] = 100.0
    x[0, 32:40] = [6.0, 3.0, -1.5, 0.5, 0.0, 2.0, -4.0, 1.0]  # amax 6 -> scale 1.0
    A = wl.act_bits(x, oracle.BF16)
    pc, sc = oracle.nvfp4_quantize_activation(A, oracle.BF16)
    assert sc.shape == (1, 3)
    assert sc[0, 2] == 0x38 and sc[0, 1] == 0x00
    # codes 7 5 11 1 0 4 14 2 -> bytes (even k low) 0x57 0x1B 0x40 0x2E
    assert pc[0, 16:20].tolist() == [0x57, 0x1B, 0x40, 0x2E]
