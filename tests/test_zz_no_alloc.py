"""fp8_weight_matmul_w8a8_noalloc on the GPU, through the C-ABI: the W8A8
matmul with its scratch in the library's fixed array agrees with
fp8_weight_matmul_w8a8_ws (caller-owned workspace) on two calls in a row,
and the calls allocate no device memory.  Kept in a file of its own that is
collected last, so it runs both in a fresh process and after the other
tests."""

import ctypes

import numpy as np
import pytest
import torch

import fp8_weight_only_nvfp4_gb300 as wq
import oracle
import workloads as wl
from gpu_util import DEV, assert_within_tolerance, fp8_dev

pytestmark = pytest.mark.gpu


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _noalloc(d, a_scale, Y, M, N, K, bs, dtype):
    """One call of the C entry point on torch's current stream."""
    st = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return wq.lib().fp8_weight_matmul_w8a8_noalloc(
        _ptr(d["A"]), _ptr(a_scale), _ptr(d["B"]), _ptr(d["s"]), _ptr(d["bias"]), _ptr(Y),
        M, N, K, bs, dtype, st)


def _with_workspace(d, a_scale, M, K, bs):
    ws = torch.empty(wq.fp8_w8a8_workspace_bytes(M, K), dtype=torch.uint8, device=DEV)
    return wq.fp8_weight_matmul_w8a8_ws(d["A"], a_scale, d["B"], d["s"], ws, d["bias"],
                                        block_size=bs)


def _case(M, N, K, bs, dtype, seed, a_scale):
    p = wl.make_fp8(M, N, K, bs, dtype, seed=seed, bias_sigma=0.1 if seed % 2 else None)
    sc = torch.full((1,), a_scale, dtype=torch.float32, device=DEV)
    Y = torch.empty(M, N, dtype=torch.bfloat16 if dtype == oracle.BF16 else torch.float16,
                    device=DEV)
    return p, fp8_dev(p), sc, Y


# Two problems issued back to back on one stream (the second overwrites the
# scratch the first one used), then one at the exact size limit
# (2 * M * K == 16 MiB) next to a ragged one.
PAIRS = [
    [(640, 384, 4096, 128, oracle.BF16, 11, 0.02), (97, 200, 1000, 64, oracle.FP16, 12, 0.0213)],
    [(2048, 128, 4096, 128, oracle.BF16, 13, 0.05), (300, 64, 5120, 128, oracle.BF16, 14, 0.01)],
]


@pytest.mark.parametrize("pair", PAIRS, ids=["two_shapes", "at_limit"])
def test_noalloc_matches_workspace_entry_point(pair):
    cases = [_case(*c) for c in pair]
    torch.cuda.synchronize()
    free0 = torch.cuda.mem_get_info()[0]
    for (p, d, sc, Y) in cases:
        assert _noalloc(d, sc, Y, p.M, p.N, p.K, p.block_size, p.dtype) == 0
    torch.cuda.synchronize()
    assert wq.device_status() == 0
    # Repeat the pair: the free device memory must not move (nothing is
    # allocated per call) and the results must repeat exactly.
    first = [Y.clone() for (_, _, _, Y) in cases]
    torch.cuda.synchronize()
    free1 = torch.cuda.mem_get_info()[0]
    for (p, d, sc, Y) in cases:
        assert _noalloc(d, sc, Y, p.M, p.N, p.K, p.block_size, p.dtype) == 0
    torch.cuda.synchronize()
    assert torch.cuda.mem_get_info()[0] == free1
    assert free1 <= free0
    assert wq.device_status() == 0
    for (p, d, sc, Y), Y1 in zip(cases, first):
        assert torch.equal(Y.view(torch.int16), Y1.view(torch.int16))
        ref = _with_workspace(d, sc, p.M, p.K, p.block_size)
        torch.cuda.synchronize()
        # Within the matmul tolerance of the existing entry point's output
        # (S from the oracle's A_deq and weights) ...
        Aq = oracle.fp8_qdq_activation(p.A, float(sc.item()), p.dtype)
        _, S = oracle.fp8_matmul(Aq, p.B, p.b_scale, p.bias, p.M, p.N, p.K, p.block_size,
                                 p.dtype)
        assert_within_tolerance(Y, ref.double().cpu().numpy(), S, p.dtype,
                                f"noalloc {p.M}x{p.N}x{p.K}")
        # ... and, being the same two launches on the same values, equal to it.
        assert torch.equal(Y.view(torch.int16), ref.view(torch.int16))


def test_noalloc_small_m_and_limit():
    """Up to 8 rows no scratch is used (same result as the fused GEMV); one row
    past the limit is refused with WQMM_ERR_UNSUPPORTED and Y is untouched."""
    p, d, sc, Y = _case(6, 256, 2048, 128, oracle.BF16, 15, 0.05)
    assert _noalloc(d, sc, Y, p.M, p.N, p.K, p.block_size, p.dtype) == 0
    ref = wq.fp8_weight_matmul_w8a8(d["A"], sc, d["B"], d["s"], d["bias"], block_size=128)
    torch.cuda.synchronize()
    assert torch.equal(Y.view(torch.int16), ref.view(torch.int16))
    K = 4096
    M = wq.NOALLOC_SCRATCH_BYTES // (2 * K) + 1
    A = torch.zeros(M, K, dtype=torch.bfloat16, device=DEV)
    B = torch.zeros(64, K, dtype=torch.uint8, device=DEV)
    s = torch.ones(64, K // 128, dtype=torch.float32, device=DEV)
    Yb = torch.full((M, 64), 7.0, dtype=torch.bfloat16, device=DEV)
    big = {"A": A, "B": B, "s": s, "bias": None}
    assert _noalloc(big, sc, Yb, M, 64, K, 128, oracle.BF16) == 2
    torch.cuda.synchronize()
    assert bool((Yb == 7.0).all())
