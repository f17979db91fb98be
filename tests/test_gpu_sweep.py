"""Seeded randomized sweep over the dispatch paths of the matmul entry points,
against the oracle within the matmul bound.

Each case draws its shape inside a family chosen to land on one path -- the
TMA decode GEMV (up to 32 rows), the register-fed and the general GEMV, the
narrow-tile GEMM (light CTAs or a cluster K split), the persistent 256-token
GEMM, the FP8 paths, the W8A8 workspace path and the FP4 x FP4 GEMM -- with
ragged sizes, block sizes, both activation types and optional bias.  Seven
seeds draw 33 shapes each; the shapes are fixed by the seed, so a failure
reproduces (the seed is part of the test id)."""

import numpy as np
import pytest
import torch

import fp8_weight_only_nvfp4_gb300 as wq
import oracle
import workloads as wl
from gpu_util import (DEV, act_to_dev, assert_within_tolerance, f32_to_dev, fp8_dev, run_fp4,
                      run_fp8, u8_to_dev)

pytestmark = pytest.mark.gpu


def _families(seed=2024):
    r = np.random.Generator(np.random.PCG64(seed))
    cases = []

    def add(kind, M, N, K, bs):
        cases.append((kind, int(M), int(N), int(K), int(bs), int(r.integers(0, 2)),
                      bool(r.integers(0, 2)), int(r.integers(0, 1 << 20)), seed))
    for _ in range(5):   # TMA decode GEMV: M <= 32, bs 16, K % 256 == 0
        add("fp4", r.integers(1, 33), r.integers(1, 700), 256 * r.integers(1, 9), 16)
    for _ in range(4):   # register-fed GEMV: other power-of-two blocks
        add("fp4", r.integers(1, 9), r.integers(1, 600), 32 * r.integers(1, 40),
            r.choice([32, 64, 128]))
    for _ in range(3):   # general GEMV: K not a multiple of 32
        add("fp4", r.integers(1, 9), r.integers(1, 300), 2 * r.integers(1, 400) + 0, 16)
    for _ in range(5):   # narrow-tile GEMM: 33..300 rows, light CTAs or a K split
        add("fp4", r.integers(33, 301), r.integers(64, 3000), 32 * r.integers(2, 60),
            r.choice([16, 32, 64]))
    for _ in range(3):   # persistent 256-token GEMM: enough tiles to fill the GPU
        add("fp4", r.integers(257, 700), r.integers(12000, 24000), 32 * r.integers(1, 6), 16)
    for _ in range(4):   # FP8: GEMV and GEMM, any K, blocks multiple of 16
        add("fp8", r.choice([r.integers(1, 9), r.integers(9, 400)]), r.integers(1, 1500),
            r.integers(16, 3000), r.choice([16, 64, 128]))
    for _ in range(2):   # FP8 persistent GEMM
        add("fp8", r.integers(300, 600), r.integers(12000, 20000), 16 * r.integers(2, 10), 128)
    for _ in range(3):   # W8A8 with a workspace
        add("w8a8", r.integers(1, 400), r.integers(1, 1200), 16 * r.integers(1, 120), 128)
    for _ in range(4):   # FP4 x FP4
        add("f4f4", r.integers(1, 700), r.integers(1, 3000), 256 * r.integers(1, 7), 16)
    return cases


SEEDS = range(2024, 2031)
CASES = [c for s in SEEDS for c in _families(s)]


def _id(c):
    kind, M, N, K, bs, dt, bias, seed, family_seed = c
    return (f"s{family_seed}-{kind}-M{M}-N{N}-K{K}-bs{bs}-{'bf16' if dt else 'fp16'}"
            f"{'-bias' if bias else ''}")


@pytest.mark.parametrize("case", CASES, ids=[_id(c) for c in CASES])
def test_sweep(case):
    kind, M, N, K, bs, dt, bias, seed, _ = case
    dtype = oracle.BF16 if dt else oracle.FP16
    sigma = 0.05 if bias else None
    if kind == "fp4":
        p = wl.make_fp4(M, N, K, bs, dtype, seed=seed, bias_sigma=sigma)
        Yr, S = oracle.fp4_matmul(p.A, p.B_packed, p.weight_scale, p.weight_scale_2, p.bias,
                                  M, N, K, bs, dtype)
        assert_within_tolerance(run_fp4(p), Yr, S, dtype, _id(case))
    elif kind == "fp8":
        p = wl.make_fp8(M, N, K, bs, dtype, seed=seed, bias_sigma=sigma)
        Yr, S = oracle.fp8_matmul(p.A, p.B, p.b_scale, p.bias, M, N, K, bs, dtype)
        assert_within_tolerance(run_fp8(p), Yr, S, dtype, _id(case))
    elif kind == "w8a8":
        p = wl.make_fp8(M, N, K, bs, dtype, seed=seed, bias_sigma=sigma)
        a_scale = 0.0213
        d = fp8_dev(p)
        ws = torch.empty(max(1, wq.fp8_w8a8_workspace_bytes(M, K)), dtype=torch.uint8,
                         device=DEV)
        Y = wq.fp8_weight_matmul_w8a8_ws(d["A"], f32_to_dev(np.array([a_scale], np.float32)),
                                         d["B"], d["s"], ws, d["bias"], block_size=bs)
        torch.cuda.synchronize()
        assert wq.device_status() == 0
        Aq = oracle.fp8_qdq_activation(p.A, a_scale, dtype)
        Yr, S = oracle.fp8_matmul(Aq, p.B, p.b_scale, p.bias, M, N, K, bs, dtype)
        assert_within_tolerance(Y, Yr, S, dtype, _id(case))
    else:
        w = wl.make_fp4(1, N, K, 16, dtype, seed=seed, bias_sigma=sigma)
        a = wl.make_fp4(1, M, K, 16, dtype, seed=seed + 1)
        Y = wq.fp4_fp4_matmul(u8_to_dev(a.B_packed), u8_to_dev(a.weight_scale),
                              u8_to_dev(w.B_packed), u8_to_dev(w.weight_scale),
                              f32_to_dev(np.array([w.weight_scale_2], np.float32)),
                              act_to_dev(w.bias, dtype) if w.bias is not None else None,
                              dtype=torch.bfloat16 if dt else torch.float16)
        torch.cuda.synchronize()
        assert wq.device_status() == 0
        Ad = oracle.fp4_dequantize(a.B_packed, a.weight_scale, 1.0, M, K, 16, dtype)
        Yr, S = oracle.fp4_matmul(Ad, w.B_packed, w.weight_scale, w.weight_scale_2, w.bias,
                                  M, N, K, 16, dtype)
        assert_within_tolerance(Y, Yr, S, dtype, _id(case))
