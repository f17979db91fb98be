"""Seeded synthetic inputs for the block-quantized weight-only matmul.

This module is shared by the tests, the smoke check and the benchmark.  It
holds no arithmetic of the method: it draws random bytes and random reals and
rounds reals to storage types with library casts (torch dtype conversion).
Both the CUDA path and the CPU oracle receive exactly the arrays made here.

Recipe (one independent PCG64 stream per tensor: seed and a tensor tag):

* activations A, bias: float64 normal draws N(0, sigma), cast to the
  activation type by torch (round to nearest even);
* NVFP4 codes: uniform random bytes, i.e. both nibbles uniform over all 16
  E2M1 codes (including 0x8, negative zero);
* E4M3 block scales: a real drawn uniform in [lo, hi] (or log-uniform:
  2^U[log2 lo, log2 hi]), rounded to float8_e4m3fn by torch, stored as bytes;
* FP8 weight: uniform over the 254 finite E4M3 bytes (0x7F and 0xFF excluded);
* FP8 block scales: float32 uniform in [lo, hi].

Shapes follow the pages' 27B-class layer shapes (hidden 5120, MLP 17408,
vocabulary 152064) and their decode (M <= 8) and 8K-token prefill workloads.
"""

from __future__ import annotations

import dataclasses
import math
from typing import Optional

import numpy as np
import torch

FP16 = 0
BF16 = 1

TAG_A, TAG_B, TAG_SCALE, TAG_BIAS, TAG_W8, TAG_BSCALE = 1, 2, 3, 4, 5, 6


def _rng(seed: int, tag: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64([int(seed), int(tag)]))


def act_bits(x: np.ndarray, dtype: int) -> np.ndarray:
    """float64 array -> uint16 bit patterns of the activation type (torch cast)."""
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32))
    t = t.to(torch.bfloat16 if dtype == BF16 else torch.float16)
    return t.view(torch.int16).numpy().view(np.uint16).copy()


def gen_activation(M: int, K: int, dtype: int, seed: int = 0, sigma: float = 1.0,
                   tag: int = TAG_A) -> np.ndarray:
    x = _rng(seed, tag).standard_normal((M, K), dtype=np.float32) * np.float32(sigma)
    return act_bits(x, dtype)


def gen_bias(N: int, dtype: int, sigma: float, seed: int = 0) -> np.ndarray:
    x = _rng(seed, TAG_BIAS).standard_normal(N, dtype=np.float32) * np.float32(sigma)
    return act_bits(x, dtype)


def gen_fp4_packed(N: int, K: int, seed: int = 0) -> np.ndarray:
    """[N, K/2] uint8; each byte holds two uniform 4-bit E2M1 codes."""
    assert K % 2 == 0
    return _rng(seed, TAG_B).integers(0, 256, size=(N, K // 2), dtype=np.uint8)


def e4m3_bytes(x: np.ndarray) -> np.ndarray:
    """Round reals to float8_e4m3fn with torch and return the raw bytes."""
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32))
    return t.to(torch.float8_e4m3fn).view(torch.uint8).numpy().copy()


def gen_e4m3_scales(N: int, S: int, lo: float, hi: float, log_uniform: bool = False,
                    seed: int = 0) -> np.ndarray:
    r = _rng(seed, TAG_SCALE)
    if log_uniform:
        x = np.exp2(r.uniform(math.log2(lo), math.log2(hi), size=(N, S)))
    else:
        x = r.uniform(lo, hi, size=(N, S))
    return e4m3_bytes(x.astype(np.float32))


def gen_fp8_weight(N: int, K: int, seed: int = 0) -> np.ndarray:
    """[N, K] uint8 uniform over the 254 finite E4M3FN bytes."""
    r = _rng(seed, TAG_W8).integers(0, 254, size=(N, K), dtype=np.int32)
    r = np.where(r >= 0x7F, r + 1, r)  # skip 0x7F; 254 -> 255 never happens
    return r.astype(np.uint8)


def gen_fp8_scale(N: int, S: int, lo: float, hi: float, seed: int = 0) -> np.ndarray:
    return _rng(seed, TAG_BSCALE).uniform(lo, hi, size=(N, S)).astype(np.float32)


def scale_cols(K: int, block_size: int) -> int:
    return (K + block_size - 1) // block_size


@dataclasses.dataclass
class Fp4Problem:
    M: int
    N: int
    K: int
    block_size: int
    dtype: int
    A: np.ndarray            # uint16 [M, K]
    B_packed: np.ndarray     # uint8 [N, K/2]
    weight_scale: np.ndarray  # uint8 [N, S]
    weight_scale_2: float    # float32 value
    bias: Optional[np.ndarray]  # uint16 [N] or None


@dataclasses.dataclass
class Fp8Problem:
    M: int
    N: int
    K: int
    block_size: int
    dtype: int
    A: np.ndarray        # uint16 [M, K]
    B: np.ndarray        # uint8 [N, K]
    b_scale: np.ndarray  # float32 [N, S]
    bias: Optional[np.ndarray]


def make_fp4(M, N, K, block_size=16, dtype=BF16, seed=0, scale_lo=2.0 ** -4,
             scale_hi=4.0, log_uniform=False, ws2=0.0125, bias_sigma=None,
             a_sigma=1.0) -> Fp4Problem:
    S = scale_cols(K, block_size)
    return Fp4Problem(
        M=M, N=N, K=K, block_size=block_size, dtype=dtype,
        A=gen_activation(M, K, dtype, seed, a_sigma),
        B_packed=gen_fp4_packed(N, K, seed),
        weight_scale=gen_e4m3_scales(N, S, scale_lo, scale_hi, log_uniform, seed),
        weight_scale_2=float(np.float32(ws2)),
        bias=None if bias_sigma is None else gen_bias(N, dtype, bias_sigma, seed),
    )


def make_fp8(M, N, K, block_size=128, dtype=BF16, seed=0, scale_lo=0.001,
             scale_hi=0.02, bias_sigma=None, a_sigma=1.0) -> Fp8Problem:
    S = scale_cols(K, block_size)
    return Fp8Problem(
        M=M, N=N, K=K, block_size=block_size, dtype=dtype,
        A=gen_activation(M, K, dtype, seed, a_sigma),
        B=gen_fp8_weight(N, K, seed),
        b_scale=gen_fp8_scale(N, S, scale_lo, scale_hi, seed),
        bias=None if bias_sigma is None else gen_bias(N, dtype, bias_sigma, seed),
    )


# The five workloads.  Names say what each one is.
def parity_small(seed=0) -> Fp4Problem:
    """NVFP4, M=1, N=256, K=512, bs=16, FP16, scales U[2^-4, 4], ws2=0.0125, bias N(0,0.1)."""
    return make_fp4(1, 256, 512, 16, FP16, seed, ws2=0.0125, bias_sigma=0.1)


def decode_gemv(M=4, seed=0) -> Fp4Problem:
    """NVFP4 decode GEMV (MTP verify), N=K=5120, bs=16, BF16, no bias."""
    return make_fp4(M, 5120, 5120, 16, BF16, seed, ws2=0.0125)


def lm_head(M=4, seed=0) -> Fp4Problem:
    """NVFP4 lm_head GEMV, N=152064, K=5120, scales log-uniform [2^-6, 4], ws2=0.01, bias N(0,0.02)."""
    return make_fp4(M, 152064, 5120, 16, BF16, seed, scale_lo=2.0 ** -6,
                    log_uniform=True, ws2=0.01, bias_sigma=0.02)


def prefill(shape="gate_up", M=8192, seed=0) -> Fp4Problem:
    """NVFP4 prefill GEMM, M=8192; gate/up N=17408 K=5120, down N=5120 K=17408; bias N(0,0.02)."""
    N, K = (17408, 5120) if shape == "gate_up" else (5120, 17408)
    return make_fp4(M, N, K, 16, BF16, seed, ws2=0.0125, bias_sigma=0.02)


def fp8_problem(M, N=5120, K=5120, seed=0, bias_sigma=None) -> Fp8Problem:
    """FP8 E4M3 weight-only, bs=128, b_scale U[0.001, 0.02], BF16."""
    return make_fp8(M, N, K, 128, BF16, seed, bias_sigma=bias_sigma)
