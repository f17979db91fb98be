"""Standalone dequantize: GPU output must be bit-exact to the oracle
(NVFP4: fp32(e2m1 * e4m3) * weight_scale_2 in fp32, RNE to the activation
type; FP8: fp32(e4m3 * b_scale), RNE)."""

import numpy as np
import pytest
import torch

import fp8_weight_only_nvfp4_gb300 as wq
import oracle
import workloads as wl
from gpu_util import bits_of, f32_to_dev, tdt, u8_to_dev, DEV

pytestmark = pytest.mark.gpu


def _fp4(N, K, bs, dtype, seed=0, log_uniform=False, lo=2.0 ** -4, hi=4.0, ws2=0.0125):
    Bp = wl.gen_fp4_packed(N, K, seed)
    ws = wl.gen_e4m3_scales(N, wl.scale_cols(K, bs), lo, hi, log_uniform, seed)
    return Bp, ws, float(np.float32(ws2))


def _check_fp4(Bp, ws, ws2, N, K, bs, dtype):
    out = wq.fp4_dequantize(u8_to_dev(Bp), u8_to_dev(ws),
                            torch.tensor([ws2], dtype=torch.float32, device=DEV),
                            block_size=bs, dtype=tdt(dtype))
    torch.cuda.synchronize()
    got = bits_of(out)
    want = oracle.fp4_dequantize(Bp, ws, ws2, N, K, bs, dtype)
    nan_w = np.isnan(torch.from_numpy(want.view(np.int16)).view(tdt(dtype)).float().numpy())
    nan_g = np.isnan(torch.from_numpy(got.view(np.int16)).view(tdt(dtype)).float().numpy())
    assert np.array_equal(nan_w, nan_g)
    diff = (got != want) & ~nan_w
    assert not diff.any(), f"{diff.sum()} mismatches, first at {np.argwhere(diff)[:3].tolist()}"


@pytest.mark.parametrize("dtype", [oracle.BF16, oracle.FP16])
def test_all_bytes_and_scales(dtype):
    """Every packed byte against every finite scale byte class (incl. subnormal
    scales, negative scales and the NaN bytes), several global scales."""
    sbytes = np.array(list(range(0, 256, 3)) + [0x7F, 0xFF, 0x7E, 0x01], dtype=np.uint8)
    N = sbytes.size
    K = 512
    Bp = np.tile(np.arange(256, dtype=np.uint8), (N, 1))
    ws = np.repeat(sbytes.reshape(N, 1), K // 16, axis=1)
    for ws2 in (1.0, 0.0125, 3.0e-5, 1234.5):
        _check_fp4(Bp, ws, float(np.float32(ws2)), N, K, 16, dtype)


@pytest.mark.parametrize("dtype", [oracle.BF16, oracle.FP16])
@pytest.mark.parametrize("N,K,bs", [
    (256, 512, 16), (257, 5120, 16), (64, 1024, 32), (33, 96, 48), (17, 40, 16),
    (5, 42, 16), (9, 6, 16), (31, 2, 16), (12, 128, 7), (7, 60, 15), (3, 34, 1), (128, 4096, 64),
])
def test_shapes_and_block_sizes(N, K, bs, dtype):
    Bp, ws, ws2 = _fp4(N, K, bs, dtype, seed=N * 7 + K)
    _check_fp4(Bp, ws, ws2, N, K, bs, dtype)


def test_prefill_weight_full_size():
    """The gate/up prefill weight (N=17408, K=5120), every element."""
    N, K, bs = 17408, 5120, 16
    Bp, ws, ws2 = _fp4(N, K, bs, oracle.BF16)
    _check_fp4(Bp, ws, ws2, N, K, bs, oracle.BF16)


def test_lm_head_weight_log_uniform_scales():
    N, K, bs = 152064 // 8, 5120, 16
    Bp, ws, ws2 = _fp4(N, K, bs, oracle.BF16, log_uniform=True, lo=2.0 ** -6, ws2=0.01)
    _check_fp4(Bp, ws, ws2, N, K, bs, oracle.BF16)


def test_empty_is_noop():
    out = torch.full((4, 0), 7, dtype=torch.bfloat16, device=DEV)
    wq.fp4_dequantize(torch.zeros(4, 0, dtype=torch.uint8, device=DEV),
                      torch.zeros(4, 0, dtype=torch.uint8, device=DEV),
                      torch.ones(1, device=DEV), out=out)
    torch.cuda.synchronize()


@pytest.mark.parametrize("dtype", [oracle.BF16, oracle.FP16])
@pytest.mark.parametrize("N,K,bs", [(64, 5120, 128), (40, 5000, 128), (9, 100, 16), (5, 77, 7),
                                    (3, 256, 8)])
def test_fp8_dequant(N, K, bs, dtype):
    B = wl.gen_fp8_weight(N, K, seed=K)
    sc = wl.gen_fp8_scale(N, wl.scale_cols(K, bs), 0.001, 0.02, seed=K)
    out = wq.fp8_dequantize(u8_to_dev(B), f32_to_dev(sc), block_size=bs, dtype=tdt(dtype))
    torch.cuda.synchronize()
    got = bits_of(out)
    want = oracle.fp8_dequantize(B, sc, N, K, bs, dtype)
    assert np.array_equal(got, want)
