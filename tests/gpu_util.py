"""Helpers shared by the GPU parity tests: move seeded numpy inputs to the
device, call the library through its binding, compare with the oracle."""

import numpy as np
import torch

import fp8_weight_only_nvfp4_gb300 as wq
import oracle

DEV = "cuda:0"


def tdt(dtype):
    return torch.bfloat16 if dtype == oracle.BF16 else torch.float16


def act_to_dev(bits, dtype):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to(DEV).view(tdt(dtype))


def u8_to_dev(a):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.uint8)).to(DEV)


def f32_to_dev(a):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(DEV)


def bits_of(t):
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def f64_of(t):
    if isinstance(t, np.ndarray):
        return t.astype(np.float64)
    return t.float().cpu().numpy().astype(np.float64)


def fp4_dev(p):
    """Device tensors for an Fp4Problem."""
    return dict(
        A=act_to_dev(p.A, p.dtype),
        B=u8_to_dev(p.B_packed),
        ws=u8_to_dev(p.weight_scale),
        ws2=torch.tensor([p.weight_scale_2], dtype=torch.float32, device=DEV),
        bias=None if p.bias is None else act_to_dev(p.bias, p.dtype),
    )


def run_fp4(p, d=None):
    d = d or fp4_dev(p)
    Y = wq.fp4_weight_matmul(d["A"], d["B"], d["ws"], d["ws2"], d["bias"], block_size=p.block_size)
    torch.cuda.synchronize()
    assert wq.device_status() == 0
    return Y


def fp8_dev(p):
    return dict(
        A=act_to_dev(p.A, p.dtype),
        B=u8_to_dev(p.B),
        s=f32_to_dev(p.b_scale),
        bias=None if p.bias is None else act_to_dev(p.bias, p.dtype),
    )


def run_fp8(p, d=None):
    d = d or fp8_dev(p)
    Y = wq.fp8_weight_matmul(d["A"], d["B"], d["s"], d["bias"], block_size=p.block_size)
    torch.cuda.synchronize()
    assert wq.device_status() == 0
    return Y


def assert_within_tolerance(Y, Yref, S, dtype, what=""):
    Yg = f64_of(Y).reshape(Yref.shape)
    err = np.abs(Yg - Yref)
    tol = oracle.tolerance(S, dtype)
    bad = ~(err <= tol)
    if bad.any():
        idx = np.argwhere(bad)[:5]
        raise AssertionError(
            f"{what}: {bad.sum()} of {bad.size} outside tolerance; max err/tol "
            f"{np.nanmax(err / tol):.3g}; first {idx.tolist()} got {Yg[bad][:5]} "
            f"want {Yref[bad][:5]}")
    return float(np.max(err / tol)) if err.size else 0.0
