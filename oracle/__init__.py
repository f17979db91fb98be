"""CPU oracle for block-quantized weight-only matmul (NVFP4 and FP8 weights).

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline legs of ``bench.py`` may import this package.  The product path
(``fp8_weight_only_nvfp4_gb300``) never imports it and never falls back to it.

The arithmetic lives in ``wqmm_oracle.cpp`` (plain C++, float64 accumulation,
explicit E2M1 and E4M3 decode tables), compiled with g++ into
``oracle/_build/liboracle.so``.  This module only marshals numpy arrays.

Function map (all cite the pages by title and section):

* ``fp4_dequantize``   -- "MatMulBlockQuantizedFp4Weight" §2 dequant formula,
  rounded per the bit-exact contract (fp32 product, fp32 x weight_scale_2,
  RNE to the activation type).
* ``fp8_dequantize``   -- "MatMulBlockQuantizedFp8Weight" §2.
* ``fp4_matmul`` / ``fp8_matmul`` (+ ``*_sampled``) -- the operator definition
  Y = A * dequant(B)^T + bias, exact decode in float64 and float64 sums, plus
  the magnitude sum S = sum_k |A[m,k] * B_dq[n,k]| used by the tolerance.
* ``nvfp4_quantize_activation`` / ``nvfp4_qdq_activation`` -- "MatMulBlockQuantizedFp4Weight"
  §6 step 1 (NVFP4 activation quantization, per-16 E4M3 scales).
* ``fp8_qdq_activation`` -- "MatMulBlockQuantizedFp8Weight" §6 (W8A8).
* ``e2m1_value``, ``e4m3_value``, ``e2m1_from_f32``, ``e4m3_from_f32``,
  ``rne_f32_to_act`` -- the format primitives.

Every function is pinned by ``tests/test_oracle_pins.py`` against values the
pages print, library routines (torch float8_e4m3fn and dtype casts), closed
forms and invariants.
"""

from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "wqmm_oracle.cpp")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "liboracle.so")

FP16 = 0
BF16 = 1

_lib = None
_lock = threading.Lock()


def build(force: bool = False) -> str:
    """Compile the oracle with g++ (no fast-math, no FMA contraction)."""
    os.makedirs(_BUILD, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["g++", "-O2", "-std=c++17", "-shared", "-fPIC", "-pthread",
           "-ffp-contract=off", "-fno-fast-math", _SRC, "-o", tmp]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        P = ctypes.c_void_p
        I64 = ctypes.c_int64
        I = ctypes.c_int
        F = ctypes.c_float
        lib.orc_hardware_threads.restype = I
        lib.orc_e2m1_value.argtypes = [I]
        lib.orc_e2m1_value.restype = ctypes.c_double
        lib.orc_e4m3_value.argtypes = [I]
        lib.orc_e4m3_value.restype = ctypes.c_double
        lib.orc_rne_f32_to_act_array.argtypes = [P, P, I64, I]
        lib.orc_act_to_double.argtypes = [ctypes.c_uint16, I]
        lib.orc_act_to_double.restype = ctypes.c_double
        lib.orc_fp4_dequantize.argtypes = [P, P, F, P, I64, I64, I, I, I]
        lib.orc_fp8_dequantize.argtypes = [P, P, P, I64, I64, I, I, I]
        lib.orc_fp4_dequantize_f64.argtypes = [P, P, F, P, I64, I64, I, I]
        lib.orc_fp8_dequantize_f64.argtypes = [P, P, P, I64, I64, I, I]
        lib.orc_fp4_matmul.argtypes = [P, P, P, F, P, I64, I64, I64, I, I, P, P, I]
        lib.orc_fp8_matmul.argtypes = [P, P, P, P, I64, I64, I64, I, I, P, P, I]
        lib.orc_fp4_matmul_sampled.argtypes = [P, P, P, F, P, I64, I, I, P, P, I64, P, P, I]
        lib.orc_fp8_matmul_sampled.argtypes = [P, P, P, P, I64, I, I, P, P, I64, P, P, I]
        lib.orc_e4m3_from_f32.argtypes = [F]
        lib.orc_e4m3_from_f32.restype = I
        lib.orc_fp8_qdq_activation.argtypes = [P, F, P, I64, I]
        lib.orc_e2m1_from_f32.argtypes = [F]
        lib.orc_e2m1_from_f32.restype = I
        lib.orc_nvfp4_quantize_act.argtypes = [P, I64, I64, I, P, P]
        lib.orc_nvfp4_qdq_act.argtypes = [P, I64, I64, I, P]
        _lib = lib
        return lib


def hardware_threads() -> int:
    return int(_load().orc_hardware_threads())


def _threads(threads):
    return hardware_threads() if threads is None else int(threads)


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def e2m1_value(code: int) -> float:
    return float(_load().orc_e2m1_value(int(code)))


def e4m3_value(byte: int) -> float:
    return float(_load().orc_e4m3_value(int(byte)))


def e4m3_from_f32(f: float) -> int:
    """E4M3FN code of a float32 value: RNE, ties to even, saturating at 448."""
    return int(_load().orc_e4m3_from_f32(float(np.float32(f))))


def fp8_qdq_activation(A, a_scale: float, dtype: int) -> np.ndarray:
    """W8A8 activation path (FP8 page §6): RNE_act(fp32(e4m3(fp32(A / a_scale)) *
    a_scale)) per element; A and the result are activation bit patterns."""
    a = _c(A, np.uint16)
    out = np.empty(a.shape, dtype=np.uint16)
    _load().orc_fp8_qdq_activation(_ptr(a), float(np.float32(a_scale)), _ptr(out), a.size,
                                   int(dtype))
    return out


def e2m1_from_f32(f: float) -> int:
    """E2M1 code of a float32 value: RNE, ties to even, saturating at 6, sign
    kept (a negative value that rounds to zero gives 0x8)."""
    return int(_load().orc_e2m1_from_f32(float(np.float32(f))))


def nvfp4_quantize_activation(A, dtype: int):
    """NVFP4 activation quantization (FP4 page §6, step 1 of the native
    path): per 16-element block of each row, scale = E4M3(fp32(amax / 6)),
    codes = E2M1(fp32(a / scale)).  A is [M, K] activation bit patterns (K
    even); returns (codes [M, K/2] uint8, two per byte with the even k in the
    low nibble; scales [M, ceil(K/16)] uint8)."""
    a = _c(A, np.uint16)
    M, K = a.shape
    codes = np.empty((M, K // 2), dtype=np.uint8)
    scales = np.empty((M, (K + 15) // 16), dtype=np.uint8)
    _load().orc_nvfp4_quantize_act(_ptr(a), M, K, int(dtype), _ptr(codes), _ptr(scales))
    return codes, scales


def nvfp4_qdq_activation(A, dtype: int) -> np.ndarray:
    """NVFP4 activation quantize-dequantize: RNE_act(e2m1(code) * e4m3(scale))
    per element (exact: at most 6 significant bits); same shape as A."""
    a = _c(A, np.uint16)
    M, K = a.shape
    out = np.empty_like(a)
    _load().orc_nvfp4_qdq_act(_ptr(a), M, K, int(dtype), _ptr(out))
    return out


def rne_f32_to_act(f32: np.ndarray, dtype: int) -> np.ndarray:
    """Round float32 values to bf16/fp16 bit patterns (uint16), RNE."""
    bits = _c(np.asarray(f32, dtype=np.float32).view(np.uint32), np.uint32)
    out = np.empty(bits.shape, dtype=np.uint16)
    _load().orc_rne_f32_to_act_array(_ptr(bits), _ptr(out), bits.size, int(dtype))
    return out


def act_to_double(bits: int, dtype: int) -> float:
    return float(_load().orc_act_to_double(int(bits), int(dtype)))


def fp4_dequantize(B_packed, weight_scale, weight_scale_2, N, K, block_size,
                   dtype, threads=None) -> np.ndarray:
    """Bit-exact dequantized [N, K] weight as uint16 activation bit patterns."""
    Bp = _c(B_packed, np.uint8)
    ws = _c(weight_scale, np.uint8)
    out = np.empty((N, K), dtype=np.uint16)
    _load().orc_fp4_dequantize(_ptr(Bp), _ptr(ws), float(np.float32(weight_scale_2)),
                               _ptr(out), N, K, block_size, dtype, _threads(threads))
    return out


def fp8_dequantize(B, b_scale, N, K, block_size, dtype, threads=None) -> np.ndarray:
    Bq = _c(B, np.uint8)
    bs = _c(b_scale, np.float32)
    out = np.empty((N, K), dtype=np.uint16)
    _load().orc_fp8_dequantize(_ptr(Bq), _ptr(bs), _ptr(out), N, K, block_size,
                               dtype, _threads(threads))
    return out


def fp4_dequantize_f64(B_packed, weight_scale, weight_scale_2, N, K, block_size,
                       threads=None) -> np.ndarray:
    Bp = _c(B_packed, np.uint8)
    ws = _c(weight_scale, np.uint8)
    out = np.empty((N, K), dtype=np.float64)
    _load().orc_fp4_dequantize_f64(_ptr(Bp), _ptr(ws), float(np.float32(weight_scale_2)),
                                   _ptr(out), N, K, block_size, _threads(threads))
    return out


def fp8_dequantize_f64(B, b_scale, N, K, block_size, threads=None) -> np.ndarray:
    Bq = _c(B, np.uint8)
    bs = _c(b_scale, np.float32)
    out = np.empty((N, K), dtype=np.float64)
    _load().orc_fp8_dequantize_f64(_ptr(Bq), _ptr(bs), _ptr(out), N, K, block_size,
                                   _threads(threads))
    return out


def fp4_matmul(A, B_packed, weight_scale, weight_scale_2, bias, M, N, K,
               block_size, dtype, threads=None):
    """Returns (Y_ref, S) as float64 [M, N] arrays."""
    A_ = _c(A, np.uint16)
    Bp = _c(B_packed, np.uint8)
    ws = _c(weight_scale, np.uint8)
    b = None if bias is None else _c(bias, np.uint16)
    Y = np.empty((M, N), dtype=np.float64)
    S = np.empty((M, N), dtype=np.float64)
    _load().orc_fp4_matmul(_ptr(A_), _ptr(Bp), _ptr(ws), float(np.float32(weight_scale_2)),
                           _ptr(b), M, N, K, block_size, dtype, _ptr(Y), _ptr(S),
                           _threads(threads))
    return Y, S


def fp8_matmul(A, B, b_scale, bias, M, N, K, block_size, dtype, threads=None):
    A_ = _c(A, np.uint16)
    Bq = _c(B, np.uint8)
    bs = _c(b_scale, np.float32)
    b = None if bias is None else _c(bias, np.uint16)
    Y = np.empty((M, N), dtype=np.float64)
    S = np.empty((M, N), dtype=np.float64)
    _load().orc_fp8_matmul(_ptr(A_), _ptr(Bq), _ptr(bs), _ptr(b), M, N, K, block_size,
                           dtype, _ptr(Y), _ptr(S), _threads(threads))
    return Y, S


def fp4_matmul_sampled(A, B_packed, weight_scale, weight_scale_2, bias, K,
                       block_size, dtype, ms, ns, threads=None):
    """(Y_ref, S) at the output positions (ms[i], ns[i]) only."""
    A_ = _c(A, np.uint16)
    Bp = _c(B_packed, np.uint8)
    ws = _c(weight_scale, np.uint8)
    b = None if bias is None else _c(bias, np.uint16)
    ms_ = _c(ms, np.int64)
    ns_ = _c(ns, np.int64)
    Y = np.empty(ms_.shape, dtype=np.float64)
    S = np.empty(ms_.shape, dtype=np.float64)
    _load().orc_fp4_matmul_sampled(_ptr(A_), _ptr(Bp), _ptr(ws),
                                   float(np.float32(weight_scale_2)), _ptr(b), K,
                                   block_size, dtype, _ptr(ms_), _ptr(ns_), ms_.size,
                                   _ptr(Y), _ptr(S), _threads(threads))
    return Y, S


def fp8_matmul_sampled(A, B, b_scale, bias, K, block_size, dtype, ms, ns,
                       threads=None):
    A_ = _c(A, np.uint16)
    Bq = _c(B, np.uint8)
    bs = _c(b_scale, np.float32)
    b = None if bias is None else _c(bias, np.uint16)
    ms_ = _c(ms, np.int64)
    ns_ = _c(ns, np.int64)
    Y = np.empty(ms_.shape, dtype=np.float64)
    S = np.empty(ms_.shape, dtype=np.float64)
    _load().orc_fp8_matmul_sampled(_ptr(A_), _ptr(Bq), _ptr(bs), _ptr(b), K,
                                   block_size, dtype, _ptr(ms_), _ptr(ns_), ms_.size,
                                   _ptr(Y), _ptr(S), _threads(threads))
    return Y, S


def tolerance(S: np.ndarray, dtype: int) -> np.ndarray:
    """Per-element matmul acceptance bound, as a function of S = sum|A*B_dq|.

    bf16 output: 8e-3 * S + 1e-3;  fp16 output: 2e-3 * S + 1e-4.
    """
    if dtype == BF16:
        return 8e-3 * S + 1e-3
    return 2e-3 * S + 1e-4
