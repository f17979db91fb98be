"""GB300-native block-quantized weight-only matmul (NVFP4 / FP8 weights).

Thin Python binding over the C-ABI library ``libwqmm.so`` (see
``include/wqmm.h``).  This module only marshals arguments: every step of the
computation runs in the library's CUDA kernels.  PyTorch supplies device
memory and the current stream.  There is no CPU fallback: if the library is
missing or fails to load, importing the entry points raises.

Raw C-ABI access (same names and arguments as the header): ``lib()``.
Torch-tensor wrappers (same names):

* ``fp4_weight_matmul(A, B_packed, weight_scale, weight_scale_2, bias=None,
  block_size=16, out=None)`` -- N = B_packed.shape[0], K = 2 * B_packed.shape[1],
  M = prod(A.shape[:-1]), Y has A's leading dims and last dim N
  ("MatMulBlockQuantizedFp4Weight - CUDA Operator Documentation" §1).
* ``fp8_weight_matmul(A, B, b_scale, bias=None, block_size=128, out=None)``
  ("MatMulBlockQuantizedFp8Weight - CUDA Operator Documentation" §1).
* ``fp8_weight_matmul_w8a8(A, a_scale, B, b_scale, bias=None, block_size=128, out=None)``,
  ``fp8_weight_matmul_w8a8_ws(A, a_scale, B, b_scale, workspace, ...)`` (prefill-sized M
  with a caller-owned workspace of ``fp8_w8a8_workspace_bytes(M, K)`` bytes) and
  ``fp8_quantize_dequantize_activation(A, a_scale)`` ("MatMulBlockQuantizedFp8Weight -
  CUDA Operator Documentation" §6, the optional W8A8 activation path).
* ``fp4_quantize_activation(A)`` and ``fp4_quantize_dequantize_activation(A)``
  ("MatMulBlockQuantizedFp4Weight - CUDA Operator Documentation" §6, step 1 of the
  native FP4 x FP4 path: packed E2M1 codes with per-16 E4M3 scales).
* ``fp4_dequantize(B_packed, weight_scale, weight_scale_2, block_size=16,
  dtype=torch.bfloat16, out=None)`` and ``fp8_dequantize(...)``.
"""

from __future__ import annotations

import ctypes
import os
import threading

__all__ = [
    "WqmmError", "lib", "library_path", "fp4_weight_matmul", "fp8_weight_matmul",
    "fp8_weight_matmul_w8a8", "fp8_weight_matmul_w8a8_ws", "fp8_w8a8_workspace_bytes",
    "fp8_weight_matmul_w8a8_noalloc", "NOALLOC_SCRATCH_BYTES",
    "fp8_quantize_dequantize_activation",
    "fp4_quantize_activation", "fp4_quantize_dequantize_activation", "fp4_fp4_matmul",
    "fp4_dequantize", "fp8_dequantize", "device_status", "FP16", "BF16",
]

FP16 = 0
BF16 = 1

# WQMM_NOALLOC_SCRATCH_BYTES of include/wqmm.h: fp8_weight_matmul_w8a8_noalloc
# takes problems with 2 * M * K up to this many bytes.
NOALLOC_SCRATCH_BYTES = 16 << 20

_PKG = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_PKG, "libwqmm.so")
_lib = None
_lock = threading.Lock()

STATUS = {
    0: "WQMM_OK", 1: "WQMM_ERR_INVALID_ARG", 2: "WQMM_ERR_UNSUPPORTED",
    3: "WQMM_ERR_MISALIGNED", 4: "WQMM_ERR_CUDA", 5: "WQMM_ERR_TIMEOUT",
}

# Exported C symbols, in header order.
SYMBOLS = ("fp4_weight_matmul", "fp8_weight_matmul", "fp8_weight_matmul_w8a8",
           "fp8_weight_matmul_w8a8_ws", "fp8_w8a8_workspace_bytes",
           "fp8_weight_matmul_w8a8_noalloc", "fp8_quantize_dequantize_activation", "fp4_quantize_activation",
           "fp4_quantize_dequantize_activation", "fp4_fp4_matmul", "fp4_dequantize",
           "fp8_dequantize",
           "wqmm_status_string", "wqmm_device_status", "wqmm_selftest_wait_timeout",
           "wqmm_version")


class WqmmError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {STATUS.get(status, status)}")


def library_path() -> str:
    return _LIB_PATH


def lib():
    """The loaded C library with argtypes set (raises if it is missing)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(_LIB_PATH):
            raise ImportError(
                f"{_LIB_PATH} is missing: build it with "
                "`python -c 'import __graft_entry__ as g; g.build()'` "
                "(or python -m fp8_weight_only_nvfp4_gb300._build)")
        L = ctypes.CDLL(_LIB_PATH)
        P, I64, I = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
        L.fp4_weight_matmul.argtypes = [P, P, P, P, P, P, I64, I64, I64, I, I, P]
        L.fp8_weight_matmul.argtypes = [P, P, P, P, P, I64, I64, I64, I, I, P]
        L.fp8_weight_matmul_w8a8.argtypes = [P, P, P, P, P, P, I64, I64, I64, I, I, P]
        L.fp8_weight_matmul_w8a8_ws.argtypes = [P, P, P, P, P, P, I64, I64, I64, I, I, P, I64,
                                                P]
        L.fp8_w8a8_workspace_bytes.argtypes = [I64, I64]
        L.fp8_w8a8_workspace_bytes.restype = I64
        L.fp8_weight_matmul_w8a8_noalloc.argtypes = [P, P, P, P, P, P, I64, I64, I64, I, I, P]
        L.fp8_quantize_dequantize_activation.argtypes = [P, P, P, I64, I, P]
        L.fp4_quantize_activation.argtypes = [P, P, P, I64, I64, I, P]
        L.fp4_quantize_dequantize_activation.argtypes = [P, P, I64, I64, I, P]
        L.fp4_fp4_matmul.argtypes = [P, P, P, P, P, P, P, I64, I64, I64, I, P]
        L.fp4_dequantize.argtypes = [P, P, P, P, I64, I64, I, I, P]
        L.fp8_dequantize.argtypes = [P, P, P, I64, I64, I, I, P]
        L.wqmm_status_string.argtypes = [I]
        L.wqmm_status_string.restype = ctypes.c_char_p
        L.wqmm_device_status.argtypes = [P]
        L.wqmm_selftest_wait_timeout.argtypes = [P]
        L.wqmm_version.argtypes = []
        for name in ("fp4_weight_matmul", "fp8_weight_matmul", "fp8_weight_matmul_w8a8",
                     "fp8_weight_matmul_w8a8_ws", "fp8_weight_matmul_w8a8_noalloc",
                     "fp8_quantize_dequantize_activation", "fp4_fp4_matmul", "fp4_dequantize",
                     "fp8_dequantize", "wqmm_device_status", "wqmm_version"):
            getattr(L, name).restype = I
        _lib = L
        return L


# ---------------------------------------------------------------------------
# torch wrappers (argument marshalling only)
# ---------------------------------------------------------------------------

def _torch():
    import torch
    return torch


def _dt(dtype) -> int:
    torch = _torch()
    if dtype == torch.bfloat16:
        return BF16
    if dtype == torch.float16:
        return FP16
    raise TypeError(f"activation dtype must be float16 or bfloat16, got {dtype}")


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream, device):
    torch = _torch()
    s = torch.cuda.current_stream(device) if stream is None else stream
    if s.device != device:
        raise ValueError(f"stream is on {s.device}, the tensors on {device}")
    return ctypes.c_void_p(s.cuda_stream)


def _check(status: int, where: str):
    if status != 0:
        raise WqmmError(status, where)


def _need(t, name, device, dtypes=None, shape=None, numel=None):
    """Validate one tensor argument before its address reaches the library:
    a CUDA tensor on `device`, contiguous, of one of `dtypes`, with exactly
    `shape` (or `numel` elements).  A wrong shape or dtype would make the
    kernels read or write outside the buffer, so nothing is passed on."""
    if t is None:
        return
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor (there is no CPU fallback)")
    if t.device != device:
        raise ValueError(f"{name} is on {t.device}, A on {device}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtypes is not None and t.dtype not in dtypes:
        raise ValueError(f"{name} must have dtype {' or '.join(str(d) for d in dtypes)}, "
                         f"got {t.dtype}")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")
    if numel is not None and t.numel() != numel:
        raise ValueError(f"{name} must have {numel} elements, got {t.numel()}")


def _act_dtypes():
    torch = _torch()
    return (torch.float16, torch.bfloat16)


def _byte_dtypes():
    torch = _torch()
    d = [torch.uint8]
    if hasattr(torch, "float8_e4m3fn"):
        d.append(torch.float8_e4m3fn)
    return tuple(d)


def _device_of(A):
    if not A.is_cuda:
        raise ValueError("A must be a CUDA tensor (there is no CPU fallback)")
    return A.device


def _scale_cols(K, block_size):
    if int(block_size) < 1:
        raise ValueError(f"block_size must be >= 1, got {block_size}")
    return (K + int(block_size) - 1) // int(block_size)


def _check_a_scale(a_scale, dev):
    _need(a_scale, "a_scale", dev, (_torch().float32,), numel=1)


def fp4_weight_matmul(A, B_packed, weight_scale, weight_scale_2, bias=None, block_size=16,
                      out=None, stream=None):
    torch = _torch()
    dev = _device_of(A)
    _need(A, "A", dev, _act_dtypes())
    if B_packed.dim() != 2:
        raise ValueError(f"B_packed must be 2-D [N, K/2], got shape {tuple(B_packed.shape)}")
    N = B_packed.shape[0]
    K = 2 * B_packed.shape[1]
    if A.dim() < 1 or A.shape[-1] != K:
        raise ValueError(f"A.shape[-1]={A.shape[-1] if A.dim() else None} != K={K}")
    S = _scale_cols(K, block_size)
    _need(B_packed, "B_packed", dev, (torch.uint8,))
    _need(weight_scale, "weight_scale", dev, _byte_dtypes(), shape=(N, S))
    _need(weight_scale_2, "weight_scale_2", dev, (torch.float32,), numel=1)
    _need(bias, "bias", dev, (A.dtype,), numel=N)
    M = A.numel() // K if K else int(torch.tensor(A.shape[:-1]).prod())
    if out is None:
        out = torch.empty(*A.shape[:-1], N, dtype=A.dtype, device=dev)
    _need(out, "out", dev, (A.dtype,), shape=tuple(A.shape[:-1]) + (N,))
    with torch.cuda.device(dev):
        st = lib().fp4_weight_matmul(_ptr(A), _ptr(B_packed), _ptr(weight_scale),
                                     _ptr(weight_scale_2), _ptr(bias), _ptr(out), M, N, K,
                                     int(block_size), _dt(A.dtype), _stream(stream, dev))
    _check(st, "fp4_weight_matmul")
    return out


def _fp8_common(A, B, b_scale, bias, block_size, out):
    torch = _torch()
    dev = _device_of(A)
    _need(A, "A", dev, _act_dtypes())
    if B.dim() != 2:
        raise ValueError(f"B must be 2-D [N, K], got shape {tuple(B.shape)}")
    N, K = B.shape
    if A.dim() < 1 or A.shape[-1] != K:
        raise ValueError(f"A.shape[-1]={A.shape[-1] if A.dim() else None} != K={K}")
    _need(B, "B", dev, _byte_dtypes())
    _need(b_scale, "b_scale", dev, (torch.float32,), shape=(N, _scale_cols(K, block_size)))
    _need(bias, "bias", dev, (A.dtype,), numel=N)
    M = A.numel() // K if K else int(torch.tensor(A.shape[:-1]).prod())
    if out is None:
        out = torch.empty(*A.shape[:-1], N, dtype=A.dtype, device=dev)
    _need(out, "out", dev, (A.dtype,), shape=tuple(A.shape[:-1]) + (N,))
    return dev, M, N, K, out


def fp8_weight_matmul(A, B, b_scale, bias=None, block_size=128, out=None, stream=None):
    torch = _torch()
    dev, M, N, K, out = _fp8_common(A, B, b_scale, bias, block_size, out)
    with torch.cuda.device(dev):
        st = lib().fp8_weight_matmul(_ptr(A), _ptr(B), _ptr(b_scale), _ptr(bias), _ptr(out), M,
                                     N, K, int(block_size), _dt(A.dtype), _stream(stream, dev))
    _check(st, "fp8_weight_matmul")
    return out


def fp8_weight_matmul_w8a8(A, a_scale, B, b_scale, bias=None, block_size=128, out=None,
                           stream=None):
    """FP8 page §6 W8A8 path: Y = (fp8_e4m3(A / a_scale) * a_scale) * dequant(B)^T (+ bias).
    a_scale is a one-element float32 CUDA tensor."""
    torch = _torch()
    dev, M, N, K, out = _fp8_common(A, B, b_scale, bias, block_size, out)
    _check_a_scale(a_scale, dev)
    with torch.cuda.device(dev):
        st = lib().fp8_weight_matmul_w8a8(_ptr(A), _ptr(a_scale), _ptr(B), _ptr(b_scale),
                                          _ptr(bias), _ptr(out), M, N, K, int(block_size),
                                          _dt(A.dtype), _stream(stream, dev))
    _check(st, "fp8_weight_matmul_w8a8")
    return out


def fp8_w8a8_workspace_bytes(M, K) -> int:
    """Workspace bytes fp8_weight_matmul_w8a8_ws needs for an [M, K] activation."""
    return int(lib().fp8_w8a8_workspace_bytes(int(M), int(K)))


def fp8_weight_matmul_w8a8_ws(A, a_scale, B, b_scale, workspace, bias=None, block_size=128,
                              out=None, stream=None):
    """FP8 page §6 W8A8 path for prefill-sized M: A_deq is written once into
    `workspace` (a contiguous CUDA tensor of at least
    fp8_w8a8_workspace_bytes(M, K) bytes, any dtype) and the FP8 weight-only
    matmul runs on it; bit-identical to fp8_quantize_dequantize_activation
    followed by fp8_weight_matmul.  Up to 8 rows this is fp8_weight_matmul_w8a8."""
    torch = _torch()
    dev, M, N, K, out = _fp8_common(A, B, b_scale, bias, block_size, out)
    _check_a_scale(a_scale, dev)
    _need(workspace, "workspace", dev)
    nbytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    with torch.cuda.device(dev):
        st = lib().fp8_weight_matmul_w8a8_ws(_ptr(A), _ptr(a_scale), _ptr(B), _ptr(b_scale),
                                             _ptr(bias), _ptr(out), M, N, K, int(block_size),
                                             _dt(A.dtype), _ptr(workspace), nbytes,
                                             _stream(stream, dev))
    _check(st, "fp8_weight_matmul_w8a8_ws")
    return out


def fp8_weight_matmul_w8a8_noalloc(A, a_scale, B, b_scale, out, bias=None, block_size=128,
                                   stream=None):
    """fp8_weight_matmul_w8a8_ws with the workspace taken from a fixed 16 MiB
    array inside the library, for callers that may not allocate device memory
    (2 * M * K <= NOALLOC_SCRATCH_BYTES when M > 8).  `out` is required, so
    nothing is allocated here either.  Calls that may overlap in time on one
    device share the array and race; the first call on a device should come
    before any stream capture."""
    torch = _torch()
    if out is None:
        raise ValueError("out is required: this entry point allocates nothing")
    dev, M, N, K, out = _fp8_common(A, B, b_scale, bias, block_size, out)
    _check_a_scale(a_scale, dev)
    with torch.cuda.device(dev):
        st = lib().fp8_weight_matmul_w8a8_noalloc(_ptr(A), _ptr(a_scale), _ptr(B), _ptr(b_scale),
                                                  _ptr(bias), _ptr(out), M, N, K,
                                                  int(block_size), _dt(A.dtype),
                                                  _stream(stream, dev))
    _check(st, "fp8_weight_matmul_w8a8_noalloc")
    return out


def fp8_quantize_dequantize_activation(A, a_scale, out=None, stream=None):
    """A_deq = fp8_e4m3(A / a_scale) * a_scale, elementwise (bit-exact contract)."""
    torch = _torch()
    dev = _device_of(A)
    _need(A, "A", dev, _act_dtypes())
    _check_a_scale(a_scale, dev)
    if out is None:
        out = torch.empty_like(A)
    _need(out, "out", dev, (A.dtype,), numel=A.numel())
    with torch.cuda.device(dev):
        st = lib().fp8_quantize_dequantize_activation(_ptr(A), _ptr(a_scale), _ptr(out),
                                                      A.numel(), _dt(A.dtype),
                                                      _stream(stream, dev))
    _check(st, "fp8_quantize_dequantize_activation")
    return out


def _rows_k(A):
    if A.dim() < 1:
        raise ValueError("A must have at least one dimension")
    K = A.shape[-1]
    return A.numel() // K if K else 0, K


def fp4_quantize_activation(A, out_packed=None, out_scale=None, stream=None):
    """NVFP4 quantization of an activation (FP4 page §6, step 1): returns
    (A_packed [..., K/2] uint8, A_scale [..., ceil(K/16)] uint8 E4M3)."""
    torch = _torch()
    dev = _device_of(A)
    _need(A, "A", dev, _act_dtypes())
    M, K = _rows_k(A)
    lead = tuple(A.shape[:-1])
    if K % 2:
        raise ValueError(f"K={K} must be even (two codes per byte)")
    if out_packed is None:
        out_packed = torch.empty(lead + (K // 2,), dtype=torch.uint8, device=dev)
    if out_scale is None:
        out_scale = torch.empty(lead + ((K + 15) // 16,), dtype=torch.uint8, device=dev)
    _need(out_packed, "out_packed", dev, (torch.uint8,), shape=lead + (K // 2,))
    _need(out_scale, "out_scale", dev, _byte_dtypes(), shape=lead + ((K + 15) // 16,))
    with torch.cuda.device(dev):
        st = lib().fp4_quantize_activation(_ptr(A), _ptr(out_packed), _ptr(out_scale), M, K,
                                           _dt(A.dtype), _stream(stream, dev))
    _check(st, "fp4_quantize_activation")
    return out_packed, out_scale


def fp4_quantize_dequantize_activation(A, out=None, stream=None):
    """e2m1(code) * e4m3(scale) of fp4_quantize_activation, in A's dtype
    (exact); feeding it to fp4_weight_matmul gives the FP4 x FP4 numerics."""
    torch = _torch()
    dev = _device_of(A)
    _need(A, "A", dev, _act_dtypes())
    M, K = _rows_k(A)
    if out is None:
        out = torch.empty_like(A)
    _need(out, "out", dev, (A.dtype,), shape=tuple(A.shape))
    with torch.cuda.device(dev):
        st = lib().fp4_quantize_dequantize_activation(_ptr(A), _ptr(out), M, K, _dt(A.dtype),
                                                      _stream(stream, dev))
    _check(st, "fp4_quantize_dequantize_activation")
    return out


def fp4_fp4_matmul(A_packed, A_scale, B_packed, weight_scale, weight_scale_2, bias=None,
                   out=None, dtype=None, stream=None):
    """FP4 x FP4 product on the block-scaled tensor core (FP4 page §6, steps
    2-3): A_packed / A_scale as returned by fp4_quantize_activation, the
    NVFP4 weight with 16-element blocks.  The output type is out.dtype, else
    bias.dtype, else `dtype` (default bfloat16).  K must be a multiple of 32."""
    torch = _torch()
    dev = _device_of(A_packed)
    if B_packed.dim() != 2:
        raise ValueError(f"B_packed must be 2-D [N, K/2], got shape {tuple(B_packed.shape)}")
    N, K = B_packed.shape[0], 2 * B_packed.shape[1]
    if A_packed.dim() < 1 or A_packed.shape[-1] * 2 != K:
        raise ValueError(f"A_packed.shape[-1] * 2 != K={K}")
    lead = tuple(A_packed.shape[:-1])
    M = A_packed.numel() // (K // 2) if K else int(torch.tensor(lead).prod())
    S = _scale_cols(K, 16)
    _need(A_packed, "A_packed", dev, (torch.uint8,))
    _need(A_scale, "A_scale", dev, _byte_dtypes(), shape=lead + (S,))
    _need(B_packed, "B_packed", dev, (torch.uint8,))
    _need(weight_scale, "weight_scale", dev, _byte_dtypes(), shape=(N, S))
    _need(weight_scale_2, "weight_scale_2", dev, (torch.float32,), numel=1)
    ydt = out.dtype if out is not None else (bias.dtype if bias is not None
                                             else (dtype or torch.bfloat16))
    _need(bias, "bias", dev, (ydt,), numel=N)
    if out is None:
        out = torch.empty(*lead, N, dtype=ydt, device=dev)
    _need(out, "out", dev, _act_dtypes(), shape=lead + (N,))
    with torch.cuda.device(dev):
        st = lib().fp4_fp4_matmul(_ptr(A_packed), _ptr(A_scale), _ptr(B_packed),
                                  _ptr(weight_scale), _ptr(weight_scale_2), _ptr(bias), _ptr(out),
                                  M, N, K, _dt(ydt), _stream(stream, dev))
    _check(st, "fp4_fp4_matmul")
    return out


def fp4_dequantize(B_packed, weight_scale, weight_scale_2, block_size=16, dtype=None,
                   out=None, stream=None):
    torch = _torch()
    dev = _device_of(B_packed)
    if B_packed.dim() != 2:
        raise ValueError(f"B_packed must be 2-D [N, K/2], got shape {tuple(B_packed.shape)}")
    N = B_packed.shape[0]
    K = 2 * B_packed.shape[1]
    _need(B_packed, "B_packed", dev, (torch.uint8,))
    _need(weight_scale, "weight_scale", dev, _byte_dtypes(),
          shape=(N, _scale_cols(K, block_size)))
    _need(weight_scale_2, "weight_scale_2", dev, (torch.float32,), numel=1)
    dtype = torch.bfloat16 if dtype is None else dtype
    if out is None:
        out = torch.empty(N, K, dtype=dtype, device=dev)
    _need(out, "out", dev, _act_dtypes(), shape=(N, K))
    with torch.cuda.device(dev):
        st = lib().fp4_dequantize(_ptr(B_packed), _ptr(weight_scale), _ptr(weight_scale_2),
                                  _ptr(out), N, K, int(block_size), _dt(out.dtype),
                                  _stream(stream, dev))
    _check(st, "fp4_dequantize")
    return out


def fp8_dequantize(B, b_scale, block_size=128, dtype=None, out=None, stream=None):
    torch = _torch()
    dev = _device_of(B)
    if B.dim() != 2:
        raise ValueError(f"B must be 2-D [N, K], got shape {tuple(B.shape)}")
    N, K = B.shape
    _need(B, "B", dev, _byte_dtypes())
    _need(b_scale, "b_scale", dev, (torch.float32,), shape=(N, _scale_cols(K, block_size)))
    dtype = torch.bfloat16 if dtype is None else dtype
    if out is None:
        out = torch.empty(N, K, dtype=dtype, device=dev)
    _need(out, "out", dev, _act_dtypes(), shape=(N, K))
    with torch.cuda.device(dev):
        st = lib().fp8_dequantize(_ptr(B), _ptr(b_scale), _ptr(out), N, K, int(block_size),
                                  _dt(out.dtype), _stream(stream, dev))
    _check(st, "fp8_dequantize")
    return out


def device_status(stream=None, device=None) -> int:
    """Synchronise the stream and return (and clear) the device error word of
    its device (the current device when neither is given)."""
    torch = _torch()
    if device is None:
        device = stream.device if stream is not None else torch.device(
            "cuda", torch.cuda.current_device())
    device = torch.device(device)
    with torch.cuda.device(device):
        return int(lib().wqmm_device_status(_stream(stream, device)))
