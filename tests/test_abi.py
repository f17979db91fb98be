"""C-ABI checks that need no GPU: the library loads, exports every function
include/wqmm.h declares, and rejects bad arguments on the host (no compute
call is made here)."""

import ctypes
import os
import re

import pytest

import fp8_weight_only_nvfp4_gb300 as wq

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _header_functions():
    text = open(os.path.join(ROOT, "include", "wqmm.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?[a-z_0-9]+\s*\*?\s*([a-z_0-9]+)\s*\(", text, flags=re.M)
    return [n for n in names if n not in ("if", "while")]


@pytest.fixture(scope="module")
def L():
    from fp8_weight_only_nvfp4_gb300 import _build
    _build.build()
    return wq.lib()


def test_header_declares_the_expected_api():
    names = _header_functions()
    assert set(names) == set(wq.SYMBOLS), names


def test_library_exports_every_declared_symbol(L):
    for name in _header_functions():
        assert hasattr(L, name), name
        assert ctypes.cast(getattr(L, name), ctypes.c_void_p).value


def test_status_strings(L):
    for code, name in wq.STATUS.items():
        assert L.wqmm_status_string(code).decode() == name
    assert L.wqmm_status_string(99).decode() == "WQMM_ERR_UNKNOWN"
    assert L.wqmm_version() == 100


P = ctypes.c_void_p
FAKE = P(0x10000)        # 16-byte aligned non-null address (never dereferenced)
FAKE_ODD = P(0x10001)


def fp4mm(L, M=4, N=16, K=32, bs=16, dt=1, A=FAKE, B=FAKE, ws=FAKE, ws2=FAKE, bias=None, Y=FAKE):
    return L.fp4_weight_matmul(A, B, ws, ws2, bias, Y, M, N, K, bs, dt, None)


def test_fp4_matmul_argument_checks(L):
    assert fp4mm(L, dt=2) == 1
    assert fp4mm(L, M=-1) == 1
    assert fp4mm(L, K=31) == 1          # odd K cannot be packed two per byte
    assert fp4mm(L, bs=0) == 1
    assert fp4mm(L, bs=8) == 2          # block size must be a multiple of 16
    assert fp4mm(L, bs=24) == 2
    assert fp4mm(L, A=None) == 1
    assert fp4mm(L, B=None) == 1
    assert fp4mm(L, ws=None) == 1
    assert fp4mm(L, ws2=None) == 1
    assert fp4mm(L, Y=None) == 1
    assert fp4mm(L, A=FAKE_ODD) == 3
    assert fp4mm(L, Y=FAKE_ODD) == 3
    assert fp4mm(L, B=FAKE_ODD) == 3
    assert fp4mm(L, bias=FAKE_ODD) == 3  # 2-byte alignment for bias
    # empty outputs return OK without touching the GPU
    assert fp4mm(L, M=0, A=None, Y=None) == 0
    assert fp4mm(L, N=0, A=None, Y=None) == 0


def test_fp8_matmul_argument_checks(L):
    f = lambda **kw: L.fp8_weight_matmul(kw.get("A", FAKE), kw.get("B", FAKE),
                                         kw.get("s", FAKE), None, kw.get("Y", FAKE),
                                         kw.get("M", 4), kw.get("N", 16), kw.get("K", 32),
                                         kw.get("bs", 128), kw.get("dt", 1), None)
    assert f(dt=-1) == 1
    assert f(K=-5) == 1
    assert f(bs=-1) == 1
    assert f(bs=100) == 2
    assert f(s=None) == 1
    assert f(s=FAKE_ODD) == 3
    assert f(M=0, A=None, Y=None) == 0


def test_dequant_argument_checks(L):
    assert L.fp4_dequantize(FAKE, FAKE, FAKE, FAKE, 4, 33, 16, 1, None) == 1   # odd K
    assert L.fp4_dequantize(FAKE, FAKE, FAKE, FAKE, 4, 32, 0, 1, None) == 1    # bs < 1
    assert L.fp4_dequantize(FAKE, FAKE, FAKE, None, 4, 32, 16, 1, None) == 1
    assert L.fp4_dequantize(FAKE, FAKE_ODD, FAKE, FAKE, 4, 32, 16, 1, None) == 3
    assert L.fp4_dequantize(None, None, None, None, 0, 32, 16, 1, None) == 0    # empty
    assert L.fp4_dequantize(None, None, None, None, 5, 0, 16, 1, None) == 0
    assert L.fp8_dequantize(FAKE, FAKE, FAKE, 4, 32, 16, 3, None) == 1
    assert L.fp8_dequantize(FAKE, None, FAKE, 4, 32, 16, 1, None) == 1
    assert L.fp8_dequantize(FAKE_ODD, FAKE, FAKE, 4, 32, 16, 1, None) == 3


def test_activation_quantize_argument_checks(L):
    """NVFP4 activation quantization: host-side checks only (no launch)."""
    q, qdq = L.fp4_quantize_activation, L.fp4_quantize_dequantize_activation
    assert q(FAKE, FAKE, FAKE, 4, 33, 1, None) == 1           # odd K
    assert q(FAKE, FAKE, FAKE, -1, 32, 1, None) == 1          # negative M
    assert q(FAKE, FAKE, FAKE, 4, 32, 2, None) == 1           # dtype
    assert q(FAKE, None, FAKE, 4, 32, 1, None) == 1           # NULL output
    assert q(FAKE_ODD, FAKE, FAKE, 4, 32, 1, None) == 3       # misaligned A
    assert q(FAKE, FAKE, FAKE_ODD, 4, 32, 0, None) == 3       # misaligned scales
    assert q(None, None, None, 0, 32, 1, None) == 0           # empty
    assert q(None, None, None, 5, 0, 1, None) == 0
    assert q(FAKE, FAKE, FAKE, 1 << 31, 32, 1, None) == 2     # too large
    assert qdq(FAKE, FAKE, 4, 31, 1, None) == 1
    assert qdq(FAKE, None, 4, 32, 1, None) == 1
    assert qdq(FAKE, FAKE_ODD, 4, 32, 1, None) == 3
    assert qdq(None, None, 0, 32, 0, None) == 0


def test_torch_wrappers_refuse_cpu_tensors(L):
    import torch
    A = torch.zeros(1, 32, dtype=torch.bfloat16)
    B = torch.zeros(16, 16, dtype=torch.uint8)
    ws = torch.zeros(16, 2, dtype=torch.uint8)
    ws2 = torch.ones(1)
    with pytest.raises(ValueError):
        wq.fp4_weight_matmul(A, B, ws, ws2)


def test_w8a8_workspace_argument_checks(L):
    """fp8_weight_matmul_w8a8_ws: the workspace is checked on the host (size,
    overlap with A or Y, alignment) before any CUDA call."""
    size = L.fp8_w8a8_workspace_bytes
    assert size(4, 32) == 0 and size(8, 32) == 0     # the fused GEMV needs none
    assert size(9, 32) == 9 * 32 * 2
    assert size(0, 32) == 0 and size(9, 0) == 0
    assert size(1 << 31, 32) == 0                     # beyond the library's limit
    A, Y, W = P(0x100000), P(0x200000), P(0x400000)
    need = 16 * 64 * 2

    def f(M=16, K=64, ws=W, nbytes=need, a=A, y=Y, **kw):
        return L.fp8_weight_matmul_w8a8_ws(a, kw.get("asc", FAKE), FAKE, FAKE, None, y, M,
                                           kw.get("N", 32), K, kw.get("bs", 128),
                                           kw.get("dt", 1), ws, nbytes, None)
    assert f(ws=None) == 1                  # M > 8 needs a workspace
    assert f(nbytes=need - 1) == 1          # too small
    assert f(ws=P(0x100000 + 64)) == 1      # overlaps A
    assert f(ws=P(0x200000 - 16)) == 1      # overlaps Y
    assert f(ws=P(0x400001)) == 3           # misaligned
    assert f(asc=None) == 1                 # NULL a_scale
    assert f(bs=100) == 2
    assert f(dt=5) == 1
    assert f(M=0, a=None, y=None, ws=None) == 0   # empty output: OK, no launch


def test_noalloc_host_checks(L):
    """fp8_weight_matmul_w8a8_noalloc: its scratch limit and argument errors
    are reported on the host, before any CUDA call."""
    text = open(os.path.join(ROOT, "include", "wqmm.h")).read()
    m = re.search(r"#define WQMM_NOALLOC_SCRATCH_BYTES \((\d+)u << (\d+)\)", text)
    assert m and int(m.group(1)) << int(m.group(2)) == wq.NOALLOC_SCRATCH_BYTES

    def f(M=16, N=32, K=64, bs=128, dt=1, A=FAKE, Y=P(0x200000), asc=FAKE):
        return L.fp8_weight_matmul_w8a8_noalloc(A, asc, FAKE, FAKE, None, Y, M, N, K, bs, dt,
                                                None)
    lim = wq.NOALLOC_SCRATCH_BYTES
    assert f(M=lim // (2 * 4096) + 1, K=4096) == 2      # 2*M*K just above the limit
    assert f(M=1 << 20, K=1 << 20) == 2
    assert f(M=1 << 31, K=64) == 2                      # beyond the library's limit
    assert f(dt=7) == 1
    assert f(M=-1) == 1
    assert f(bs=0) == 1
    assert f(bs=100) == 2
    assert f(A=None) == 1
    assert f(asc=None) == 1
    assert f(Y=FAKE_ODD) == 3
    assert f(M=0, A=None, Y=None) == 0                   # empty output: no launch


def test_fp4_fp4_matmul_host_checks(L):
    """fp4_fp4_matmul: argument errors are reported before any CUDA call."""
    def f(M=16, N=32, K=256, dt=1, A=FAKE, As=FAKE, B=FAKE, Ws=FAKE, g=FAKE, bias=None, Y=FAKE):
        return L.fp4_fp4_matmul(A, As, B, Ws, g, bias, Y, M, N, K, dt, None)
    assert f(dt=3) == 1
    assert f(K=255) == 1              # odd K
    assert f(M=-1) == 1
    assert f(K=48) == 2               # K must be a multiple of 32
    assert f(K=1 << 31) == 2
    assert f(A=None) == 1
    assert f(As=None) == 1
    assert f(g=None) == 1
    assert f(Y=None) == 1
    assert f(Ws=FAKE_ODD) == 3
    assert f(As=FAKE_ODD) == 3
    assert f(bias=FAKE_ODD) == 3
    assert f(M=0, A=None, Y=None) == 0
    assert f(N=0, B=None, Y=None) == 0


def test_plain_c_caller(L, tmp_path):
    """The header and library used from C (gcc, no Python in the call path)."""
    import shutil
    import subprocess
    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("gcc not available")
    exe = tmp_path / "abi_host_checks"
    lib_dir = os.path.dirname(wq.library_path())
    r = subprocess.run([gcc, "-std=c99", "-Wall", "-Werror", "-I", os.path.join(ROOT, "include"),
                        os.path.join(ROOT, "tests", "c", "abi_host_checks.c"), "-L", lib_dir,
                        "-lwqmm", f"-Wl,-rpath,{lib_dir}", "-o", str(exe)],
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    r = subprocess.run([str(exe)], capture_output=True, text=True)
    assert r.returncode == 0, r.stdout + r.stderr
    assert r.stdout.strip() == "ok"
