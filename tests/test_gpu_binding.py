"""The Python binding refuses arguments that would make the kernels read or
write outside a buffer: wrong dtypes, scale tensors shaped for another block
size, short outputs or biases.  Nothing reaches the library in these cases."""

import pytest
import torch

import fp8_weight_only_nvfp4_gb300 as wq

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


def _fp4(M=4, N=32, K=64, bs=16):
    A = torch.randn(M, K, device=DEV, dtype=torch.bfloat16)
    B = torch.zeros(N, K // 2, dtype=torch.uint8, device=DEV)
    ws = torch.full((N, (K + bs - 1) // bs), 0x38, dtype=torch.uint8, device=DEV)
    ws2 = torch.ones(1, dtype=torch.float32, device=DEV)
    return A, B, ws, ws2


def test_fp4_matmul_rejects_bad_arguments():
    A, B, ws, ws2 = _fp4()
    wq.fp4_weight_matmul(A, B, ws, ws2)          # well formed: runs
    torch.cuda.synchronize()
    bad = [
        dict(weight_scale=ws[:, :2]),                                    # scales for bs = 32
        dict(weight_scale=ws.to(torch.int32)),
        dict(weight_scale_2=ws2.double()),
        dict(weight_scale_2=torch.ones(2, dtype=torch.float32, device=DEV)),
        dict(bias=torch.zeros(32, dtype=torch.float16, device=DEV)),     # A is BF16
        dict(bias=torch.zeros(31, dtype=torch.bfloat16, device=DEV)),
        dict(out=torch.empty(4, 31, dtype=torch.bfloat16, device=DEV)),
        dict(out=torch.empty(4, 32, dtype=torch.float16, device=DEV)),
        dict(A=A.float()),
        dict(A=A[:, :32]),
        dict(B_packed=B.view(torch.int8)),
        dict(block_size=0),
    ]
    base = dict(A=A, B_packed=B, weight_scale=ws, weight_scale_2=ws2)
    for change in bad:
        kw = dict(base, **change)
        with pytest.raises(ValueError):
            wq.fp4_weight_matmul(kw.pop("A"), kw.pop("B_packed"), kw.pop("weight_scale"),
                                 kw.pop("weight_scale_2"), **kw)


def test_fp8_matmul_rejects_bad_arguments():
    A = torch.randn(4, 256, device=DEV, dtype=torch.float16)
    B = torch.zeros(32, 256, dtype=torch.uint8, device=DEV)
    s = torch.ones(32, 2, dtype=torch.float32, device=DEV)
    wq.fp8_weight_matmul(A, B, s, block_size=128)
    torch.cuda.synchronize()
    for kw in (dict(b_scale=s.bfloat16()), dict(b_scale=s[:, :1].contiguous()),
               dict(block_size=64), dict(out=torch.empty(4, 32, dtype=torch.bfloat16,
                                                         device=DEV))):
        args = dict(A=A, B=B, b_scale=s, block_size=128)
        args.update(kw)
        with pytest.raises(ValueError):
            wq.fp8_weight_matmul(args.pop("A"), args.pop("B"), args.pop("b_scale"), **args)
    with pytest.raises(ValueError):
        wq.fp8_weight_matmul_w8a8(A, torch.ones(2, device=DEV), B, s, block_size=128)


def test_quantize_and_dequantize_reject_bad_outputs():
    A = torch.randn(8, 64, device=DEV, dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        wq.fp4_quantize_activation(A, out_scale=torch.empty(8, 3, dtype=torch.uint8, device=DEV))
    with pytest.raises(ValueError):
        wq.fp4_quantize_dequantize_activation(A, out=torch.empty(8, 63, dtype=torch.bfloat16,
                                                                  device=DEV))
    _, B, ws, ws2 = _fp4()
    with pytest.raises(ValueError):
        wq.fp4_dequantize(B, ws, ws2, out=torch.empty(32, 63, dtype=torch.bfloat16, device=DEV))
    with pytest.raises(ValueError):
        wq.fp4_dequantize(B, ws[:, :1].contiguous(), ws2)
