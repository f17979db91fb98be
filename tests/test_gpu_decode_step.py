"""The decode step's GEMV shapes and a replayed graph of them.

A 27B-class decode step ("MatMulBlockQuantizedFp4Weight - CUDA Operator
Documentation" §4: one GEMV launch per projection, the step measured as a
whole) chains four hidden x hidden projections, gate and up (MLP x hidden)
and down (hidden x MLP) per layer.  These tests check every output of the
gate/up and down shapes at M <= 8 against the oracle, and a short chain of
mixed shapes captured once as a CUDA graph and replayed: every layer's output
against the oracle applied to the input that layer actually read, and the
replays against each other bit for bit."""

import numpy as np
import pytest
import torch

import fp8_weight_only_nvfp4_gb300 as wq
import oracle
import workloads as wl
from gpu_util import DEV, act_to_dev, assert_within_tolerance, bits_of, fp4_dev, run_fp4

pytestmark = pytest.mark.gpu

HIDDEN, MLP = 5120, 17408


def _ref(p):
    return oracle.fp4_matmul(p.A, p.B_packed, p.weight_scale, p.weight_scale_2, p.bias, p.M, p.N,
                             p.K, p.block_size, p.dtype)


@pytest.mark.parametrize("M", [1, 4, 8])
@pytest.mark.parametrize("N,K", [(MLP, HIDDEN), (HIDDEN, MLP)], ids=["gate_up", "down"])
def test_decode_step_shape_every_output(M, N, K):
    p = wl.make_fp4(M, N, K, 16, oracle.BF16, seed=40 + M + (N > K), ws2=0.0125)
    Y = run_fp4(p)
    Yr, S = _ref(p)
    assert_within_tolerance(Y, Yr, S, p.dtype, f"M={M} N={N} K={K}")


def test_replayed_graph_chain_of_mixed_shapes():
    """q -> o -> up -> down -> q' (hidden, hidden, MLP x hidden, hidden x MLP,
    hidden): each launch reads the previous launch's output, all captured in
    one CUDA graph on a side stream and replayed twice."""
    M = 4
    shapes = [(HIDDEN, HIDDEN), (HIDDEN, HIDDEN), (MLP, HIDDEN), (HIDDEN, MLP), (HIDDEN, HIDDEN)]
    # weight_scale_2 = 1 / (rms weight * sqrt(K)) keeps the chained values near
    # unit scale (the rms of an E2M1 code times a scale uniform in [2^-4, 4] is
    # about 6.8).
    probs = [wl.make_fp4(M, N, K, 16, oracle.BF16, seed=60 + i, ws2=1.0 / (6.8 * K ** 0.5),
                         bias_sigma=0.02 if i % 2 else None)
             for i, (N, K) in enumerate(shapes)]
    devs = [fp4_dev(p) for p in probs]
    x0 = act_to_dev(wl.gen_activation(M, HIDDEN, oracle.BF16, 61), oracle.BF16)
    outs = [torch.empty(M, N, dtype=torch.bfloat16, device=DEV) for (N, _) in shapes]
    stream = torch.cuda.Stream(DEV)

    def step():
        cur = x0
        for d, y in zip(devs, outs):
            wq.fp4_weight_matmul(cur, d["B"], d["ws"], d["ws2"], d["bias"], 16, out=y,
                                 stream=stream)
            cur = y

    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        step()                       # one-time library setup outside the capture
        stream.synchronize()
        with torch.cuda.graph(g, stream=stream):
            step()
    replays = []
    for _ in range(2):
        for y in outs:
            y.fill_(float("nan"))
        g.replay()
        stream.synchronize()
        assert wq.device_status() == 0
        replays.append([bits_of(y) for y in outs])
    for a, b in zip(replays[0], replays[1]):
        assert np.array_equal(a, b)
    inp = bits_of(x0)
    for i, (p, y) in enumerate(zip(probs, outs)):
        q = wl.Fp4Problem(p.M, p.N, p.K, 16, p.dtype, inp, p.B_packed, p.weight_scale,
                          p.weight_scale_2, p.bias)
        Yr, S = _ref(q)
        assert_within_tolerance(y, Yr, S, q.dtype, f"chain layer {i} {p.N}x{p.K}")
        inp = replays[0][i]
