"""The resident layer inside a CUDA graph: route + forward issue no host
synchronisation and allocate nothing, so a decode step can be captured once
and replayed (the launch-overhead remedy of the DeepSpeed-Inference article,
part 3.3).  A replay on new token values must give the same bits as the
eager calls on those values, and match the oracle."""
import numpy as np
import pytest
import torch

import mixture_experts_layer_gemm_gb300 as moe
import oracle
import workloads as wl
from gpu_util import TOL, f64, from_device, max_token_rel_l2, to_device

pytestmark = pytest.mark.gpu

SHAPE = wl.LayerShape("graph-swiglu", m=512, p=1024, E=8, k=2, expert=wl.SWIGLU, act="bf16",
                      weight="bf16")


def _capture(layers, xs, ys):
    """One graph holding route + forward of every (layer, x, y) in order."""
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):  # warm-up: kernel attributes, tensor maps
        for ml, x, y in zip(layers, xs, ys):
            ml.route(x)
            ml.forward(x, y)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for ml, x, y in zip(layers, xs, ys):
            ml.route(x)
            ml.forward(x, y)
    return g


@pytest.mark.parametrize("tokens", [(1, 4, 16), (64, 300), (1, 700)])
def test_graph_replay_equals_eager(tokens):
    layer = wl.make_layer(SHAPE, seed=11)
    max_t = max(tokens)
    layers = [moe.MoELayer(layer, max_t) for _ in tokens]
    xs = [torch.empty((T, SHAPE.m), dtype=torch.bfloat16, device="cuda") for T in tokens]
    ys = [torch.empty((T, SHAPE.m), dtype=torch.bfloat16, device="cuda") for T in tokens]
    for x, T in zip(xs, tokens):
        x.copy_(to_device(wl.make_tokens(SHAPE, T, seed=T)))
    g = _capture(layers, xs, ys)
    for rep in range(3):
        new = [wl.make_tokens(SHAPE, T, seed=1000 * rep + T + 1) for T in tokens]
        for x, xn in zip(xs, new):
            x.copy_(to_device(xn))
        g.replay()
        torch.cuda.synchronize()
        got = [from_device(y) for y in ys]
        routed = [(from_device(ml.topk_ids[:T * SHAPE.k]).reshape(T, SHAPE.k),
                   from_device(ml.topk_w[:T * SHAPE.k]).reshape(T, SHAPE.k))
                  for ml, T in zip(layers, tokens)]
        for ml, x, y in zip(layers, xs, ys):  # eager on the same values
            ml.route(x)
            ml.forward(x, y)
        torch.cuda.synchronize()
        for ml, y, yg in zip(layers, ys, got):
            np.testing.assert_array_equal(from_device(y), yg)
            assert ml.sync_check()[0] == moe.MOE_OK
    # the last replay against the oracle, on the routing the replay produced
    # (routing parity itself is checked in the parity tests)
    for xn, yg, (ids, w) in zip(new, got, routed):
        ref = oracle.layer(f64(xn), layer.w1, layer.w2, layer.w3, ids, w, oracle.SWIGLU)
        assert max_token_rel_l2(yg, ref)[0] <= TOL["bf16"]
    for ml in layers:
        ml.close()


def test_sync_check_refuses_a_capturing_stream():
    layer = wl.make_layer(SHAPE, seed=12)
    ml = moe.MoELayer(layer, 4)
    x = to_device(wl.make_tokens(SHAPE, 4, seed=1))
    y = torch.empty_like(x)
    ml.route(x)
    ml.forward(x, y)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        ml.route(x)
        ml.forward(x, y)
        status, _ = ml.sync_check()
        assert status == moe.MOE_ERR_INVALID_ARG
    g.replay()
    torch.cuda.synchronize()
    ml.route(x)  # an eager call moves the layer back to an ordinary stream
    assert ml.sync_check()[0] == moe.MOE_OK
    ml.close()
