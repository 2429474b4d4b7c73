"""moe_forward_static_scratch: the forward pass for callers that cannot
allocate device memory while they run -- a serving engine whose allocator
already holds all free device memory, a loop that cannot take cudaMalloc's
implicit synchronisation -- with its scratch in a static array inside the
library.

It runs the decode kernels with the decode launch plan, so with moe_forward
held to the decode regime the two must give the same bits.  Checked through
the C ABI for calls in a row, on a small layer and on a Phi-3.5-MoE-shaped one
(m=4096, p=6400, E=16), whose T = 1 plans split the up projection (the split
partial sums sit in the static array too), against moe_forward bit for bit and against the fp64
oracle per token; and for its size limit.  This file is collected last so
that a run stopping at the first failure has run every other test first; it
passes alone in a fresh process too."""
import numpy as np
import pytest
import torch

import mixture_experts_layer_gemm_gb300 as moe
import oracle
import workloads as wl
from gpu_util import TOL, from_device, max_token_rel_l2, oracle_quantized, to_device

pytestmark = pytest.mark.gpu

SHAPE = wl.LayerShape("noalloc-swiglu", m=512, p=1024, E=8, k=2, expert=wl.SWIGLU, act="bf16",
                      weight="bf16")


def _forward_both(ml, x_np):
    """Route once, then moe_forward (held to the decode regime) and the
    static-scratch forward on the same routing; both outputs as bf16 bits,
    with the routing the library chose."""
    x = to_device(x_np)
    T = x_np.shape[0]
    ml.route(x)
    y_ref = torch.empty((T, ml.shape.m), dtype=torch.bfloat16, device="cuda")
    y_new = torch.full((T, ml.shape.m), float("nan"), dtype=torch.bfloat16, device="cuda")
    ml.forward(x, y_ref)
    moe.moe_forward_static_scratch(ml.handle, x, ml.routing, y_new)
    torch.cuda.synchronize()
    assert ml.sync_check()[0] == moe.MOE_OK
    n = T * ml.shape.k
    ids = from_device(ml.topk_ids[:n]).reshape(T, ml.shape.k)
    w = from_device(ml.topk_w[:n]).reshape(T, ml.shape.k).astype(np.float64)
    return from_device(y_ref), from_device(y_new), ids, w


def _check_calls(ml, layer, tokens, seed, device="cpu", quantized=None):
    """Two or more calls in a row: same bits as moe_forward, oracle parity."""
    tol = TOL[layer.shape.weight]
    for call, T in enumerate(tokens):
        x = wl.make_tokens(layer.shape, T, seed=seed + call, device=device)
        runs0 = ml.stats().gemv_runs
        y_ref, y_new, ids, w = _forward_both(ml, x)
        assert ml.stats().gemv_runs == runs0 + 2, "both forwards take the decode kernels"
        np.testing.assert_array_equal(y_new, y_ref, err_msg=f"call {call}, T = {T}")
        ref = oracle.layer(x, layer.w1, layer.w2, layer.w3, ids, w, oracle.SWIGLU)
        rel, glob = max_token_rel_l2(y_new, ref)
        assert rel <= tol, (call, T, rel, glob)
        if quantized is not None:  # against the oracle on the library's own int8 codes
            q = quantized
            refq = oracle.layer(x, q["w1"], q["w2"], q["w3"], ids, w, oracle.SWIGLU,
                                scales=(q["s1"], q["s2"], q["s3"]))
            relq, _ = max_token_rel_l2(y_new, refq)
            assert relq <= 1e-2, (call, T, relq)


@pytest.mark.parametrize("weight", ["bf16", "i8"])
def test_static_scratch_matches_forward_twice(weight):
    shape = SHAPE if weight == "bf16" else SHAPE.with_weight("i8")
    layer = wl.make_layer(shape, seed=31)
    ml = moe.MoELayer(layer, 64)
    ml.set_regime(moe.REGIME_DECODE)
    q = oracle_quantized(layer) if weight == "i8" else None
    assert ml.plan(1).splits_up > 1 and ml.plan(16).splits_up == 1
    _check_calls(ml, layer, (16, 1, 9), seed=40, quantized=q)
    ml.close()


@pytest.mark.parametrize("weight", ["bf16", "i8"])
def test_static_scratch_split_up_projection(weight):
    """Phi-3.5-MoE-shaped layer at T = 1, 4, 1: the T = 1 plan splits the up
    projection, so its gate and up partial sums live in the static array."""
    shape = wl.PHI35 if weight == "bf16" else wl.PHI35.with_weight("i8")
    layer = wl.make_layer(shape, seed=34, device="cuda")
    ml = moe.MoELayer(layer, 16)
    ml.set_regime(moe.REGIME_DECODE)
    plans = {T: ml.plan(T) for T in (1, 4)}
    assert all(moe.PATHS[p.path] == "gemv" for p in plans.values())
    assert plans[1].splits_up > 1, plans[1].splits_up
    q = oracle_quantized(layer) if weight == "i8" else None
    _check_calls(ml, layer, (1, 4, 1), seed=50, device="cuda", quantized=q)
    ml.close()


def test_static_scratch_rejects_requests_beyond_its_size():
    layer = wl.make_layer(wl.LayerShape("noalloc-wide", m=4096, p=14336, E=8, k=2,
                                        expert=wl.SWIGLU, act="bf16", weight="bf16"), seed=32,
                          device="cuda")
    ml = moe.MoELayer(layer, 64)
    x = to_device(wl.make_tokens(layer.shape, 64, seed=33, device="cuda"))
    ml.route(x)
    y = torch.empty((64, 4096), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(moe.MoeError) as ei:
        moe.moe_forward_static_scratch(ml.handle, x, ml.routing, y)
    assert ei.value.status == moe.MOE_ERR_INVALID_ARG
    assert "static scratch holds" in str(ei.value)
    ml.close()
