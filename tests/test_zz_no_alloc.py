"""moe_forward_static_scratch: the forward pass for callers that cannot
allocate device memory while they run (its scratch is a static array inside
the library).  Checked through the C ABI against moe_forward on the same
routing, for two calls in a row, and for its size limit.  This file is
collected last so that a run stopping at the first failure has run every
other test first; it passes alone in a fresh process too."""
import numpy as np
import pytest
import torch

import mixture_experts_layer_gemm_gb300 as moe
import workloads as wl
from gpu_util import max_token_rel_l2, to_device, from_device

pytestmark = pytest.mark.gpu

SHAPE = wl.LayerShape("noalloc-swiglu", m=512, p=1024, E=8, k=2, expert=wl.SWIGLU, act="bf16",
                      weight="bf16")


def _forward_both(ml, x_np):
    x = to_device(x_np)
    T = x_np.shape[0]
    ml.route(x)
    y_ref = torch.empty((T, SHAPE.m), dtype=torch.bfloat16, device="cuda")
    y_new = torch.full((T, SHAPE.m), float("nan"), dtype=torch.bfloat16, device="cuda")
    ml.forward(x, y_ref)
    moe.moe_forward_static_scratch(ml.handle, x, ml.routing, y_new)
    torch.cuda.synchronize()
    assert ml.sync_check()[0] == moe.MOE_OK
    return from_device(y_ref), from_device(y_new)


@pytest.mark.parametrize("weight", ["bf16", "i8"])
def test_static_scratch_matches_forward_twice(weight):
    shape = SHAPE if weight == "bf16" else SHAPE.with_weight("i8")
    layer = wl.make_layer(shape, seed=31)
    ml = moe.MoELayer(layer, 64)
    for call, T in enumerate((16, 9)):  # two calls in a row, different batches
        x = wl.make_tokens(shape, T, seed=40 + call)
        y_ref, y_new = _forward_both(ml, x)
        rel, _ = max_token_rel_l2(y_new, wl.bf16_bits_to_f32(y_ref).astype(np.float64))
        assert rel <= 1e-2, (call, rel)
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
