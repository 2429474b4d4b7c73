"""Failure detection without a GPU fault: a device wait that can never be
satisfied runs out its poll budget, reports MOE_FLAG_WAIT_TIMEOUT through the
error word, and the context stays usable for ordinary layer work afterwards.
Bad routing data is covered by the parity tests (flags, no faults)."""
import numpy as np
import pytest
import torch

import mixture_experts_layer_gemm_gb300 as moe
import workloads as wl
from gpu_util import Run

pytestmark = pytest.mark.gpu

SHAPE = wl.LayerShape("failure-swiglu", m=256, p=512, E=8, k=2, expert=wl.SWIGLU, act="bf16",
                      weight="bf16")


@pytest.mark.parametrize("polls", [1, 1000, 100000])
def test_bounded_wait_reports_timeout_and_context_survives(polls):
    st, flags = moe.moe_selftest_bounded_wait(polls)
    assert st == moe.MOE_ERR_TIMEOUT
    assert flags & moe.MOE_FLAG_WAIT_TIMEOUT
    # the same context still runs a layer, twice with the same bits
    layer = wl.make_layer(SHAPE, seed=3)
    ml = moe.MoELayer(layer, 32)
    x = wl.make_tokens(SHAPE, 32, seed=4)
    a, b = Run(ml, x), Run(ml, x)
    np.testing.assert_array_equal(a.y_np, b.y_np)
    assert ml.sync_check()[0] == moe.MOE_OK
    ml.close()


def test_selftest_on_a_side_stream():
    s = torch.cuda.Stream()
    st, flags = moe.moe_selftest_bounded_wait(64, stream=s)
    assert st == moe.MOE_ERR_TIMEOUT and flags == moe.MOE_FLAG_WAIT_TIMEOUT
