"""Seeded random shapes through the whole path, each against the oracle: the
combinations of hidden size, FFN size, expert count, top-k, expert form,
numeric type, batch size and regime that the fixed-shape parity tests do not
pick -- partial vector widths of the combine, last router CTAs with fewer than
16 tokens, a last gather block with fewer than four rows, reduction splits and
128-token tiles of the batch down projection.  Shapes stay inside what the
library accepts (bf16 m, p multiples of 64, int8 of 128, fp32 m of 4; layers
without 128-row tensor-core blocks keep T k <= 512)."""
import numpy as np
import pytest

import mixture_experts_layer_gemm_gb300 as moe
import workloads as wl
from gpu_util import TOL, Run, max_token_rel_l2, oracle_quantized
from test_gpu_parity import check_routing, oracle_y

pytestmark = pytest.mark.gpu


def _cases(n=48, seed=2026):
    rng = np.random.default_rng(seed)
    cases = []
    while len(cases) < n:
        kind = str(rng.choice(["f32", "bf16", "i8"], p=[0.25, 0.5, 0.25]))
        expert = wl.SWIGLU if rng.random() < 0.6 else wl.RELU2
        if kind == "f32":
            m, p = int(rng.integers(1, 48)) * 4, int(rng.integers(1, 64)) * 4
        elif kind == "bf16":
            m, p = int(rng.integers(1, 8)) * 64, int(rng.integers(1, 12)) * 64
        else:
            m, p = int(rng.integers(1, 5)) * 128, int(rng.integers(1, 7)) * 128
        E = int(rng.integers(1, 65))
        k = int(rng.integers(1, min(E, 8) + 1))
        rows_up = 2 * p if expert == wl.SWIGLU else p
        tc = kind != "f32" and m % 128 == 0 and rows_up % 128 == 0
        T = int(rng.integers(1, (300 if tc else max(1, 512 // k)) + 1))
        regime = moe.REGIME_AUTO
        if kind != "f32":
            r = rng.random()
            if r < 0.3 and T * k <= 512:
                regime = moe.REGIME_DECODE
            elif r < 0.6 and tc:
                regime = moe.REGIME_BATCH
        cases.append((kind, expert, m, p, E, k, T, regime))
    return cases


def _id(c):
    kind, expert, m, p, E, k, T, regime = c
    return f"{kind}-{expert}-m{m}-p{p}-E{E}-k{k}-T{T}-r{regime}"


@pytest.mark.parametrize("case", _cases(), ids=_id)
def test_random_shape_matches_oracle(case):
    kind, expert, m, p, E, k, T, regime = case
    act = "f32" if kind == "f32" else "bf16"
    shape = wl.LayerShape(f"fuzz-{kind}", m=m, p=p, E=E, k=k, expert=expert, act=act, weight=kind)
    layer = wl.make_layer(shape, seed=m + 7 * p + 13 * E + k)
    x = wl.make_tokens(shape, T, seed=T + 11)
    ml = moe.MoELayer(layer, T, with_logits=True)
    ml.set_regime(regime)
    run = Run(ml, x)
    assert ml.sync_check()[0] == moe.MOE_OK
    ids, w = check_routing(run, layer, x)
    ref = oracle_y(layer, x, ids, w, oracle_quantized(layer) if kind == "i8" else None)
    rel, _ = max_token_rel_l2(run.y_np, ref)
    assert rel <= (1e-2 if kind == "i8" else TOL[kind]), rel
    ml.close()
