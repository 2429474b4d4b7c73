"""Parity at the full layer sizes the pages name, in the launch configuration
the benchmark times: Mixtral-8x7B-shaped (m=4096, p=14336, E=8, top-2,
SwiGLU, bf16 and int8 weights) at the decode batches T = 1, 4, 16, 64, and
Phi-3.5-MoE-shaped (m=4096, p=6400, E=16) with uniform and temporally local
routing.  The oracle evaluates a seeded sample of tokens one by one; routing
tables are checked in full."""
import numpy as np
import pytest
import torch

import mixture_experts_layer_gemm_gb300 as moe
import oracle
import workloads as wl
from gpu_util import Run, max_token_rel_l2, oracle_quantized
from test_gpu_parity import check_routing

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def mixtral():
    return wl.make_layer(wl.MIXTRAL, seed=0, device="cuda")


@pytest.fixture(scope="module")
def mixtral_lib(mixtral):
    ml = moe.MoELayer(mixtral, 64, with_logits=True)
    yield ml
    ml.close()


@pytest.fixture(scope="module")
def mixtral_q(mixtral):
    """The oracle's own int8 codes and scales of the Mixtral-shaped experts."""
    return oracle_quantized(mixtral)


@pytest.fixture(scope="module")
def phi():
    return wl.make_layer(wl.PHI35, seed=0, device="cuda")


def _sample(T, n, seed):
    if T <= n:
        return np.arange(T)
    return np.sort(np.random.default_rng(seed).choice(T, size=n, replace=False))


def _check(ml, layer, T, seed, n_sample, tol, locality=0.0, quantized=None):
    x = wl.make_tokens(layer.shape, T, seed=seed, locality=locality, device="cuda")
    run = Run(ml, x)
    assert ml.sync_check()[0] == moe.MOE_OK
    ids, w = check_routing(run, layer, x)
    toks = _sample(T, n_sample, seed)
    ref = oracle.layer(x, layer.w1, layer.w2, layer.w3, ids, w, oracle.SWIGLU, tokens=toks)
    rel, glob = max_token_rel_l2(run.y_np[toks], ref)
    assert rel <= tol, (rel, glob)
    if quantized is not None:
        q = quantized
        refq = oracle.layer(x, q["w1"], q["w2"], q["w3"], ids, w, oracle.SWIGLU,
                            scales=(q["s1"], q["s2"], q["s3"]), tokens=toks)
        relq, _ = max_token_rel_l2(run.y_np[toks], refq)
        assert relq <= 1e-2, (relq, rel)
    return run


@pytest.mark.parametrize("T", wl.DECODE_TOKENS)
def test_mixtral_decode_bf16(mixtral, mixtral_lib, T):
    run = _check(mixtral_lib, mixtral, T, seed=100 + T, n_sample=8, tol=1e-2)
    assert run.counts.sum() == 2 * T


def test_mixtral_decode_int8(mixtral, mixtral_q):
    shape = wl.MIXTRAL.with_weight("i8")
    layer = wl.Layer(shape, mixtral.w_router, None, mixtral.w1, mixtral.w2, mixtral.w3)
    ml = moe.MoELayer(layer, 64, with_logits=True)
    q = mixtral_q
    codes, scales = moe.moe_layer_read_expert(ml.handle, 5, 2, (shape.p, shape.m), np.int8)
    np.testing.assert_array_equal(codes, q["w2"][5])
    np.testing.assert_array_equal(scales, q["s2"][5])
    for T in (1, 16, 64):
        _check(ml, layer, T, seed=200 + T, n_sample=6, tol=3e-2, quantized=q)
    ml.close()


@pytest.mark.parametrize("T,locality", [(1, 0.0), (8, 0.0), (64, 0.0), (64, 0.5)])
def test_phi35_decode(phi, T, locality):
    ml = moe.MoELayer(phi, 64, with_logits=True)
    run = _check(ml, phi, T, seed=300 + T, n_sample=8, tol=1e-2, locality=locality)
    if locality:
        # copied rows keep their predecessor's expert set exactly
        x = wl.make_tokens(phi.shape, T, seed=300 + T, locality=locality, device="cuda")
        same = [t for t in range(1, T) if np.array_equal(x[t], x[t - 1])]
        assert same and all(np.array_equal(run.ids[t], run.ids[t - 1]) for t in same)
    ml.close()


@pytest.mark.parametrize("T", [512, 2048, 8192])
def test_mixtral_batch_zipf(mixtral, T):
    """Batch / prefill with Zipf(1.2) expert popularity (router bias)."""
    shape = wl.MIXTRAL.with_zipf(1.2)
    layer = wl.Layer(shape, mixtral.w_router, wl.zipf_bias(shape.E, 1.2), mixtral.w1, mixtral.w2,
                     mixtral.w3)
    ml = moe.MoELayer(layer, T, with_logits=True)
    run = _check(ml, layer, T, seed=400 + T, n_sample=8, tol=1e-2)
    assert run.counts[0] == run.counts.max()
    ml.close()


@pytest.mark.parametrize("T", [512, 2048])
def test_mixtral_batch_zipf_int8(mixtral, mixtral_q, T):
    """The batch regime with int8 weights (tensor cores, codes widened in
    tensor memory): against the original weights at 3e-2 and the oracle's own
    dequantised weights at 1e-2."""
    shape = wl.MIXTRAL.with_zipf(1.2).with_weight("i8")
    layer = wl.Layer(shape, mixtral.w_router, wl.zipf_bias(shape.E, 1.2), mixtral.w1, mixtral.w2,
                     mixtral.w3)
    ml = moe.MoELayer(layer, T, with_logits=True)
    _check(ml, layer, T, seed=450 + T, n_sample=6, tol=3e-2, quantized=mixtral_q)
    ml.close()


@pytest.mark.parametrize("T", [512, 4096])
def test_phi35_batch(phi, T):
    ml = moe.MoELayer(phi, T, with_logits=True)
    _check(ml, phi, T, seed=500 + T, n_sample=8, tol=1e-2)
    ml.close()
