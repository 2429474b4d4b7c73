"""The seeded input recipe (workloads.py) does what it states.

These pin the synthetic inputs that stand in for the pages' workloads: the
Zipf router bias, the N(0, 1/fan_in) weight scales that make the router
uniform, bf16 rounding to nearest even, the temporal-locality tokens, the
paged decode routing trace and its reuse rates, and reproducibility from the
seed.  Statistical checks use sample sizes whose tolerance is several standard
errors wide, so they are deterministic for the fixed seeds used here."""
import math

import numpy as np

import workloads as wl

SMALL = wl.LayerShape("recipe", m=512, p=1024, E=8, k=2, expert=wl.SWIGLU, act="bf16", weight="bf16")


def test_zipf_bias_is_a_normalised_power_law():
    b = wl.zipf_bias(8, 1.2).astype(np.float64)
    P = np.exp(b)
    assert abs(P.sum() - 1.0) < 1e-6
    assert np.all(np.diff(P) < 0)  # expert 0 hottest
    for e in range(8):
        assert abs(P[e] / P[0] - (e + 1) ** -1.2) < 1e-6
    # the popularity quoted (approximately) for the skewed batch workload
    assert np.allclose(P, [0.43, 0.19, 0.12, 0.08, 0.06, 0.05, 0.04, 0.04], atol=0.006)
    assert np.allclose(wl.zipf_bias(4, 0.0), math.log(0.25))  # s = 0: uniform


def test_bf16_rounding_is_to_nearest_even():
    one = np.float32(1.0)
    ulp = np.float32(2.0 ** -7)  # bf16 spacing in [1, 2)
    cases = {
        float(one): 0x3F80,
        float(one + ulp / 2): 0x3F80,          # tie, even neighbour below
        float(one + 3 * ulp / 2): 0x3F82,      # tie, even neighbour above
        float(one + ulp / 2 + 2 ** -20): 0x3F81,
        -2.0: 0xC000,
    }
    for v, bits in cases.items():
        got = int(wl.f32_to_bf16_bits(np.array([v], np.float32))[0])
        assert got == bits, (v, hex(got))
    x = np.random.default_rng(0).standard_normal(4096).astype(np.float32)
    back = wl.bf16_bits_to_f32(wl.f32_to_bf16_bits(x))
    assert np.all(np.abs(back - x) <= np.abs(x) * 2.0 ** -8)


def test_weight_scales_make_a_uniform_router():
    layer = wl.make_layer(SMALL, seed=3)
    f = lambda a: wl.bf16_bits_to_f32(np.asarray(a)).astype(np.float64)
    m, p = SMALL.m, SMALL.p
    assert abs(f(layer.w_router).std() * math.sqrt(m) - 1.0) < 0.05
    assert abs(f(layer.w1[0]).std() * math.sqrt(m) - 1.0) < 0.01
    assert abs(f(layer.w3[5]).std() * math.sqrt(m) - 1.0) < 0.01
    assert abs(f(layer.w2[7]).std() * math.sqrt(p) - 1.0) < 0.01
    assert layer.b_router is None
    x = f(wl.make_tokens(SMALL, 2048, seed=4))
    assert abs(x.mean()) < 0.01 and abs(x.std() - 1.0) < 0.01
    logits = x @ f(layer.w_router)
    assert abs(logits.std() - 1.0) < 0.1
    # every expert is someone's first choice at a similar rate
    first = np.bincount(np.argmax(logits, axis=1), minlength=SMALL.E) / 2048
    assert first.min() > 0.06 and first.max() < 0.2


def test_zipf_shape_carries_the_bias():
    layer = wl.make_layer(SMALL.with_zipf(1.2), seed=3)
    assert np.array_equal(layer.b_router, wl.zipf_bias(8, 1.2))


def test_draws_are_reproducible_from_the_seed():
    a, b, c = (wl.make_layer(SMALL, seed=s) for s in (5, 5, 6))
    assert np.array_equal(a.w1[2], b.w1[2]) and np.array_equal(a.w_router, b.w_router)
    assert not np.array_equal(a.w1[2], c.w1[2])
    assert not np.array_equal(a.w1[0], a.w1[1])  # experts draw from their own streams
    assert np.array_equal(wl.make_tokens(SMALL, 64, seed=1), wl.make_tokens(SMALL, 64, seed=1))


def test_temporal_locality_copies_the_previous_row():
    x = wl.make_tokens(SMALL, 4000, seed=9, locality=0.5)
    same = np.all(x[1:] == x[:-1], axis=1)
    assert abs(same.mean() - 0.5) < 0.03
    assert not np.any(np.all(wl.make_tokens(SMALL, 4000, seed=9)[1:] == wl.make_tokens(SMALL, 4000, seed=9)[:-1],
                             axis=1))


def test_paged_trace_reuse_rates_and_weights():
    E, k = 8, 2
    ids, w = wl.make_topk_trace(E, k, steps=64, layers=32, batch=16, seed=0)
    assert ids.shape == (64, 32, 16, 2) and w.shape == ids.shape
    assert ids.min() >= 0 and ids.max() < E
    assert np.all(ids[..., 0] != ids[..., 1])  # distinct experts per row
    assert np.allclose(w.sum(-1), 1.0, atol=1e-6) and np.all(w[..., 0] >= w[..., 1])
    # a row repeats the previous layer's set with p = 0.44, plus the chance that a
    # fresh or token-copied set happens to coincide with it
    key = lambda a: np.sort(a, axis=-1)
    same_layer = np.all(key(ids[:, 1:]) == key(ids[:, :-1]), axis=-1).mean()
    assert 0.43 <= same_layer < 0.44 + 0.56 * 0.5 * 0.6
    # layer 0 rows repeat the previous step's set with p = 0.5 (plus chance agreement)
    same_step = np.all(key(ids[1:, 0]) == key(ids[:-1, 0]), axis=-1).mean()
    assert abs(same_step - (0.5 + 0.5 / 28)) < 0.06
