"""Pins of the fp64 CPU oracle to facts outside itself (CPU only, no GPU).

Each test ties one oracle function to something it does not compute itself:
a library routine on a special case, brute force on tiny inputs, a closed form
printed on the pages, an invariant, or a hand-worked golden value.  The inputs
are chosen so that a dropped term, a wrong sign or index, or a transposed
operand in the oracle fails at least one of them (m != p everywhere).
"""
import itertools
import json
import os

import numpy as np
import pytest

import oracle
import workloads as wl

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rng(seed):
    return np.random.default_rng(seed)


def _f64(a):
    """Exact fp64 value of an fp32 or bf16-pattern array."""
    if a.dtype == np.uint16:
        return wl.bf16_bits_to_f32(a).astype(np.float64)
    return a.astype(np.float64)


def _silu(z):
    return z / (1.0 + np.exp(-z))


# --------------------------------------------------------------------------
# router GEMM
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_router_logits_match_numpy_matmul(dtype):
    r = _rng(1)
    T, m, E = 7, 40, 6
    x = r.standard_normal((T, m)).astype(np.float32)
    w = r.standard_normal((m, E)).astype(np.float32)
    b = r.standard_normal(E)
    if dtype == "bf16":
        x, w = wl.f32_to_bf16_bits(x), wl.f32_to_bf16_bits(w)
    logits, mag = oracle.router_logits(x, w, b, with_abssum=True)
    ref = _f64(x) @ _f64(w) + b
    np.testing.assert_allclose(logits, ref, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(mag, np.abs(_f64(x)) @ np.abs(_f64(w)), rtol=1e-12)


def test_router_logits_one_hot():
    m, E = 5, 3
    x = np.zeros((1, m), np.float32)
    x[0, 3] = 2.0
    w = np.zeros((m, E), np.float32)
    w[3, 1] = -1.5
    w[2, 2] = 7.0  # multiplied by x[0,2] = 0
    logits = oracle.router_logits(x, w)
    np.testing.assert_array_equal(logits, [[0.0, -3.0, 0.0]])


# --------------------------------------------------------------------------
# top-k
def _brute_topk(l, k):
    """Max-sum k-subset, lexicographically smallest id set among ties; then
    ordered by (logit desc, id asc)."""
    E = len(l)
    best, best_sum = None, None
    for sub in itertools.combinations(range(E), k):  # lexicographic order
        s = sum(l[e] for e in sub)
        if best is None or s > best_sum:
            best, best_sum = sub, s
    return sorted(best, key=lambda e: (-l[e], e))


@pytest.mark.parametrize("E,k", [(2, 1), (4, 2), (8, 2), (8, 3), (6, 6), (16, 2)])
def test_topk_brute_force_with_ties(E, k):
    r = _rng(E * 10 + k)
    # small integer logits force many exact ties; add a few continuous rows
    L = np.concatenate([r.integers(-2, 3, size=(60, E)).astype(np.float64),
                        r.standard_normal((20, E))])
    L[0] = 0.0  # all tied
    ids, w = oracle.topk(L, k)
    for t in range(L.shape[0]):
        assert list(ids[t]) == _brute_topk(list(L[t]), k), t


@pytest.mark.parametrize("E,k", [(8, 1), (8, 2), (16, 2), (5, 4)])
def test_topk_weights_equal_renormalised_full_softmax(E, k):
    L = _rng(3).standard_normal((50, E)) * 3.0
    ids, w = oracle.topk(L, k)
    sm = np.exp(L - L.max(axis=1, keepdims=True))
    sm /= sm.sum(axis=1, keepdims=True)
    picked = np.take_along_axis(sm, ids.astype(np.int64), axis=1)
    np.testing.assert_allclose(w, picked / picked.sum(axis=1, keepdims=True), rtol=1e-12)
    np.testing.assert_allclose(w.sum(axis=1), 1.0, atol=1e-12)
    assert np.all(np.diff(w, axis=1) <= 0)  # slot 0 carries the largest weight


def test_topk_k2_sigmoid_and_k1_unit_weight():
    L = _rng(4).standard_normal((40, 8))
    ids, w = oracle.topk(L, 2)
    gap = L[np.arange(40), ids[:, 0]] - L[np.arange(40), ids[:, 1]]
    np.testing.assert_allclose(w[:, 0], 1.0 / (1.0 + np.exp(-gap)), rtol=1e-13)
    _, w1 = oracle.topk(L, 1)
    np.testing.assert_array_equal(w1, 1.0)


def test_topk_distinct_and_in_range():
    L = _rng(5).integers(0, 2, size=(100, 8)).astype(np.float64)
    ids, _ = oracle.topk(L, 3)
    assert ids.min() >= 0 and ids.max() < 8
    for row in ids:
        assert len(set(row)) == 3


# --------------------------------------------------------------------------
# histogram / scan / stable scatter
@pytest.mark.parametrize("T,k,E", [(1, 1, 1), (16, 2, 8), (33, 2, 8), (64, 3, 16), (5, 2, 64)])
def test_permute_matches_stable_sort(T, k, E):
    ids = _rng(T + E).integers(0, E, size=(T, k)).astype(np.int32)
    counts, offsets, gather, scatter = oracle.permute(ids, E)
    flat = ids.reshape(-1)
    np.testing.assert_array_equal(counts, np.bincount(flat, minlength=E))
    np.testing.assert_array_equal(offsets, np.concatenate([[0], np.cumsum(counts)]))
    np.testing.assert_array_equal(gather, np.argsort(flat, kind="stable"))
    # invariants: sum of counts = T*k, bijection, inverse pair, sorted segments
    assert counts.sum() == T * k
    assert sorted(gather) == list(range(T * k))
    np.testing.assert_array_equal(scatter[gather], np.arange(T * k))
    for e in range(E):
        seg = gather[offsets[e]:offsets[e + 1]]
        assert np.all(flat[seg] == e) and np.all(np.diff(seg) > 0)


def test_permute_then_unpermute_is_identity():
    T, k, E, m = 20, 2, 8, 9
    ids = _rng(9).integers(0, E, size=(T, k)).astype(np.int32)
    _, _, gather, scatter = oracle.permute(ids, E)
    rows = _rng(10).standard_normal((T * k, m))
    permuted = rows[gather]
    np.testing.assert_array_equal(permuted[scatter], rows)


def test_permute_rejects_out_of_range_ids():
    with pytest.raises(oracle.OracleError):
        oracle.permute(np.array([[0, 8]], np.int32), 8)


# --------------------------------------------------------------------------
# int8 quantiser
def test_quantize_golden_columns():
    cases = json.load(open(os.path.join(GOLDEN, "int8_quant_cases.json")))["cases"]
    rows = max(len(c["column"]) for c in cases)
    W = np.zeros((rows, len(cases)), np.float32)
    for j, c in enumerate(cases):
        W[:len(c["column"]), j] = c["column"]
        # pad rows repeat a zero, which quantises to 0 under any scale
    q, s = oracle.quantize_cols(W)
    for j, c in enumerate(cases):
        assert s[j] == np.float32(c["scale"]), c["note"]
        assert list(q[:len(c["column"]), j]) == c["codes"], c["note"]


def test_quantize_error_bound_and_extremes():
    W = wl.f32_to_bf16_bits(_rng(11).standard_normal((64, 24)).astype(np.float32) * 0.05)
    q, s = oracle.quantize_cols(W)
    Wf = _f64(W)
    err = np.abs(Wf - q.astype(np.float64) * s.astype(np.float64))
    # half a step, plus the fp32 rounding of a quotient of magnitude <= 127
    assert np.all(err <= s.astype(np.float64) * (0.5 + 128 * 2.0 ** -24))
    assert np.all(np.abs(q).max(axis=0) == 127)


# --------------------------------------------------------------------------
# expert MLP
@pytest.mark.parametrize("kind", [oracle.RELU2, oracle.SWIGLU])
def test_op_count_matches_closed_form(kind):
    """HARMOEny write-up, part 3.2: |O| = q p (2m-1) + q m (2p-1) for q tokens
    through the two-matrix expert; the gated form has one more m x p product."""
    T, m, p, E, k = 11, 6, 10, 4, 2
    r = _rng(12)
    x = r.standard_normal((T, m)).astype(np.float32)
    w1 = [r.standard_normal((m, p)).astype(np.float32) for _ in range(E)]
    w2 = [r.standard_normal((p, m)).astype(np.float32) for _ in range(E)]
    w3 = [r.standard_normal((m, p)).astype(np.float32) for _ in range(E)] \
        if kind == oracle.SWIGLU else None
    ids = np.array([r.choice(E, size=k, replace=False) for _ in range(T)], np.int32)
    weights = np.full((T, k), 0.5)
    _, ops = oracle.layer(x, w1, w2, w3, ids, weights, kind, count_ops=True)
    for e in range(E):
        q = int((ids == e).sum())
        n_up = 2 if kind == oracle.SWIGLU else 1
        O = n_up * q * p * (2 * m - 1) + q * m * (2 * p - 1)
        assert ops[e, 0] + ops[e, 1] == O
        assert ops[e, 2] == q * p                      # one activation per hidden unit
        assert ops[e, 3] == (q * p if kind == oracle.SWIGLU else 0)


@pytest.mark.parametrize("kind,dtype", [(oracle.RELU2, "f32"), (oracle.SWIGLU, "bf16"),
                                        (oracle.RELU2, "bf16")])
def test_single_expert_layer_is_dense_mlp(kind, dtype):
    """E = 1, k = 1: the layer reduces to a dense MLP (numpy fp64 matmul)."""
    T, m, p = 9, 12, 20
    r = _rng(13)
    cast = (lambda a: a) if dtype == "f32" else wl.f32_to_bf16_bits
    x = cast(r.standard_normal((T, m)).astype(np.float32))
    w1 = cast(r.standard_normal((m, p)).astype(np.float32))
    w2 = cast(r.standard_normal((p, m)).astype(np.float32))
    w3 = cast(r.standard_normal((m, p)).astype(np.float32)) if kind == oracle.SWIGLU else None
    ids = np.zeros((T, 1), np.int32)
    y = oracle.layer(x, [w1], [w2], None if w3 is None else [w3], ids, np.ones((T, 1)), kind)
    X, W1, W2 = _f64(x), _f64(w1), _f64(w2)
    if kind == oracle.SWIGLU:
        H = _silu(X @ W1) * (X @ _f64(w3))
    else:
        H = np.maximum(X @ W1, 0.0)
    np.testing.assert_allclose(y, H @ W2, rtol=1e-11, atol=1e-11)


def test_identical_experts_make_output_routing_independent():
    T, m, p, E, k = 10, 8, 14, 5, 2
    r = _rng(14)
    x = r.standard_normal((T, m)).astype(np.float32)
    w1 = r.standard_normal((m, p)).astype(np.float32)
    w2 = r.standard_normal((p, m)).astype(np.float32)
    w3 = r.standard_normal((m, p)).astype(np.float32)
    logits = r.standard_normal((T, E))
    ids, w = oracle.topk(logits, k)
    y = oracle.layer(x, [w1] * E, [w2] * E, [w3] * E, ids, w, oracle.SWIGLU)
    for t in range(T):
        _, out = oracle.expert(x[t], w1, w2, w3, oracle.SWIGLU)
        np.testing.assert_allclose(y[t], out, rtol=1e-12, atol=1e-12)


def test_weighted_combine_of_distinct_experts():
    """y_t = sum_j w_j expert_{e_j}(x_t): checked against separate expert calls."""
    T, m, p, E, k = 6, 7, 9, 4, 3
    r = _rng(15)
    x = wl.f32_to_bf16_bits(r.standard_normal((T, m)).astype(np.float32))
    w1 = [wl.f32_to_bf16_bits(r.standard_normal((m, p)).astype(np.float32)) for _ in range(E)]
    w2 = [wl.f32_to_bf16_bits(r.standard_normal((p, m)).astype(np.float32)) for _ in range(E)]
    ids, w = oracle.topk(r.standard_normal((T, E)), k)
    y = oracle.layer(x, w1, w2, None, ids, w, oracle.RELU2)
    ysub = oracle.layer(x, w1, w2, None, ids, w, oracle.RELU2, tokens=[4, 1])
    for t in range(T):
        ref = sum(w[t, j] * oracle.expert(x[t], w1[ids[t, j]], w2[ids[t, j]])[1]
                  for j in range(k))
        np.testing.assert_allclose(y[t], ref, rtol=1e-12, atol=1e-12)
    np.testing.assert_array_equal(ysub, y[[4, 1]])


def test_one_hot_expert_picks_single_entries():
    m, p = 4, 6
    x = np.zeros(m, np.float32)
    x[1] = 2.0
    w1 = np.zeros((m, p), np.float32)
    w1[1, 5] = 3.0
    w1[2, 0] = 9.0          # x[2] = 0: must not contribute
    w2 = np.zeros((p, m), np.float32)
    w2[5, 3] = -0.5
    w2[0, 0] = 4.0          # h[0] = 0: must not contribute
    h, out = oracle.expert(x, w1, w2)
    np.testing.assert_array_equal(h, [0, 0, 0, 0, 0, 6.0])
    np.testing.assert_array_equal(out, [0, 0, 0, -3.0])
    # ReLU clips a negative pre-activation
    w1[1, 5] = -3.0
    h, out = oracle.expert(x, w1, w2)
    np.testing.assert_array_equal(out, 0.0)
    # gated form: silu(x.W1) * (x.W3) with closed-form silu(6) = 6 / (1 + e^-6)
    w1[1, 5] = 3.0
    w3 = np.zeros((m, p), np.float32)
    w3[1, 5] = 0.25
    h, out = oracle.expert(x, w1, w2, w3, kind=oracle.SWIGLU)
    assert h[5] == pytest.approx(6.0 / (1.0 + np.exp(-6.0)) * 0.5, rel=1e-15)
    assert out[3] == pytest.approx(-0.5 * h[5], rel=1e-15)


def test_int8_expert_uses_code_times_scale():
    m, p = 8, 10
    r = _rng(16)
    w1 = wl.f32_to_bf16_bits(r.standard_normal((m, p)).astype(np.float32))
    w2 = wl.f32_to_bf16_bits(r.standard_normal((p, m)).astype(np.float32))
    q1, s1 = oracle.quantize_cols(w1)
    q2, s2 = oracle.quantize_cols(w2)
    x = r.standard_normal(m).astype(np.float32)
    h, out = oracle.expert(x, q1, q2, scales=(s1, s2, None))
    D1 = q1.astype(np.float64) * s1.astype(np.float64)
    D2 = q2.astype(np.float64) * s2.astype(np.float64)
    np.testing.assert_allclose(out, np.maximum(x.astype(np.float64) @ D1, 0) @ D2,
                               rtol=1e-12, atol=1e-12)


def test_nonfinite_input_is_rejected():
    x = np.array([[1.0, np.nan]], np.float32)
    with pytest.raises(oracle.OracleError):
        oracle.router_logits(x, np.ones((2, 3), np.float32))


# --------------------------------------------------------------------------
# set-associative expert cache
def _lru_model(n_index, n_way, layers, experts):
    """Independent model: one list per set, most recent at the end."""
    sets = [[] for _ in range(n_index)]
    slots = [[None] * n_way for _ in range(n_index)]
    hits, where = [], []
    for l, e in zip(layers, experts):
        s = l % n_index
        key = (l, e)
        if key in sets[s]:
            hits.append(1)
            sets[s].remove(key)
        else:
            hits.append(0)
            if None in slots[s]:
                slots[s][slots[s].index(None)] = key
            else:
                victim = sets[s].pop(0)
                slots[s][slots[s].index(victim)] = key
        sets[s].append(key)
        where.append(s * n_way + slots[s].index(key))
    return hits, where


def test_cache_replay_hand_trace():
    # 2 sets x 2 ways.  Layer 0 and 2 share set 0, layer 1 uses set 1.
    layers = [0, 0, 0, 0, 0, 1, 2, 0]
    experts = [1, 2, 3, 2, 1, 1, 1, 2]
    hit, slot = oracle.cache_replay(2, 2, layers, experts)
    # (0,1) m->w0; (0,2) m->w1; (0,3) m evicts LRU (0,1) ->w0; (0,2) hit w1;
    # (0,1) m evicts LRU (0,3) ->w0; (1,1) m set1 w0; (2,1) m set0 evicts (0,2) ->w1;
    # (0,2) m evicts LRU (0,1) ->w0
    assert list(hit) == [0, 0, 0, 1, 0, 0, 0, 0]
    assert list(slot) == [0, 1, 0, 1, 0, 2, 1, 0]


def test_cache_replay_matches_independent_model():
    r = _rng(17)
    layers = r.integers(0, 32, size=3000)
    experts = r.integers(0, 8, size=3000)
    for n_index, n_way in [(12, 4), (7, 8), (1, 1), (14, 4)]:
        hit, slot = oracle.cache_replay(n_index, n_way, layers, experts)
        h2, s2 = _lru_model(n_index, n_way, list(layers), list(experts))
        assert list(hit) == h2 and list(slot) == s2


# --------------------------------------------------------------------------
# the cache driven by layer calls, with cross-layer prefetch
def test_cache_calls_without_prefetch_equal_query_replay():
    """Prefetch off: the call replay is the query replay of each call's experts
    in ascending id (the pinned function above)."""
    r = _rng(23)
    E, n_calls = 8, 400
    layers = r.integers(0, 20, size=n_calls)
    counts = r.integers(0, 3, size=(n_calls, E)) * (r.random((n_calls, E)) < 0.4)
    ql, qe = [], []
    for l, c in zip(layers, counts):
        for e in range(E):
            if c[e] > 0:
                ql.append(l)
                qe.append(e)
    for n_index, n_way in [(12, 4), (5, 2), (1, 3)]:
        lay, exp_, kind, slot = oracle.cache_replay_calls(n_index, n_way, layers, counts, 20, 0)
        hit, slot2 = oracle.cache_replay(n_index, n_way, ql, qe)
        assert list(lay) == ql and list(exp_) == qe
        assert list(kind) == list(hit) and list(slot) == list(slot2)


def test_cache_calls_hand_trace_prefetch_used():
    # 2 sets x 2 ways, layers 0 and 1, prefetch 2.  Call 0 (layer 0, experts
    # 0 and 1) misses twice into set 0, then prefetches (1,0) and (1,1) into
    # set 1; call 1 (layer 1, same experts) finds both prefetched (kind 3);
    # call 2 repeats layer 1: plain hits.
    counts = np.array([[2, 1, 0], [1, 1, 0], [1, 1, 0]])
    lay, exp_, kind, slot = oracle.cache_replay_calls(2, 2, [0, 1, 1], counts, 2, 2)
    assert list(lay) == [0, 0, 1, 1, 1, 1, 1, 1]
    assert list(exp_) == [0, 1, 0, 1, 0, 1, 0, 1]
    assert list(kind) == [0, 0, 2, 2, 3, 3, 1, 1]
    assert list(slot) == [0, 1, 2, 3, 2, 3, 2, 3]


def test_cache_calls_hand_trace_prefetch_evicted():
    # 2 sets x 2 ways, 3 layers, prefetch 2.
    # call 0, layer 0, counts (1,0,2): (0,0) miss w0, (0,2) miss w1; prefetch for
    #   layer 1 by count: e2 then e0 -> set 1 w0, w1.
    # call 1, layer 1, counts (0,3,1): (1,1) miss evicts LRU (1,2) -> slot 2;
    #   (1,2) now misses, evicts LRU (1,0) -> slot 3; prefetch for layer 2:
    #   e1 (3 tokens) then e2 -> set 0, evicting (0,0) then (0,2).
    # call 2, layer 0, counts (1,1,0): both miss (evicting (2,1), (2,2));
    #   prefetch e0, e1 (tie, lower id first) for layer 1: (1,0) evicts (1,1)
    #   at slot 2, then (1,1) is gone and evicts (1,2) at slot 3.
    counts = np.array([[1, 0, 2], [0, 3, 1], [1, 1, 0]])
    lay, exp_, kind, slot = oracle.cache_replay_calls(2, 2, [0, 1, 0], counts, 3, 2)
    assert list(lay) == [0, 0, 1, 1, 1, 1, 2, 2, 0, 0, 1, 1]
    assert list(exp_) == [0, 2, 2, 0, 1, 2, 1, 2, 0, 1, 0, 1]
    assert list(kind) == [0, 0, 2, 2, 0, 0, 2, 2, 0, 0, 2, 2]
    assert list(slot) == [0, 1, 2, 3, 2, 3, 0, 1, 0, 1, 2, 3]


@pytest.mark.parametrize("a,L,S", [(2, 6, 4), (3, 4, 3), (1, 8, 2)])
def test_cache_calls_closed_form_repeated_expert_set(a, L, S):
    """Every layer picks the same a experts at every step, each layer owns a
    set of at least a ways.  Without prefetch: L a misses then hits.  With
    prefetch >= a: only layer 0 misses at step 0; layers 1..L-1 find their a
    experts prefetched (kind 3); everything after is a plain hit; (L-1) a
    prefetch inserts in total."""
    E = 8
    counts = np.zeros((S * L, E), np.int32)
    counts[:, :a] = np.arange(a, 0, -1)
    layers = np.tile(np.arange(L), S)
    _, _, k0, _ = oracle.cache_replay_calls(L, a, layers, counts, L, 0)
    assert (k0 == 0).sum() == L * a and (k0 == 1).sum() == (S - 1) * L * a
    _, _, k1, _ = oracle.cache_replay_calls(L, a, layers, counts, L, a)
    assert (k1 == 0).sum() == a
    assert (k1 == 3).sum() == (L - 1) * a
    assert (k1 == 2).sum() == (L - 1) * a
    assert (k1 == 1).sum() == (S - 1) * L * a


def test_cache_calls_prefetch_invariants():
    r = _rng(29)
    E, n_layers = 8, 32
    n_calls = 32 * 20
    layers = np.tile(np.arange(n_layers), 20)
    counts = (r.random((n_calls, E)) < 0.3) * r.integers(1, 5, size=(n_calls, E))
    for n_index, n_way, pf in [(12, 4, 2), (12, 4, 8), (7, 2, 1), (1, 4, 4)]:
        lay, exp_, kind, slot = oracle.cache_replay_calls(n_index, n_way, layers, counts,
                                                          n_layers, pf)
        assert np.all(slot // n_way == lay % n_index)  # every entry in its layer's set
        if n_index == 1:
            assert not np.any(kind >= 2)  # the next layer shares the set: no prefetch
        # a first use of a prefetched entry follows a prefetch insert of the same
        # (layer, expert) into the same slot
        last = {}
        for l, e, k, s in zip(lay, exp_, kind, slot):
            if k == 2:
                last[(l, e)] = s
            elif k == 3:
                assert last.get((l, e)) == s
                del last[(l, e)]
        # prefetch inserts per call never exceed the prefetch count
        demand = kind != 2
        assert (kind == 2).sum() <= pf * n_calls
        assert demand.sum() == int((counts > 0).sum())
