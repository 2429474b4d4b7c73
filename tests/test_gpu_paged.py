"""Paged expert weights (expert-cache article, sections 2.2 and 3.2): experts in
pinned host memory, brought into an N-index x M-way set-associative GPU slot
pool on a copy stream.  Checked against (a) resident layers with the same
weights -- outputs must be bit-identical -- and (b) the oracle's replay of the
same lookups through an LRU set-associative cache -- hits and slots must match
exactly."""
import numpy as np
import pytest
import torch

import mixture_experts_layer_gemm_gb300 as moe
import oracle
import workloads as wl
from gpu_util import Run, to_device

pytestmark = pytest.mark.gpu

SHAPE = wl.LayerShape("paged-swiglu", m=512, p=1024, E=8, k=2, expert=wl.SWIGLU, act="bf16",
                      weight="bf16")


def _expert_bytes(shape):
    probe = moe.MoELayer(wl.make_layer(shape, seed=99), 4)
    nbytes = probe.info().expert_bytes
    probe.close()
    return nbytes


def _run_pair(shape, n_layers, sets, ways, schedule, page_bytes=0, regime=moe.REGIME_AUTO,
              topk_trace=None, prefetch=0, counts_out=None):
    eb = _expert_bytes(shape)
    pool = moe.moe_pool_create(eb * sets * ways, eb, ways, page_bytes)
    if prefetch:
        moe.moe_pool_set_prefetch(pool, prefetch)
    layers = [wl.make_layer(shape, seed=200 + i) for i in range(n_layers)]
    max_t = max(T for _, T in schedule)
    paged = [moe.MoELayer(layers[i], max_t, pool=pool, layer_id=i) for i in range(n_layers)]
    resident = [moe.MoELayer(layers[i], max_t) for i in range(n_layers)]
    for ml in paged + resident:
        ml.set_regime(regime)
    queries = []
    for step, (li, T) in enumerate(schedule):
        x = wl.make_tokens(shape, T, seed=300 + step)
        if topk_trace is None:
            rp, rr = Run(paged[li], x), Run(resident[li], x)
        else:
            ids, w = topk_trace[step]
            rp = Run(paged[li], x, routing="topk", ids=ids, w=w)
            rr = Run(resident[li], x, routing="topk", ids=ids, w=w)
        np.testing.assert_array_equal(rp.y_np, rr.y_np)
        assert paged[li].sync_check()[0] == moe.MOE_OK
        queries += [(li, e) for e in range(shape.E) if rp.counts[e] > 0]
        if counts_out is not None:
            counts_out.append(rp.counts.copy())
    log = moe.moe_pool_query_log(pool)
    stats = [ml.stats() for ml in paged]
    for ml in paged + resident:
        ml.close()
    moe.moe_pool_destroy(pool)
    return eb, queries, log, stats


def _check_log(queries, log, sets, ways):
    layers = np.array([q[0] for q in queries], np.int32)
    experts = np.array([q[1] for q in queries], np.int32)
    hit, slot = oracle.cache_replay(sets, ways, layers, experts)
    np.testing.assert_array_equal(log[0], layers)
    np.testing.assert_array_equal(log[1], experts)
    np.testing.assert_array_equal(log[2], hit)
    np.testing.assert_array_equal(log[3], slot)
    return hit


def test_paged_equals_resident_and_lru_replay():
    sets, ways = 2, 2
    schedule = [(0, 16), (1, 3), (2, 16), (0, 5), (1, 16), (2, 1), (0, 16), (1, 2)]
    eb, queries, log, stats = _run_pair(SHAPE, 3, sets, ways, schedule)
    hit = _check_log(queries, log, sets, ways)
    misses = sum(int(s.slot_misses) for s in stats)
    assert misses == int((hit == 0).sum())
    assert sum(int(s.slot_hits) for s in stats) == int(hit.sum())
    h2d = sum(int(s.h2d_bytes) for s in stats)
    assert misses * eb <= h2d <= misses * (eb + 768)


def test_paged_with_small_pages_and_reuse():
    """One set, 4 ways, a layer revisited with few experts: hits happen and
    16 KB pages split every expert into many copies."""
    sets, ways = 1, 4
    T = 2
    trace = []
    for step in range(6):
        ids = np.array([[0, 1], [1, 2]], np.int32) if step % 2 == 0 else np.array([[2, 0], [0, 1]], np.int32)
        trace.append((ids, np.full((T, 2), 0.5, np.float32)))
    schedule = [(0, T)] * 6
    eb, queries, log, stats = _run_pair(SHAPE, 1, sets, ways, schedule, page_bytes=16384,
                                        topk_trace=trace)
    hit = _check_log(queries, log, sets, ways)
    assert hit.sum() > 0 and int(stats[0].slot_hits) == int(hit.sum())


def test_paged_int8():
    shape = SHAPE.with_weight("i8")
    schedule = [(0, 16), (1, 16), (0, 4), (1, 1)]
    _, queries, log, _ = _run_pair(shape, 2, 1, 2, schedule)
    _check_log(queries, log, 1, 2)


def test_paged_tensor_core_path():
    schedule = [(0, 200), (1, 64), (0, 100)]
    _, queries, log, _ = _run_pair(SHAPE, 2, 2, 2, schedule, regime=moe.REGIME_BATCH)
    _check_log(queries, log, 2, 2)


def test_pool_too_small_for_layer_is_rejected():
    eb = _expert_bytes(SHAPE)
    pool = moe.moe_pool_create(eb, eb // 2, 1, 0)  # slots of half an expert
    with pytest.raises(moe.MoeError) as ei:
        moe.MoELayer(wl.make_layer(SHAPE, seed=5), 4, pool=pool, layer_id=0)
    assert ei.value.status == moe.MOE_ERR_INVALID_ARG
    moe.moe_pool_destroy(pool)


def test_paged_step_time_within_overlap_bounds():
    """Copies and compute overlap: a paged call's time lies between
    max(copy, compute) and copy + compute (the GPU-only form of the decode
    latency model max(comm, T_gpu) of the MoE-Lightning note)."""
    eb = _expert_bytes(SHAPE)
    pool = moe.moe_pool_create(eb * 2, eb, 2, 0)
    layers = [moe.MoELayer(wl.make_layer(SHAPE, seed=400 + i), 16, pool=pool, layer_id=i)
              for i in range(3)]
    xs = [to_device(wl.make_tokens(SHAPE, 16, seed=500 + i)) for i in range(3)]
    y = torch.empty((16, SHAPE.m), dtype=torch.bfloat16, device="cuda")
    for ml, x in zip(layers, xs):  # warm-up
        ml.route(x)
        ml.forward(x, y)
    torch.cuda.synchronize()
    for ml in layers:
        ml.set_timing(True)
        ml.timings(reset=True)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(4):
        for ml, x in zip(layers, xs):
            ml.route(x)
            ml.forward(x, y)
    e1.record()
    torch.cuda.synchronize()
    wall = e0.elapsed_time(e1)
    tim = [ml.timings(reset=True) for ml in layers]
    copy = sum(t["copy"][0] for t in tim)
    compute = sum(sum(v[0] for k, v in t.items() if k != "copy") for t in tim)
    assert copy > 0 and compute > 0
    # event timing adds a little; the host synchronises once per paged call
    assert 0.9 * max(copy, compute) <= wall
    for ml in layers:
        ml.close()
    moe.moe_pool_destroy(pool)


def test_routing_ahead_on_a_side_stream():
    """A step routes all its paged layers first on a side stream and then runs
    their forward calls on the compute stream: each paged call reads its token
    counts on the routing stream and the compute stream waits for that read.
    Outputs equal resident layers' bit for bit and the lookups equal the
    oracle's LRU replay."""
    sets, ways, n_layers, T = 2, 2, 4, 8
    eb = _expert_bytes(SHAPE)
    pool = moe.moe_pool_create(eb * sets * ways, eb, ways, 0)
    layers = [wl.make_layer(SHAPE, seed=600 + i) for i in range(n_layers)]
    paged = [moe.MoELayer(layers[i], T, pool=pool, layer_id=i) for i in range(n_layers)]
    resident = [moe.MoELayer(layers[i], T) for i in range(n_layers)]
    side, main = torch.cuda.Stream(), torch.cuda.current_stream()
    queries = []
    for step in range(3):
        xs = [to_device(wl.make_tokens(SHAPE, T, seed=700 + 10 * step + i)) for i in range(n_layers)]
        ys = [torch.empty((T, SHAPE.m), dtype=torch.bfloat16, device="cuda") for _ in range(n_layers)]
        side.wait_stream(main)  # inputs written, earlier forwards done with the tables
        for ml, x in zip(paged, xs):
            ml.route(x, stream=side)
        for ml, x, y in zip(paged, xs, ys):
            ml.forward(x, y, stream=main)
        torch.cuda.synchronize()
        for i, (ml, x, y) in enumerate(zip(paged, xs, ys)):
            assert ml.sync_check()[0] == moe.MOE_OK
            counts = ml.counts.cpu().numpy()
            queries += [(i, e) for e in range(SHAPE.E) if counts[e] > 0]
            yr = torch.empty_like(y)
            resident[i].route(x)
            resident[i].forward(x, yr)
            torch.cuda.synchronize()
            assert torch.equal(y.view(torch.int16), yr.view(torch.int16)), (step, i)
    _check_log(queries, moe.moe_pool_query_log(pool), sets, ways)
    for ml in paged + resident:
        ml.close()
    moe.moe_pool_destroy(pool)


def _check_calls(schedule, counts, log, sets, ways, n_layers, prefetch, stats):
    lay, exp_, kind, slot = oracle.cache_replay_calls(sets, ways, [li for li, _ in schedule],
                                                      np.array(counts), n_layers, prefetch)
    np.testing.assert_array_equal(log[0], lay)
    np.testing.assert_array_equal(log[1], exp_)
    np.testing.assert_array_equal(log[2], kind)
    np.testing.assert_array_equal(log[3], slot)
    for li in range(n_layers):
        mine = lay == li
        assert int(stats[li].prefetch_hits) == int(((kind == oracle.PREFETCH_HIT) & mine).sum())
        assert int(stats[li].slot_misses) == int(((kind == oracle.MISS) & mine).sum())
    # a prefetch insert for layer l + 1 is issued (and counted) by layer l
    issued = sum(int(st.prefetch_copies) for st in stats)
    assert issued == int((kind == oracle.PREFETCH).sum())
    return kind


def test_cross_layer_prefetch_matches_oracle_and_resident():
    """Layers reuse their predecessor's experts: prefetched experts serve the
    next layer's lookups (kind 3), outputs stay bit-identical to resident layers
    and the pool log equals the oracle's call replay."""
    sets, ways, n_layers, T = 3, 2, 4, 2
    trace, schedule = [], []
    base = [np.array([[0, 1], [1, 0]], np.int32), np.array([[2, 3], [3, 2]], np.int32)]
    for step in range(3):
        for li in range(n_layers):
            ids = base[(li // 2 + step) % 2]  # pairs of consecutive layers share experts
            trace.append((ids, np.full((T, 2), 0.5, np.float32)))
            schedule.append((li, T))
    counts = []
    eb, _, log, stats = _run_pair(SHAPE, n_layers, sets, ways, schedule, topk_trace=trace,
                                  prefetch=2, counts_out=counts)
    kind = _check_calls(schedule, counts, log, sets, ways, n_layers, 2, stats)
    assert (kind == oracle.PREFETCH_HIT).sum() > 0


@pytest.mark.parametrize("prefetch", [1, 8])
def test_cross_layer_prefetch_random_trace(prefetch):
    """A seeded decode trace (copy the previous layer's choice with p = 0.44,
    else the previous step's, else fresh) through 6 layers and 4 sets x 2 ways."""
    sets, ways, n_layers, T, steps = 4, 2, 6, 3, 3
    tr = wl.make_topk_trace(SHAPE.E, SHAPE.k, steps, n_layers, T, seed=7)
    trace, schedule = [], []
    for st_ in range(steps):
        for li in range(n_layers):
            trace.append((tr[0][st_, li], tr[1][st_, li]))
            schedule.append((li, T))
    counts = []
    _, _, log, stats = _run_pair(SHAPE, n_layers, sets, ways, schedule, topk_trace=trace,
                                 prefetch=prefetch, counts_out=counts)
    _check_calls(schedule, counts, log, sets, ways, n_layers, prefetch, stats)


def test_prefetch_count_is_validated():
    eb = _expert_bytes(SHAPE)
    pool = moe.moe_pool_create(eb * 2, eb, 1, 0)
    with pytest.raises(moe.MoeError):
        moe.moe_pool_set_prefetch(pool, -1)
    moe.moe_pool_set_prefetch(pool, 0)
    moe.moe_pool_destroy(pool)


def test_duplicate_layer_id_in_a_pool_is_rejected():
    eb = _expert_bytes(SHAPE)
    pool = moe.moe_pool_create(eb * 4, eb, 2, 0)
    a = moe.MoELayer(wl.make_layer(SHAPE, seed=5), 4, pool=pool, layer_id=3)
    with pytest.raises(moe.MoeError) as ei:
        moe.MoELayer(wl.make_layer(SHAPE, seed=6), 4, pool=pool, layer_id=3)
    assert ei.value.status == moe.MOE_ERR_INVALID_ARG
    a.close()
    b = moe.MoELayer(wl.make_layer(SHAPE, seed=6), 4, pool=pool, layer_id=3)  # id free again
    b.close()
    moe.moe_pool_destroy(pool)


def test_injected_page_copy_failure_rolls_back_the_slot(monkeypatch):
    """MOE_FAULT_COPY_FAIL=n: the n-th page copy is not issued, the forward that
    needed it returns MOE_ERR_CUDA, the half-filled slot is emptied, and the
    next calls copy that expert again and match the resident layer bit for bit."""
    monkeypatch.setenv("MOE_FAULT_COPY_FAIL", "2")  # the third page copy (one page per expert here)
    eb = _expert_bytes(SHAPE)
    pool = moe.moe_pool_create(eb * 8, eb, 4, 0)
    monkeypatch.delenv("MOE_FAULT_COPY_FAIL")
    layer = wl.make_layer(SHAPE, seed=71)
    paged = moe.MoELayer(layer, 16, pool=pool, layer_id=0)
    resident = moe.MoELayer(layer, 16)
    ids = np.array([[0, 1], [2, 3]], np.int32)  # four experts: copies 0, 1, 2 (fails), ...
    w = np.full((2, 2), 0.5, np.float32)
    x = wl.make_tokens(SHAPE, 2, seed=72)
    with pytest.raises(moe.MoeError) as ei:
        Run(paged, x, routing="topk", ids=ids, w=w)
    assert ei.value.status == moe.MOE_ERR_CUDA
    torch.cuda.synchronize()
    for _ in range(2):
        rp = Run(paged, x, routing="topk", ids=ids, w=w)
        rr = Run(resident, x, routing="topk", ids=ids, w=w)
        np.testing.assert_array_equal(rp.y_np, rr.y_np)
    log = moe.moe_pool_query_log(pool)
    # call 1: experts 0, 1 copied, expert 2 failed (logged as a miss); call 2:
    # 0, 1 hit, 2 missed again (the slot was emptied), 3 missed; call 3: all hit
    assert list(log[1]) == [0, 1, 2, 0, 1, 2, 3, 0, 1, 2, 3]
    assert list(log[2]) == [0, 0, 0, 1, 1, 0, 0, 1, 1, 1, 1]
    paged.close()
    resident.close()
    moe.moe_pool_destroy(pool)


def test_host_wait_deadline_returns_timeout_and_the_layer_recovers():
    """A paged forward waits on the host for the token counts with a deadline
    (MOE_OPT_HOST_TIMEOUT_MS).  Device work queued ahead of the counts copy
    that outlasts it makes the call return MOE_ERR_TIMEOUT before any slot is
    looked up; with the limit restored the next calls match the resident
    layer bit for bit."""
    eb = _expert_bytes(SHAPE)
    pool = moe.moe_pool_create(eb * 8, eb, 4, 0)
    layer = wl.make_layer(SHAPE, seed=81)
    paged = moe.MoELayer(layer, 16, pool=pool, layer_id=0)
    resident = moe.MoELayer(layer, 16)
    ids = np.array([[0, 1], [2, 3]], np.int32)
    w = np.full((2, 2), 0.5, np.float32)
    x = wl.make_tokens(SHAPE, 2, seed=82)
    xd = to_device(x)
    y = torch.empty((2, SHAPE.m), dtype=torch.bfloat16, device="cuda")
    paged.route_from_topk(to_device(ids.reshape(-1)), to_device(w.reshape(-1)), T=2)
    paged.set_host_timeout_ms(0)
    torch.cuda._sleep(200_000_000)  # about 0.1 s of device time ahead of the counts copy
    with pytest.raises(moe.MoeError) as ei:
        paged.forward(xd, y)
    assert ei.value.status == moe.MOE_ERR_TIMEOUT
    torch.cuda.synchronize()
    with pytest.raises(moe.MoeError) as ei:
        paged.set_host_timeout_ms(-2)
    assert ei.value.status == moe.MOE_ERR_INVALID_ARG
    paged.set_host_timeout_ms(120000)
    for _ in range(2):
        rp = Run(paged, x, routing="topk", ids=ids, w=w)
        rr = Run(resident, x, routing="topk", ids=ids, w=w)
        np.testing.assert_array_equal(rp.y_np, rr.y_np)
    log = moe.moe_pool_query_log(pool)
    # the timed-out call looked nothing up: four misses, then four hits
    assert list(log[1]) == [0, 1, 2, 3, 0, 1, 2, 3]
    assert list(log[2]) == [0, 0, 0, 0, 1, 1, 1, 1]
    paged.close()
    resident.close()
    moe.moe_pool_destroy(pool)
