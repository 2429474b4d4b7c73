"""Expert parallelism with token rebalancing (HARMOEny write-up, 三 3.1-3.3),
host logic only: the rebalancing plan on hand-built request tables whose
outcome is worked out by hand, invariants on random tables, the threshold q
against the expert-cost formula it comes from, and the whole dispatch ->
per-rank experts -> gather -> combine path on two gloo ranks on the host,
whose result must equal the single-rank oracle bit for bit (the per-rank
expert MLPs are the oracle's, so only the data movement is under test)."""
import os
import socket
import sys

import numpy as np
import pytest
import torch.multiprocessing as mp

from mixture_experts_layer_gemm_gb300 import expert_parallel as ep

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_threshold_balances_expert_compute_and_weight_transfer():
    # |O| = q p (2m - 1) + q m (2p - 1) ~ 4 q m p flops at phi flop/s against
    # |E| = 2 m p dtype bytes at beta bytes/s: equal at q = phi dtype / (2 beta)
    phi, dtype, beta, m, p = 1.9e15, 2.0, 2.0e11, 4096, 14336
    q = ep.harmoeny_threshold(phi, dtype, beta)
    t_transfer = 2 * m * p * dtype / beta
    ops_exact = q * p * (2 * m - 1) + q * m * (2 * p - 1)
    assert ops_exact / phi == pytest.approx(t_transfer, rel=1.0 / min(m, p))
    assert 4 * q * m * p / phi == pytest.approx(t_transfer, rel=1e-12)
    with pytest.raises(ValueError):
        ep.harmoeny_threshold(phi, dtype, 0.0)


def test_expert_home_is_contiguous_blocks():
    np.testing.assert_array_equal(ep.expert_home(8, 2), [0, 0, 0, 0, 1, 1, 1, 1])
    np.testing.assert_array_equal(ep.expert_home(8, 4), [0, 0, 1, 1, 2, 2, 3, 3])
    with pytest.raises(ValueError):
        ep.expert_home(6, 4)


def test_hot_expert_moves_to_the_idle_rank():
    # two ranks, experts 0, 1 on rank 0 and 2, 3 on rank 1; expert 0 is hot
    n = np.array([[100, 0, 10, 0],     # rank 0 sends 100 pairs to expert 0
                  [60, 0, 10, 20]])    # rank 1 sends 60 to expert 0
    # loads: rank 0 computes 160, rank 1 computes 40; mean 100.
    # step 1: target rank 0; source rank 0 (100 > 60); expert 0, c = 100 >= q;
    # destination rank 1, capacity 100 - 40 = 60: move 60 of (0 -> 0, expert 0).
    # step 2: loads 100 / 100: target rank 0 (tie -> lower), source rank 1
    # (60 > 40), expert 0, c = 60; the least loaded rank is rank 0 again (tie
    # -> lower), the target itself: no progress, stop.
    plan = ep.rebalance(n, world=2, q=16)
    assert plan.moves == [(0, 0, 0, 1, 60, 100)]
    np.testing.assert_array_equal(plan.load(), [100, 100])
    np.testing.assert_array_equal(plan.alloc[0, 0], [40, 60])
    np.testing.assert_array_equal(plan.alloc[1, 0], [60, 0])
    assert plan.fetch == [[], [0]]   # rank 1 computes expert 0 without holding it


def test_moves_below_the_threshold_are_not_taken():
    n = np.array([[100, 0, 10, 0], [60, 0, 10, 20]])
    plan = ep.rebalance(n, world=2, q=101)   # the largest group is 100 < q
    assert plan.moves == []
    np.testing.assert_array_equal(plan.load(), [160, 40])
    assert plan.fetch == [[], []]


def test_capacity_limits_a_move():
    # four ranks: rank 0 computes 90 of expert 0 from rank 0; the others 10
    n = np.zeros((4, 4), np.int64)
    n[0, 0] = 90
    n[1, 1] = n[2, 2] = n[3, 3] = 10
    plan = ep.rebalance(n, world=4, q=5)
    # mean 30: each idle rank takes 20 of expert 0 in turn (ranks 1, 2, 3)
    assert plan.moves == [(0, 0, 0, 1, 20, 90), (0, 0, 0, 2, 20, 70), (0, 0, 0, 3, 20, 50)]
    np.testing.assert_array_equal(plan.load(), [30, 30, 30, 30])


@pytest.mark.parametrize("seed", range(6))
def test_rebalance_invariants_on_random_tables(seed):
    rng = np.random.default_rng(seed)
    world, E = [(2, 8), (4, 8), (4, 16)][seed % 3]
    pop = rng.dirichlet(np.full(E, 0.3))               # skewed expert popularity
    n = np.stack([rng.multinomial(rng.integers(50, 400), pop) for _ in range(world)])
    q = float(rng.integers(1, 40))
    plan = ep.rebalance(n, world, q)
    np.testing.assert_array_equal(plan.alloc.sum(axis=2), n)     # every pair placed once
    assert (plan.alloc >= 0).all()
    home = ep.expert_home(E, world)
    before = np.bincount(home, weights=n.sum(axis=0), minlength=world)
    assert plan.load().max() <= before.max()
    for s, e, g, d, moved, group in plan.moves:
        assert group >= q and 0 < moved <= group and g != d
    for g in range(world):
        for e in plan.fetch[g]:
            assert home[e] != g and plan.alloc[:, e, g].sum() > 0


def test_destinations_cut_each_expert_into_runs():
    ids = np.array([[0, 2], [0, 1], [2, 0], [0, 3]])
    n = ep.request_table([ids, np.zeros((0, 2), int)], E=4)
    plan = ep.RebalancePlan(alloc=np.zeros((2, 4, 2), np.int64), moves=[], fetch=[[], []])
    plan.alloc[0, 0] = [2, 2]          # expert 0: first two pairs stay, next two go to rank 1
    plan.alloc[0, 1, 0] = 1
    plan.alloc[0, 2, 1] = 2
    plan.alloc[0, 3, 1] = 1
    np.testing.assert_array_equal(plan.alloc.sum(axis=2)[0], n[0])
    dest = ep.destinations(ids, 0, plan)
    # flat pairs: e0 e2 e0 e1 e2 e0 e0 e3 -> expert 0 at 0, 2, 5, 6
    np.testing.assert_array_equal(dest, [0, 1, 0, 0, 1, 1, 1, 1])


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, q_thresh, out_q):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    import torch
    import torch.distributed as dist

    import oracle
    import workloads as wl
    from mixture_experts_layer_gemm_gb300 import expert_parallel as ep_

    dist.init_process_group("gloo", rank=rank, world_size=world)
    shape = wl.TINY_FP32.with_zipf(1.2)        # a skewed router: hot experts
    layer = wl.make_layer(shape, seed=3)
    x = wl.make_tokens(shape, 24, seed=10 + rank)  # each rank's own tokens
    ids, w = oracle.topk(oracle.router_logits(x, layer.w_router, layer.b_router), shape.k)

    def compute(rows, experts, weights):  # the rank's expert MLPs (the oracle's here)
        r = rows.numpy()
        if not len(r):
            return torch.zeros((0, shape.m), dtype=torch.float64)
        y = oracle.layer(r, layer.w1, layer.w2, layer.w3, experts.numpy()[:, None],
                         weights.numpy()[:, None], oracle.RELU2)
        return torch.from_numpy(y)

    y, plan = ep_.ep_forward(torch.from_numpy(x), torch.from_numpy(ids.astype(np.int64)),
                             torch.from_numpy(w), shape.E, q_thresh, compute)
    ref = oracle.layer(x, layer.w1, layer.w2, layer.w3, ids, w, oracle.RELU2)
    dist.destroy_process_group()
    out_q.put((rank, bool(np.array_equal(y.numpy(), ref)), float(np.abs(y.numpy() - ref).max()),
               plan.moves, plan.load().tolist()))


@pytest.mark.parametrize("q_thresh", [1.0, 1e9])
def test_two_rank_dispatch_and_combine_equal_the_single_rank_oracle(q_thresh):
    ctx = mp.get_context("spawn")
    out_q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q_thresh, out_q)) for r in range(2)]
    for p in procs:
        p.start()
    out = sorted(out_q.get(timeout=300) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, equal, err, moves, load in out:
        assert equal, (rank, err)
    moves, load = out[0][3], out[0][4]
    assert out[1][3] == moves                 # both ranks took the same plan
    if q_thresh < 2:
        assert moves, "the Zipf-skewed routing should make the hot expert's rank move pairs"
    else:
        assert moves == []
