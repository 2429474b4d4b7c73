"""Expert parallelism across ranks with token rebalancing: the host-side
planning and the data movement around the expert MLPs.

Follows the HARMOEny write-up (yejing.asia): part 二 (experts split across
GPUs, one all-to-all that sends every (token, slot) to the GPU holding its
expert and one that brings the results back, and the idle GPUs a hot expert
leaves), part 三 3.1 (token rebalance: greedy moves of requests from the most
loaded GPU to the least loaded one while a move carries at least q requests),
3.2 (the threshold q = phi * dtype / (2 beta) above which a moved expert's
weight transfer hides under its compute, and the prefetch of moved experts)
and 3.3 (the six steps: route, metadata sync, rebalance, dispatch, expert
compute with prefetch, gather).

Readings of points the write-up leaves open (each stated where the code
implements it):
  - load of a GPU: the number of (token, slot) pairs it will compute;
  - expert placement: E / world consecutive experts per rank (expert e on
    rank e // (E / world)); world must divide E;
  - "the remaining request capacity" of the least loaded GPU: the mean load
    over GPUs minus its load, rounded down;
  - which requests of a (source, expert) group move: the plan fixes how many
    of the group go to each GPU; the group's pairs, in flat index order
    t * k + j, are cut into consecutive runs in ascending destination rank;
  - the loop also stops when no move can make progress (capacity 0, or the
    least loaded GPU is the target), so it always ends.

Everything here is host logic: routing tables in, destinations and exchange
orders out, with the exchanges done by torch.distributed all-to-all on the
tensors given (gloo on the host in the tests).  The expert MLPs themselves run
in the function the caller passes (the library's forward pass on a GPU).
"""
from __future__ import annotations

import dataclasses
from typing import Callable, List, Sequence

import numpy as np


def harmoeny_threshold(flops_per_s: float, dtype_bytes: float, link_bytes_per_s: float) -> float:
    """q > phi * dtype / (2 beta): the tokens an expert needs for its compute,
    |O| ~ 4 q m p flops at phi flop/s, to cover the transfer of its weights,
    |E| = 2 m p dtype bytes at beta bytes/s (HARMOEny write-up, 三 3.2)."""
    if flops_per_s <= 0 or dtype_bytes <= 0 or link_bytes_per_s <= 0:
        raise ValueError("flops, dtype bytes and link bandwidth must be positive")
    return flops_per_s * dtype_bytes / (2.0 * link_bytes_per_s)


def expert_home(E: int, world: int) -> np.ndarray:
    """Rank holding each expert: E / world consecutive experts per rank."""
    if world < 1 or E % world:
        raise ValueError(f"world = {world} must divide E = {E}")
    return np.arange(E) // (E // world)


def request_table(ids_per_rank: Sequence[np.ndarray], E: int) -> np.ndarray:
    """n[s, e] = (token, slot) pairs of rank s routed to expert e (the
    metadata each rank shares in step 2: E counts per rank)."""
    world = len(ids_per_rank)
    n = np.zeros((world, E), np.int64)
    for s, ids in enumerate(ids_per_rank):
        ids = np.asarray(ids).reshape(-1)
        if ids.size and (ids.min() < 0 or ids.max() >= E):
            raise ValueError("expert id out of range")
        n[s] = np.bincount(ids, minlength=E)
    return n


@dataclasses.dataclass
class RebalancePlan:
    """alloc[s, e, g]: pairs of source rank s for expert e computed on rank g.
    moves: (source, expert, from rank, to rank, pairs moved, pairs of the
    group chosen) in the order taken; the group has at least q pairs, the
    move at most the destination's capacity.
    fetch[g]: experts rank g computes without holding them (to prefetch)."""
    alloc: np.ndarray
    moves: List[tuple]
    fetch: List[List[int]]

    def load(self) -> np.ndarray:
        return self.alloc.sum(axis=(0, 1))


def rebalance(n: np.ndarray, world: int, q: float, max_moves: int = 10_000) -> RebalancePlan:
    """Token rebalance of the HARMOEny write-up, 三 3.1, on the request table
    n[s, e].  Starting from every pair on its expert's home rank, repeat:
      1. the target g: the rank with the most pairs to compute;
      2. the source s: the rank sending g the most pairs;
      3. the expert e: the expert of g that s's pairs choose most, and c the
         number of those pairs (s -> g, expert e);
      4. stop if c < q (a move that small does not pay for its prefetch);
      5. the destination d: the rank with the fewest pairs; move
         min(c, capacity of d) of them to d, capacity = floor(mean load) -
         load(d);
      6. update the loads and go again.
    Ties go to the lower rank / expert id.  Also stops when no move can make
    progress.  Deterministic: every rank computes the same plan from the same
    table."""
    n = np.asarray(n, np.int64)
    S, E = n.shape
    if S != world:
        raise ValueError("request table must have one row per rank")
    home = expert_home(E, world)
    alloc = np.zeros((world, E, world), np.int64)
    for s in range(world):
        for e in range(E):
            alloc[s, e, home[e]] = n[s, e]
    moves: List[tuple] = []
    total = int(n.sum())
    mean = total // world
    for _ in range(max_moves):
        load = alloc.sum(axis=(0, 1))
        g = int(np.argmax(load))                       # 1. most loaded rank
        to_g = alloc[:, :, g]                          # [s, e] pairs computed on g
        s = int(np.argmax(to_g.sum(axis=1)))           # 2. its largest source
        e = int(np.argmax(to_g[s]))                    # 3. that source's busiest expert on g
        c = int(to_g[s, e])
        if c < q or c == 0:                            # 4. no gain left
            break
        d = int(np.argmin(load))                       # 5. least loaded rank
        cap = mean - int(load[d])
        moved = min(c, cap)
        if d == g or moved <= 0:
            break
        alloc[s, e, g] -= moved                        # 6. update
        alloc[s, e, d] += moved
        moves.append((s, e, g, d, moved, c))
    fetch = [sorted({int(e) for e in range(E) if home[e] != g and alloc[:, e, g].sum() > 0})
             for g in range(world)]
    return RebalancePlan(alloc=alloc, moves=moves, fetch=fetch)


def destinations(ids_local: np.ndarray, rank: int, plan: RebalancePlan) -> np.ndarray:
    """Destination rank of each local (token, slot) pair, in flat index order:
    the pairs of each expert, in flat index order, are cut into consecutive
    runs of plan.alloc[rank, e, g] pairs for g = 0, 1, ...  (reading stated in
    the module header)."""
    ids = np.asarray(ids_local).reshape(-1)
    world = plan.alloc.shape[2]
    dest = np.empty(ids.size, np.int64)
    for e in np.unique(ids):
        idx = np.nonzero(ids == e)[0]                  # flat index order
        runs = plan.alloc[rank, e]
        if int(runs.sum()) != idx.size:
            raise ValueError(f"plan holds {int(runs.sum())} pairs of expert {e}, rank has {idx.size}")
        dest[idx] = np.repeat(np.arange(world), runs)
    return dest


def library_compute(layer_k1, device="cuda"):
    """ep_forward's compute through this library: the received pairs are
    routed as a batch of one-slot tokens (route_from_topk with their expert
    ids and routing weights) on a layer holding the same experts with k = 1,
    whose forward pass returns weight * expert(row) for each.  Returns fp32
    host rows (the layer's output type widened)."""
    import torch

    def compute(rows, experts, weights):
        n = int(rows.shape[0])
        if n == 0:
            return torch.zeros((0, layer_k1.shape.m), dtype=torch.float32)
        x = rows.to(device).contiguous()
        ids = experts.to(torch.int32).to(device)
        w = weights.to(torch.float32).to(device)
        layer_k1.route_from_topk(ids, w, T=n)
        y = torch.empty_like(x)
        layer_k1.forward(x, y)
        torch.cuda.synchronize(device)
        return y.float().cpu()

    return compute


def ep_forward(x_local, ids_local, w_local, E: int, q: float, compute: Callable, group=None):
    """The six steps of the HARMOEny write-up (三 3.3) on one rank.

    x_local [T x m] float tensor, ids_local / w_local [T x k] (step 1, the
    router, already ran).  compute(rows, experts, weights) -> [n x m] returns
    weight * expert(row) for received pairs (the library's expert MLPs on a
    GPU).  Returns y_local [T x m] = sum over slots j, ascending, of the
    pair outputs, and the plan.  All ranks must call it together."""
    import torch
    import torch.distributed as dist

    world = dist.get_world_size(group)
    rank = dist.get_rank(group)
    T, k = ids_local.shape
    m = x_local.shape[1]
    ids = ids_local.reshape(-1).cpu().numpy().astype(np.int64)
    # 2. metadata sync: E pair counts per rank
    counts = torch.from_numpy(np.bincount(ids, minlength=E).astype(np.int64))
    gathered = [torch.zeros(E, dtype=torch.int64) for _ in range(world)]
    dist.all_gather(gathered, counts, group=group)
    n = np.stack([t.numpy() for t in gathered])
    # 3. rebalance (the same plan on every rank)
    plan = rebalance(n, world, q)
    # 4. dispatch: pairs sorted by destination, flat index order inside
    dest = destinations(ids, rank, plan)
    order = np.argsort(dest, kind="stable")
    send_counts = np.bincount(dest, minlength=world)
    recv_counts = torch.zeros(world, dtype=torch.int64)
    dist.all_to_all_single(recv_counts, torch.from_numpy(send_counts.astype(np.int64)), group=group)
    recv_counts = recv_counts.numpy()
    order_t = torch.from_numpy(order)
    send_rows = x_local[order_t // k]
    send_meta = torch.stack([torch.from_numpy(ids[order]).to(torch.float64),
                             w_local.reshape(-1)[order_t].to(torch.float64)], dim=1)
    n_recv = int(recv_counts.sum())
    recv_rows = torch.empty((n_recv, m), dtype=x_local.dtype)
    recv_meta = torch.empty((n_recv, 2), dtype=torch.float64)
    sc, rc = [int(v) for v in send_counts], [int(v) for v in recv_counts]
    dist.all_to_all_single(recv_rows, send_rows, rc, sc, group=group)
    dist.all_to_all_single(recv_meta, send_meta, rc, sc, group=group)
    # 5. expert compute on this rank (experts of plan.fetch[rank] come from
    # another rank's weights: the prefetch of 三 3.2)
    out = compute(recv_rows, recv_meta[:, 0].to(torch.int64), recv_meta[:, 1])
    out = torch.as_tensor(out)
    # 6. gather: results go back in the order they came, then to flat order
    back = torch.empty((ids.size, m), dtype=out.dtype)
    dist.all_to_all_single(back, out.contiguous(), sc, rc, group=group)
    pair_out = torch.empty_like(back)
    pair_out[order_t] = back
    y = pair_out.reshape(T, k, m)[:, 0].clone()
    for j in range(1, k):  # combine in slot order
        y += pair_out.reshape(T, k, m)[:, j]
    return y, plan
