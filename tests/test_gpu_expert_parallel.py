"""Expert parallelism with the library computing each rank's experts on the
GPU (HARMOEny write-up, 三 3.3): two gloo ranks, collectives on the host,
share cuda:0 -- their kernels never wait on each other; every run here has
one GPU.  Each rank routes its own tokens with the library, the plan moves
pairs of the hot expert between ranks (or none), the received pairs run
through a k = 1 copy of the layer (library_compute), and the combined
output must match the fp64 oracle on the library's routing (1e-5, fp32
layer) and the single-rank forward pass of the same tokens."""
import os
import socket
import sys

import numpy as np
import pytest
import torch.multiprocessing as mp

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, q_thresh, out_q):
    sys.path.insert(0, ROOT)
    sys.path.insert(0, os.path.join(ROOT, "tests"))
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    import dataclasses

    import torch
    import torch.distributed as dist

    import mixture_experts_layer_gemm_gb300 as moe
    import oracle
    import workloads as wl
    from gpu_util import max_token_rel_l2, to_device
    from mixture_experts_layer_gemm_gb300 import expert_parallel as ep

    dist.init_process_group("gloo", rank=rank, world_size=world)
    torch.cuda.set_device(0)
    T = 24
    shape = wl.TINY_FP32.with_zipf(1.2)
    layer = wl.make_layer(shape, seed=3)
    x = wl.make_tokens(shape, T, seed=10 + rank)
    ml = moe.MoELayer(layer, T)
    xd = to_device(x)
    ml.route(xd)
    y_single = torch.empty_like(xd)
    ml.forward(xd, y_single)
    torch.cuda.synchronize()
    ids = ml.topk_ids[:T * shape.k].cpu().reshape(T, shape.k).to(torch.int64)
    w = ml.topk_w[:T * shape.k].cpu().reshape(T, shape.k)
    k1 = moe.MoELayer(dataclasses.replace(layer, shape=dataclasses.replace(shape, k=1)), world * T * shape.k)
    y, plan = ep.ep_forward(torch.from_numpy(x), ids, w, shape.E, q_thresh, ep.library_compute(k1))
    ref = oracle.layer(x, layer.w1, layer.w2, layer.w3, ids.numpy(), w.numpy().astype(np.float64),
                       oracle.RELU2)
    rel, _ = max_token_rel_l2(y.numpy(), ref)
    single = y_single.cpu().numpy()
    diff = float(np.abs(y.numpy() - single).max() / np.abs(single).max())
    ok = ml.sync_check()[0] == moe.MOE_OK and k1.sync_check()[0] == moe.MOE_OK
    ml.close()
    k1.close()
    dist.destroy_process_group()
    out_q.put((rank, rel, diff, ok, plan.moves))


@pytest.mark.parametrize("q_thresh", [1.0, 1e9])
def test_two_ranks_on_one_gpu_match_the_oracle_and_the_single_rank_forward(q_thresh):
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
    for rank, rel, diff, ok, moves in out:
        assert ok, rank
        assert rel <= 1e-5, (rank, rel)
        # per-pair fp32 results summed in slot order, as the single-rank combine
        assert diff <= 1e-6, (rank, diff)
    assert out[0][4] == out[1][4]
    if q_thresh < 2:
        assert out[0][4], "the Zipf-skewed routing should move pairs of the hot expert"
    else:
        assert out[0][4] == []
