"""The benchmark's multi-process logic on CPU: world_size-2 gloo ranks agree on the max-over-ranks time
and the whole-job aggregation (sequence-sharded replicas, no data-path collective)."""
import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, ws, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(ws),
                      LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=ws)
    try:
        bench.barrier(ws)
        t = bench.reduce_max(1.5 + rank, ws)      # rank 1 is the slow one
        out[rank] = t
        assert bench.dist_env() == (ws, rank, rank)
    finally:
        dist.destroy_process_group()


def test_reduce_max_over_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    mgr = ctx.Manager()
    out = mgr.dict()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    assert out[0] == out[1] == pytest.approx(2.5)


def test_single_rank_helpers_need_no_process_group():
    assert bench.reduce_max(3.25, 1) == 3.25
    bench.barrier(1)
    args = bench.parse_args([])
    assert args.gpus == 1 and args.impl == "ours" and args.warmup >= 3


def test_algorithmic_bytes_model_counts_every_weight_once_per_pass():
    import workloads as WL
    w = WL.workload("dsv3_b1")
    model = bench.algorithmic_bytes(w, WL.context_lengths(w))
    shapes = w.weight_shapes()
    ws = 2
    # weight bytes read per decode step by the streaming kernels (embedding and norms excluded)
    step_w = sum(shapes[k][0] * shapes[k][1] for k in ("q_a", "kv_a", "q_b", "kv_b", "o", "gate", "up", "down",
                                                     "lm_head")) * ws
    per_step = sum(b for k, (b, n) in model.items() if k not in ("fc", "attention"))
    assert abs(per_step - step_w) / step_w < 0.01
    assert model["fc"][1] == 1 and model["attention"][1] == w.gamma
