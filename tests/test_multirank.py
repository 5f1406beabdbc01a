"""The benchmark's multi-rank logic on CPU: two gloo ranks rendezvous on
127.0.0.1, each draws its own sequences (weak scaling with no data shared and
no collective on the path), and the job's time is the largest over the ranks."""
import os
import socket
import sys

import numpy as np
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, q):
    sys.path.insert(0, ROOT)
    import torch.distributed as dist

    import bench
    from chunked_weight_mlp_place_b300 import inputs

    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=world)
    try:
        t = bench.max_over_ranks(10.0 + 5.0 * rank, dist, "cpu")
        w = inputs.workload("tiny")
        x = inputs.generate(w, seed=bench.rank_seed(rank), n_tokens=8, want=("X",))["X"]
        cu = inputs.doc_boundaries(4096, seed=rank, mix="short")
        q.put((rank, t, x, cu))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_draw_their_own_inputs_and_time_the_slowest():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    got = {}
    for _ in procs:
        r, t, x, cu = q.get(timeout=120)
        got[r] = (t, x, cu)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert got[0][0] == got[1][0] == 15.0                        # max over ranks, on every rank
    assert not np.array_equal(got[0][1], got[1][1])              # each rank its own sequences
    assert not np.array_equal(got[0][2], got[1][2])              # and its own document packing
    import bench
    assert bench.max_over_ranks(3.5, None, "cpu") == 3.5         # one rank: no collective


def test_reference_arm_prints_on_rank_zero_only(capsys):
    import argparse

    import bench
    from chunked_weight_mlp_place_b300 import inputs

    args = argparse.Namespace(rule="mse", docs=None, layers=0, steps=1, warmup=0)
    w = inputs.workload("tiny")
    bench.run_reference(args, w, 1, 2)
    assert capsys.readouterr().out == ""
    bench.run_reference(args, w, 0, 2)
    out = capsys.readouterr().out.strip().splitlines()
    assert len(out) == 1 and '"impl": "reference"' in out[0] and '"n_gpus": 2' in out[0]
