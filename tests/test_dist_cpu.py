"""The bench's multi-process host logic on CPU: two gloo ranks started the way
torchrun starts them (RANK, WORLD_SIZE, MASTER_ADDR/PORT in the environment).
The timing reduction must give every rank the slowest rank's time, the
barrier must pass, and the reference arm must leave rank 1 without work or
output."""
import io
import json
import os
import socket
import contextlib

import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, results):
    os.environ.update({"RANK": str(rank), "WORLD_SIZE": str(world), "LOCAL_RANK": str(rank),
                       "MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port)})
    import bench
    import synth
    import torch.distributed as dist
    w, r, _ = bench.dist_setup()
    assert (w, r) == (world, rank)
    slowest = bench.max_over_ranks(1.5 + rank, w)
    bench.barrier(w)
    buf = io.StringIO()
    with contextlib.redirect_stdout(buf):
        rc = bench.run_reference(type("A", (), {"warmup": 0, "steps": 1, "ref_seconds": 0.0, "gpus": world})(),
                                 synth.WORKLOADS["pr1_min_tanh2"], w, r)
    results[rank] = (slowest, rc, buf.getvalue())
    dist.destroy_process_group()


def test_two_gloo_ranks():
    world, port = 2, _free_port()
    with mp.Manager() as mgr:
        results = mgr.dict()
        mp.start_processes(_rank, args=(world, port, results), nprocs=world, start_method="spawn")
        res = dict(results)
    assert res[0][0] == res[1][0] == 2.5          # the slowest rank's time on both
    assert res[0][1] == 0 and res[1][1] == 0
    line = json.loads(res[0][2].strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["n_gpus"] == 2
    assert res[1][2] == ""                        # rank 1 does no work and prints nothing
