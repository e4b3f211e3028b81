"""The multi-GPU path of bench.py on CPU: two gloo ranks on 127.0.0.1.

The inner loop does not shard (chunk i+1 needs chunk i's update), so N GPUs run
N independent replicas, one sequence each with seed 1000 + rank.  The only
collectives are the timing barrier and the max over ranks of the elapsed time;
throughput is all ranks' tokens over the slowest rank's time.
"""
import os
import socket
import sys

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, out):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    from ttt_inputs import SHAPES, sequence_tokens
    ms = 100.0 + 50.0 * rank                     # the slower rank decides
    slowest = bench.max_over_ranks(ms, dist, "cpu")
    tokens = sequence_tokens(SHAPES["tiny"], rank)
    dist.barrier()
    out[rank] = (slowest, int(tokens[:64].sum()), bench.replica_tokens_per_s(world, 3, 512, slowest / 1e3))
    dist.destroy_process_group()


def test_two_gloo_ranks_time_by_the_slowest_and_draw_distinct_sequences():
    world, port = 2, _free_port()
    with mp.Manager() as man:
        out = man.dict()
        mp.start_processes(_rank, args=(world, port, out), nprocs=world, start_method="spawn")
        res = dict(out)
    assert res[0][0] == res[1][0] == 150.0
    assert res[0][1] != res[1][1]                   # seed 1000 + rank
    assert res[0][2] == pytest.approx(2 * 3 * 512 / 0.150)


def test_reference_arm_runs_on_rank_zero_only(monkeypatch, capsys):
    sys.path.insert(0, ROOT)
    import bench
    monkeypatch.setenv("RANK", "1")
    args = bench.argparse.Namespace(workload="tiny", warmup=0, steps=1, cpu_tokens=16, gpus=2)
    assert bench.run_reference(args) == 0
    assert capsys.readouterr().out == ""


def test_single_process_reductions_are_identities():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(12.5, None, "cpu") == 12.5
    assert bench.replica_tokens_per_s(1, 5, 131072, 1.0) == 5 * 131072
