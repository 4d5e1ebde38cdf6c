"""The N > 1 host logic of the benchmark on CPU: two gloo ranks, no GPU.

Every rank runs its own full weight pass (independent problems, no collective on the data
path); the job's step time is the slowest rank's and the job's weight bytes are the sum over
ranks, so the reported GB/s is the whole job's.  The reference arm runs on rank 0 only.
"""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    import sys
    import torch.distributed as dist
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    sys.path.insert(0, root)
    import bench
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=world)
    try:
        ms = [2.5, 3.25][rank]            # the two ranks' step times
        nbytes = [1000, 1000][rank]       # each rank streams its own full pass
        ms_max, total = bench.aggregate_ranks(ms, nbytes, True)
        gbps = bench.weight_gbps(total, ms_max)
        out.put((rank, ms_max, total, gbps))
    finally:
        dist.destroy_process_group()


def test_two_ranks_aggregate_max_time_and_summed_bytes():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    got = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, ms_max, total, gbps in got:
        assert ms_max == 3.25                     # the slowest rank sets the step time
        assert total == 2000                      # both ranks' bytes count
        assert gbps == pytest.approx(2000 / 3.25e-3 / 1e9)


def test_single_rank_is_identity():
    import sys
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    import bench
    assert bench.aggregate_ranks(1.5, 123, False) == (1.5, 123)


def test_reference_arm_runs_on_rank_zero_only(capsys):
    import sys
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    import argparse
    import bench
    bench.run_reference(argparse.Namespace(M=8, steps=1, warmup=3), rank=1)   # returns at once
    assert capsys.readouterr().out == ""
