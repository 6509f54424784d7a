"""The multi-GPU form of the path is N independent replicas (no collective on the data path):
bench.py's whole-job throughput is the units all ranks processed over the slowest rank's
time, and the reference arm runs on rank 0 only. Checked with two gloo ranks on the CPU."""
import os
import socket

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, ws, port, out):
    import sys
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(ws), LOCAL_RANK=str(rank))
    import torch.distributed as dist
    dist.init_process_group("gloo", rank=rank, world_size=ws)
    import bench
    # rank r took (r + 1) seconds for 100 tokens
    out[rank] = (bench.max_over_ranks(rank + 1.0), bench.replica_throughput(100, rank + 1.0))
    # the reference arm: ranks other than 0 leave at once, with no work and no output
    if rank != 0:
        import argparse
        bench.run_reference(argparse.Namespace(workload="decode_bf16", steps=1, warmup=3))
    dist.barrier()
    dist.destroy_process_group()


def test_two_replicas_max_time_and_whole_job_throughput():
    ws = 2
    with mp.get_context("spawn").Manager() as m:
        out = m.dict()
        mp.start_processes(_rank, args=(ws, _free_port(), out), nprocs=ws, join=True,
                           start_method="spawn")
        res = dict(out)
    for r in range(ws):
        t_max, value = res[r]
        assert t_max == 2.0                       # the slowest rank
        assert value == pytest.approx(100 * ws / 2.0)


def test_single_process_needs_no_group():
    import sys
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(3.5) == 3.5
    assert bench.replica_throughput(10, 2.0) == 5.0
