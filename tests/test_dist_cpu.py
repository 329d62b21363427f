"""Multi-rank host logic of bench.py on CPU (gloo, world size 2): the max-over-ranks timing
and the reference arm running on rank 0 only."""
import io
import os
import socket
import sys
from contextlib import redirect_stdout

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    sys.path.insert(0, ROOT)
    import torch
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    got = bench.max_over_ranks([10.0 + rank, 5.0 - rank], torch.device("cpu"), world)
    buf = io.StringIO()
    with redirect_stdout(buf):
        bench.main(["--impl", "reference", "--steps", "1", "--warmup", "0", "--workload", "vit14_f32",
                    "--gpus", str(world)])
    dist.destroy_process_group()
    out[rank] = (got, buf.getvalue())


def test_two_rank_host_logic():
    world = 2
    mgr = mp.Manager()
    out = mgr.dict()
    mp.start_processes(_worker, args=(world, _free_port(), out), nprocs=world, start_method="spawn")
    assert out[0][0] == [11.0, 5.0] and out[1][0] == [11.0, 5.0]
    assert '"impl": "reference"' in out[0][1]
    assert out[1][1] == ""   # only rank 0 runs and prints the reference arm
