"""The multi-process plumbing of bench.py on CPU (gloo, world size 2): rank
set-up from the torchrun environment, the max over ranks of the timed
region, the barrier, and the reference arm printing from rank 0 only."""
import io
import os
import socket
import sys
from contextlib import redirect_stdout

import pytest
import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), LOCAL_RANK=str(rank),
                      WORLD_SIZE=str(world))
    sys.path.insert(0, ROOT)
    import bench
    dist, r, ws, local = bench.dist_init()
    assert dist is not None and (r, ws, local) == (rank, world, rank)
    assert dist.get_backend() == "gloo"
    dev = torch.device("cpu")
    m = bench.max_over_ranks(dist, 10.0 + 3.5 * rank, dev)
    bench.barrier(dist, dev)
    dist.destroy_process_group()
    # the reference arm prints one line on rank 0 and nothing elsewhere
    # (a cheap stand-in for the oracle sample keeps this test fast)
    bench.cpu_baseline = lambda w, seconds_hint=0: {"value": 1.0, "unit": "GB/s", "cores": 1, "kind": "oracle",
                                                     "sample": "test"}
    buf = io.StringIO()
    with redirect_stdout(buf):
        bench.run_reference(type("A", (), {"steps": 1, "warmup": 3, "gpus": world})())
    q.put((rank, m, buf.getvalue()))


def test_two_gloo_ranks_take_the_max_and_only_rank0_reports():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    got = {}
    for _ in range(world):
        rank, m, out = q.get(timeout=120)
        got[rank] = (m, out)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert got[0][0] == got[1][0] == 13.5
    assert '"impl": "reference"' in got[0][1] and got[1][1] == ""
