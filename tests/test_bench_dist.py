"""Multi-rank host logic of bench.py on CPU with the gloo backend (world size 2):
barrier, max-over-ranks time, whole-job rate, and that the CPU reference arm
runs on rank 0 only."""
import io
import os
import socket
import sys
from contextlib import redirect_stdout

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, outdir):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    import bench
    r, ws = bench.dist_init("gloo")
    assert (r, ws) == (rank, world)
    bench.barrier()
    t = bench.reduce_max(1.0 + rank)            # rank times 1 s and 2 s
    units = bench.reduce_sum(10.0 * (rank + 1))  # 10 and 20 units
    rate = bench.whole_job_rate(units, t)
    buf = io.StringIO()
    with redirect_stdout(buf):
        bench.reference(bench.parse_args(["--impl", "reference", "--workload", "tiny",
                                          "--steps", "1", "--warmup", "3",
                                          "--ref-rows-per-head", "2"]))
    with open(os.path.join(outdir, f"rank{rank}.txt"), "w") as f:
        f.write(f"{t} {units} {rate}\n")
        f.write(buf.getvalue())
    dist.destroy_process_group()


def test_two_rank_gloo(tmp_path):
    port = _free_port()
    mp.start_processes(_worker, args=(2, port, str(tmp_path)), nprocs=2, join=True,
                       start_method="spawn")
    r0 = open(tmp_path / "rank0.txt").read().splitlines()
    r1 = open(tmp_path / "rank1.txt").read().splitlines()
    for lines in (r0, r1):
        t, units, rate = map(float, lines[0].split())
        assert t == 2.0 and units == 30.0 and rate == 15.0
    # the reference arm prints one JSON line on rank 0 and nothing elsewhere
    assert len(r0) == 2 and '"impl": "reference"' in r0[1]
    assert len(r1) == 1
