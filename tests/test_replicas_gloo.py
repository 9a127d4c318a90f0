"""The multi-process (replica) harness of bench.py on CPU with gloo, world
size 2: the path shards by sequence with no collective on the data path, so
the only exchanges are the barrier and the max over ranks of the timed
region.  Rendezvous on 127.0.0.1."""
import json
import os
import socket
import subprocess
import sys

import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE="2", LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench
    ws, r, local = bench.dist_env()
    dist = bench.init_dist(ws)
    bench.barrier(dist)
    got = bench.max_over_ranks(dist, 10.0 + 5.0 * rank)   # rank 1 is the slow one
    bench.barrier(dist)
    out[rank] = (ws, r, local, got)
    dist.destroy_process_group()


def test_barrier_and_max_over_ranks_world_size_2():
    port = _free_port()
    with mp.get_context("spawn").Manager() as mgr:
        out = mgr.dict()
        mp.spawn(_rank_main, args=(port, out), nprocs=2, join=True)
        res = dict(out)
    assert res[0] == (2, 0, 0, 15.0)
    assert res[1] == (2, 1, 1, 15.0)


def test_reference_arm_under_torchrun_rank0_prints_one_line():
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), "bench.py", "--impl",
           "reference", "--gpus", "2", "--workload", "tiny_fp32", "--steps", "2", "--warmup", "3"]
    p = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=600,
                       env={**os.environ, "OMP_NUM_THREADS": "2"})
    assert p.returncode == 0, p.stderr[-2000:]
    lines = [l for l in p.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["value"] > 0
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["cpu_baseline"]["kind"] == "oracle"
