"""The multi-rank path of bench.py on CPU (gloo, world size 2): replicas only, so the ranks exchange
nothing but the barrier and the max over ranks of the timed interval, and rank 0 alone prints."""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    # CPU ranks even on a machine with GPUs (before anything initialises CUDA in this process)
    os.environ.update({"MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port), "RANK": str(rank),
                       "WORLD_SIZE": str(world), "LOCAL_RANK": str(rank), "CUDA_VISIBLE_DEVICES": ""})
    sys.path.insert(0, ROOT)
    import bench

    d = bench.Dist()
    try:
        d.barrier()
        got = d.max(10.0 + rank)  # each rank's interval; the job's time is the slowest rank's
        with open(os.path.join(out_dir, "rank%d" % rank), "w") as f:
            f.write(repr(got))
    finally:
        d.close()


def test_max_over_ranks_gloo(tmp_path):
    port = _free_port()
    mp.start_processes(_rank_main, args=(2, port, str(tmp_path)), nprocs=2, join=True, start_method="spawn")
    for r in range(2):
        assert float((tmp_path / ("rank%d" % r)).read_text()) == 11.0


def test_reference_arm_two_ranks_prints_once():
    # launched the way the driver launches N > 1: rank 0 runs the oracle arm and prints one line,
    # rank 1 exits 0 without work
    pytest.importorskip("torch.distributed.run")
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2", "--master-addr",
           "127.0.0.1", "--master-port", str(port), os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2",
           "--steps", "1", "--warmup", "3", "--config", "tiny"]
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="")
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=600, env=env)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, r.stdout
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["value"] > 0
