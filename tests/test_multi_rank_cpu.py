"""The benchmark's multi-process host logic on CPU: two gloo ranks (no GPU).

Each GPU runs an independent replica of the step (the convolution shards by
batch with no exchange on the hot path), so what N > 1 adds is host logic: the
max-over-ranks time, the whole-job throughput and the reference arm printing
from rank 0 only.
"""
import json
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, ws, port, out_dir):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(ws), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    import bench
    dist.init_process_group("gloo", init_method="env://", rank=rank, world_size=ws)
    try:
        assert bench.dist_env() == (ws, rank, rank)
        ms = 10.0 + 5.0 * rank            # rank 1 is the slow one
        ms_max = bench.max_over_ranks(ms, ws)
        value = bench.whole_job_tflops(2e12, ws, ms_max)
        with open(os.path.join(out_dir, "rank%d.json" % rank), "w") as f:
            json.dump({"ms_max": ms_max, "value": value}, f)
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_whole_job_value_two_gloo_ranks(tmp_path):
    import torch.multiprocessing as mp
    ws, port = 2, _free_port()
    mp.start_processes(_rank_main, args=(ws, port, str(tmp_path)), nprocs=ws, join=True,
                       start_method="spawn")
    got = [json.load(open(tmp_path / ("rank%d.json" % r))) for r in range(ws)]
    for g in got:
        assert g["ms_max"] == 15.0                               # every rank sees the slowest
        assert g["value"] == pytest.approx(2e12 * 2 / 15e-3 / 1e12)


def test_reference_arm_prints_once_under_torchrun(tmp_path):
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port),
           os.path.join(ROOT, "bench.py"), "--impl", "reference", "--workload", "tiny",
           "--gpus", "2", "--steps", "1", "--warmup", "3"]
    env = dict(os.environ, OMP_NUM_THREADS="1")
    r = subprocess.run(cmd, capture_output=True, text=True, timeout=600, cwd=ROOT, env=env)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, r.stdout
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle"
