"""The multi-process host logic of the benchmark on CPU (gloo, world size 2):
the rendezvous on 127.0.0.1, the barrier, the max over ranks of the timed
region, the whole-job rate that counts every replica, and the reference arm,
which only rank 0 runs. Attention heads are independent, so N GPUs run N
replicas and no data moves between them; these are the only multi-rank steps."""
import json
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402

WORKER = """
import json, sys
sys.path.insert(0, {root!r})
import bench
d = bench.Dist()
d.init("gloo")
d.barrier()
m = d.max(10.0 * d.rank + 1.0)   # rank 1 holds the longer time
d.barrier()
print(json.dumps({{"rank": d.rank, "world": d.world, "max": m}}))
d.close()
"""


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def test_two_gloo_ranks_agree_on_the_max():
    port = _free_port()
    procs = []
    for rank in range(2):
        env = dict(os.environ, RANK=str(rank), WORLD_SIZE="2", LOCAL_RANK=str(rank), MASTER_ADDR="127.0.0.1",
                   MASTER_PORT=str(port))
        procs.append(subprocess.Popen([sys.executable, "-c", WORKER.format(root=ROOT)], env=env,
                                      stdout=subprocess.PIPE, stderr=subprocess.PIPE, text=True))
    outs = []
    for p in procs:
        try:
            outs.append(p.communicate(timeout=180))
        except subprocess.TimeoutExpired:
            for q in procs:
                q.kill()
            raise
    for p, (_, err) in zip(procs, outs):
        assert p.returncode == 0, err[-2000:]
    res = sorted((json.loads(o.strip().splitlines()[-1]) for o, _ in outs), key=lambda r: r["rank"])
    assert [r["rank"] for r in res] == [0, 1]
    assert all(r["world"] == 2 and r["max"] == 11.0 for r in res)


def test_single_process_dist_is_a_no_op():
    d = bench.Dist()
    d.init("gloo")  # WORLD_SIZE unset: no process group
    d.barrier()
    assert d.max(3.5) == 3.5 and not d.pg


def test_whole_job_rate_counts_every_replica():
    # 2.75e11 FLOP per replica, 4 replicas, 0.25 ms per step (the slowest rank)
    assert bench.aggregate_tflops(2.75e11, 4, 0.25) == pytest.approx(2.75e11 * 4 / 0.25e-3 / 1e12)
    assert bench.aggregate_tflops(2.75e11, 1, 0.25) == pytest.approx(1100.0)


def test_reference_arm_on_a_non_zero_rank_exits_without_output():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                        "--warmup", "0"], cwd=ROOT, env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    assert r.stdout.strip() == ""
