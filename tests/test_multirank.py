"""The multi-rank path of bench.py, on CPU: two gloo ranks on 127.0.0.1.

bench.py runs one process per GPU.  Heads are independent (weak scaling, no data-path collective):
each rank draws its own inputs, the job's time is the slowest rank's, the job's throughput is world x
per-rank units / that time, and rank 0 alone prints the JSON line.  These tests run that host logic
with the gloo backend and no GPU: the rank setup from the launcher's environment, the max over ranks,
the per-rank seeds, and the reference arm launched by torch.distributed.run with two ranks.
"""
import json
import os
import socket
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

RANK_SCRIPT = """
import json, sys
sys.path.insert(0, {root!r})
import bench
import torch.distributed as dist
from local_linear_attention_flashlla_gb300.inputs import workload
world, rank, local = bench.dist_setup(None)
slowest = bench.ranks_max(10.0 + rank, "cpu")
seed = bench.rank_workload(workload("lm_bf16", B=1, H=1, n=8, d=16), rank).seed
print(json.dumps({{"rank": rank, "world": world, "backend": dist.get_backend(), "slowest": slowest, "seed": seed}}))
dist.destroy_process_group()
"""


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def test_two_gloo_ranks_share_the_slowest_time():
    port = _free_port()
    procs = []
    for rank in range(2):
        env = dict(os.environ, MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE="2",
                   LOCAL_RANK=str(rank), CUDA_VISIBLE_DEVICES="")
        procs.append(subprocess.Popen([sys.executable, "-c", RANK_SCRIPT.format(root=ROOT)], cwd=ROOT, env=env,
                                      stdout=subprocess.PIPE, stderr=subprocess.PIPE, text=True))
    res = []
    for p in procs:
        out, err = p.communicate(timeout=300)
        assert p.returncode == 0, err[-2000:]
        res.append(json.loads(out.strip().splitlines()[-1]))
    res.sort(key=lambda r: r["rank"])
    assert [r["rank"] for r in res] == [0, 1]
    assert all(r["world"] == 2 and r["backend"] == "gloo" for r in res)
    assert all(r["slowest"] == 11.0 for r in res)      # every rank sees the slowest rank's time
    assert res[0]["seed"] != res[1]["seed"]              # each rank draws its own inputs


def test_job_throughput_counts_every_rank():
    sys.path.insert(0, ROOT)
    import bench
    # 2 ranks x 1000 units x 10 steps in 500 ms of the slowest rank
    assert bench.job_throughput(2, 1000, 10, 500.0) == 40000.0
    assert bench.job_throughput(1, 1000, 10, 500.0) == 20000.0


def test_reference_arm_with_two_ranks_prints_one_line():
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2", "--master-addr",
           "127.0.0.1", "--master-port", str(port), "bench.py", "--impl", "reference", "--gpus", "2", "--steps", "1",
           "--warmup", "0", "--batch", "1"]
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="")
    r = subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-3000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, r.stdout[-2000:]
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle" and d["e2e"]["h2d_bytes_per_step"] == 0
