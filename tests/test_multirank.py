"""Multi-rank host logic of bench.py on CPU (gloo, world size 2).

The data path shards into independent replicas (one per GPU, no exchange),
so the only collectives are the bench's own: the job's step time is the
slowest rank's (max over ranks), the whole-job rate counts every rank's
units, and the reference arm runs and prints on rank 0 only while the
other ranks exit 0 without work.  Ranks are separate processes started the
way torchrun starts them (RANK / WORLD_SIZE / LOCAL_RANK / MASTER_* in the
environment, rendezvous on 127.0.0.1).
"""
import json
import os
import socket
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

WORKER = r'''
import contextlib, io, json, sys
sys.path.insert(0, ROOT_DIR)
import torch.distributed as dist
import bench
rank, world, local = bench.dist_env()
dist.init_process_group("gloo", rank=rank, world_size=world)
ms = [1.5, 2.5][rank]
worst = bench.max_over_ranks(ms, world)
out = {"rank": rank, "world": world, "local": local, "max": worst, "rate": bench.job_rate(world, 1000, worst)}
class Args:
    steps = 1
    warmup = 0
buf = io.StringIO()
with contextlib.redirect_stdout(buf):
    if rank != 0:
        bench.run_reference(Args, rank, world)   # must return at once, printing nothing
out["ref_stdout"] = buf.getvalue()
dist.barrier()
dist.destroy_process_group()
print(json.dumps(out))
'''


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _env(rank, world, port):
    env = dict(os.environ, RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank),
               MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    env.pop("CUDA_VISIBLE_DEVICES", None)
    return env


def test_two_ranks_reduce_to_the_slowest_and_count_every_rank():
    port = _free_port()
    code = WORKER.replace("ROOT_DIR", repr(ROOT))
    procs = [subprocess.Popen([sys.executable, "-c", code], env=_env(r, 2, port), cwd=ROOT,
                              stdout=subprocess.PIPE, stderr=subprocess.PIPE, text=True) for r in range(2)]
    outs = [p.communicate(timeout=300) for p in procs]
    for p, (o, e) in zip(procs, outs):
        assert p.returncode == 0, e[-2000:]
    res = sorted((json.loads(o.strip().splitlines()[-1]) for o, _ in outs), key=lambda r: r["rank"])
    assert [r["rank"] for r in res] == [0, 1] and all(r["world"] == 2 for r in res)
    assert all(r["max"] == 2.5 for r in res)                      # both ranks see the slowest
    assert all(abs(r["rate"] - 2 * 1000 / 2.5e-3) < 1e-6 for r in res)
    assert res[1]["ref_stdout"] == ""


def test_reference_arm_under_torchrun_prints_one_line_from_rank_0():
    """bench.py --impl reference launched by torchrun with 2 ranks on CPU:
    rank 0 times the oracle and prints the JSON line, rank 1 exits 0."""
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), "bench.py", "--impl", "reference",
           "--gpus", "2", "--steps", "1", "--warmup", "0"]
    env = dict(os.environ)
    env.pop("CUDA_VISIBLE_DEVICES", None)
    r = subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-3000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, r.stdout
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle"
