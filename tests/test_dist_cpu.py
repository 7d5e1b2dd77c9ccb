"""The multi-rank path of bench.py on CPU: two gloo ranks on 127.0.0.1.

Each rank decodes its own batch (weak scaling, per-rank seed); the step time
is the maximum over ranks and the bytes are summed; the reference arm runs on
rank 0 only. No data-path collective exists: only the timing reduction.
"""
import json
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

WORKER = r"""
import json, os, sys
sys.path.insert(0, sys.argv[1])
import bench
world, rank, local = bench.dist_setup(2)
spec = bench.rank_spec("llama8b", rank)
out = {
    "world": world, "rank": rank, "seed": spec.seed,
    "max": bench.max_over_ranks(10.0 + rank, world),
    "sum": bench.sum_over_ranks(1.5 * (rank + 1), world),
}
bench.barrier(world)
import torch.distributed as dist
dist.destroy_process_group()
print("RESULT " + json.dumps(out), flush=True)
"""


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def test_two_gloo_ranks_reduce_timing_and_shard_seeds():
    port = _free_port()
    procs = []
    for rank in range(2):
        env = dict(os.environ, RANK=str(rank), LOCAL_RANK=str(rank), WORLD_SIZE="2",
                   MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), CUDA_VISIBLE_DEVICES="")
        procs.append(subprocess.Popen([sys.executable, "-c", WORKER, ROOT], env=env,
                                      stdout=subprocess.PIPE, stderr=subprocess.PIPE, text=True))
    results = []
    for p in procs:
        try:
            out, err = p.communicate(timeout=180)
        except subprocess.TimeoutExpired:
            p.kill()
            pytest.fail("a gloo rank did not finish")
        assert p.returncode == 0, err
        line = [ln for ln in out.splitlines() if ln.startswith("RESULT ")][-1]
        results.append(json.loads(line[len("RESULT "):]))
    by_rank = {r["rank"]: r for r in results}
    assert by_rank[0]["world"] == by_rank[1]["world"] == 2
    assert by_rank[0]["max"] == by_rank[1]["max"] == 11.0
    assert by_rank[0]["sum"] == by_rank[1]["sum"] == 4.5
    assert by_rank[0]["seed"] != by_rank[1]["seed"]


def test_reference_arm_runs_on_rank_zero_only(monkeypatch):
    sys.path.insert(0, ROOT)
    import bench

    calls = []
    monkeypatch.setattr(bench, "oracle_baseline", lambda *a, **k: calls.append(1))

    class Args:
        steps, warmup, gpus, config = 1, 0, 2, "tiny"

    bench.run_reference(Args, world=2, rank=1)   # other ranks exit without work
    assert calls == []


def _bench_env(**extra):
    env = {k: v for k, v in os.environ.items()
           if k not in ("WORLD_SIZE", "RANK", "LOCAL_RANK", "MASTER_ADDR", "MASTER_PORT")}
    env.update(CUDA_VISIBLE_DEVICES="", OMP_NUM_THREADS="1", **extra)
    return env


def test_gpus_flag_without_a_launcher_starts_that_many_ranks():
    """`bench.py --gpus 2` with no launcher relaunches itself under
    torch.distributed.run with two ranks (gloo here); the reference arm then
    prints one line, from rank 0, for two GPUs."""
    cmd = [sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2",
           "--steps", "1", "--warmup", "0", "--config", "tiny"]
    r = subprocess.run(cmd, env=_bench_env(), cwd=ROOT, capture_output=True, text=True,
                       timeout=600)
    assert r.returncode == 0, r.stderr[-3000:]
    lines = [json.loads(ln) for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, r.stdout
    assert lines[0]["impl"] == "reference" and lines[0]["n_gpus"] == 2


def test_gpus_flag_must_match_the_launcher():
    cmd = [sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2",
           "--steps", "1", "--warmup", "0", "--config", "tiny"]
    r = subprocess.run(cmd, env=_bench_env(WORLD_SIZE="1", RANK="0", LOCAL_RANK="0"), cwd=ROOT,
                       capture_output=True, text=True, timeout=300)
    assert r.returncode != 0
    assert "--gpus 2 but the launcher started 1 ranks" in r.stderr
