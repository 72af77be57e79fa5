"""The multi-rank path of bench.py on the CPU (gloo, world size 2): each rank's timing is
reduced to the slowest rank's, the job's throughput counts every rank's tokens, every rank
draws its own token shard, and under torchrun the reference arm prints one line from rank 0."""
import hashlib
import json
import os
import socket
import subprocess
import sys

import pytest

import moe_synth as S

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def torchrun(args, timeout=240):
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node=2",
           "--master-addr=127.0.0.1", f"--master-port={free_port()}"] + args
    env = dict(os.environ, OMP_NUM_THREADS="2")
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=timeout, env=env)
    assert r.returncode == 0, r.stderr[-2000:]
    return [json.loads(l) for l in r.stdout.splitlines() if l.startswith("{")]


def test_max_over_ranks_and_shards_gloo(tmp_path):
    out = str(tmp_path / "rank")
    torchrun([os.path.join("tests", "_ranks_worker.py"), out])
    lines = [json.load(open(f"{out}.{r}.json")) for r in range(2)]
    assert [d["rank"] for d in lines] == [0, 1] and all(d["world"] == 2 for d in lines)
    assert all(d["max_ms"] == 15.0 for d in lines)                     # the slowest rank's time
    assert all(d["tokens_per_s"] == pytest.approx(64 * 2 * 3 / 15e-3) for d in lines)
    assert lines[0]["x"] != lines[1]["x"] and lines[0]["ids"] != lines[1]["ids"]   # own shards
    import bench
    for d in lines:                                                      # deterministic shards
        x, ids, _ = bench.rank_inputs(S.CONFIGS["tiny"], d["rank"])
        assert hashlib.sha1(x.tobytes()).hexdigest() == d["x"]
        assert hashlib.sha1(ids.tobytes()).hexdigest() == d["ids"]


def test_reference_arm_under_torchrun_prints_one_line():
    lines = torchrun(["bench.py", "--impl", "reference", "--workload", "tiny", "--steps", "1", "--warmup", "3"])
    assert len(lines) == 1
    d = lines[0]
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle"
