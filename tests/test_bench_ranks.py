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


def test_backward_roofline_arithmetic():
    import bench
    peaks = {"hbm_gbs": 6791.7, "bf16_tflops": 1916.3}
    c2 = S.CONFIGS["qwen3_30b_a3b"]
    w = bench.backward_work(c2)
    assert w["flops"] == 12 * 4096 * 8 * 2048 * 768
    # BF16 weights read (E*3IH*2) and FP32 weight gradients written (E*3IH*4) dominate
    assert 3.8e9 < w["bytes"] < 3.85e9
    r = bench.backward_roofline(w, 1.6705, peaks, "measured")
    assert r["bound"] == "hbm" and r["unit"] == "GB/s"           # 0.56 ms of bytes vs 0.32 ms of FLOPs
    assert r["frac"] == pytest.approx(w["bytes"] / 1.6705e-3 / 6791.7e9, abs=1e-4)
    assert r["bound_ms"] == pytest.approx(1e3 * w["bytes"] / 6791.7e9, abs=1e-3)
    big = bench.backward_roofline(bench.backward_work(S.CONFIGS["large"]), 20.0, peaks, "measured")
    assert big["bound"] == "tensor" and big["unit"] == "TFLOP/s"


def test_forward_stage_roofline_arithmetic():
    import bench
    peaks = {"hbm_gbs": 6791.7, "bf16_tflops": 1916.3}
    c2 = S.CONFIGS["qwen3_30b_a3b"]
    w = bench.stage_work(c2)
    # per token: X read once, k quantised copies (codes + scales + g), row maps, pair rows
    assert w["route_sort_quant"]["bytes"] == 4096 * 13536
    # the combine: k rows of y read (gathered through the pair rows), one output row written
    assert w["combine"]["bytes"] == 32768 * (4096 + 4) + 4096 * 4096
    # FC1 at 4096 tokens streams every expert's weights once: 201 MB of codes + 25 MB of scales
    assert w["fc1_swiglu"]["bytes"] == 128 * 1536 * (1024 + 128 + 4) + 32768 * (1024 + 128 + 4) + 32768 * (1536 + 12)
    assert w["fc1_swiglu"]["flops"] == 2 * 32768 * 2048 * 1536
    r = bench.roofline_of("fc1_swiglu", w["fc1_swiglu"], 0.0953, peaks, "measured")
    assert r["bound"] == "hbm" and r["frac"] == pytest.approx(w["fc1_swiglu"]["bytes"] / 95.3e-6 / 6791.7e9, abs=1e-4)
    big = bench.stage_work(S.CONFIGS["large"])["fc1_swiglu"]
    rb = bench.roofline_of("fc1_swiglu", big, 1.41, peaks, "measured")
    assert rb["bound"] == "tensor" and rb["peak"] == pytest.approx(1916.3 * bench.FP4_OVER_BF16, abs=0.1)


def test_layer_roofline_arithmetic():
    import bench
    peaks = {"hbm_gbs": 6791.7, "bf16_tflops": 1916.3}
    r = bench.layer_roofline(S.CONFIGS["qwen3_30b_a3b"], peaks, "measured", 0.2554)
    per = r["stage_bound_us"]
    assert set(per) == {"route_sort_quant", "fc1_swiglu", "requant", "fc2", "combine"}
    assert list(per) == bench.step_stages(S.CONFIGS["qwen3_30b_a3b"])
    # the fused FC2 (timed beside the step) takes I <= 768 and E <= 512
    assert bench.fused_fc2_supported(S.CONFIGS["qwen3_30b_a3b"]) and not bench.fused_fc2_supported(S.CONFIGS["large"])
    # at 4096 tokens every stage is bound by its bytes: FC1's weight stream is ~46 us
    assert 45 < per["fc1_swiglu"] < 48 and 7 < per["route_sort_quant"] < 9
    assert r["bound_ms"] == pytest.approx(sum(per.values()) / 1e3, abs=1e-3)
    assert r["frac"] == pytest.approx(r["bound_ms"] / 0.2554, abs=1e-3)


def test_batch_invariance_glue_on_cpu():
    # bench.batch_invariance driven by a stand-in library on host tensors: a per-token
    # computation passes, one that depends on the batch size fails
    import torch
    import bench

    class Lib:
        def __init__(self, batch_dependent):
            self.batch_dependent = batch_dependent

        def alloc_workspace(self, T, H, I, E, k, dev):
            return torch.empty(1)

        def moe_route_sort_amax(self, x, ids, pw, E, offs, ws):
            self.x = x

        def moe_expert_forward_nvfp4(self, w, T, k, offs, out, ws):
            scale = float(T) if self.batch_dependent else 2.0
            out.copy_((self.x.float() * scale).to(torch.bfloat16))

    cfg = S.CONFIGS["tiny"]
    x = torch.randn(cfg.T, cfg.H).to(torch.bfloat16)
    ids = torch.zeros(cfg.T, cfg.k, dtype=torch.int32)
    pw = torch.ones(cfg.T, cfg.k)
    ok = Lib(False)
    out = (x.float() * 2.0).to(torch.bfloat16)
    r = bench.batch_invariance(ok, torch, cfg, None, x, ids, pw, out, "cpu")
    # sizes 1, 7 and T/2 = 32 (64 is not below T): each as a prefix and as 3 random windows
    assert r["bitwise_equal"] and r["batches"] == r["batches_equal"] == 12 and r["decode_calls"] == 32
    bad = Lib(True)
    out = (x.float() * cfg.T).to(torch.bfloat16)
    r = bench.batch_invariance(bad, torch, cfg, None, x, ids, pw, out, "cpu")
    assert not r["bitwise_equal"] and r["decode_equal"] == 0
