#!/usr/bin/env python
"""NVFP4 MoE expert-forward throughput on GB300.

One step = the whole hot path on one batch through the C ABI's one-call layer
entry, moe_layer_forward_nvfp4: the route sort (+ per-token amax + pad + NVFP4
quantise, as moe_route_sort_amax) and the expert forward (FC1 + SwiGLU x prob,
requant, FC2, fixed-order combine, as moe_expert_forward_nvfp4), with the
quantised weights resident.  The per-stage attribution times the stage calls.  Default workload: the Qwen3-30B-A3B-shaped layer
(hidden 2048, expert intermediate 768, 128 experts, top-8, 4096 tokens,
balanced routing), seeded synthetic data.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

Prints one JSON line (rank 0).  Under torchrun each rank runs its own token
shard with the same weights (weak scaling, no collective on the data path);
the timing is the max over ranks.  `--impl reference` times the CPU oracle on
the host cores instead (bounded sample per step).
"""

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import moe_synth as S  # noqa: E402

FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
FP4_OVER_BF16 = 13.5 / 2.25     # nominal dense FP4 : BF16 tensor ratio on GB300
FLUSH_BYTES = 512 << 20         # > L2 (129 MB)


FUSED_FC2_MAX_I = 768   # moe_fc2_requant_max_intermediate(): FC2 with the requantisation fused in


def fused_fc2_supported(cfg):
    return cfg.I <= FUSED_FC2_MAX_I and cfg.E <= 512


def kernels_per_step(cfg):
    """Launches of one step: the route sort is one block-sort kernel for up to 8192 (token,
    slot) pairs and E <= 256, else a histogram and a scan kernel; then quantise-scatter, the
    scale-tile kernel, FC1, requant, FC2, combine."""
    return (1 if cfg.T * cfg.k <= 8192 and cfg.E <= 256 else 2) + 6


def step_stages(cfg):
    """The stages one step runs, in order."""
    return ["route_sort_quant", "fc1_swiglu", "requant", "fc2", "combine"]


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=500)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--workload", default="qwen3_30b_a3b", choices=sorted(S.CONFIGS))
    ap.add_argument("--tokens", type=int, default=0,
                    help="run the workload's layer with this many tokens instead (small profiling cases)")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--minimal", action="store_true",
                    help="time the steps and their stages only (no e2e, router, masked, backward, invariance, "
                         "extra workloads or CPU baseline): the command the ncu captures run")
    ap.add_argument("--no-extra-workloads", action="store_true",
                    help="time only the headline workload (skip the 16384-token skewed and large layers)")
    ap.add_argument("--oracle-sample", default=None, help=argparse.SUPPRESS)
    ap.add_argument("--oracle-seconds", type=float, default=5.0, help=argparse.SUPPRESS)
    ap.add_argument("--oracle-tokens", type=int, default=0, help=argparse.SUPPRESS)
    ap.add_argument("--oracle-experts", type=int, default=8, help=argparse.SUPPRESS)
    return ap.parse_args()


# Source files each stage's kernels are built from (for matching stored ncu captures).
STAGE_SOURCES = {
    "route_sort_quant": ["quant.cu", "nvfp4_quant.cuh", "ptx.cuh", "common.cuh"],
    "fc1_swiglu": ["gemm.cu", "nvfp4_quant.cuh", "ptx.cuh", "common.cuh"],
    "requant": ["quant.cu", "nvfp4_quant.cuh", "ptx.cuh", "common.cuh"],
    "fc2": ["gemm.cu", "nvfp4_quant.cuh", "ptx.cuh", "common.cuh"],
    "fc2_requant": ["gemm.cu", "nvfp4_quant.cuh", "ptx.cuh", "common.cuh"],
    "combine": ["combine.cu", "common.cuh"],
}


def source_digest(stage):
    """SHA-1 over the CUDA sources a stage's kernels are compiled from: identifies the
    kernels a stored ncu capture was taken from."""
    import hashlib
    h = hashlib.sha1()
    csrc = os.path.join(ROOT, "nvfp4_moe_expert_gb300", "csrc")
    for name in STAGE_SOURCES[stage]:
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(name.encode() + b"\0" + f.read())
    return h.hexdigest()


def stored_traffic(cfg):
    """DRAM bytes per launch (ncu dram__bytes_read.sum + dram__bytes_write.sum) of each
    stage, from profiles/ncu_traffic.json, for the stages whose capture was taken from
    these exact sources on this workload (other stages report null)."""
    p = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    if not os.path.exists(p):
        return {}
    with open(p) as f:
        d = json.load(f)
    if d.get("workload") != cfg.name or d.get("tokens", cfg.T) != cfg.T:
        return {}
    out = {}
    for stage, rec in d.get("kernels", {}).items():
        if stage in STAGE_SOURCES and rec.get("source_digest") == source_digest(stage):
            out[stage] = rec["bytes"]
    return out


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def describe(cfg):
    return {
        "workload": f"{cfg.name}: hidden {cfg.H}, expert intermediate {cfg.I} (FC1 out {2 * cfg.I}), "
                    f"{cfg.E} experts, top-{cfg.k}, {cfg.T} tokens per GPU, {cfg.routing} routing"
                    + (f", {cfg.outlier_frac:.0%} x20 outlier channels" if cfg.outlier_frac else ""),
        "tokens": cfg.T, "hidden": cfg.H, "intermediate": cfg.I, "experts": cfg.E, "top_k": cfg.k,
        "l2": "flushed by a 512 MB write between timed steps",
        "weights": "pre-quantised NVFP4, resident in HBM (weight quantisation timed separately)",
    }


# ---------------------------------------------------------------- algorithmic work
def stage_work(cfg):
    """Algorithmic bytes and FLOPs per launch of each stage (real rows only, no padding)."""
    T, H, I, E, k = cfg.T, cfg.H, cfg.I, cfg.E, cfg.k
    R = T * k
    row_q = lambda C: C // 2 + C // 16 + 4          # codes + block scales + g of one NVFP4 row
    return {
        # X read, k routed copies written, ids/probs read, row map/probability/maxima and each
        # pair's row written
        "route_sort_quant": {"bytes": T * (2 * H + k * row_q(H) + 8 * k + 16 * k), "flops": 0},
        "fc1_swiglu": {"bytes": E * 2 * I * row_q(H) + R * row_q(H) + R * (2 * I + 4 + 8),
                       "flops": 2 * R * H * 2 * I},
        "requant": {"bytes": R * (2 * I + 4 + 4) + R * row_q(I), "flops": 0},
        "fc2": {"bytes": E * H * row_q(I) + R * row_q(I) + R * 2 * H, "flops": 2 * R * I * H},
        # FC2 with the requantisation fused in: W2, h and its maxima/row map read, y written
        "fc2_requant": {"bytes": E * H * row_q(I) + R * (2 * I + 8) + R * 2 * H, "flops": 2 * R * I * H},
        "combine": {"bytes": R * (2 * H + 4) + T * 2 * H, "flops": 0},
    }


def roofline_of(name, work, ms, peaks, peak_kind):
    hbm = float(peaks["hbm_gbs"])
    fp4 = float(peaks["bf16_tflops"]) * FP4_OVER_BF16
    b, f = work["bytes"], work["flops"]
    t_mem = b / (hbm * 1e9)
    t_cmp = f / (fp4 * 1e12) if f else 0.0
    if t_cmp > t_mem:
        ach = f / (ms * 1e-3) / 1e12
        return {"kernel": name, "bound": "tensor", "achieved": round(ach, 2), "peak": round(fp4, 1),
                "unit": "TFLOP/s", "frac": round(ach / fp4, 4), "traffic": None,
                "peak_source": f"{peak_kind} bf16 x {FP4_OVER_BF16:g} (nominal FP4/BF16 ratio)",
                "algorithmic": f"{f:.4g} FLOP per launch"}
    ach = b / (ms * 1e-3) / 1e9
    return {"kernel": name, "bound": "hbm", "achieved": round(ach, 1), "peak": hbm, "unit": "GB/s",
            "frac": round(ach / hbm, 4), "traffic": None, "peak_source": f"{peak_kind} copy bandwidth",
            "algorithmic": f"{b:.4g} bytes per launch"}


def batch_invariance(M, torch, cfg, weights, x, ids, pw, out, dev, sizes=(1, 7, 64), n_decode=32, n_windows=3):
    """Spot check of bitwise batch invariance on this workload: the first n tokens and n_windows
    random contiguous windows of each size n run as batches of their own, and n_decode tokens
    spread over the batch run one at a time (decode-shaped calls); each must give the same BF16
    output bits as in the full batch `out` (the full sweep over 256 sequences of 64-2048 tokens
    is tests/test_gpu_invariance.py)."""
    T, H, I, E, k = cfg.T, cfg.H, cfg.I, cfg.E, cfg.k
    offs_n = torch.empty(E + 1, dtype=torch.int32, device=dev)

    def run(lo, hi):
        n = hi - lo
        ws_n = M.alloc_workspace(n, H, I, E, k, dev)
        out_n = torch.empty((n, H), dtype=torch.bfloat16, device=dev)
        M.moe_route_sort_amax(x[lo:hi], ids[lo:hi], pw[lo:hi], E, offs_n, ws_n)
        M.moe_expert_forward_nvfp4(weights, n, k, offs_n, out_n, ws_n)
        return bool(torch.equal(out_n.view(torch.int16), out[lo:hi].view(torch.int16)))

    rng = np.random.default_rng(T)
    calls = []
    for n in sorted(set(tuple(sizes) + (T // 2,))):
        if 0 < n < T:
            calls.append((0, n))
            calls += [(int(lo), int(lo) + n) for lo in rng.integers(1, T - n + 1, n_windows)]
    equal = [run(lo, hi) for lo, hi in calls]
    step = max(1, T // n_decode)
    decode = [run(t, t + 1) for t in range(0, T, step)][:n_decode]
    return {"bitwise_equal": all(equal) and all(decode), "batches": len(calls), "batches_equal": sum(equal),
            "decode_calls": len(decode), "decode_equal": sum(decode),
            "what": f"prefix + random-window sub-batches of {sorted(set(sizes + (T // 2,)))} tokens, 1-token calls"}


def layer_roofline(cfg, peaks, peak_kind, ms_per_step):
    """The step's roofline: the sum over its stages of each stage's bound time (the larger of
    algorithmic bytes / copy bandwidth and FLOPs / FP4 peak), against the measured step time."""
    hbm = float(peaks["hbm_gbs"])
    fp4 = float(peaks["bf16_tflops"]) * FP4_OVER_BF16
    work = stage_work(cfg)
    per = {n: max(work[n]["bytes"] / (hbm * 1e9), work[n]["flops"] / (fp4 * 1e12)) for n in step_stages(cfg)}
    bound_ms = 1e3 * sum(per.values())
    return {"frac": round(bound_ms / ms_per_step, 4), "bound_ms": round(bound_ms, 4),
            "measured_ms": round(ms_per_step, 4),
            "stage_bound_us": {n: round(1e6 * t, 1) for n, t in per.items()}, "peak_note": "of " + peak_kind}


def backward_work(cfg):
    """Algorithmic FLOPs and bytes of one moe_expert_backward_ste call: four BF16 GEMMs
    (2RHI, 2R(2I)H, 2RHI, 2R(2I)H FLOPs); the BF16 weights read once, the FP32
    weight gradients written once, x, dOut, the saved h and gate/up (BF16) read, dX and
    dprob written."""
    T, H, I, E, k = cfg.T, cfg.H, cfg.I, cfg.E, cfg.k
    R = T * k
    flops = 12 * R * H * I
    nbytes = (E * 3 * I * H * 2 + E * 3 * I * H * 4 + 2 * T * H * 2 + R * I * 2 + R * 2 * I * 2
              + T * H * 2 + R * 4)
    return {"flops": flops, "bytes": nbytes}


def backward_roofline(work, ms, peaks, peak_kind):
    """The binding bound of the backward (BF16 tensor peak or HBM copy bandwidth) and the
    fraction of it that `ms` per call reaches."""
    hbm = float(peaks["hbm_gbs"])
    bf16 = float(peaks["bf16_tflops"])
    t_mem = work["bytes"] / (hbm * 1e9)
    t_cmp = work["flops"] / (bf16 * 1e12)
    out = {"algorithmic": f"{work['flops']:.4g} FLOP (12 T k H I) and {work['bytes']:.4g} bytes per call",
           "bound_ms": round(1e3 * max(t_mem, t_cmp), 4), "peak_note": "of " + peak_kind}
    if t_cmp > t_mem:
        ach = work["flops"] / (ms * 1e-3) / 1e12
        return out | {"bound": "tensor", "achieved": round(ach, 2), "peak": bf16, "unit": "TFLOP/s",
                      "frac": round(ach / bf16, 4)}
    ach = work["bytes"] / (ms * 1e-3) / 1e9
    return out | {"bound": "hbm", "achieved": round(ach, 1), "peak": hbm, "unit": "GB/s",
                  "frac": round(ach / hbm, 4)}


# ---------------------------------------------------------------- clocks
class ClockSampler:
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.QUERY}", "--format=csv,noheader,nounits",
                 "-lms", "50", "-f", self.path], stdout=subprocess.DEVNULL, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        time.sleep(0.3)

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.1)
        self.proc.terminate()
        self.proc.wait()
        rows = []
        with open(self.path) as f:
            for line in f:
                p = [v.strip() for v in line.split(",")]
                if len(p) >= 9:
                    rows.append(p)
        os.unlink(self.path)
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i] == "Active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows)}


# ---------------------------------------------------------------- CPU oracle timing
def oracle_sample_rate(cfg, seconds=12.0, n_experts=8, T=None):
    """Time the CPU oracle on a bounded sample of the workload: every (token, slot)
    pair of the first T tokens routed to the first n experts (their weights quantised
    beforehand, untimed), repeated until about `seconds` of CPU work (at least one pass).
    Returns (tokens/s, sample description)."""
    from oracle import moe as OM
    ids, w = S.make_routing(cfg, T)
    x = S.make_x(cfg, T)
    n_experts = max(1, min(cfg.E, n_experts))
    w1, w2 = S.make_weights(cfg, experts=n_experts)
    wq = OM.quantize_weights(w1, w2)
    for e in range(n_experts):
        wq.expert(e)
    groups = []
    for e in range(n_experts):
        t_e, s_e = np.nonzero(ids == e)
        if len(t_e):
            groups.append((x[t_e], np.zeros((len(t_e), 1), np.int32) + e, w[t_e, s_e][:, None]))
    pairs = sum(len(g[0]) for g in groups)
    reps = 0
    t0 = time.perf_counter()
    while True:
        for xe, ie, we in groups:
            OM.moe_forward(xe, ie, we, wq)
        reps += 1
        dt = time.perf_counter() - t0
        if dt >= seconds or reps >= 1000:
            break
    tokens_per_s = pairs * reps / cfg.k / dt
    n_tok = cfg.T if T is None else T
    desc = (f"{cfg.name}: every routed (token, slot) pair of experts 0..{n_experts - 1} among the first "
            f"{n_tok} tokens ({pairs} pairs), {reps} passes in {dt:.1f} s; tokens/s = pairs/s / top-{cfg.k}")
    return tokens_per_s, desc


def cpu_model():
    """The host CPU's model name (lscpu, else /proc/cpuinfo, else the platform string)."""
    try:
        r = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10)
        for line in r.stdout.splitlines():
            if line.strip().startswith("Model name:"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.lower().startswith(("model name", "hardware")):
                    return line.split(":", 1)[1].strip()
    except OSError:
        pass
    import platform
    return platform.processor() or platform.machine()


def oracle_sample_subprocess(name, seconds, tokens=0, experts=8, threads=None):
    """oracle_sample_rate in a child process (threads=1: numpy's BLAS held to one thread)."""
    env = dict(os.environ)
    if threads is not None:
        for v in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS", "BLIS_NUM_THREADS"):
            env[v] = str(threads)
    cmd = [sys.executable, os.path.abspath(__file__), "--oracle-sample", name, "--oracle-seconds", str(seconds),
           "--oracle-tokens", str(tokens), "--oracle-experts", str(experts)]
    r = subprocess.run(cmd, capture_output=True, text=True, env=env, timeout=600)
    if r.returncode != 0:
        return None
    return json.loads(r.stdout.strip().splitlines()[-1])


def cpu_baselines(cfg):
    """The oracle on the host cores: the headline workload (all cores, and one thread), the
    small 64-token layer in full, and bounded samples of 2048-token slices of the skewed
    16384-token workload and of the large layer."""
    v, desc = oracle_sample_rate(cfg, seconds=10.0)
    out = {"value": round(v, 3), "unit": "tokens/s", "cores": os.cpu_count(), "kind": "oracle", "sample": desc,
           "cpu_model": cpu_model()}
    one = oracle_sample_subprocess(cfg.name, 5.0, threads=1)
    if one:
        out["single_thread"] = {"value": round(one["value"], 3), "cores": 1, "sample": one["sample"]}
    extra = {}
    for name, tokens, experts in (("tiny", 0, 8), ("qwen3_30b_a3b_skew", 2048, 4), ("large", 2048, 1)):
        if name in S.CONFIGS:
            r = oracle_sample_subprocess(name, 4.0, tokens=tokens, experts=experts)
            if r:
                extra[name] = {"value": round(r["value"], 3), "unit": "tokens/s", "sample": r["sample"]}
    out["workloads"] = extra
    return out


def max_over_ranks(x, world, device=None):
    """The largest of every rank's value of x (a job's time is its slowest rank's).  NCCL
    reduces device tensors, gloo host tensors."""
    if world == 1:
        return float(x)
    import torch
    import torch.distributed as dist
    dev = device if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([float(x)], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_tokens_per_s(tokens_per_rank, world, steps, total_ms):
    """Whole-job throughput: every rank's tokens over the slowest rank's time."""
    return tokens_per_rank * world * steps / (total_ms * 1e-3)


def rank_inputs(cfg, rank):
    """This rank's token shard (weak scaling: each rank draws its own seeded tokens and routing;
    the experts' weights are the same on every rank)."""
    x = S.make_x(cfg, stream=rank)
    ids, w = S.make_routing(cfg, stream=rank)
    return x, ids, w


def run_reference(args, cfg, rank, world):
    if rank != 0:
        return None
    from oracle import moe as OM
    budget = 150.0
    per_step = budget / max(1, args.steps + args.warmup)
    ids, w = S.make_routing(cfg)
    x = S.make_x(cfg)
    # experts per step sized from one calibration expert
    w1, w2 = S.make_weights(cfg, experts=1)
    wq = OM.quantize_weights(w1, w2)
    wq.expert(0)
    t_e, s_e = np.nonzero(ids == 0)
    t0 = time.perf_counter()
    OM.moe_forward(x[t_e], np.zeros((len(t_e), 1), np.int32), w[t_e, s_e][:, None], wq)
    one = time.perf_counter() - t0
    n_e = int(max(1, min(cfg.E, per_step / max(one, 1e-3))))
    w1, w2 = S.make_weights(cfg, experts=n_e)
    wq = OM.quantize_weights(w1, w2)
    for e in range(n_e):
        wq.expert(e)
    groups = []
    for e in range(n_e):
        t_e, s_e = np.nonzero(ids == e)
        groups.append((x[t_e], np.zeros((len(t_e), 1), np.int32) + e, w[t_e, s_e][:, None]))
    pairs = sum(len(g[0]) for g in groups)

    def step():
        for xe, ie, we in groups:
            OM.moe_forward(xe, ie, we, wq)

    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step()
    dt = time.perf_counter() - t0
    value = pairs * args.steps / cfg.k / dt
    sample = (f"each step: the CPU oracle on every routed (token, slot) pair of experts 0..{n_e - 1} of the "
              f"{cfg.name} workload ({pairs} pairs); tokens/s = pairs/s / top-{cfg.k}")
    return {
        "impl": "reference", "metric": "nvfp4_moe_expert_forward_tokens_per_s", "value": round(value, 3),
        "unit": "tokens/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(dt / args.steps * 1e3, 3), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64 (GEMM) / f32 (quantiser, epilogue)", "data": "synthetic",
        "config": describe(cfg),
        "cpu_baseline": {"value": round(value, 3), "unit": "tokens/s", "cores": os.cpu_count(),
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": round(value, 3), "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


# ---------------------------------------------------------------- GPU arm
def stage_times(M, torch, cfg, weights, x, ids, pw, offs, ws, out, flush, stream, n):
    """Mean CUDA-event time (ms) of each stage over n passes of the step called stage by
    stage (events on the launching stream between the stages), L2 flushed between passes."""
    T, E, k = cfg.T, cfg.E, cfg.k
    calls = {
        "route_sort_quant": lambda: M.moe_route_sort_amax(x, ids, pw, E, offs, ws),
        "fc1_swiglu": lambda: M.moe_fc1_swiglu_nvfp4(weights, T, k, offs, ws),
        "requant": lambda: M.moe_requant_nvfp4(weights, T, k, offs, ws),
        "fc2": lambda: M.moe_fc2_nvfp4(weights, T, k, offs, ws),
        "fc2_requant": lambda: M.moe_fc2_requant_nvfp4(weights, T, k, offs, ws),
        "combine": lambda: M.moe_combine_bf16(weights, T, k, out, ws),
    }
    names = step_stages(cfg)
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(len(names) + 1)] for _ in range(n)]
    for i in range(n):
        e = evs[i]
        e[0].record(stream)
        for j, name in enumerate(names):
            calls[name]()
            e[j + 1].record(stream)
        flush.zero_()
    torch.cuda.synchronize()
    return {name: statistics.mean(evs[i][j].elapsed_time(evs[i][j + 1]) for i in range(n))
            for j, name in enumerate(names)}


def fused_fc2_timing(M, torch, cfg, weights, x, ids, pw, offs, ws, flush, stream, n, stage_ms, peaks, peak_kind):
    """moe_fc2_requant_nvfp4 (the FC2 input's requantisation fused into FC2, same bits as the
    requant and FC2 stages) timed on its own after a route sort and FC1, L2 flushed between
    calls, against the two stages' times."""
    if not fused_fc2_supported(cfg):
        return None
    T, E, k = cfg.T, cfg.E, cfg.k
    M.moe_route_sort_amax(x, ids, pw, E, offs, ws)
    M.moe_fc1_swiglu_nvfp4(weights, T, k, offs, ws)
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(n)]
    for i in range(n):
        flush.zero_()
        ev[i][0].record(stream)
        M.moe_fc2_requant_nvfp4(weights, T, k, offs, ws)
        ev[i][1].record(stream)
    torch.cuda.synchronize()
    if M.nvfp4_get_device_error() != 0:
        raise RuntimeError("device error in the fused FC2")
    ms = statistics.mean(a.elapsed_time(b) for a, b in ev)
    r = roofline_of("fc2_requant", stage_work(cfg)["fc2_requant"], ms, peaks, peak_kind)
    return {"ms": round(ms, 4), "bound": r["bound"], "frac": r["frac"],
            "requant_plus_fc2_ms": round(stage_ms["requant"] + stage_ms["fc2"], 4),
            "note": "moe_fc2_requant_nvfp4, not used by the step: slower than the two stages here"}


def time_steps(M, torch, weights, cfg, x, ids, pw, offs, ws, out, flush, stream, K, W):
    """CUDA-event time (ms) of each of K steps (moe_layer_forward_nvfp4), after W warm-up
    steps, L2 flushed between steps outside the events."""
    T, E, k = cfg.T, cfg.E, cfg.k

    def step():
        M.moe_layer_forward_nvfp4(weights, x, ids, pw, offs, out, ws)

    for _ in range(W):
        step()
        flush.zero_()
    torch.cuda.synchronize()
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    for i in range(K):
        starts[i].record(stream)
        step()
        ends[i].record(stream)
        flush.zero_()
    torch.cuda.synchronize()
    return [a.elapsed_time(b) for a, b in zip(starts, ends)]


def extra_workload(M, torch, name, dev, stream, flush, K, W, peaks, peak_kind, to_dev):
    """Throughput of one of the compute-bound workloads (the 16384-token skewed layer, the
    large 4096/1536 layer): step time, each stage's time against its roofline (FP4 tensor
    peak for the GEMMs, copy bandwidth for the rest) and a batch-invariance spot check."""
    cfg = S.CONFIGS[name]
    T, H, I, E, k = cfg.T, cfg.H, cfg.I, cfg.E, cfg.k
    w1, w2 = S.make_weights_device(cfg, dev)
    weights = M.quantize_moe_weights(w1, w2)
    del w1, w2
    x = to_dev(S.make_x(cfg))
    ids_np, w_np = S.make_routing(cfg)
    ids = torch.from_numpy(ids_np).to(dev)
    pw = torch.from_numpy(w_np).to(dev)
    ws = M.alloc_workspace(T, H, I, E, k, dev)
    offs = torch.empty(E + 1, dtype=torch.int32, device=dev)
    out = torch.empty((T, H), dtype=torch.bfloat16, device=dev)
    ms = time_steps(M, torch, weights, cfg, x, ids, pw, offs, ws, out, flush, stream, K, W)
    st = stage_times(M, torch, cfg, weights, x, ids, pw, offs, ws, out, flush, stream, min(K, 20))
    if M.nvfp4_get_device_error() != 0:
        raise RuntimeError(f"device error in the {name} workload")
    work = stage_work(cfg)
    stages = {}
    for n in step_stages(cfg):
        r = roofline_of(n, work[n], st[n], peaks, peak_kind)
        # [ms, roofline fraction, bound]: "tensor" = of the FP4 peak, "hbm" = of the copy bandwidth
        stages[n] = [round(st[n], 4), r["frac"], r["bound"]]
    step_ms = statistics.mean(ms)
    M.moe_route_sort_amax(x, ids, pw, E, offs, ws)
    M.moe_expert_forward_nvfp4(weights, T, k, offs, out, ws)
    fused = fused_fc2_timing(M, torch, cfg, weights, x, ids, pw, offs, ws, flush, stream, min(K, 20), st, peaks,
                             peak_kind)
    M.moe_route_sort_amax(x, ids, pw, E, offs, ws)
    M.moe_expert_forward_nvfp4(weights, T, k, offs, out, ws)
    inv = batch_invariance(M, torch, cfg, weights, x, ids, pw, out, dev, sizes=(1, 64), n_decode=8, n_windows=2)
    res = {"tokens_per_s": round(T / (step_ms * 1e-3), 1), "ms_per_step": round(step_ms, 4), "steps": K,
           "layer_roofline_frac": layer_roofline(cfg, peaks, peak_kind, step_ms)["frac"],
           "bitwise_invariant": inv["bitwise_equal"],
           "stages_ms_frac_bound": stages}
    if fused:
        res["fused_fc2_requant_ms"] = [fused["ms"], fused["frac"], fused["requant_plus_fc2_ms"]]
    del weights, ws, out, x
    torch.cuda.empty_cache()
    return res


def run_ours(args, cfg, rank, world, local_rank):
    import torch
    import torch.distributed as dist
    import nvfp4_moe_expert_gb300 as M
    from nvfp4_moe_expert_gb300 import build as B

    B.build()
    M.lib()
    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream()

    def to_dev(bits):
        return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).to(dev)

    x_np, ids_np, w_np = rank_inputs(cfg, rank)
    w1_np, w2_np = S.make_weights(cfg)
    w1, w2 = to_dev(w1_np), to_dev(w2_np)
    del w1_np, w2_np
    # S0: weight quantisation, timed on its own
    M.quantize_moe_weights(w1, w2)
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ev0.record(stream)
    weights = M.quantize_moe_weights(w1, w2)
    ev1.record(stream)
    torch.cuda.synchronize()
    wq_ms = ev0.elapsed_time(ev1)

    T, H, I, E, k = cfg.T, cfg.H, cfg.I, cfg.E, cfg.k
    x = to_dev(x_np)
    ids = torch.from_numpy(ids_np).to(dev)
    pw = torch.from_numpy(w_np).to(dev)
    ws = M.alloc_workspace(T, H, I, E, k, dev)
    offs = torch.empty(E + 1, dtype=torch.int32, device=dev)
    out = torch.empty((T, H), dtype=torch.bfloat16, device=dev)
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)

    def step():
        M.moe_layer_forward_nvfp4(weights, x, ids, pw, offs, out, ws)

    for _ in range(args.warmup):
        step()
        flush.zero_()
    if M.nvfp4_get_device_error() != 0:
        raise RuntimeError("device error during warm-up")

    # ---- timed region: K steps, L2 flushed between steps (outside the events)
    K = args.steps
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    visible = os.environ.get("CUDA_VISIBLE_DEVICES", "")
    sampler = ClockSampler(visible.split(",")[local_rank] if visible else local_rank)
    sampler.start()
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    for i in range(K):
        starts[i].record(stream)
        step()
        ends[i].record(stream)
        flush.zero_()
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    clocks = sampler.stop()
    step_ms = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    total_ms = max_over_ranks(sum(step_ms), world, dev)
    if M.nvfp4_get_device_error() != 0:
        raise RuntimeError("device error during the timed steps")
    value = job_tokens_per_s(T, world, K, total_ms)

    # ---- per-stage attribution (separate pass, same launches, events between stages)
    names = step_stages(cfg)
    n_attr = min(K, 100)
    stage_ms = stage_times(M, torch, cfg, weights, x, ids, pw, offs, ws, out, flush, stream, n_attr)
    peaks, peak_kind = load_peaks()
    work = stage_work(cfg)
    kernels = {n: roofline_of(n, work[n], stage_ms[n], peaks, peak_kind) | {"ms": round(stage_ms[n], 4)}
               for n in names}
    traffic = stored_traffic(cfg)
    for n in names:
        if n in traffic:
            kernels[n]["traffic"] = traffic[n]
    fused = fused_fc2_timing(M, torch, cfg, weights, x, ids, pw, offs, ws, flush, stream, min(K, 50), stage_ms,
                             peaks, peak_kind)
    dominant = max(names, key=lambda n: stage_ms[n])
    roof = dict(kernels[dominant])
    roof["peak_note"] = "of " + peak_kind
    if args.minimal:
        return {"metric": "nvfp4_moe_expert_forward_tokens_per_s", "value": round(value, 1), "unit": "tokens/s",
                "n_gpus": world, "steps": K, "warmup": args.warmup, "ms_per_step": round(total_ms / K, 4),
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "config": describe(cfg),
                "roofline": roof, "kernels": kernels, "clocks": clocks, "minimal": True}

    # ---- router step (produces the step's routing; timed on its own, not part of the step)
    router = None
    if cfg.E % 16 == 0 and 16 <= cfg.E <= 256 and cfg.H % 64 == 0:
        wr = to_dev(S.make_router_weights(cfg))
        for _ in range(5):                 # warm-up: the first calls after the step run slow
            M.moe_router_topk(x, wr, k)
            flush.zero_()
        rev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(n_attr)]
        for i in range(n_attr):
            rev[i][0].record(stream)
            M.moe_router_topk(x, wr, k)
            rev[i][1].record(stream)
            flush.zero_()
        torch.cuda.synchronize()
        r_ms = statistics.mean(a.elapsed_time(b) for a, b in rev)
        r_bytes = T * H * 2 + E * H * 2 + T * k * 8
        r_flops = 2 * T * H * E
        bf16 = float(peaks["bf16_tflops"])
        hbm = float(peaks["hbm_gbs"])
        if r_flops / (bf16 * 1e12) > r_bytes / (hbm * 1e9):
            ach = r_flops / (r_ms * 1e-3) / 1e12
            router = {"bound": "tensor", "achieved": round(ach, 2), "peak": bf16, "unit": "TFLOP/s",
                      "frac": round(ach / bf16, 4)}
        else:
            ach = r_bytes / (r_ms * 1e-3) / 1e9
            router = {"bound": "hbm", "achieved": round(ach, 1), "peak": hbm, "unit": "GB/s",
                      "frac": round(ach / hbm, 4)}
        router |= {"ms": round(r_ms, 4), "algorithmic": f"{r_bytes:.4g} bytes, {r_flops:.4g} FLOP per launch",
                   "peak_note": "of " + peak_kind,
                   "note": "moe_router_topk: BF16 router GEMM + top-k + softmax over the chosen, "
                           "T x E logits; timed on its own (the step takes routing as an input)"}
        if M.nvfp4_get_device_error() != 0:
            raise RuntimeError("device error in the router step")

    # ---- the same step in the fixed-capacity layout (expert e at rows [e*C, (e+1)*C)), C the
    # smallest multiple of 128 that holds the fullest expert; timed on its own
    counts = np.bincount(ids_np.ravel(), minlength=E)
    C = 128 * ((int(counts.max()) + 127) // 128)
    ws_m = M.alloc_workspace_masked(T, H, cfg.I, E, k, C)
    out_m = torch.empty_like(out)
    M.moe_layer_forward_nvfp4_masked(weights, x, ids, pw, C, offs, out_m, ws_m)
    mev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(n_attr)]
    for i in range(n_attr):
        mev[i][0].record(stream)
        M.moe_layer_forward_nvfp4_masked(weights, x, ids, pw, C, offs, out_m, ws_m)
        mev[i][1].record(stream)
        flush.zero_()
    torch.cuda.synchronize()
    if M.nvfp4_get_device_error() != 0:
        raise RuntimeError("device error in the masked-layout step")
    m_ms = statistics.mean(a.elapsed_time(b) for a, b in mev)
    masked = {"ms_per_step": round(m_ms, 4), "tokens_per_s": round(T / (m_ms * 1e-3), 1), "capacity": C,
              "rows": E * C, "contiguous_rows": int(sum((c + 127) // 128 * 128 for c in counts)),
              "bitwise_equal_to_contiguous": bool(torch.equal(out_m.view(torch.int16), out.view(torch.int16))),
              "note": "route sort + expert forward in the fixed-capacity layout (moe_layer_forward_nvfp4_masked); "
                      "timed on its own"}
    # the contiguous step's output is recomputed so `out` holds it again for the checks below
    M.moe_route_sort_amax(x, ids, pw, E, offs, ws)
    M.moe_expert_forward_nvfp4(weights, T, k, offs, out, ws)
    invariance = batch_invariance(M, torch, cfg, weights, x, ids, pw, out, dev)
    if M.nvfp4_get_device_error() != 0:
        raise RuntimeError("device error in the batch-invariance check")

    # ---- end to end through the public API with host buffers (pinned), copies inside the timed region.
    # A serving loop: every step copies its own inputs in and its output back, on two copy
    # streams, with device buffers double-buffered so that step i's copies overlap the compute of
    # steps i-1 and i+1.  The timed region covers every copy of every step.
    x_h = x.cpu().pin_memory()
    ids_h = ids.cpu().pin_memory()
    pw_h = pw.cpu().pin_memory()
    out_h = [torch.empty((T, H), dtype=torch.bfloat16).pin_memory() for _ in range(2)]
    x_d = [torch.empty_like(x) for _ in range(2)]
    ids_d = [torch.empty_like(ids) for _ in range(2)]
    pw_d = [torch.empty_like(pw) for _ in range(2)]
    out_d = [torch.empty_like(out) for _ in range(2)]
    h2d_s, d2h_s = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    ev = lambda: torch.cuda.Event()
    h2d_done, comp_done, d2h_done = [ev(), ev()], [ev(), ev()], [ev(), ev()]
    for b in range(2):   # every buffer starts "free"
        comp_done[b].record(stream)
        d2h_done[b].record(stream)

    def e2e_step(i):
        b = i & 1
        with torch.cuda.stream(h2d_s):
            h2d_s.wait_event(comp_done[b])           # step i-2's compute has read this buffer
            x_d[b].copy_(x_h, non_blocking=True)
            ids_d[b].copy_(ids_h, non_blocking=True)
            pw_d[b].copy_(pw_h, non_blocking=True)
            h2d_done[b].record(h2d_s)
        stream.wait_event(h2d_done[b])
        stream.wait_event(d2h_done[b])                # step i-2's output has been copied out
        M.moe_layer_forward_nvfp4(weights, x_d[b], ids_d[b], pw_d[b], offs, out_d[b], ws)
        comp_done[b].record(stream)
        with torch.cuda.stream(d2h_s):
            d2h_s.wait_event(comp_done[b])
            out_h[b].copy_(out_d[b], non_blocking=True)
            d2h_done[b].record(d2h_s)

    for i in range(4):
        e2e_step(i)
    K2 = min(K, 200)
    torch.cuda.synchronize()
    e_s, e_e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e_s.record(stream)
    h2d_s.wait_event(e_s)
    d2h_s.wait_event(e_s)
    for i in range(K2):
        e2e_step(i)
    stream.wait_event(d2h_done[(K2 - 1) & 1])
    stream.wait_event(d2h_done[K2 & 1])
    e_e.record(stream)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(e_s.elapsed_time(e_e) / K2, world, dev)
    if not torch.equal(out_h[(K2 - 1) & 1].view(torch.int16), out.cpu().view(torch.int16)):
        raise SystemExit("bench: end-to-end output differs from the device-resident run")
    h2d = x.numel() * 2 + ids.numel() * 4 + pw.numel() * 4
    d2h = out.numel() * 2

    # ---- straight-through backward of the same layer (timed on its own, not part of the step):
    # a forward that saves FC1's FP32 values, then moe_expert_backward_ste on a seeded dOut
    backward = backward_step(M, torch, cfg, weights, w1, w2, x, ids, pw, ws, offs, flush, stream, dev, to_dev,
                             min(K, 20), peaks, peak_kind)
    del w1, w2

    # ---- the compute-bound workloads: 16384 tokens with skewed routing, and the large layer
    workloads = {}
    if not args.no_extra_workloads:
        del ws, ws_m
        torch.cuda.empty_cache()
        for name in ("qwen3_30b_a3b_skew", "large"):
            workloads[name] = extra_workload(M, torch, name, dev, stream, flush, min(K, 20), max(3, args.warmup),
                                             peaks, peak_kind, to_dev)

    line = {
        "metric": "nvfp4_moe_expert_forward_tokens_per_s", "value": round(value, 1), "unit": "tokens/s",
        "n_gpus": world, "steps": K, "warmup": args.warmup, "ms_per_step": round(total_ms / K, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "nvfp4 (e2m1 x ue4m3 block-scaled) MMA, f32 accumulate/epilogue, bf16 in/out",
        "data": "synthetic (seeded; random-init weights of the layer's shape)",
        "config": describe(cfg),
        "roofline": roof,
        "e2e": {"value": round(T * world / (e2e_ms * 1e-3), 1), "unit": "tokens/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "note": "pinned host X/ids/probs in and output out every step; two copy streams, "
                        "double-buffered device buffers"},
        "gpu_launches": kernels_per_step(cfg) * K,
        "clocks": clocks,
        "kernels": kernels,
        "fused_fc2_requant": fused,
        "weight_quant_ms": round(wq_ms, 3),
        "router_step": router,
        "masked_step": masked,
        "backward_step": backward,
        # last, where a tail of the output shows them: the compute-bound workloads' stage
        # fractions, the headline layer's roofline and the invariance check
        "workloads": workloads,
        "layer_roofline": layer_roofline(cfg, peaks, peak_kind, total_ms / K),
        "batch_invariance": invariance,
    }
    return line


def backward_step(M, torch, cfg, weights, w1, w2, x, ids, pw, ws, offs, flush, stream, dev, to_dev, n, peaks,
                  peak_kind):
    """CUDA-event time of moe_expert_backward_ste (four BF16 grouped GEMMs, the SwiGLU x prob
    derivative, two row gathers and the slot-order sum) on this workload, L2 flushed between calls."""
    T, H, I, E, k = cfg.T, cfg.H, cfg.I, cfg.E, cfg.k
    wt = M.MoEWeightsBF16(w1, w2)
    lay = M.moe_workspace_layout_query(T, H, I, E, k)
    gu = torch.empty((lay.rows_cap, 2 * I), dtype=torch.bfloat16, device=dev)
    dout = to_dev(S.make_grad_out(cfg))
    out = torch.empty((T, H), dtype=torch.bfloat16, device=dev)
    dx = torch.empty((T, H), dtype=torch.bfloat16, device=dev)
    dw1 = torch.empty((E, 2 * I, H), dtype=torch.float32, device=dev)
    dw2 = torch.empty((E, H, I), dtype=torch.float32, device=dev)
    dprob = torch.empty((T, k), dtype=torch.float32, device=dev)
    bws = M.alloc_backward_workspace(T, H, I, E, k, dev)
    M.moe_route_sort_amax(x, ids, pw, E, offs, ws)
    M.moe_fc1_swiglu_save_nvfp4(weights, T, k, offs, ws, gu)
    M.moe_requant_nvfp4(weights, T, k, offs, ws)
    M.moe_fc2_nvfp4(weights, T, k, offs, ws)
    M.moe_combine_bf16(weights, T, k, out, ws)

    def bwd():
        M.moe_expert_backward_ste(wt, T, k, x, dout, offs, ws, gu, dx, dw1, dw2, dprob, bws)

    for _ in range(3):
        bwd()
        flush.zero_()
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(n)]
    for i in range(n):
        ev[i][0].record(stream)
        bwd()
        ev[i][1].record(stream)
        flush.zero_()
    torch.cuda.synchronize()
    if M.nvfp4_get_device_error() != 0:
        raise RuntimeError("device error in the backward step")
    ms = statistics.mean(a.elapsed_time(b) for a, b in ev)
    work = backward_work(cfg)
    tflops = work["flops"] / (ms * 1e-3) / 1e12
    return {"ms": round(ms, 4), "tokens_per_s": round(T / (ms * 1e-3), 1),
            **backward_roofline(work, ms, peaks, peak_kind),
            "gemm_tflops": round(tflops, 2),
            "finite": bool(torch.isfinite(dw1).all() and torch.isfinite(dw2).all()),
            "note": "moe_expert_backward_ste: STE gradients dX, dW1, dW2, dprob from the saved BF16 "
                    "originals; timed on its own after a forward that saves FC1's values"}


def main():
    args = parse()
    if args.oracle_sample:
        c = S.CONFIGS[args.oracle_sample]
        v, desc = oracle_sample_rate(c, args.oracle_seconds, args.oracle_experts, args.oracle_tokens or None)
        print(json.dumps({"value": v, "sample": desc}), flush=True)
        return
    cfg = S.CONFIGS[args.workload]
    if args.tokens > 0:
        cfg = S.shrink(cfg, T=args.tokens)
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1 and args.impl == "ours":
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(local_rank)
        dist.init_process_group(backend="nccl" if torch.cuda.is_available() else "gloo")
    if args.impl == "reference":
        line = run_reference(args, cfg, rank, world)
    else:
        line = run_ours(args, cfg, rank, world, local_rank)
        if rank == 0 and world == 1 and not args.no_cpu_baseline and not args.minimal:
            tail = {key: line.pop(key) for key in ("workloads", "layer_roofline", "batch_invariance")}
            line["cpu_baseline"] = cpu_baselines(cfg)
            line.update(tail)
    if rank == 0 and line is not None:
        print(json.dumps(line), flush=True)
    if world > 1 and args.impl == "ours":
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
