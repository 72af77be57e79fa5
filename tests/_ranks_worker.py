"""One rank of the multi-rank host-logic test (launched by tests/test_bench_ranks.py through
torch.distributed.run with the gloo backend on the CPU): writes its result to <argv[1]>.<rank>.json."""
import hashlib
import json
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import torch.distributed as dist  # noqa: E402

import bench  # noqa: E402
import moe_synth as S  # noqa: E402

dist.init_process_group("gloo")
rank, world = dist.get_rank(), dist.get_world_size()
slowest = bench.max_over_ranks(10.0 + 5.0 * rank, world)
x, ids, w = bench.rank_inputs(S.CONFIGS["tiny"], rank)
# one file per rank (the ranks share stdout, where their lines could interleave)
with open(f"{sys.argv[1]}.{rank}.json", "w") as f:
    json.dump({"rank": rank, "world": world, "max_ms": slowest,
               "tokens_per_s": bench.job_tokens_per_s(64, world, 3, slowest),
               "x": hashlib.sha1(x.tobytes()).hexdigest(), "ids": hashlib.sha1(ids.tobytes()).hexdigest()}, f)
dist.destroy_process_group()
