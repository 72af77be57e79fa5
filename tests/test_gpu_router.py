"""GPU parity of moe_router_topk (the router step) against the oracle (oracle/router.py).

* logits: against the exact FP64 logits of the BF16 inputs, within the FP32 accumulation
  bound |error| <= 2^-12 * sum_h |x_h w_h| (H additions of at most 2^-24 relative error each,
  H <= 4096), and relative L2 <= 1e-5 over the whole matrix;
* selection: the decision is taken in the kernel's precision, so the ids must equal the
  oracle's top-k (logit desc, id asc) applied to the kernel's own FP32 logits, exactly; ids
  that differ from the top-k of the exact logits are allowed only where the exact logits of
  the swapped experts are within twice the accumulation bound of each other (a near tie);
* probabilities: against the oracle's softmax of the chosen logits, computed in FP64 from the
  kernel's own FP32 logits: |error| <= 4e-6 * p + 1e-7 (FP32 exp and division);
* batch invariance: a token's logits, ids and probabilities are bitwise the same whatever T
  and whatever the other tokens are.
"""

import numpy as np
import pytest
import torch

import moe_synth as S
import nvfp4_moe_expert_gb300 as M
from nvfp4_moe_expert_gb300 import build as B
from oracle import formats as F
from oracle import router as R
from _helpers import bf16_to_torch

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    B.build()
    M.lib()


def run(x_bits, w_bits, k):
    ids, w, logits = M.moe_router_topk(bf16_to_torch(x_bits), bf16_to_torch(w_bits), k, with_logits=True)
    assert M.nvfp4_get_device_error() == 0
    return ids.cpu().numpy(), w.cpu().numpy(), logits.cpu().numpy()


def check(x_bits, w_bits, k):
    ids, p, lg = run(x_bits, w_bits, k)
    exact = R.router_logits_f64(x_bits, w_bits)
    xf = F.bf16_bits_to_f32(x_bits).astype(np.float64)
    wf = F.bf16_bits_to_f32(w_bits).astype(np.float64)
    bound = 2.0 ** -12 * (np.abs(xf) @ np.abs(wf).T)
    err = np.abs(lg.astype(np.float64) - exact)
    assert np.all(err <= bound), float((err / np.maximum(bound, 1e-30)).max())
    assert np.linalg.norm(lg - exact) <= 1e-5 * np.linalg.norm(exact)
    # selection and probabilities in the kernel's own precision
    lg64 = lg.astype(np.float64)
    assert np.array_equal(ids, R.topk_order(lg64, k))
    ref_p = R.topk_probs(lg64, ids)
    assert np.all(np.abs(p - ref_p) <= 4e-6 * ref_p + 1e-7)
    # against the exact logits: equal except at near ties
    ids_x = R.topk_order(exact, k)
    bad = np.nonzero(np.any(ids != ids_x, axis=1))[0]
    for t in bad:
        swapped = np.setxor1d(ids[t], ids_x[t])
        if swapped.size == 0:          # same set, different order: order decided by a near tie
            swapped = np.concatenate([ids[t], ids_x[t]])
        vals = exact[t, swapped]
        assert vals.max() - vals.min() <= 2 * bound[t].max(), (t, ids[t], ids_x[t])
    return ids, p, lg, len(bad)


# H = 192 and 320 split H/64 unevenly over the four K quarters (192: the first quarter is
# empty); E = 48 leaves the upper half of the lanes with one logit each
@pytest.mark.parametrize("T,H,E,k", [(1, 256, 16, 4), (77, 256, 16, 4), (128, 512, 32, 8), (300, 1024, 64, 8),
                                     (129, 256, 256, 32), (50, 192, 16, 4), (200, 320, 48, 5)])
def test_router_small_shapes(T, H, E, k):
    cfg = S.LayerConfig("router_test", H=H, I=128, E=E, k=k, T=T, seed=T + H + E)
    check(S.make_x(cfg), S.make_router_weights(cfg), k)


def test_router_qwen3_shape():
    cfg = S.CONFIGS["qwen3_30b_a3b"]
    ids, p, lg, n_near_ties = check(S.make_x(cfg), S.make_router_weights(cfg), cfg.k)
    assert n_near_ties <= cfg.T // 100         # near ties are rare on continuous inputs


def test_router_ties_lower_id_first():
    cfg = S.LayerConfig("router_ties", H=256, I=128, E=32, k=6, T=64, seed=11)
    x = S.make_x(cfg)
    w = S.make_router_weights(cfg)
    w[7] = w[3]                                 # experts 3 and 7, 12 and 20 give identical logits
    w[20] = w[12]
    ids, p, lg = run(x, w, cfg.k)
    assert np.array_equal(lg[:, 3], lg[:, 7]) and np.array_equal(lg[:, 12], lg[:, 20])
    for t in range(cfg.T):
        row = list(ids[t])
        for a, b in ((3, 7), (12, 20)):
            if a in row and b in row:
                assert row.index(a) < row.index(b)
                assert p[t, row.index(a)] == p[t, row.index(b)]
            else:
                assert b not in row or a in row      # the higher id never wins a tie alone
    assert np.array_equal(ids, R.topk_order(lg.astype(np.float64), cfg.k))


def test_router_batch_invariance():
    cfg = S.shrink(S.CONFIGS["qwen3_30b_a3b"], T=1000)
    x = S.make_x(cfg)
    w = S.make_router_weights(cfg)
    ids, p, lg = run(x, w, cfg.k)
    for T in (1, 37, 128, 300, 999):
        i2, p2, l2 = run(x[:T], w, cfg.k)
        assert np.array_equal(i2, ids[:T]) and np.array_equal(p2.view(np.uint32), p[:T].view(np.uint32))
        assert np.array_equal(l2.view(np.uint32), lg[:T].view(np.uint32))
    perm = np.random.default_rng(1).permutation(1000)
    i3, p3, l3 = run(np.ascontiguousarray(x[perm]), w, cfg.k)
    assert np.array_equal(i3, ids[perm]) and np.array_equal(p3.view(np.uint32), p[perm].view(np.uint32))
    assert np.array_equal(l3.view(np.uint32), lg[perm].view(np.uint32))


def test_router_feeds_the_expert_forward():
    # the router's outputs are valid inputs of the route sort + expert forward
    cfg = S.CONFIGS["tiny"]
    cfg = S.shrink(cfg, E=16, k=2)
    x = S.make_x(cfg)
    wr = S.make_router_weights(cfg)
    ids, p, _ = M.moe_router_topk(bf16_to_torch(x), bf16_to_torch(wr), cfg.k)
    w1, w2 = S.make_weights(cfg)
    layer = M.MoELayer(bf16_to_torch(w1.reshape(-1, cfg.H)).view(cfg.E, 2 * cfg.I, cfg.H),
                       bf16_to_torch(w2.reshape(-1, cfg.I)).view(cfg.E, cfg.H, cfg.I))
    out = layer.forward(bf16_to_torch(x), ids, p)
    assert M.nvfp4_get_device_error() == 0
    assert torch.isfinite(out.float()).all()
    assert torch.allclose(p.sum(dim=1), torch.ones(cfg.T, device=p.device), rtol=0, atol=2e-6)
