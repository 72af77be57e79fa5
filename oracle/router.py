"""Router step: FP32-output router GEMM, deterministic top-k, renormalised probabilities.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__``).

Sources: page "Finishing RL training faster: bitwise consistency, high
performance, agent-driven" (spke.com/ko/ai/article/3192):

* section 4.1 "Dense GEMM": the router gate uses one FP32-output GEMM for every
  batch size (no small-batch kernel switch), so a token's scores do not depend
  on its neighbours;
* section 2 (the conditions beyond the four dimensions): top-k and MoE routing
  turn a 1-ulp difference upstream into a different expert set, so ties and the
  output order must be fixed too;
* section 4.4 (the "R3 unnecessary" paragraph): with the single FP32-output
  router kernel the recomputed routing matches the rollout's.

Readings taken: logits[t, e] = sum_h x[t, h] * W_r[e, h] on the
BF16 values, here exact (FP64 of exactly representable products); the k
selected experts are the k largest logits, a larger logit first and, on equal
logits, the lower expert id first (softmax is monotonic, so this is the order
of the probabilities); the probabilities are the softmax over all experts
renormalised over the k chosen, which equals the softmax over the k chosen
logits, p_j = exp(l_j - l_1) / sum_i exp(l_i - l_1), here in FP64.

Every function is pinned by ``tests/test_oracle_router.py``.
"""

import numpy as np

from .formats import bf16_bits_to_f32


def router_logits_f64(x_bits, w_bits):
    """logits [T, E] (FP64) of BF16 activations x [T, H] and router weights W_r [E, H] (uint16 bits)."""
    x = bf16_bits_to_f32(np.asarray(x_bits)).astype(np.float64)
    w = bf16_bits_to_f32(np.asarray(w_bits)).astype(np.float64)
    return x @ w.T


def topk_order(logits, k):
    """Expert ids [T, k] of the k largest logits per row: larger logit first, lower id first on ties."""
    logits = np.asarray(logits)
    T, E = logits.shape
    if not 1 <= k <= E:
        raise ValueError("k out of range")
    out = np.empty((T, k), dtype=np.int32)
    ids = np.arange(E)
    for t in range(T):
        # lexicographic sort on (-logit, id): np.lexsort sorts by the last key first
        order = np.lexsort((ids, -logits[t]))
        out[t] = order[:k]
    return out


def topk_probs(logits, ids):
    """Softmax of each row's selected logits, in slot order (FP64)."""
    sel = np.take_along_axis(np.asarray(logits, dtype=np.float64), np.asarray(ids, dtype=np.int64), axis=1)
    z = np.exp(sel - sel[:, :1])
    return z / z.sum(axis=1, keepdims=True)


def router_topk(x_bits, w_bits, k):
    """(ids int32 [T, k], probs float64 [T, k], logits float64 [T, E]) of the router step."""
    logits = router_logits_f64(x_bits, w_bits)
    ids = topk_order(logits, k)
    return ids, topk_probs(logits, ids), logits
