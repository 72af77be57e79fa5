"""Pins of the router-step oracle (oracle/router.py) against closed forms, brute force and
the routing rule of the input generator; no GPU."""

from fractions import Fraction

import numpy as np
import pytest

import moe_synth as S
from oracle import formats as F
from oracle import router as R


def bits(a):
    return S.f32_to_bf16_bits(np.asarray(a, dtype=np.float32))


def test_logits_exact_on_small_rows():
    rng = np.random.default_rng(3)
    x = bits(rng.standard_normal((5, 64)))
    w = bits(rng.standard_normal((7, 64)) / 8)
    got = R.router_logits_f64(x, w)
    xf, wf = F.bf16_bits_to_f32(x), F.bf16_bits_to_f32(w)
    for t in range(5):
        for e in range(7):
            exact = sum(Fraction(float(a)) * Fraction(float(b)) for a, b in zip(xf[t], wf[e]))
            assert abs(Fraction(got[t, e]) - exact) <= Fraction(1, 2 ** 45) * (1 + abs(exact))


def test_logits_one_hot_weights_select_columns():
    rng = np.random.default_rng(4)
    x = bits(rng.standard_normal((9, 32)))
    w = np.zeros((6, 32), np.uint16)
    for e in range(6):
        w[e, 5 * e % 32] = 0x3F80                      # 1.0 in BF16
    got = R.router_logits_f64(x, w)
    xf = F.bf16_bits_to_f32(x).astype(np.float64)
    for e in range(6):
        assert np.array_equal(got[:, e], xf[:, 5 * e % 32])


def brute_topk(row, k):
    return [e for _, e in sorted(((-v, e) for e, v in enumerate(row)))[:k]]


def test_topk_matches_brute_force_and_breaks_ties_by_lower_id():
    rng = np.random.default_rng(5)
    logits = rng.integers(-3, 4, size=(50, 12)).astype(np.float64)   # many ties
    for k in (1, 3, 12):
        ids = R.topk_order(logits, k)
        for t in range(50):
            assert list(ids[t]) == brute_topk(logits[t], k)
    row = np.array([[1.0, 2.0, 2.0, 0.5, 2.0]])
    assert list(R.topk_order(row, 3)[0]) == [1, 2, 4]


def test_topk_permutation_covariance_without_ties():
    rng = np.random.default_rng(6)
    logits = rng.standard_normal((20, 16))
    perm = rng.permutation(16)
    ids = R.topk_order(logits, 5)
    ids_p = R.topk_order(logits[:, perm], 5)
    assert np.array_equal(perm[ids_p], ids)


def test_probs_equal_renormalised_full_softmax():
    rng = np.random.default_rng(7)
    logits = rng.standard_normal((30, 16)) * 3
    ids = R.topk_order(logits, 4)
    p = R.topk_probs(logits, ids)
    full = np.exp(logits - logits.max(axis=1, keepdims=True))
    full /= full.sum(axis=1, keepdims=True)
    sel = np.take_along_axis(full, ids.astype(np.int64), axis=1)
    assert np.allclose(p, sel / sel.sum(axis=1, keepdims=True), rtol=1e-14, atol=0)
    assert np.allclose(p.sum(axis=1), 1.0, rtol=1e-15)
    assert np.all(np.diff(p, axis=1) <= 0)             # slot order = descending probability


def test_probs_special_cases():
    logits = np.array([[0.5, 0.5, 0.5, -1.0]])
    ids = R.topk_order(logits, 3)
    assert list(ids[0]) == [0, 1, 2]
    assert np.array_equal(R.topk_probs(logits, ids), np.full((1, 3), 1 / 3))
    assert np.array_equal(R.topk_probs(logits, R.topk_order(logits, 1)), np.ones((1, 1)))


def test_rule_matches_the_input_generator():
    # make_routing draws logits on sub-stream 3 and selects by (probability desc, id asc);
    # the oracle's top-k on the same logits (logit desc, id asc) must give the same ids
    cfg = S.shrink(S.CONFIGS["qwen3_30b_a3b"], T=64)
    ids_gen, w_gen = S.make_routing(cfg)
    logits = S._rng(cfg.seed, 3).standard_normal((cfg.T, cfg.E)).astype(np.float64)
    ids = R.topk_order(logits, cfg.k)
    assert np.array_equal(ids, ids_gen)
    assert np.allclose(R.topk_probs(logits, ids), w_gen, rtol=1e-6, atol=0)


def test_router_weights_generator():
    cfg = S.CONFIGS["tiny"]
    w = S.make_router_weights(cfg)
    assert w.shape == (cfg.E, cfg.H) and w.dtype == np.uint16
    assert np.array_equal(w, S.make_router_weights(cfg))
    wf = F.bf16_bits_to_f32(w)
    assert abs(float(wf.std()) * np.sqrt(cfg.H) - 1.0) < 0.1
