"""Straight-through (STE) backward of the MoE expert layer.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__``).

Source: page "miniTE diagnoses and narrows the cross-engine execution gap of
NVFP4 RL" (onedev.kr/papers/1404), section "How it differs": the backward is a
straight-through approximation that runs BF16 GEMMs on the saved original BF16
activations and weights, so no quantisation runs backward; the same page's
results paragraph measures the BF16 backward's gradients against an FP32
reference by relative L2 (largest difference 0.001663 over its module cells).

What the backward computes (the plainest reading of the page, each quantiser
taken as the identity, every other op differentiated where it ran):

* combine: out[t] = sum over slots of y[t, j], so each slot's output gradient
  is dout[t];
* FC2: y = h W2[e]^T, so dh = dout[t] W2[e] and dW2[e] = sum over the expert's
  pairs of dout[t]^T h (h the saved BF16 activation, W2 the BF16 original);
* SwiGLU x prob: h = silu(a) * u * p with a, u the forward's own FC1 outputs
  (the BF16 gate and up values the SwiGLU ran on): da = dh * p * u * silu'(a),
  du = dh * p * silu(a), dp = sum_i dh_i * silu(a_i) * u_i, where
  silu(a) = a * sigma(a) and silu'(a) = sigma(a) * (1 + a * (1 - sigma(a)));
* FC1: [a, u] = x W1[e]^T, so dx(t, j) = [da, du] W1[e] and
  dW1[e] = sum over the expert's pairs of [da, du]^T x[t];
* dX[t] = sum over slots of dx(t, j), in slot order.

Precision: FP64 on the given values (``bf16_stages=False``, the exact reading
that the page's FP32 reference approximates).  ``bf16_stages=True`` also rounds
to BF16 where a BF16 GEMM pipeline hands a tensor on (a reading: the page
names no rounding points): dh (a BF16 GEMM output), [da, du] (the BF16 operand of the FC1
dgrad and wgrad GEMMs), each slot's dx (a BF16 GEMM output), and dX, summed in
FP32 in slot order and rounded once.  The weight gradients and dp stay FP64.

Parity: pinned (tests/test_oracle_backward.py) by central finite differences
of the unquantised layer on tiny shapes, by float64 autograd of the same layer
on larger ones, by the special cases p = 0 and h = 0 and an empty expert, and
by the BF16 rounding bound between the two precisions.
"""

import numpy as np

from .formats import bf16_bits_to_f32, round_to_bf16_bits
from .moe import route_sort, combine_slots


def _bf16(v):
    """Round FP64/FP32 values to the nearest BF16 value (ties to even), as FP64."""
    return bf16_bits_to_f32(round_to_bf16_bits(np.asarray(v, np.float64).astype(np.float32))).astype(np.float64)


def silu_and_derivative(a):
    """(silu(a), silu'(a)) in FP64: silu(a) = a sigma(a), silu' = sigma (1 + a (1 - sigma))."""
    a = np.asarray(a, np.float64)
    with np.errstate(over="ignore"):
        s = 1.0 / (1.0 + np.exp(-a))
    return a * s, s * (1.0 + a * (1.0 - s))


def moe_backward_ste(dout, x, topk_ids, topk_w, w1, w2, gu, h, bf16_stages=False):
    """STE gradients of the expert layer.

    dout [T, H], x [T, H]: values (BF16 inputs passed as their float values);
    topk_ids [T, k] int, topk_w [T, k]; w1 [E, 2I, H] (gate rows then up
    rows), w2 [E, H, I]; gu [T, k, 2I]: the forward's FC1 outputs of each
    (token, slot), gate then up; h [T, k, I]: the forward's SwiGLU x prob
    activation of each (token, slot).

    Returns a dict: dx [T, H], dw1 [E, 2I, H], dw2 [E, H, I], dprob [T, k]
    and the intermediates dh [T, k, I], dgu [T, k, 2I], dx_slots [T, k, H].
    """
    dout = np.asarray(dout, np.float64)
    x = np.asarray(x, np.float64)
    ids = np.asarray(topk_ids)
    p_all = np.asarray(topk_w, np.float64)
    w1 = np.asarray(w1, np.float64)
    w2 = np.asarray(w2, np.float64)
    gu = np.asarray(gu, np.float64)
    h = np.asarray(h, np.float64)
    T, H = x.shape
    k = ids.shape[1]
    E, two_i, _ = w1.shape
    I = two_i // 2
    rnd = _bf16 if bf16_stages else (lambda v: v)

    dh_all = np.zeros((T, k, I))
    dgu_all = np.zeros((T, k, 2 * I))
    dxs_all = np.zeros((T, k, H))
    dprob = np.zeros((T, k))
    dw1 = np.zeros((E, 2 * I, H))
    dw2 = np.zeros((E, H, I))
    counts, offsets, order = route_sort(ids, E)
    for e in range(E):
        pairs = order[offsets[e]:offsets[e + 1]]
        if len(pairs) == 0:
            continue
        toks, slots = pairs // k, pairs % k
        dy = dout[toks]                                   # each slot's gradient is dout[t]
        # FC2 dgrad and wgrad on the BF16 originals.
        dh = rnd(dy @ w2[e])                              # [n, I]
        dw2[e] = dy.T @ h[toks, slots]                    # [H, I]
        # SwiGLU x prob, at the forward's own gate/up values.
        a = gu[toks, slots, :I]
        u = gu[toks, slots, I:]
        p = p_all[toks, slots][:, None]
        silu, dsilu = silu_and_derivative(a)
        da = dh * p * u * dsilu
        du = dh * p * silu
        dprob[toks, slots] = np.sum(dh * silu * u, axis=1)
        dgu = rnd(np.concatenate([da, du], axis=1))       # [n, 2I]
        # FC1 dgrad and wgrad.
        dxs = rnd(dgu @ w1[e])                            # [n, H]
        dw1[e] = dgu.T @ x[toks]                          # [2I, H]
        dh_all[toks, slots] = dh
        dgu_all[toks, slots] = dgu
        dxs_all[toks, slots] = dxs
    if bf16_stages:
        bits = round_to_bf16_bits(dxs_all.astype(np.float32))     # already BF16 values: exact
        dx = bf16_bits_to_f32(combine_slots(bits)).astype(np.float64)
    else:
        dx = np.zeros((T, H))
        for j in range(k):
            dx = dx + dxs_all[:, j, :]
    return dict(dx=dx, dw1=dw1, dw2=dw2, dprob=dprob, dh=dh_all, dgu=dgu_all, dx_slots=dxs_all)


def forward_saved_activations(x, topk_ids, topk_w, w1, w2):
    """Unquantised FP64 forward of the layer, keeping what the backward needs.

    Returns (out [T, H], gu [T, k, 2I], h [T, k, I]) with gu = x W1[e]^T and
    h = silu(gate) * up * p, no rounding anywhere.  With these saved values the
    STE backward is the exact gradient of ``out`` (the finite-difference and
    autograd pins rely on it).
    """
    x = np.asarray(x, np.float64)
    ids = np.asarray(topk_ids)
    p_all = np.asarray(topk_w, np.float64)
    w1 = np.asarray(w1, np.float64)
    w2 = np.asarray(w2, np.float64)
    T, H = x.shape
    k = ids.shape[1]
    I = w1.shape[1] // 2
    gu = np.zeros((T, k, 2 * I))
    h = np.zeros((T, k, I))
    out = np.zeros((T, H))
    for t in range(T):
        for j in range(k):
            e = ids[t, j]
            g = w1[e] @ x[t]
            silu, _ = silu_and_derivative(g[:I])
            gu[t, j] = g
            h[t, j] = silu * g[I:] * p_all[t, j]
            out[t] += w2[e] @ h[t, j]
    return out, gu, h
