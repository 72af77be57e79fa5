"""MoE expert forward: route sort, FC1, SwiGLU x prob, requant, FC2, fixed-order combine.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__``).

Sources:

* page "miniTE diagnoses and narrows the cross-engine execution gap of NVFP4
  RL" (onedev.kr/papers/1404), section "How it differs": per-token activation
  outer scale g^x and per-row weight outer scale g^w are multiplied in an FP32
  epilogue before the BF16 cast; the router probability is applied to the
  SwiGLU activation before FC2; the expert combine order is kept through
  padding, quantisation and cast;
* the same page, section "How to use it": tokens are sorted by expert, the
  per-token amax is taken during the sort and reused to quantise, and the FC2
  quantisation maxima come from the producer of the router-weighted
  activation;
* page "Finishing RL training faster: bitwise consistency, high performance,
  agent-driven" (spke.com/ko/ai/article/3192), section 4.4 "Expert GEMM: two
  layouts, same row result": SiLU(gate)*up computed in FP32, only the product
  rounded to BF16, then quantised; each row's result is independent of its
  neighbours; section 4.5 "Cross-GPU reduction": expert outputs are summed in
  FP32 in top-k slot order.

Readings where the pages are silent: the GEMM
accumulation is exact (FP64 on the exactly dequantised operands q*s, outer
scales applied afterwards, (acc*g^x)*g^w, one rounding to BF16); W1's rows are
gate rows 0..I-1 then up rows I..2I-1; SiLU(a) = a / (1 + exp(-a)) evaluated in
FP64 and rounded once to FP32; h = bf16( f32( f32(silu * up) * p ) ); the
combine is an FP32 left-to-right sum from 0 over slots 0..k-1, then BF16; the
rows of one expert are its (token, slot) pairs in token-then-slot order.

Parity: pinned (tests/test_oracle_moe.py) by brute-force loops on tiny
shapes, closed forms of the GEMM, the dense-MLP special case (E=1, k=1, p=1)
against an unquantised FP64 SwiGLU MLP, and permutation / k=1 invariants of
the combine.
"""

import numpy as np

from .formats import bf16_bits_to_f32, round_to_bf16_bits
from .quant import quantize_rows, dequantize_rows


def route_sort(topk_ids, num_experts):
    """Counting sort of the (token, slot) pairs by expert, stable in token-then-slot order.

    Returns (counts [E], offsets [E+1] (unpadded), order): ``order[offsets[e]:
    offsets[e+1]]`` are the pair indices p = token*k + slot routed to expert e,
    ascending.
    """
    ids = np.asarray(topk_ids)
    flat = ids.reshape(-1).astype(np.int64)
    if np.any(flat < 0) or np.any(flat >= num_experts):
        raise ValueError("route_sort: expert id out of range")
    counts = np.bincount(flat, minlength=num_experts)
    order = np.argsort(flat, kind="stable")
    offsets = np.concatenate([[0], np.cumsum(counts)]).astype(np.int64)
    return counts, offsets, order


def qgemm_f64(a_codes, a_scales, w_codes, w_scales):
    """acc[m, n] = sum_k (q_a s_a)[m, k] * (q_w s_w)[n, k], in FP64 (outer scales excluded)."""
    a = dequantize_rows(a_codes, a_scales)
    w = dequantize_rows(w_codes, w_scales)
    return a @ w.T


def epilogue_f64(acc, g_rows, g_cols):
    """Pre-cast epilogue value v = (acc * g^x[row]) * g^w[col], in FP64."""
    return (acc * np.asarray(g_rows, np.float64)[:, None]) * np.asarray(g_cols, np.float64)[None, :]


def silu_f32(gate_bits):
    """silu(a) = a / (1 + exp(-a)) of BF16 values (bits), evaluated in FP64 and rounded
    once to FP32."""
    with np.errstate(over="ignore", invalid="ignore"):
        a = bf16_bits_to_f32(gate_bits).astype(np.float64)
        return (a / (1.0 + np.exp(-a))).astype(np.float32)


def swiglu_prob(gate_bits, up_bits, prob):
    """h = bf16( f32( f32(silu(gate) * up) * p ) ); gate/up BF16 bits, p FP32 per row."""
    silu = silu_f32(gate_bits)                                     # FP64, one rounding
    u = bf16_bits_to_f32(up_bits)
    t1 = (silu * u).astype(np.float32)                             # FP32 product
    t2 = (t1 * np.asarray(prob, np.float32)[:, None]).astype(np.float32)
    return round_to_bf16_bits(t2)


def combine_slots(y_bits):
    """out[t] = bf16( (((0 + y[t,0]) + y[t,1]) + ...) + y[t,k-1] ) with FP32 adds."""
    y_bits = np.asarray(y_bits, dtype=np.uint16)
    T, k, H = y_bits.shape
    acc = np.zeros((T, H), dtype=np.float32)
    for j in range(k):
        acc = (acc + bf16_bits_to_f32(y_bits[:, j, :])).astype(np.float32)
    return round_to_bf16_bits(acc)


class MoEWeightsQ:
    """BF16 expert weights and their per-row NVFP4 quantisation (computed on demand).

    w1_bits: uint16 [E, 2I, H] (gate rows 0..I-1, up rows I..2I-1)
    w2_bits: uint16 [E, H, I]
    """

    def __init__(self, w1_bits, w2_bits):
        self.w1_bits = np.asarray(w1_bits, dtype=np.uint16)
        self.w2_bits = np.asarray(w2_bits, dtype=np.uint16)
        self.E, two_i, self.H = self.w1_bits.shape
        self.I = two_i // 2
        if self.w2_bits.shape != (self.E, self.H, self.I):
            raise ValueError("MoEWeightsQ: W2 must be [E, H, I]")
        self._cache = {}

    def expert(self, e):
        """((codes1, scales1, g1), (codes2, scales2, g2)) for expert e."""
        if e not in self._cache:
            q1 = quantize_rows(bf16_bits_to_f32(self.w1_bits[e]))
            q2 = quantize_rows(bf16_bits_to_f32(self.w2_bits[e]))
            self._cache[e] = (q1, q2)
        return self._cache[e]


def quantize_weights(w1_bits, w2_bits):
    return MoEWeightsQ(w1_bits, w2_bits)


def moe_forward(x_bits, topk_ids, topk_w, wq, keep=False):
    """The layer: BF16 X [T, H] (bits), top-k ids/probs [T, k] -> BF16 out [T, H] (bits).

    With ``keep`` also returns the intermediates, indexed by pair p = t*k + s:
    ``xq`` (codes, scales, g^x per token), ``v1`` FC1 pre-cast FP64 [R, 2I],
    ``gu`` FC1 BF16 bits [R, 2I], ``h`` BF16 bits [R, I], ``hq`` (codes,
    scales, g2) [R, ...], ``v2`` FC2 pre-cast FP64 [R, H], ``y`` BF16 bits
    [T, k, H], plus the sort (counts, offsets, order).
    """
    x_bits = np.asarray(x_bits, dtype=np.uint16)
    topk_ids = np.asarray(topk_ids)
    topk_w = np.asarray(topk_w, dtype=np.float32)
    T, H = x_bits.shape
    k = topk_ids.shape[1]
    E, I = wq.E, wq.I
    if H != wq.H:
        raise ValueError("moe_forward: hidden size mismatch")

    # Per-token quantisation, once per token, shared by its k routed rows.
    xq = quantize_rows(bf16_bits_to_f32(x_bits))
    counts, offsets, order = route_sort(topk_ids, E)

    R = T * k
    y = np.zeros((T, k, H), dtype=np.uint16)
    inter = None
    if keep:
        inter = dict(
            xq=xq, counts=counts, offsets=offsets, order=order,
            v1=np.zeros((R, 2 * I)), gu=np.zeros((R, 2 * I), np.uint16),
            h=np.zeros((R, I), np.uint16),
            hq=(np.zeros((R, I), np.uint8), np.zeros((R, I // 16), np.uint8),
                np.zeros(R, np.float32)),
            v2=np.zeros((R, H)),
        )
    for e in range(E):
        pairs = order[offsets[e]:offsets[e + 1]]
        if len(pairs) == 0:
            continue
        toks, slots = pairs // k, pairs % k
        (c1, s1, g1), (c2, s2, g2w) = wq.expert(e)
        # FC1 (gate + up) and its FP32 epilogue, cast to BF16.
        v1 = epilogue_f64(qgemm_f64(xq[0][toks], xq[1][toks], c1, s1), xq[2][toks], g1)
        gu = round_to_bf16_bits(v1)
        # SwiGLU times the router probability, rounded once to BF16.
        h = swiglu_prob(gu[:, :I], gu[:, I:], topk_w[toks, slots])
        # Requantise; the maxima are those of the produced activation.
        h_f32 = bf16_bits_to_f32(h)
        hq = quantize_rows(h_f32, amax=np.abs(h_f32).max(axis=1))
        # FC2 and its epilogue.
        v2 = epilogue_f64(qgemm_f64(hq[0], hq[1], c2, s2), hq[2], g2w)
        y[toks, slots] = round_to_bf16_bits(v2)
        if keep:
            inter["v1"][pairs] = v1
            inter["gu"][pairs] = gu
            inter["h"][pairs] = h
            inter["hq"][0][pairs] = hq[0]
            inter["hq"][1][pairs] = hq[1]
            inter["hq"][2][pairs] = hq[2]
            inter["v2"][pairs] = v2
    out = combine_slots(y)
    if keep:
        inter["y"] = y
        return out, inter
    return out


def dense_swiglu_mlp_f64(x, w1, w2):
    """Unquantised FP64 SwiGLU MLP: (silu(x W_gate^T) * (x W_up^T)) W2^T.

    Used only as the special-case pin: with one expert, top-1 and probability
    1 the quantised layer must approximate it within the NVFP4 error.
    """
    x = np.asarray(x, np.float64)
    w1 = np.asarray(w1, np.float64)
    w2 = np.asarray(w2, np.float64)
    I = w1.shape[0] // 2
    gate = x @ w1[:I].T
    up = x @ w1[I:].T
    with np.errstate(over="ignore"):
        h = gate / (1.0 + np.exp(-gate)) * up
    return h @ w2.T
