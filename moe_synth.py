"""Seeded synthetic inputs for the NVFP4 MoE expert forward.

This module only draws inputs; it holds none of the layer's arithmetic and is
the one piece of code that both the CPU oracle and the CUDA path are fed from.

Workloads (sizes of the Qwen3-30B-A3B-style MoE layers the miniTE summary
measures on, section "How it works" / "Assumptions and limits"; the real
weights and the DAPO-Math text are not available, so seeded synthetic tensors
of the same shapes stand in for them):

* ``tiny``   hidden 256, expert intermediate 128, 8 experts, top-2, 64 tokens
* ``qwen3_30b_a3b``   hidden 2048, intermediate 768, 128 experts, top-8, 4096
  tokens, balanced routing
* ``qwen3_30b_a3b_skew``   same layer, 16384 tokens, Zipf(s=1.1) expert bias
  on the router logits, 1% of hidden channels scaled x20 (activation outliers)
* ``large``   hidden 4096, intermediate 1536, 128 experts, top-8, 32768
  tokens, Zipf routing, 1% outlier channels, weights N(0, 0.015)

Recipe: numpy PCG64 (throughput runs of the large layers may draw the
weights on the GPU instead, make_weights_device); sub-streams seed+0 (X), +1 (W1), +2 (W2), +3 (router
logits), +4 (outlier channels), +5 (sequence lengths), +6 (router weights for
the router step, W_r ~ N(0, 1/H) so that logits of N(0,1) inputs are about
N(0,1)), +7 (the output gradient of the backward, dOut ~ N(0, 1)).  Values are
drawn in
float32 and rounded to BF16 (round-to-nearest-even on the bit pattern).
Routing: softmax over experts in FP64, top-k by (probability descending,
expert id ascending), probabilities renormalised over the k chosen experts in
FP64, then rounded to FP32.
"""

from dataclasses import dataclass, replace

import numpy as np


@dataclass(frozen=True)
class LayerConfig:
    name: str
    H: int                   # hidden size
    I: int                   # expert intermediate size (FC1 has 2I outputs)
    E: int                   # experts
    k: int                   # top-k
    T: int                   # tokens
    routing: str = "uniform"  # "uniform" or "zipf"
    outlier_frac: float = 0.0
    w_std: float = 0.02
    seed: int = 0


CONFIGS = {
    "tiny": LayerConfig("tiny", H=256, I=128, E=8, k=2, T=64),
    "qwen3_30b_a3b": LayerConfig("qwen3_30b_a3b", H=2048, I=768, E=128, k=8, T=4096),
    "qwen3_30b_a3b_skew": LayerConfig("qwen3_30b_a3b_skew", H=2048, I=768, E=128, k=8,
                                      T=16384, routing="zipf", outlier_frac=0.01),
    "large": LayerConfig("large", H=4096, I=1536, E=128, k=8, T=32768, routing="zipf",
                         outlier_frac=0.01, w_std=0.015),
}


def _rng(seed, sub):
    return np.random.Generator(np.random.PCG64(seed + sub))


def f32_to_bf16_bits(a):
    """Round binary32 values to BF16 (RNE) and return the uint16 bit patterns."""
    # 32-bit arithmetic: a carry past 2^32 (only from negative NaN patterns) is dropped by
    # the final 16-bit truncation either way, so the bits equal a 64-bit computation's
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32)
    rounded = (u + np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))) >> np.uint32(16)
    return rounded.astype(np.uint16)


def bf16_bits_as_f32(bits):
    return (np.asarray(bits, np.uint16).astype(np.uint32) << 16).view(np.float32)


def outlier_channels(cfg):
    n = int(round(cfg.outlier_frac * cfg.H))
    if n == 0:
        return np.zeros(0, dtype=np.int64)
    return np.sort(_rng(cfg.seed, 4).choice(cfg.H, size=n, replace=False))


def make_x(cfg, T=None, stream=0):
    """BF16 activations [T, H] as uint16 bits; X ~ N(0,1), outlier channels x20."""
    T = cfg.T if T is None else T
    rng = _rng(cfg.seed + 1000 * stream, 0)
    x = rng.standard_normal((T, cfg.H), dtype=np.float32)
    ch = outlier_channels(cfg)
    if len(ch):
        x[:, ch] *= np.float32(20.0)
    return f32_to_bf16_bits(x)


def make_weights(cfg, experts=None):
    """BF16 expert weights as uint16 bits: W1 [E, 2I, H] (gate rows, then up rows), W2 [E, H, I].

    ``experts`` limits the draw to the first n experts' worth of the stream
    (the same values the full draw gives for those experts).
    """
    E = cfg.E if experts is None else experts
    w1 = np.empty((E, 2 * cfg.I, cfg.H), dtype=np.uint16)
    w2 = np.empty((E, cfg.H, cfg.I), dtype=np.uint16)
    r1, r2 = _rng(cfg.seed, 1), _rng(cfg.seed, 2)
    std = np.float32(cfg.w_std)
    for e in range(E):   # one expert at a time keeps the float32 temporaries small
        w1[e] = f32_to_bf16_bits(r1.standard_normal((2 * cfg.I, cfg.H), dtype=np.float32) * std)
        w2[e] = f32_to_bf16_bits(r2.standard_normal((cfg.H, cfg.I), dtype=np.float32) * std)
    return w1, w2


def make_weights_device(cfg, device, seed_offset=0):
    """BF16 expert weights drawn on the GPU (torch tensors W1 [E, 2I, H], W2 [E, H, I]),
    N(0, w_std) rounded to BF16: the same distribution as make_weights from torch's seeded
    device generator (sub-streams seed+1 and seed+2), for throughput runs of layers whose
    host-side draw would take a minute.  The values differ from make_weights'."""
    import torch
    out = []
    for sub, shape in ((1, (cfg.E, 2 * cfg.I, cfg.H)), (2, (cfg.E, cfg.H, cfg.I))):
        g = torch.Generator(device=device)
        g.manual_seed(cfg.seed + sub + seed_offset)
        w = torch.empty(shape, dtype=torch.bfloat16, device=device)
        for e in range(cfg.E):   # one expert at a time keeps the float32 temporary small
            w[e] = (torch.randn(shape[1:], generator=g, device=device, dtype=torch.float32)
                    * cfg.w_std).to(torch.bfloat16)
        out.append(w)
    return tuple(out)


def make_routing(cfg, T=None, stream=0):
    """Top-k expert ids (int32 [T, k]) and renormalised probabilities (float32 [T, k])."""
    T = cfg.T if T is None else T
    rng = _rng(cfg.seed + 1000 * stream, 3)
    logits = rng.standard_normal((T, cfg.E)).astype(np.float64)
    if cfg.routing == "zipf":
        rank = np.arange(1, cfg.E + 1, dtype=np.float64)
        logits = logits + (-1.1 * np.log(rank))[None, :]
    elif cfg.routing != "uniform":
        raise ValueError(cfg.routing)
    z = logits - logits.max(axis=1, keepdims=True)
    probs = np.exp(z)
    probs /= probs.sum(axis=1, keepdims=True)
    # stable sort on -prob: equal probabilities keep ascending expert id
    order = np.argsort(-probs, axis=1, kind="stable")[:, :cfg.k]
    top = np.take_along_axis(probs, order, axis=1)
    top = top / top.sum(axis=1, keepdims=True)
    return order.astype(np.int32), top.astype(np.float32)


def make_router_weights(cfg):
    """BF16 router weights W_r [E, H] as uint16 bits, N(0, 1/H) (rows = experts)."""
    rng = _rng(cfg.seed, 6)
    w = rng.standard_normal((cfg.E, cfg.H), dtype=np.float32) * np.float32(1.0 / np.sqrt(cfg.H))
    return f32_to_bf16_bits(w)


def make_grad_out(cfg, T=None, stream=0):
    """BF16 output gradient dOut [T, H] as uint16 bits, N(0, 1)."""
    T = cfg.T if T is None else T
    rng = _rng(cfg.seed + 1000 * stream, 7)
    return f32_to_bf16_bits(rng.standard_normal((T, cfg.H), dtype=np.float32))


def make_layer(cfg, T=None, experts=None):
    """Everything a forward needs: dict of x, w1, w2, topk_ids, topk_w (numpy)."""
    x = make_x(cfg, T)
    ids, w = make_routing(cfg, T)
    w1, w2 = make_weights(cfg, experts)
    return dict(x=x, w1=w1, w2=w2, topk_ids=ids, topk_w=w)


def sequence_lengths(cfg, n_seq=256, lo=64, hi=2048):
    """Lengths of the batch-invariance sweep's sequences, uniform on {lo..hi}."""
    return _rng(cfg.seed, 5).integers(lo, hi + 1, size=n_seq)


def shrink(cfg, **kw):
    return replace(cfg, **kw)
