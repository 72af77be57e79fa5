"""Shared test plumbing: numpy <-> torch moves of BF16 bit patterns, tolerances."""

import numpy as np
import torch


def bf16_to_torch(bits, device="cuda"):
    """uint16 bit patterns (numpy) -> torch.bfloat16 tensor on `device`."""
    t = torch.from_numpy(np.ascontiguousarray(bits, dtype=np.uint16).view(np.int16))
    return t.view(torch.bfloat16).to(device)


def torch_to_bf16_bits(t):
    """torch.bfloat16 tensor -> numpy uint16 bit patterns."""
    return t.detach().contiguous().cpu().view(torch.int16).numpy().view(np.uint16)


def rel_l2(a, b):
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    den = np.linalg.norm(b)
    return float(np.linalg.norm(a - b) / (den if den > 0 else 1.0))


def bf16_ulp_distance(a_bits, b_bits):
    """Distance in BF16 units in the last place between two arrays of bit patterns."""
    def ordered(x):
        x = np.asarray(x, np.uint16).astype(np.int32)
        return np.where(x & 0x8000, 0x8000 - (x & 0x7FFF), 0x8000 + (x & 0x7FFF))
    return np.abs(ordered(a_bits) - ordered(b_bits))


# Tolerances, stated once:
#  GEMM stages given identical quantised inputs: FP32 accumulation on the tensor
#  cores vs the exact FP64 sum, relative L2 of the pre-cast values <= 1e-5, and
#  the BF16 outputs within 1 unit in the last place.
GEMM_REL_L2 = 1e-5
GEMM_BF16_ULP = 1
#  end-to-end layer vs the oracle: relative L2 <= 1e-2, FC2 requant code flips <= 0.1%
LAYER_REL_L2 = 1e-2
FC2_CODE_FLIP_RATE = 1e-3


def bf16_ulp(x):
    """Unit in the last place of BF16 at the magnitude of each FP32 value (2^-133 at 0)."""
    return np.spacing(np.abs(np.asarray(x, np.float32))).astype(np.float64) * 65536.0


def h_bound(gate_gpu, up_gpu, gate_ref, up_ref, prob, h_gpu, h_ref):
    """Per-element bound on |h_gpu - h_ref| for h = bf16(f32(f32(silu(gate) * up) * p)) when the
    two sides' BF16 gate/up inputs differ (FC1's 1-ulp cast differences).  With s = silu
    evaluated in FP64 at each side's own gate:
        |h_gpu - h_ref| <= |p| (|s(g') - s(g)| |u'| + |s(g)| |u' - u|)       (the inputs)
                           + (ulp(h_gpu) + ulp(h_ref)) / 2                   (the BF16 roundings)
                           + 2^-21 (|h_gpu| + |h_ref|)                       (three FP32 roundings)
    All arguments are FP32/FP64 values (gate and up already decoded from BF16)."""
    def silu(a):
        a = np.asarray(a, np.float64)
        with np.errstate(over="ignore"):
            return a / (1.0 + np.exp(-a))
    g1, u1 = np.asarray(gate_gpu, np.float64), np.asarray(up_gpu, np.float64)
    g0, u0 = np.asarray(gate_ref, np.float64), np.asarray(up_ref, np.float64)
    p = np.abs(np.asarray(prob, np.float64))
    hg, hr = np.asarray(h_gpu, np.float64), np.asarray(h_ref, np.float64)
    inputs = p * (np.abs(silu(g1) - silu(g0)) * np.abs(u1) + np.abs(silu(g0)) * np.abs(u1 - u0))
    return inputs + 0.5 * (bf16_ulp(hg) + bf16_ulp(hr)) + 2.0 ** -21 * (np.abs(hg) + np.abs(hr))
