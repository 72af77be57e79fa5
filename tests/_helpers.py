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
