"""The SiLU the FC1 epilogue applies (its shared-memory range of the table and its closed
forms outside it, run by the epilogue's own device function) equals the oracle's SiLU, FP64
then one rounding to FP32, bit for bit at all 65,536 BF16 gate values ("Finishing RL
training faster: bitwise consistency, high performance, agent-driven", section 4.4)."""

import numpy as np
import pytest
import torch

import nvfp4_moe_expert_gb300 as M
from nvfp4_moe_expert_gb300 import build as B
from oracle import moe as OM

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    B.build()
    M.lib()


def test_device_table_equals_oracle_silu():
    dev = M.nvfp4_silu_table().cpu().numpy().view(np.uint32)
    ref = OM.silu_f32(np.arange(65536, dtype=np.uint32).astype(np.uint16)).view(np.uint32)
    nan_d = np.isnan(dev.view(np.float32))
    assert np.array_equal(nan_d, np.isnan(ref.view(np.float32)))
    assert np.array_equal(dev[~nan_d], ref[~nan_d])


def test_table_is_there_before_any_forward():
    # a fresh stream, no FC1 launched on it: the table is part of the loaded library
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        out = M.nvfp4_silu_table(stream=s)
    s.synchronize()
    assert out.cpu().numpy().view(np.uint32)[0x3F80] == np.float32(1.0 / (1.0 + np.exp(-1.0))).view(np.uint32)
