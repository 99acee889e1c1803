"""Exhaustive fp32 -> bf16 check of the all-gather cast: every one of the 2^32
binary32 bit patterns goes through dpg_allgather_params (16 launches of 2^28
elements) and must equal the oracle's round-to-nearest-even conversion (NaN
inputs must give a NaN; its payload and sign are not unique)."""
import numpy as np
import pytest
import torch

import oracle
import zero_optimizer_step_gb300 as dpg
from parity_util import np_bf16

pytestmark = pytest.mark.gpu

CHUNK = 1 << 28


def test_all_fp32_patterns():
    from zero_optimizer_step_gb300 import build
    build.build()
    plan = dpg.dpg_plan_buckets([CHUNK], 1 << 40, 1)
    assert plan.total_padded == CHUNK
    out = torch.empty(CHUNK, dtype=torch.bfloat16, device="cuda")
    for c in range(1 << 32 >> 28):
        base = (c << 28) - (1 << 32 if c >= 8 else 0)      # same bits as a signed int32
        bits = torch.arange(base, base + CHUNK, dtype=torch.int32, device="cuda")
        dpg.dpg_allgather_params(plan, bits.view(torch.float32), [out])
        got = np_bf16(out)
        pats = (np.arange(CHUNK, dtype=np.uint64) + (c << 28)).astype(np.uint32)
        ref = oracle.f32_to_bf16(pats.view(np.float32))
        nan_in = ((pats & 0x7F800000) == 0x7F800000) & ((pats & 0x7FFFFF) != 0)
        assert np.array_equal(got[~nan_in], ref[~nan_in]), f"chunk {c}"
        g_nan = got[nan_in]
        assert np.all((g_nan & 0x7F80) == 0x7F80) and np.all((g_nan & 0x7F) != 0), f"chunk {c}"
