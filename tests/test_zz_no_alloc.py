"""dpg_step_noalloc: the allocation-free variant of dpg_step.

Some callers cannot let a library allocate device memory -- their device
memory belongs to another allocator (a framework's caching pool or a fixed
budget), or they cannot accept cudaMalloc/cudaFree synchronising the device in
the middle of a step.  dpg_step_noalloc serves them from one static device
array compiled into the library.  These tests call it through the C ABI and
check, on two calls in a row, that it gives what dpg_step gives (master/m/v
within 2 ulp, bf16 parameters within 1 ulp, norms within 1e-5 relative, equal
non-finite counts -- the same bars as every other parity test), and that a
plan too large for the static array is refused before any device work.

The file is named so that pytest collects it last; it passes alone in a fresh
process (where its first call performs the one-time address lookup) and after
the other tests.
"""
import ctypes

import numpy as np
import pytest
import torch

import zero_optimizer_step_gb300 as dpg
from parity_util import BF16_ULP, F32_ULP, NORM_RTOL, np_bf16, np_f32, ulp_bf16, ulp_f32
from workloads import (CONFIGS, KIND_GRAD, KIND_MASTER, flat_grads_bf16, master_f32,
                       random_param_list, segments, stream_seed)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    from zero_optimizer_step_gb300 import build
    build.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"


def _case(name):
    if name == "tiny":
        c = CONFIGS["tiny"]
        return c.numels, c.cap_bytes, c.R, 1, list(c.fixed_tokens), c.grad_std
    rng = np.random.Generator(np.random.Philox(4242))
    if name == "R8_ragged":
        return random_param_list(rng, 60, 300_000), 1 << 20, 8, 1, None, 1e-3
    return random_param_list(rng, 40, 200_000), 1 << 19, 4, 2, None, 1e-3   # R4_acc_K2


@pytest.mark.parametrize("name", ["tiny", "R8_ragged", "R4_acc_K2"])
def test_noalloc_matches_dpg_step_on_two_calls_in_a_row(name):
    numels, cap, R, K, tokens, std = _case(name)
    plan = dpg.dpg_plan_buckets(numels, cap, R)
    N = plan.total_padded
    segs = segments(plan.param_offset, numels)
    dev = "cuda"
    w0 = master_f32(N, stream_seed(11, KIND_MASTER), device=dev)
    st = {side: dict(w=w0.clone(), m=torch.zeros(N, device=dev), v=torch.zeros(N, device=dev),
                     p=torch.empty(N, dtype=torch.bfloat16, device=dev),
                     sq=torch.full((plan.n_buckets,), -1.0, device=dev),
                     nf=torch.full((plan.n_buckets,), -1, dtype=torch.int64, device=dev))
          for side in ("noalloc", "step")}
    for call in (1, 2):
        micro = [[flat_grads_bf16(segs, N, std, stream_seed(11 + call, KIND_GRAD, r, k), device=dev)
                  for k in range(K)] for r in range(R)]
        tok = tokens or [3000 + 97 * call + 13 * i for i in range(R * K)]
        hp = dpg.HParams(step=call, weight_decay=0.01 * (call - 1))
        for side, fn in (("noalloc", dpg.dpg_step_noalloc), ("step", dpg.dpg_step)):
            s = st[side]
            if K > 1:
                acc = [torch.empty(N, device=dev) for _ in range(R)]
                for k in range(K - 1):
                    for r in range(R):
                        dpg.dpg_accumulate(plan, micro[r][k], acc[r], first=(k == 0))
                fn(plan, acc, tok, hp, s["w"], s["m"], s["v"], [s["p"]],
                   last_micro=[micro[r][K - 1] for r in range(R)], bucket_sqnorm=s["sq"],
                   bucket_nonfinite=s["nf"])
            else:
                fn(plan, [micro[r][0] for r in range(R)], tok, hp, s["w"], s["m"], s["v"],
                   [s["p"]], bucket_sqnorm=s["sq"], bucket_nonfinite=s["nf"])
        torch.cuda.synchronize()
        a, b = st["noalloc"], st["step"]
        for k in ("w", "m", "v"):
            assert ulp_f32(np_f32(a[k]), np_f32(b[k])) <= F32_ULP, (call, k)
        assert ulp_bf16(np_bf16(a["p"]), np_bf16(b["p"])) <= BF16_ULP, call
        sa, sb = np_f32(a["sq"]).astype(np.float64), np_f32(b["sq"]).astype(np.float64)
        assert np.all(np.abs(sa - sb) <= NORM_RTOL * np.abs(sb)), call
        assert np.all(sb >= 0)
        np.testing.assert_array_equal(a["nf"].cpu().numpy(), b["nf"].cpu().numpy())


def test_noalloc_refuses_plans_beyond_its_scratch():
    # 2000 one-parameter buckets of 123 tiles each: every CTA visits hundreds of
    # buckets, so the norm partials alone need tens of MB.  All buffers are NULL:
    # the call must stop at the size check (and would stop at the NULL checks
    # otherwise), so nothing can reach the device.
    plan = dpg.dpg_plan_buckets([500_000] * 2000, 1 << 20, 1)
    assert plan.n_buckets == 2000
    hp = dpg.HParams().c()
    tok = np.array([100], np.int64)
    before = dpg.dpg_launch_count()
    rc = dpg.lib().dpg_step_noalloc(plan.handle, dpg._ptrs([0]), dpg.DPG_BF16, None,
                                    tok.ctypes.data, 1, ctypes.byref(hp), None, None, None,
                                    dpg._ptrs([0]), 1, 1 << 20, None, None)
    assert rc == dpg.DPG_ERR_INVALID_ARG
    msg = dpg.lib().dpg_last_error().decode()
    assert "scratch" in msg and str(dpg.DPG_NOALLOC_SCRATCH_BYTES) in msg, msg
    assert dpg.dpg_launch_count() == before
