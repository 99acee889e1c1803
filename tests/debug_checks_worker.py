"""Run by tests/test_gpu_debug_checks.py in a process of its own, with
DPG_LIBRARY=debug (the index-checking library) and DPG_TEST_HOOKS=1.

* Parity cases (ragged lists, the accumulation path, the 10,000-tensor list,
  pack/unpack) give the oracle's results and record no failed check.
* With the check bound lowered below the plan's total, the fused pass's
  chunks of the last bucket and the pack items fail their checks: each
  records its kernel code, and the accesses they guard are skipped (those
  elements keep their old values), with no fault; with the bound restored, a
  step records nothing.
Prints "debug checks ok" at the end.
"""
import os
import sys

import numpy as np
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
sys.path.insert(0, os.path.join(ROOT, "tests"))

import zero_optimizer_step_gb300 as dpg                          # noqa: E402
from parity_util import StepCase, assert_parity, run_case        # noqa: E402
from workloads import (CONFIGS, KIND_GRAD, KIND_MASTER, flat_grads_bf16, master_f32,  # noqa: E402
                       random_param_list, segments, stream_seed)

assert dpg.LIB_PATH.endswith("libdpg_debug.so"), dpg.LIB_PATH


def clean(plan):
    built, first = dpg.dpg_debug_checks(plan)
    assert built, "the loaded library has no index checks"
    assert first == 0, f"a check failed: code {first >> 32}, CTA {first & 0xFFFFFFFF}"


rng = np.random.Generator(np.random.Philox(5))
cases = [StepCase(numels=random_param_list(rng, 40, 200_000), cap_bytes=1 << 19, R=4, seed=11),
         StepCase(numels=random_param_list(rng, 30, 100_000), cap_bytes=1 << 18, R=2, K=3,
                  seed=12),
         StepCase(numels=CONFIGS["sweep"].numels, cap_bytes=4096, R=8, seed=13, b_split=700)]
for c in cases:
    res = run_case(c)
    assert_parity(res)
    clean(res.plan)

# pack / unpack of many parameters
numels = random_param_list(rng, 300, 70_000)
plan = dpg.dpg_plan_buckets(numels, 1 << 20, 2)
params = [torch.randn(int(n), device="cuda").to(torch.bfloat16) for n in numels]
flat = torch.empty(plan.total_padded, dtype=torch.bfloat16, device="cuda")
dpg.dpg_pack(plan, params, flat)
back = [torch.empty_like(p) for p in params]
dpg.dpg_unpack(plan, flat, back)
torch.cuda.synchronize()
assert all(torch.equal(a.view(torch.int16), b.view(torch.int16)) for a, b in zip(params, back))
clean(plan)

# a check made to fail: the bound lowered by one vector below the plan's
# total, so every chunk of the last bucket (whose end is past the bound)
# fails its check and is skipped, and the other buckets are updated
numels = [5000, 3000]
plan = dpg.dpg_plan_buckets(numels, 8000, 2)
N = plan.total_padded
assert plan.n_buckets == 2
last = int(plan.bucket_offset[-1])
segs = segments(plan.param_offset, numels)
g = [flat_grads_bf16(segs, N, 1e-3, stream_seed(17, KIND_GRAD, r), device="cuda") for r in range(2)]
w0 = master_f32(N, stream_seed(17, KIND_MASTER), device="cuda")
w, m, v = w0.clone(), torch.zeros(N, device="cuda"), torch.zeros(N, device="cuda")
p = torch.empty(N, dtype=torch.bfloat16, device="cuda")
sq = torch.empty(plan.n_buckets, device="cuda")
dpg.dpg_debug_set_limit(N - 8)
try:
    dpg.dpg_step(plan, g, [100, 200], dpg.HParams(), w, m, v, [p], bucket_sqnorm=sq)
    torch.cuda.synchronize()
finally:
    dpg.dpg_debug_set_limit(-1)
built, first = dpg.dpg_debug_checks(plan)
assert built and first >> 32 == 1, hex(first)
assert torch.equal(w[last:].view(torch.int32), w0[last:].view(torch.int32)), "skipped access ran"
assert not torch.equal(w[:last].view(torch.int32), w0[:last].view(torch.int32))
dpg.dpg_step(plan, g, [100, 200], dpg.HParams(step=2), w, m, v, [p], bucket_sqnorm=sq)
clean(plan)

# a pack item made to fail its check
params = [torch.randn(n, device="cuda").to(torch.bfloat16) for n in numels]
flat = torch.zeros(N, dtype=torch.bfloat16, device="cuda")
dpg.dpg_debug_set_limit(8)
try:
    dpg.dpg_pack(plan, params, flat)
    torch.cuda.synchronize()
finally:
    dpg.dpg_debug_set_limit(-1)
built, first = dpg.dpg_debug_checks(plan)
assert first >> 32 == 4, hex(first)
assert not flat.view(torch.int16).any(), "a refused item was copied"
print("debug checks ok")
