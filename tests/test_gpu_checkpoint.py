"""Checkpoint, resume and resharding of the optimizer state on the GPU
("Distributed Training and Parallelism", Reproduction and debugging:
checkpoint ownership, resumability, mesh reconfiguration).

* dpg_export_state / dpg_import_state equal the oracle's canonical layout
  bit for bit (import zeroes padding);
* resume: export after step t, import into fresh buffers, step t+1 -- equal
  bit for bit to running step t+1 without the checkpoint;
* reshard to another bucket cap (same R): the canonical state after the next
  step is bit-identical to the unresharded run (Adam is elementwise and each
  element's rank-ordered sum is unchanged);
* reshard to another R (mesh reconfiguration, 4 -> 8 replicas): the next
  step on the new layout matches the oracle run on the oracle's own layout.
"""
import numpy as np
import pytest
import torch

import oracle
import zero_optimizer_step_gb300 as dpg
from parity_util import np_bf16, np_f32, ulp_f32
from workloads import random_param_list

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    from zero_optimizer_step_gb300 import build
    build.build()
    oracle.build()


def _numels(seed, n=40, mx=120_000):
    return random_param_list(np.random.Generator(np.random.Philox(seed)), n, mx)


def _param_grads(numels, R, seed, std=1e-3):
    g = torch.Generator().manual_seed(seed)
    return [[(torch.randn(int(n), generator=g) * std).to(torch.bfloat16) for n in numels]
            for _ in range(R)]


def _flats(plan, per_param):
    out = []
    for grads in per_param:
        f = torch.empty(plan.total_padded, dtype=torch.bfloat16, device="cuda")
        dpg.dpg_pack(plan, [x.cuda() for x in grads], f)
        out.append(f)
    return out


@pytest.mark.parametrize("seed", range(3))
def test_export_import_match_oracle(seed):
    numels = _numels(50 + seed)
    numels[0] = 3 * 32768 + 3            # a parameter spanning several items
    rng = np.random.Generator(np.random.Philox(seed))
    cap, R = int(rng.integers(1000, 1 << 20)), int(rng.choice([1, 2, 4, 8]))
    plan = dpg.dpg_plan_buckets(numels, cap, R)
    oplan = oracle.plan_buckets(numels, cap, R)
    flats = [torch.randn(plan.total_padded, generator=torch.Generator().manual_seed(k)).cuda()
             for k in range(3)]
    canon = [torch.full((plan.canon_total,), float("nan"), device="cuda") for _ in range(3)]
    dpg.dpg_export_state(plan, flats, canon)
    back = [torch.full((plan.total_padded,), float("nan"), device="cuda") for _ in range(3)]
    dpg.dpg_import_state(plan, canon, back)
    torch.cuda.synchronize()
    for f, c, b in zip(flats, canon, back):
        ref_c = oracle.export_state(oplan, np_f32(f))
        np.testing.assert_array_equal(np_f32(c).view(np.uint32), ref_c.view(np.uint32))
        ref_b = oracle.import_state(oplan, ref_c)
        np.testing.assert_array_equal(np_f32(b).view(np.uint32), ref_b.view(np.uint32))


def _run_steps(plan, per_param_steps, tokens, state, t0):
    for k, per_param in enumerate(per_param_steps):
        view = torch.empty(plan.total_padded, dtype=torch.bfloat16, device="cuda")
        dpg.dpg_step(plan, _flats(plan, per_param), tokens, dpg.HParams(step=t0 + k), *state, [view])
    return state


def _state(plan, seed):
    w = torch.randn(plan.canon_total, generator=torch.Generator().manual_seed(seed)) * 0.02
    canon = [w.cuda(), torch.zeros(plan.canon_total, device="cuda"),
             torch.zeros(plan.canon_total, device="cuda")]
    flat = [torch.empty(plan.total_padded, device="cuda") for _ in range(3)]
    dpg.dpg_import_state(plan, canon, flat)
    return flat


def _export(plan, flat):
    canon = [torch.empty(plan.canon_total, device="cuda") for _ in range(3)]
    dpg.dpg_export_state(plan, flat, canon)
    torch.cuda.synchronize()
    return [np_f32(c) for c in canon]


def test_resume_is_bit_identical():
    numels = _numels(60)
    R, tok = 4, [3100, 2900, 4000, 3500]
    plan = dpg.dpg_plan_buckets(numels, 1 << 19, R)
    steps = [_param_grads(numels, R, 100 + t) for t in range(2)]
    straight = _run_steps(plan, steps, tok, _state(plan, 1), 1)       # steps 1, 2
    first = _run_steps(plan, steps[:1], tok, _state(plan, 1), 1)        # step 1
    ckpt = _export(plan, first)
    fresh = [torch.full((plan.total_padded,), float("nan"), device="cuda") for _ in range(3)]
    dpg.dpg_import_state(plan, [torch.from_numpy(c).cuda() for c in ckpt], fresh)
    resumed = _run_steps(plan, steps[1:], tok, fresh, 2)                # step 2
    for a, b in zip(_export(plan, straight), _export(plan, resumed)):
        np.testing.assert_array_equal(a.view(np.uint32), b.view(np.uint32))


def test_reshard_to_another_cap_is_bit_identical():
    numels = _numels(61)
    R, tok = 4, [3000, 3001, 3002, 3003]
    pa = dpg.dpg_plan_buckets(numels, 1 << 20, R)
    pb = dpg.dpg_plan_buckets(numels, 3000, R)       # many small buckets
    assert pb.n_buckets > pa.n_buckets
    steps = [_param_grads(numels, R, 200 + t) for t in range(2)]
    a = _run_steps(pa, steps, tok, _state(pa, 2), 1)
    a1 = _run_steps(pa, steps[:1], tok, _state(pa, 2), 1)
    ckpt = _export(pa, a1)
    fb = [torch.empty(pb.total_padded, device="cuda") for _ in range(3)]
    dpg.dpg_import_state(pb, [torch.from_numpy(c).cuda() for c in ckpt], fb)
    b = _run_steps(pb, steps[1:], tok, fb, 2)
    for x, y in zip(_export(pa, a), _export(pb, b)):
        np.testing.assert_array_equal(x.view(np.uint32), y.view(np.uint32))


def test_reshard_to_more_replicas_matches_oracle():
    numels = _numels(62)
    pa = dpg.dpg_plan_buckets(numels, 1 << 19, 4)
    pc = dpg.dpg_plan_buckets(numels, 1 << 18, 8)
    oc = oracle.plan_buckets(numels, 1 << 18, 8)
    a1 = _run_steps(pa, [_param_grads(numels, 4, 300)], [3000] * 4, _state(pa, 3), 1)
    ckpt = _export(pa, a1)
    fc = [torch.empty(pc.total_padded, device="cuda") for _ in range(3)]
    dpg.dpg_import_state(pc, [torch.from_numpy(c).cuda() for c in ckpt], fc)
    grads8 = _param_grads(numels, 8, 301)
    tok8 = [3000 + 10 * r for r in range(8)]
    _run_steps(pc, [grads8], tok8, fc, 2)
    got = _export(pc, fc)
    # oracle: import the same canonical state into its own layout and step
    w, m, v = (oracle.import_state(oc, c) for c in ckpt)
    hflats = [oracle.pack(oc, [np_bf16(x) for x in grads8[r]]) for r in range(8)]
    oracle.step(oc.bucket_offset, oc.bucket_padded, hflats, tok8, w, m, v, t=2)
    for g_, r_ in zip(got, (w, m, v)):
        assert ulp_f32(g_, oracle.export_state(oc, r_)) == 0
