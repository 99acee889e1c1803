"""The staged (bulk-copy + mbarrier) variant of the fused pass.

* Parity: dpg_step_staged against the oracle on the same inputs, bit-exact
  expected (bars: 2 ulp fp32, 1 ulp bf16, norms 1e-5), for R = 1, 2, 4, 8,
  ragged buckets (partial units, empty second halves of tiles at R = 8),
  several views.
* Failure detection without a GPU fault: a test-only hook makes one CTA's
  unit never be fetched, so its bounded wait (50 ms here) runs out; the
  kernel records DPG_ERR_DEVICE_TIMEOUT, drains its copies in flight and
  returns; dpg_check_device_status reports it, and the next call on the same
  context runs normally and is exact again.
"""
import numpy as np
import pytest
import torch

import oracle
import zero_optimizer_step_gb300 as dpg
from parity_util import (BF16_ULP, F32_ULP, StepCase, check_norms, np_bf16, np_f32, ulp_bf16,
                         ulp_f32)
from workloads import (KIND_GRAD, KIND_MASTER, flat_grads_bf16, master_f32, random_param_list,
                       segments, stream_seed)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    from zero_optimizer_step_gb300 import build
    build.build()
    oracle.build()


def _case(numels, cap, R, seed=5, n_views=1):
    plan = dpg.dpg_plan_buckets(numels, cap, R)
    op = oracle.plan_buckets(numels, cap, R)
    N = op.total_padded
    segs = segments(op.param_offset, numels)
    grads = [flat_grads_bf16(segs, N, 1e-2, stream_seed(seed, KIND_GRAD, r)) for r in range(R)]
    w0 = master_f32(N, stream_seed(seed, KIND_MASTER))
    tok = [3000 + 11 * r for r in range(R)]
    return plan, op, grads, w0, tok


def _device(plan, grads, w0, tok, fn, n_views=1, t=1):
    N = plan.total_padded
    d = [w0.cuda(), torch.zeros(N, device="cuda"), torch.zeros(N, device="cuda")]
    views = [torch.full((N,), float("nan"), dtype=torch.bfloat16, device="cuda")
             for _ in range(n_views)]
    sq = torch.full((max(1, plan.n_buckets),), -1.0, device="cuda")
    nf = torch.full((max(1, plan.n_buckets),), -1, dtype=torch.int64, device="cuda")
    fn(plan, [g.cuda() for g in grads], tok, dpg.HParams(step=t), *d, views, bucket_sqnorm=sq,
       bucket_nonfinite=nf)
    return d, views, sq, nf


def _oracle(op, grads, w0, tok, n_views=1, t=1):
    N = op.total_padded
    w, m, v = np_f32(w0).copy(), np.zeros(N, np.float32), np.zeros(N, np.float32)
    views, red, sq = oracle.step(op.bucket_offset, op.bucket_padded, [np_bf16(g) for g in grads],
                                 tok, w, m, v, n_views=n_views, t=t, want_reduced=True)
    return w, m, v, views, sq, red


def _check(plan, op, grads, w0, tok, n_views=1):
    d, views, sq, nf = _device(plan, grads, w0, tok, dpg.dpg_step_staged, n_views)
    dpg.dpg_check_device_status(plan)
    w, m, v, rviews, rsq, red = _oracle(op, grads, w0, tok, n_views)
    for got, ref in zip(d, (w, m, v)):
        assert ulp_f32(np_f32(got), ref) == 0
    for gv, rv in zip(views, rviews):
        assert ulp_bf16(np_bf16(gv), rv) == 0
    check_norms(np_f32(sq)[: op.n_buckets], rsq)
    nfr = [int(np.sum(~np.isfinite(red[o:o + p]))) for o, p in zip(op.bucket_offset, op.bucket_padded)]
    np.testing.assert_array_equal(nf.cpu().numpy()[: op.n_buckets], nfr)


def test_staged_tiny():
    numels = [64 * 32, 32, 32 * 10]
    _check(*_case(numels, 2048, 4))


@pytest.mark.parametrize("R", [1, 2, 4, 8])
def test_staged_parity_ragged(R):
    rng = np.random.Generator(np.random.Philox(40 + R))
    numels = random_param_list(rng, 60, 150_000)
    _check(*_case(numels, int(rng.integers(3000, 1 << 20)), R, seed=R), n_views=2)


def test_staged_many_small_buckets():
    rng = np.random.Generator(np.random.Philox(77))
    numels = random_param_list(rng, 800, 3000)
    _check(*_case(numels, 1000, 8))


def test_staged_matches_direct_path_on_gpt2_sized_list():
    from workloads import CONFIGS
    cfg = CONFIGS["gpt2"]
    plan = dpg.dpg_plan_buckets(cfg.numels, cfg.cap_bytes, cfg.R)
    N = plan.total_padded
    segs = segments(plan.param_offset, cfg.numels)
    grads = [flat_grads_bf16(segs, N, 1e-3, stream_seed(3, KIND_GRAD, r), device="cuda")
             for r in range(cfg.R)]
    w0 = master_f32(N, stream_seed(3, KIND_MASTER), device="cuda")
    tok = [3500] * cfg.R
    outs = []
    for fn in (dpg.dpg_step, dpg.dpg_step_staged):
        d = [w0.clone(), torch.zeros(N, device="cuda"), torch.zeros(N, device="cuda")]
        p = torch.empty(N, dtype=torch.bfloat16, device="cuda")
        fn(plan, grads, tok, dpg.HParams(), *d, [p])
        outs.append((d, p))
    dpg.dpg_check_device_status(plan)
    torch.cuda.synchronize()
    for a, b in zip(outs[0][0], outs[1][0]):
        assert torch.equal(a.view(torch.int32), b.view(torch.int32))
    assert torch.equal(outs[0][1].view(torch.int16), outs[1][1].view(torch.int16))


def test_staged_wait_times_out_and_context_survives(monkeypatch):
    numels = [40_000, 123_456, 7_777]
    plan, op, grads, w0, tok = _case(numels, 1 << 20, 4)
    before = dpg.dpg_launch_count()
    # the hook is refused unless the process opted in through the environment
    monkeypatch.delenv("DPG_TEST_HOOKS", raising=False)
    with pytest.raises(dpg.DpgError) as e:
        dpg.dpg_set_staged_fault(skip_unit=3, timeout_ns=50_000_000)
    assert e.value.status == dpg.DPG_ERR_INVALID_ARG
    monkeypatch.setenv("DPG_TEST_HOOKS", "1")
    dpg.dpg_set_staged_fault(skip_unit=3, timeout_ns=50_000_000)
    _device(plan, grads, w0, tok, dpg.dpg_step_staged)
    with pytest.raises(dpg.DpgError) as e:
        dpg.dpg_check_device_status(plan)
    assert e.value.status == dpg.DPG_ERR_DEVICE_TIMEOUT
    assert dpg.dpg_launch_count() > before
    # the hook was consumed; the same context runs the next step normally
    _check(plan, op, grads, w0, tok)
