"""Per-bucket updates overlapped with a producer, as a backward pass would feed
them ("Parallelisms" -- Gradient bucketing: a bucket is reduced as soon as
its gradients are ready).

A producer stream writes each bucket's replica gradients in backward-ready
order (bucket 0 first), each after a GPU spin, and records an event; an
update stream waits on each event and launches that bucket's fused update
(programmatic launches on, the default), either through the library's
event-gated entry (dpg_reduce_scatter_adam_when_ready) or bucket by bucket
from Python.  The result -- master, moments,
parameters, reduced gradient and per-bucket norms -- must be the bits of one
whole-plan launch on the finished gradients: a kernel of the update stream
never reads a bucket before its event, whatever the launch mode.  It is also
compared with the CPU oracle's step on the same gradients: 0 ulp for master,
moments and parameters, the reduced gradient bit for bit, norms within 1e-5.
"""
import numpy as np
import pytest
import torch

import oracle
import zero_optimizer_step_gb300 as dpg
from parity_util import check_norms, np_bf16, np_f32, ulp_bf16, ulp_f32
from workloads import (KIND_GRAD, KIND_MASTER, flat_grads_bf16, master_f32, random_param_list,
                       segments, stream_seed)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    from zero_optimizer_step_gb300 import build
    build.build()


def _state(N, w0, nb):
    return dict(w=w0.clone(), m=torch.zeros(N, device="cuda"), v=torch.zeros(N, device="cuda"),
                p=torch.empty(N, dtype=torch.bfloat16, device="cuda"),
                red=torch.full((N,), float("nan"), device="cuda"),
                sq=torch.full((nb,), float("nan"), device="cuda"),
                nf=torch.full((nb,), -1, dtype=torch.int64, device="cuda"))


@pytest.mark.parametrize("native", [True, False])
@pytest.mark.parametrize("programmatic", [True, False])
def test_event_gated_bucket_updates_equal_one_step(programmatic, native):
    R = 4
    numels = random_param_list(np.random.Generator(np.random.Philox(77)), 60, 400_000)
    plan = dpg.dpg_plan_buckets(numels, 1 << 20, R)
    N, nb = plan.total_padded, plan.n_buckets
    assert nb >= 6
    segs = segments(plan.param_offset, numels)
    src = [flat_grads_bf16(segs, N, 1e-3, stream_seed(77, KIND_GRAD, r), device="cuda")
           for r in range(R)]
    w0 = master_f32(N, stream_seed(77, KIND_MASTER), device="cuda")
    tok = [3100, 2900, 4000, 3500]
    hp = dpg.HParams(step=1)

    ref = _state(N, w0, nb)
    dpg.dpg_reduce_scatter_adam(plan, src, tok, hp, ref["w"], ref["m"], ref["v"], [ref["p"]],
                                bucket_sqnorm=ref["sq"], bucket_nonfinite=ref["nf"],
                                reduced_grad=ref["red"])
    torch.cuda.synchronize()

    grads = [torch.full((N,), float("nan"), dtype=torch.bfloat16, device="cuda") for _ in range(R)]
    got = _state(N, w0, nb)
    producer, updater = torch.cuda.Stream(), torch.cuda.Stream()
    events = [torch.cuda.Event() for _ in range(nb)]
    off = [int(x) for x in plan.bucket_offset] + [N]
    torch.cuda.synchronize()
    dpg.dpg_set_programmatic_launch(programmatic)
    try:
        with torch.cuda.stream(producer):
            for b in range(nb):
                torch.cuda._sleep(200_000)            # ~0.1 ms of "backward" per bucket
                for r in range(R):
                    grads[r][off[b]:off[b + 1]].copy_(src[r][off[b]:off[b + 1]])
                events[b].record(producer)
        if native:                                # the library's event-gated entry
            dpg.dpg_reduce_scatter_adam_when_ready(
                plan, grads, tok, hp, got["w"], got["m"], got["v"], [got["p"]],
                ready_events=events, bucket_sqnorm=got["sq"], bucket_nonfinite=got["nf"],
                reduced_grad=got["red"], stream=updater)
        else:                                     # the same schedule from Python
            with torch.cuda.stream(updater):
                for b in range(nb):
                    updater.wait_event(events[b])
                    dpg.dpg_reduce_scatter_adam(plan, grads, tok, hp, got["w"], got["m"],
                                                got["v"], [got["p"]], bucket_sqnorm=got["sq"],
                                                bucket_nonfinite=got["nf"],
                                                reduced_grad=got["red"], b0=b, b1=b + 1,
                                                stream=updater)
        torch.cuda.synchronize()
    finally:
        dpg.dpg_set_programmatic_launch(True)
    for k in ("w", "m", "v", "p", "red", "sq", "nf"):
        assert torch.equal(got[k].view(torch.uint8), ref[k].view(torch.uint8)), k

    # and directly against the oracle, on host copies of the finished gradients
    op = oracle.plan_buckets(numels, 1 << 20, R)
    np.testing.assert_array_equal(op.bucket_offset, plan.bucket_offset)
    w, m, v = np_f32(w0).copy(), np.zeros(N, np.float32), np.zeros(N, np.float32)
    views, red, sq = oracle.step(op.bucket_offset, op.bucket_padded, [np_bf16(g) for g in src],
                                 np.asarray(tok, np.int64), w, m, v, t=1, want_reduced=True)
    assert ulp_f32(np_f32(got["red"]), red) == 0, "reduced gradient not bit-exact"
    for name, ref_arr in (("w", w), ("m", m), ("v", v)):
        assert ulp_f32(np_f32(got[name]), ref_arr) == 0, name
    assert ulp_bf16(np_bf16(got["p"]), views[0]) == 0, "bf16 parameters"
    check_norms(np_f32(got["sq"]), sq)
    assert np.all(got["nf"].cpu().numpy() == 0)
