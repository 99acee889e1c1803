"""Launch shape and launch mode do not change results.

By default the fused passes launch one small CTA per 1024-element chunk; a
grid cap (dpg_set_fused_max_ctas) switches every one of them to the
persistent grid-stride kernels.  For each entry point and input mode, the
capped run must give the same bits as the default run (the chunked runs are
checked against the oracle elsewhere), and per-bucket norms within their
relative 1e-5 bar.

By default the chunked and streaming kernels are launched with programmatic
stream serialization (each waits on the device for its predecessor before
touching memory); chains of launches where every kernel reads what the one
just before it wrote must give the same bits with it switched off.
"""
import numpy as np
import pytest
import torch

import zero_optimizer_step_gb300 as dpg
from parity_util import np_f32
from workloads import (KIND_GRAD, KIND_MASTER, flat_grads_bf16, flat_values_f32, master_f32,
                       random_param_list, segments, stream_seed)

pytestmark = pytest.mark.gpu

NORM_RTOL = 1e-5


@pytest.fixture(scope="module", autouse=True)
def built():
    from zero_optimizer_step_gb300 import build
    build.build()


@pytest.fixture
def setup():
    R = 4
    numels = random_param_list(np.random.Generator(np.random.Philox(91)), 40, 120_000)
    plan = dpg.dpg_plan_buckets(numels, 1 << 18, R)
    N = plan.total_padded
    segs = segments(plan.param_offset, numels)
    bf = [flat_grads_bf16(segs, N, 1e-3, stream_seed(91, KIND_GRAD, r), device="cuda")
          for r in range(R)]
    bf2 = [flat_grads_bf16(segs, N, 1e-3, stream_seed(92, KIND_GRAD, r), device="cuda")
           for r in range(R)]
    f32 = [flat_values_f32(segs, N, 1e-3, stream_seed(93, KIND_GRAD, r), device="cuda")
           for r in range(R)]
    w0 = master_f32(N, stream_seed(91, KIND_MASTER), device="cuda")
    tok = [2500 + 7 * r for r in range(R)]
    return plan, bf, bf2, f32, w0, tok


def _state(plan, w0):
    N = plan.total_padded
    return dict(w=w0.clone(), m=torch.zeros(N, device="cuda"), v=torch.zeros(N, device="cuda"),
                p=torch.empty(N, dtype=torch.bfloat16, device="cuda"),
                sq=torch.empty(plan.n_buckets, device="cuda"),
                nf=torch.empty(plan.n_buckets, dtype=torch.int64, device="cuda"),
                red=torch.empty(N, device="cuda"))


def _run_both(fn, cap):
    outs = []
    for c in (0, cap):
        dpg.dpg_set_fused_max_ctas(c)
        try:
            outs.append(fn())
        finally:
            dpg.dpg_set_fused_max_ctas(0)
        torch.cuda.synchronize()
    return outs


def _same(a, b, keys):
    for k in keys:
        assert torch.equal(a[k].view(torch.uint8), b[k].view(torch.uint8)), k


def _norms_close(a, b):
    sa, sb = np_f32(a["sq"]).astype(np.float64), np_f32(b["sq"]).astype(np.float64)
    assert np.all(np.abs(sa - sb) <= NORM_RTOL * np.abs(sb))
    assert torch.equal(a["nf"], b["nf"])


@pytest.mark.parametrize("cap", [1, 37])
@pytest.mark.parametrize("mode", ["bf16", "f32", "acc", "fold2"])
def test_step_modes_same_bits_under_a_grid_cap(setup, cap, mode):
    plan, bf, bf2, f32, w0, tok = setup

    def run():
        s = _state(plan, w0)
        kw = dict(bucket_sqnorm=s["sq"], bucket_nonfinite=s["nf"])
        if mode == "bf16":
            dpg.dpg_reduce_scatter_adam(plan, bf, tok, dpg.HParams(step=2), s["w"], s["m"], s["v"],
                                        [s["p"]], reduced_grad=s["red"], **kw)
        elif mode == "f32":
            dpg.dpg_step(plan, f32, tok, dpg.HParams(), s["w"], s["m"], s["v"], [s["p"]], **kw)
        elif mode == "acc":
            dpg.dpg_step(plan, f32, tok * 2, dpg.HParams(), s["w"], s["m"], s["v"], [s["p"]],
                         last_micro=bf, **kw)
        else:
            dpg.dpg_step_fold2(plan, f32, bf, bf2, tok * 3, dpg.HParams(), s["w"], s["m"], s["v"],
                               [s["p"]], **kw)
        return s

    a, b = _run_both(run, cap)
    _same(a, b, ("w", "m", "v", "p") + (("red",) if mode == "bf16" else ()))
    _norms_close(a, b)


@pytest.mark.parametrize("cap", [1, 37])
def test_ddp_pieces_same_bits_under_a_grid_cap(setup, cap):
    plan, bf, _, _, w0, tok = setup

    def run():
        s = _state(plan, w0)
        dpg.dpg_allreduce_grads(plan, bf, tok, s["red"], bucket_sqnorm=s["sq"],
                                bucket_nonfinite=s["nf"])
        dpg.dpg_adam_from_reduced(plan, s["red"], dpg.HParams(), s["w"], s["m"], s["v"], [s["p"]])
        return s

    a, b = _run_both(run, cap)
    _same(a, b, ("red", "w", "m", "v", "p"))
    _norms_close(a, b)


def _run_launch_modes(fn):
    outs = []
    for on in (False, True):
        dpg.dpg_set_programmatic_launch(on)
        try:
            outs.append(fn())
        finally:
            dpg.dpg_set_programmatic_launch(True)
        torch.cuda.synchronize()
    return outs


@pytest.mark.parametrize("chain", ["accumulate", "per_bucket", "clipped", "gathers"])
def test_programmatic_launch_same_bits(setup, chain):
    plan, bf, bf2, f32, w0, tok = setup
    N, R = plan.total_padded, len(bf)

    def run():
        s = _state(plan, w0)
        if chain == "accumulate":
            # acc <- g0, += g1, += (g2 + g3), then the fused step reads acc at once
            accs = [torch.empty(N, device="cuda") for _ in range(R)]
            for r in range(R):
                dpg.dpg_accumulate(plan, bf[r], accs[r], True)
                dpg.dpg_accumulate(plan, bf2[r], accs[r], False)
                dpg.dpg_accumulate_pair(plan, bf[r], bf2[r], accs[r], False)
            dpg.dpg_step(plan, accs, tok * 5, dpg.HParams(), s["w"], s["m"], s["v"], [s["p"]],
                         last_micro=bf2, bucket_sqnorm=s["sq"], bucket_nonfinite=s["nf"])
            s["red"] = accs[R - 1]
        elif chain == "per_bucket":
            # two steps, one launch per bucket; step 2 reads the state step 1 wrote
            for t in (1, 2):
                for b in range(plan.n_buckets):
                    dpg.dpg_reduce_scatter_adam(plan, bf, tok, dpg.HParams(step=t), s["w"], s["m"],
                                                s["v"], [s["p"]], b0=b, b1=b + 1)
            dpg.dpg_step(plan, bf2, tok, dpg.HParams(step=3), s["w"], s["m"], s["v"], [s["p"]],
                         bucket_sqnorm=s["sq"], bucket_nonfinite=s["nf"])
        elif chain == "clipped":
            # norm pass -> finalize -> coefficient -> update, twice
            for t in (1, 2):
                dpg.dpg_step_clipped(plan, bf, tok, dpg.HParams(step=t), 1e-4, s["w"], s["m"],
                                     s["v"], [s["p"]], bucket_sqnorm=s["sq"],
                                     bucket_nonfinite=s["nf"], reduced_grad=s["red"])
        else:
            # the step writes the shards; each gather reads them right after
            views = [torch.zeros(N, dtype=torch.bfloat16, device="cuda") for _ in range(2)]
            dpg.dpg_step(plan, bf, tok, dpg.HParams(), s["w"], s["m"], s["v"], [s["p"]],
                         bucket_sqnorm=s["sq"], bucket_nonfinite=s["nf"])
            for b in range(plan.n_buckets):
                dpg.dpg_gather_params_bf16(plan, s["p"], views, b0=b, b1=b + 1)
            dpg.dpg_allgather_params(plan, s["w"], [s["p"]])
            s["g0"], s["g1"] = views
        return s

    a, b = _run_launch_modes(run)
    keys = ("w", "m", "v", "p", "sq", "nf") + (("red",) if chain in ("accumulate", "clipped") else ())
    keys += ("g0", "g1") if chain == "gathers" else ()
    _same(a, b, keys)
