"""The step inside a CUDA graph.

After dpg_plan_upload, the entry points issue only kernel launches on the
caller's stream (no allocation, no synchronisation), so a whole step can be
captured once and replayed.  A replay must equal the eager call bit for bit.
The hyper-parameters (and with them the step t) are fixed at capture, as for
any captured launch argument.
"""
import numpy as np
import pytest
import torch

import zero_optimizer_step_gb300 as dpg
from workloads import (KIND_GRAD, KIND_MASTER, flat_grads_bf16, master_f32, random_param_list,
                       segments, stream_seed)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    from zero_optimizer_step_gb300 import build
    build.build()


def _setup(R=4, seed=61):
    numels = random_param_list(np.random.Generator(np.random.Philox(seed)), 40, 100_000)
    plan = dpg.dpg_plan_buckets(numels, 1 << 18, R)
    dpg.dpg_plan_upload(plan)
    N = plan.total_padded
    segs = segments(plan.param_offset, numels)
    g = [flat_grads_bf16(segs, N, 1e-3, stream_seed(seed, KIND_GRAD, r), device="cuda")
         for r in range(R)]
    w0 = master_f32(N, stream_seed(seed, KIND_MASTER), device="cuda")
    tok = [3000 + r for r in range(R)]
    return plan, g, w0, tok


def _buffers(plan, w0):
    N, nb = plan.total_padded, plan.n_buckets
    return dict(w=w0.clone(), m=torch.zeros(N, device="cuda"), v=torch.zeros(N, device="cuda"),
                p=torch.empty(N, dtype=torch.bfloat16, device="cuda"),
                sq=torch.empty(nb, device="cuda"),
                nf=torch.empty(nb, dtype=torch.int64, device="cuda"))


def _same(a, b):
    for k in a:
        assert torch.equal(a[k].view(torch.uint8), b[k].view(torch.uint8)), k


def test_captured_step_equals_eager_step():
    plan, g, w0, tok = _setup()
    hp = dpg.HParams(step=1)
    eager, graph = _buffers(plan, w0), _buffers(plan, w0)
    # warm the library's per-kernel launch-geometry cache outside the capture
    scratch = _buffers(plan, w0)
    dpg.dpg_step(plan, g, tok, hp, scratch["w"], scratch["m"], scratch["v"], [scratch["p"]],
                 bucket_sqnorm=scratch["sq"], bucket_nonfinite=scratch["nf"])
    torch.cuda.synchronize()

    s = torch.cuda.Stream()
    gr = torch.cuda.CUDAGraph()
    with torch.cuda.graph(gr, stream=s):
        dpg.dpg_step(plan, g, tok, hp, graph["w"], graph["m"], graph["v"], [graph["p"]],
                     bucket_sqnorm=graph["sq"], bucket_nonfinite=graph["nf"],
                     stream=torch.cuda.current_stream())
    gr.replay()
    dpg.dpg_step(plan, g, tok, hp, eager["w"], eager["m"], eager["v"], [eager["p"]],
                 bucket_sqnorm=eager["sq"], bucket_nonfinite=eager["nf"])
    torch.cuda.synchronize()
    _same(eager, graph)


def test_captured_accumulation_cycle_replays():
    """Two replays of a captured K = 3 cycle (accumulate, accumulate, fused
    step with the last microbatch) equal two eager cycles with the same
    hyper-parameters."""
    plan, g, w0, tok = _setup(R=2, seed=62)
    N = plan.total_padded
    hp = dpg.HParams(step=1)
    tok3 = tok * 3

    def cycle(buf, acc):
        for r in range(2):
            dpg.dpg_accumulate(plan, g[r], acc[r], first=True, stream=torch.cuda.current_stream())
            dpg.dpg_accumulate(plan, g[r], acc[r], first=False, stream=torch.cuda.current_stream())
        dpg.dpg_step(plan, acc, tok3, hp, buf["w"], buf["m"], buf["v"], [buf["p"]], last_micro=g,
                     bucket_sqnorm=buf["sq"], bucket_nonfinite=buf["nf"],
                     stream=torch.cuda.current_stream())

    eager, graph = _buffers(plan, w0), _buffers(plan, w0)
    acc_e = [torch.empty(N, device="cuda") for _ in range(2)]
    acc_g = [torch.empty(N, device="cuda") for _ in range(2)]
    cycle(_buffers(plan, w0), [torch.empty(N, device="cuda") for _ in range(2)])   # warm-up
    torch.cuda.synchronize()
    s = torch.cuda.Stream()
    gr = torch.cuda.CUDAGraph()
    with torch.cuda.graph(gr, stream=s):
        cycle(graph, acc_g)
    for _ in range(2):
        # poison the norm outputs: each replay must write them again (the
        # finalize's per-bucket arrival counters are back at zero after every
        # launch, replayed or not)
        for buf in (graph, eager):
            buf["sq"].fill_(float("nan"))
            buf["nf"].fill_(-1)
        gr.replay()
        cycle(eager, acc_e)
        torch.cuda.synchronize()
        assert torch.isfinite(graph["sq"]).all() and (graph["nf"] >= 0).all()
    _same(eager, graph)
