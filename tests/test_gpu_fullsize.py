"""Full-size parity: the benchmark's workloads at their real sizes, run exactly
as the benchmark runs them (one dpg_step over every bucket, accumulation
microbatches through dpg_accumulate), checked against the oracle on samples
it can compute one by one:
  * whole buckets (first, last, two seeded random ones): every element of
    master/m/v/param plus the bucket's squared norm;
  * a contiguous window of the largest bucket;
  * 200,000 seeded random elements anywhere in the flat buffer.
Inputs are drawn on the GPU by torch's seeded generator; the oracle gets host
copies of the sampled slices taken before the step.
"""
import numpy as np
import pytest
import torch

import oracle
import zero_optimizer_step_gb300 as dpg
from parity_util import BF16_ULP, F32_ULP, check_norms, np_bf16, np_f32, ulp_bf16, ulp_f32
from workloads import (CONFIGS, KIND_GRAD, KIND_MASTER, flat_grads_bf16, master_f32, segments,
                       stream_seed, token_counts)

pytestmark = pytest.mark.gpu

WINDOW = 1 << 22
N_RANDOM = 200_000


@pytest.fixture(scope="module", autouse=True)
def built():
    from zero_optimizer_step_gb300 import build
    build.build()
    oracle.build()


def _gather(t: torch.Tensor, sel) -> torch.Tensor:
    return torch.cat([t[a:b] for a, b in sel["ranges"]] + [t[sel["idx"]]]).cpu()


@pytest.mark.parametrize("name", ["gpt2", "llama1b", "llama8b16l"])
def test_fullsize_sampled(name):
    cfg = CONFIGS[name]
    plan = dpg.dpg_plan_buckets(cfg.numels, cfg.cap_bytes, cfg.R)
    oplan = oracle.plan_buckets(cfg.numels, cfg.cap_bytes, cfg.R)
    np.testing.assert_array_equal(oplan.param_offset, plan.param_offset)
    np.testing.assert_array_equal(oplan.bucket_padded, plan.bucket_padded)
    N, R, K = oplan.total_padded, cfg.R, cfg.K
    segs = segments(oplan.param_offset, cfg.numels)
    rng = np.random.Generator(np.random.Philox(cfg.seed))
    largest = int(np.argmax(oplan.bucket_padded))
    whole = sorted({0, oplan.n_buckets - 1,
                    *[int(b) for b in rng.choice(oplan.n_buckets, 2, replace=False)]} - {largest})
    ranges = [(int(oplan.bucket_offset[b]), int(oplan.bucket_offset[b] + oplan.bucket_padded[b]))
              for b in whole]
    lo = int(oplan.bucket_offset[largest] + rng.integers(0, max(1, oplan.bucket_padded[largest] - WINDOW)))
    ranges.append((lo, min(lo + WINDOW, int(oplan.bucket_offset[largest] + oplan.bucket_padded[largest]))))
    idx = torch.from_numpy(np.sort(rng.integers(0, N, N_RANDOM)).astype(np.int64)).cuda()
    sel = dict(ranges=ranges, idx=idx)

    dev = "cuda"
    tokens = token_counts(cfg)
    w = master_f32(N, stream_seed(cfg.seed, KIND_MASTER), device=dev)
    m = torch.zeros(N, device=dev)
    v = torch.zeros(N, device=dev)
    param = torch.empty(N, dtype=torch.bfloat16, device=dev)
    sq = torch.empty(oplan.n_buckets, device=dev)
    nf = torch.empty(oplan.n_buckets, dtype=torch.int64, device=dev)
    h_w0, h_m0, h_v0 = _gather(w, sel).numpy(), _gather(m, sel).numpy(), _gather(v, sel).numpy()
    h_micro = [[None] * K for _ in range(R)]
    acc = [torch.empty(N, device=dev) for _ in range(R)] if K > 1 else None
    g = [None] * R
    for k in range(K):
        for r in range(R):
            g[r] = None
            g[r] = flat_grads_bf16(segs, N, cfg.grad_std, stream_seed(cfg.seed, KIND_GRAD, r, k),
                                   device=dev)
            h_micro[r][k] = np_bf16(_gather(g[r], sel))
            if k < K - 1:
                dpg.dpg_accumulate(plan, g[r], acc[r], first=(k == 0))
    hp = dpg.HParams(step=1)
    if K > 1:
        dpg.dpg_step(plan, acc, tokens, hp, w, m, v, [param], last_micro=g, bucket_sqnorm=sq,
                     bucket_nonfinite=nf)
    else:
        dpg.dpg_step(plan, g, tokens, hp, w, m, v, [param], bucket_sqnorm=sq, bucket_nonfinite=nf)
    torch.cuda.synchronize()
    got = dict(w=_gather(w, sel).numpy(), m=_gather(m, sel).numpy(), v=_gather(v, sel).numpy(),
               p=np_bf16(_gather(param, sel)))
    del g, acc

    # oracle on the gathered elements (the update is elementwise)
    hw, hm, hv = h_w0.copy(), h_m0.copy(), h_v0.copy()
    if K > 1:
        accs = [np.empty(hw.size, np.float32) for _ in range(R)]
        for k in range(K - 1):
            for r in range(R):
                oracle.accumulate(h_micro[r][k], accs[r], first=(k == 0))
        gr = oracle.reduce(accs, oracle.grad_scale(tokens), last=[h_micro[r][K - 1] for r in range(R)])
    else:
        gr = oracle.reduce([h_micro[r][0] for r in range(R)], oracle.grad_scale(tokens))
    oracle.adam(gr, hw, hm, hv, t=1)
    assert ulp_f32(got["w"], hw) <= F32_ULP
    assert ulp_f32(got["m"], hm) <= F32_ULP
    assert ulp_f32(got["v"], hv) <= F32_ULP
    assert ulp_bf16(got["p"], oracle.f32_to_bf16(hw)) <= BF16_ULP
    # whole sampled buckets: their squared norms
    gsq = sq.cpu().numpy()
    pos = 0
    for b, (a, e) in zip(whole, ranges):
        ref = float(np.sum(gr[pos:pos + (e - a)].astype(np.float64) ** 2))
        check_norms(gsq[b:b + 1], np.array([ref]))
        pos += e - a
    assert nf.sum().item() == 0


def test_fullsize_deferred_llama8b16l():
    """The deferred schedule the benchmark also times on the 4.5B list: every
    replica's K = 4 bf16 microbatches held at once (16 buffers of 4.5B
    elements) and summed inside one dpg_step_deferred pass; sampled outputs
    against the oracle's one-microbatch-at-a-time accumulation path."""
    torch.cuda.empty_cache()         # the other full-size cases' cached blocks
    cfg = CONFIGS["llama8b16l"]
    plan = dpg.dpg_plan_buckets(cfg.numels, cfg.cap_bytes, cfg.R)
    N, R, K = plan.total_padded, cfg.R, cfg.K
    segs = segments(plan.param_offset, cfg.numels)
    rng = np.random.Generator(np.random.Philox(cfg.seed + 7))
    b = int(rng.integers(0, plan.n_buckets))
    ranges = [(int(plan.bucket_offset[b]), int(plan.bucket_offset[b] + plan.bucket_padded[b]))]
    idx = torch.from_numpy(np.sort(rng.integers(0, N, N_RANDOM)).astype(np.int64)).cuda()
    sel = dict(ranges=ranges, idx=idx)
    dev = "cuda"
    tokens = token_counts(cfg)
    w = master_f32(N, stream_seed(cfg.seed, KIND_MASTER), device=dev)
    m, v = torch.zeros(N, device=dev), torch.zeros(N, device=dev)
    param = torch.empty(N, dtype=torch.bfloat16, device=dev)
    sq = torch.empty(plan.n_buckets, device=dev)
    h_w0 = _gather(w, sel).numpy()
    gd = [[flat_grads_bf16(segs, N, cfg.grad_std, stream_seed(cfg.seed, KIND_GRAD, r, k), device=dev)
           for k in range(K)] for r in range(R)]
    h_micro = [[np_bf16(_gather(gd[r][k], sel)) for k in range(K)] for r in range(R)]
    dpg.dpg_step_deferred(plan, gd, tokens, dpg.HParams(step=1), w, m, v, [param], bucket_sqnorm=sq)
    torch.cuda.synchronize()
    got = dict(w=_gather(w, sel).numpy(), m=_gather(m, sel).numpy(), v=_gather(v, sel).numpy(),
               p=np_bf16(_gather(param, sel)))
    del gd
    torch.cuda.empty_cache()

    hw = h_w0.copy()
    hm, hv = np.zeros_like(hw), np.zeros_like(hw)
    accs = [np.empty(hw.size, np.float32) for _ in range(R)]
    for k in range(K - 1):
        for r in range(R):
            oracle.accumulate(h_micro[r][k], accs[r], first=(k == 0))
    gr = oracle.reduce(accs, oracle.grad_scale(tokens), last=[h_micro[r][K - 1] for r in range(R)])
    oracle.adam(gr, hw, hm, hv, t=1)
    for name, ref in (("w", hw), ("m", hm), ("v", hv)):
        assert ulp_f32(got[name], ref) == 0, name
    assert ulp_bf16(got["p"], oracle.f32_to_bf16(hw)) == 0
    e = ranges[0][1] - ranges[0][0]
    check_norms(sq.cpu().numpy()[b:b + 1], np.array([float(np.sum(gr[:e].astype(np.float64) ** 2))]))
