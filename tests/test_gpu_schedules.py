"""DDP (NO_SHARD) against ZeRO-2 on the GPU.

* dpg_allreduce_grads equals the oracle's all-reduce bit for bit (bf16,
  fp32 and fp32 + last-microbatch inputs), and equals the reduce-scatter
  shards of the fused step concatenated -- all-reduce = reduce-scatter then
  all-gather ("Parallelism Starts With the Bottleneck", Allreduce equals
  reducescatter plus allgather);
* dpg_adam_from_reduced equals the oracle's Adam;
* the DDP schedule (all-reduce, then every replica's own optimizer step on
  its full state) leaves every replica bit-identical to the others and to
  the ZeRO-2 step ("Parallelisms", ZeRO-1: the same update, the second
  all-reduce phase repurposed; "Distributed Training and Parallelism":
  matching a single-device update).
"""
import numpy as np
import pytest
import torch

import oracle
import zero_optimizer_step_gb300 as dpg
from parity_util import check_norms, np_bf16, np_f32, ulp_f32
from workloads import (KIND_GRAD, KIND_MASTER, flat_grads_bf16, flat_values_f32, master_f32,
                       random_param_list, segments, stream_seed)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    from zero_optimizer_step_gb300 import build
    build.build()
    oracle.build()


def _setup(R, mode, seed=3):
    numels = random_param_list(np.random.Generator(np.random.Philox(seed)), 40, 100_000)
    plan = dpg.dpg_plan_buckets(numels, 1 << 19, R)
    op = oracle.plan_buckets(numels, 1 << 19, R)
    N = op.total_padded
    segs = segments(op.param_offset, numels)
    if mode == "f32":
        grads = [flat_values_f32(segs, N, 1e-3, stream_seed(seed, KIND_GRAD, r)) for r in range(R)]
        last = None
    else:
        grads = [flat_grads_bf16(segs, N, 1e-3, stream_seed(seed, KIND_GRAD, r)) for r in range(R)]
        last = None
        if mode == "acc":
            last = grads
            grads = [flat_values_f32(segs, N, 1e-3, stream_seed(seed + 1, KIND_GRAD, r))
                     for r in range(R)]
    tok = [3000 + 7 * r for r in range(R)]
    return plan, op, grads, last, tok


def _host(x):
    return np_f32(x) if x.dtype == torch.float32 else np_bf16(x)


@pytest.mark.parametrize("R,mode", [(8, "bf16"), (3, "bf16"), (4, "f32"), (4, "acc")])
def test_allreduce_matches_oracle_and_reduce_scatter(R, mode):
    plan, op, grads, last, tok = _setup(R, mode)
    N = op.total_padded
    dg = [g.cuda() for g in grads]
    dl = None if last is None else [x.cuda() for x in last]
    red = torch.full((N,), float("nan"), device="cuda")
    sq = torch.empty(op.n_buckets, device="cuda")
    dpg.dpg_allreduce_grads(plan, dg, tok, red, last_micro=dl, bucket_sqnorm=sq)
    ref = oracle.allreduce([_host(g) for g in grads], oracle.grad_scale(tok),
                           last=None if last is None else [np_bf16(x) for x in last])[0]
    torch.cuda.synchronize()
    assert ulp_f32(np_f32(red), ref) == 0
    check_norms(np_f32(sq), np.array([np.sum(ref[o:o + p].astype(np.float64) ** 2)
                                      for o, p in zip(op.bucket_offset, op.bucket_padded)]))
    # the fused step's reduce-scatter shards, concatenated, are the same buffer
    rs = torch.full((N,), float("nan"), device="cuda")
    w, m, v = (torch.zeros(N, device="cuda") for _ in range(3))
    dpg.dpg_reduce_scatter_adam(plan, dg, tok, dpg.HParams(), w, m, v, [], last_micro=dl,
                                reduced_grad=rs)
    torch.cuda.synchronize()
    assert torch.equal(rs.view(torch.int32), red.view(torch.int32))


def test_adam_from_reduced_matches_oracle():
    plan, op, grads, _, tok = _setup(4, "bf16", seed=9)
    N = op.total_padded
    g = oracle.allreduce([np_bf16(x) for x in grads], oracle.grad_scale(tok))[0]
    w0 = master_f32(N, stream_seed(9, KIND_MASTER))
    d = [w0.cuda(), torch.zeros(N, device="cuda"), torch.zeros(N, device="cuda")]
    view = torch.empty(N, dtype=torch.bfloat16, device="cuda")
    for t in (1, 2, 3):
        dpg.dpg_adam_from_reduced(plan, torch.from_numpy(g).cuda(), dpg.HParams(step=t), *d, [view])
    hw, hm, hv = np_f32(w0).copy(), np.zeros(N, np.float32), np.zeros(N, np.float32)
    for t in (1, 2, 3):
        oracle.adam(g, hw, hm, hv, t=t)
    torch.cuda.synchronize()
    for got, ref in zip(d, (hw, hm, hv)):
        assert ulp_f32(np_f32(got), ref) == 0
    np.testing.assert_array_equal(np_bf16(view), oracle.f32_to_bf16(hw))


def test_ddp_replicas_equal_zero2_bit_for_bit():
    R = 4
    plan, op, grads, _, tok = _setup(R, "bf16", seed=11)
    N = op.total_padded
    dg = [g.cuda() for g in grads]
    w0 = master_f32(N, stream_seed(11, KIND_MASTER), device="cuda")
    # ZeRO-2: one fused step over the sharded state
    z = [w0.clone(), torch.zeros(N, device="cuda"), torch.zeros(N, device="cuda")]
    zp = torch.empty(N, dtype=torch.bfloat16, device="cuda")
    # DDP: every replica holds a full copy of the state and updates it itself
    reps = [[w0.clone(), torch.zeros(N, device="cuda"), torch.zeros(N, device="cuda")]
            for _ in range(R)]
    rp = [torch.empty(N, dtype=torch.bfloat16, device="cuda") for _ in range(R)]
    red = torch.empty(N, device="cuda")
    for t in (1, 2):
        dpg.dpg_step(plan, dg, tok, dpg.HParams(step=t), *z, [zp])
        dpg.dpg_allreduce_grads(plan, dg, tok, red)
        for r in range(R):
            dpg.dpg_adam_from_reduced(plan, red, dpg.HParams(step=t), *reps[r], [rp[r]])
    torch.cuda.synchronize()
    for r in range(R):
        for a, b in zip(reps[r], z):
            assert torch.equal(a.view(torch.int32), b.view(torch.int32))
        assert torch.equal(rp[r].view(torch.int16), zp.view(torch.int16))
