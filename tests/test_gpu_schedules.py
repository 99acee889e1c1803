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


def test_zero3_gather_copies_bucket_range_only():
    plan, op, _, _, _ = _setup(2, "bf16", seed=13)
    N = op.total_padded
    g = torch.Generator().manual_seed(13)
    param = torch.randn(N, generator=g).to(torch.bfloat16).cuda()
    nan_bits = torch.tensor(0x7FC1, dtype=torch.int16)
    views = [torch.full((N,), int(nan_bits), dtype=torch.int16, device="cuda") for _ in range(3)]
    b0, b1 = 1, max(2, op.n_buckets - 1)
    dpg.dpg_gather_params_bf16(plan, param, [v.view(torch.bfloat16) for v in views], b0=b0, b1=b1)
    torch.cuda.synchronize()
    lo, hi = op.bucket_offset[b0], op.bucket_offset[b1 - 1] + op.bucket_padded[b1 - 1]
    pb = param.view(torch.int16).cpu()
    for v in views:
        h = v.cpu()
        assert torch.equal(h[lo:hi], pb[lo:hi])
        assert bool((h[:lo] == nan_bits).all()) and bool((h[hi:] == nan_bits).all())


def test_zero3_schedule_equals_zero2_views():
    """ZeRO-3: the step writes only the sharded bf16 parameters (one buffer);
    before use, every replica all-gathers the full layer from the shards.
    Each gathered replica equals the ZeRO-2 step's own per-replica view and
    the oracle's cast of the master weights."""
    R = 4
    plan, op, grads, _, tok = _setup(R, "bf16", seed=17)
    N = op.total_padded
    dg = [g.cuda() for g in grads]
    w0 = master_f32(N, stream_seed(17, KIND_MASTER), device="cuda")
    z2 = [w0.clone(), torch.zeros(N, device="cuda"), torch.zeros(N, device="cuda")]
    z2v = [torch.empty(N, dtype=torch.bfloat16, device="cuda") for _ in range(R)]
    z3 = [w0.clone(), torch.zeros(N, device="cuda"), torch.zeros(N, device="cuda")]
    shards = torch.empty(N, dtype=torch.bfloat16, device="cuda")
    z3v = [torch.full((N,), float("nan"), dtype=torch.bfloat16, device="cuda") for _ in range(R)]
    for t in (1, 2):
        dpg.dpg_step(plan, dg, tok, dpg.HParams(step=t), *z2, z2v)
        dpg.dpg_step(plan, dg, tok, dpg.HParams(step=t), *z3, [shards])
        for b in range(op.n_buckets):  # layer by layer, as a forward pass would
            dpg.dpg_gather_params_bf16(plan, shards, z3v, b0=b, b1=b + 1)
    torch.cuda.synchronize()
    w, m, v = np_f32(w0).copy(), np.zeros(N, np.float32), np.zeros(N, np.float32)
    for t in (1, 2):
        oracle.step(op.bucket_offset, op.bucket_padded, [np_bf16(g) for g in grads], tok, w, m, v,
                    n_views=1, t=t)
    ref = oracle.f32_to_bf16(w)
    for a, b in zip(z2v, z3v):
        assert torch.equal(a.view(torch.int16), b.view(torch.int16))
        np.testing.assert_array_equal(np_bf16(b), ref)


def test_pinned_host_gradients_read_in_place():
    """Gradient inputs in page-locked host memory are read by the kernels over
    the host link; every output equals the device-resident run bit for bit
    (fused step with and without accumulation, all-reduce)."""
    R = 4
    plan, op, grads, last, tok = _setup(R, "acc", seed=19)
    N = op.total_padded
    w0 = master_f32(N, stream_seed(19, KIND_MASTER), device="cuda")
    h_acc = [x.pin_memory() for x in grads]
    h_last = [x.pin_memory() for x in last]
    outs = []
    for acc, last in (([x.cuda() for x in h_acc], [x.cuda() for x in h_last]), (h_acc, h_last)):
        d = [w0.clone(), torch.zeros(N, device="cuda"), torch.zeros(N, device="cuda")]
        p = torch.empty(N, dtype=torch.bfloat16, device="cuda")
        sq = torch.empty(op.n_buckets, device="cuda")
        red = torch.empty(N, device="cuda")
        a0 = torch.empty(N, device="cuda")
        dpg.dpg_accumulate(plan, last[0], a0, first=True)
        dpg.dpg_step(plan, acc, tok, dpg.HParams(), *d, [p], last_micro=last, bucket_sqnorm=sq)
        dpg.dpg_allreduce_grads(plan, acc, tok, red, last_micro=last)
        torch.cuda.synchronize()
        outs.append([*d, p, sq, red, a0])
    for a, b in zip(*outs):
        assert torch.equal(a.view(torch.uint8), b.view(torch.uint8))


@pytest.mark.parametrize("max_ctas", [1, 7, 40])
def test_fused_grid_cap_gives_the_same_bits(max_ctas):
    """A capped grid changes only which CTA visits which tile: every output
    is the same bits, and the per-bucket norms stay within their bar."""
    R = 4
    plan, op, grads, _, tok = _setup(R, "bf16", seed=23)
    N = op.total_padded
    dg = [g.cuda() for g in grads]
    w0 = master_f32(N, stream_seed(23, KIND_MASTER), device="cuda")
    outs = []
    for cap in (0, max_ctas):
        dpg.dpg_set_fused_max_ctas(cap)
        try:
            d = [w0.clone(), torch.zeros(N, device="cuda"), torch.zeros(N, device="cuda")]
            p = torch.empty(N, dtype=torch.bfloat16, device="cuda")
            sq = torch.empty(op.n_buckets, device="cuda")
            red = torch.empty(N, device="cuda")
            dpg.dpg_reduce_scatter_adam(plan, dg, tok, dpg.HParams(), *d, [p], bucket_sqnorm=sq,
                                        reduced_grad=red)
            torch.cuda.synchronize()
        finally:
            dpg.dpg_set_fused_max_ctas(0)
        outs.append((d, p, sq, red))
    (d0, p0, sq0, r0), (d1, p1, sq1, r1) = outs
    for a, b in zip(d0 + [p0, r0], d1 + [p1, r1]):
        assert torch.equal(a.view(torch.uint8), b.view(torch.uint8))
    ref = oracle.reduce([np_bf16(x) for x in grads], oracle.grad_scale(tok))
    check_norms(np_f32(sq1), np.array([np.sum(ref[o:o + q].astype(np.float64) ** 2)
                                       for o, q in zip(op.bucket_offset, op.bucket_padded)]))
