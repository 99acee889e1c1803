"""One rank's update of the ZeRO-2 split on the GPU ("Parallelisms" -- ZeRO-2).

For every rank r of R = 2, 4, 8 (and a generic R = 3): the slices the
exchange would deliver are copied locally from all R replica buffers
(sharded.loopback_receive), then the library's fused update runs on the shard
plan (dpg_plan_shards) with those R slice buffers as its replicas.  Its
master/m/v shard and bf16 parameter shard must equal, bit for bit, shard r of
the single-device dpg_step over all R replicas and of the CPU oracle's step;
the per-bucket norms of the R shards must add up to the bucket's norm.
"""
import numpy as np
import pytest
import torch

import oracle
import zero_optimizer_step_gb300 as dpg
from parity_util import np_bf16, np_f32
from workloads import KIND_GRAD, KIND_MASTER, flat_grads_bf16, master_f32, random_param_list, segments, stream_seed
from zero_optimizer_step_gb300.sharded import ShardedStep, loopback_receive

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    from zero_optimizer_step_gb300 import build
    build.build()


@pytest.mark.parametrize("R", [2, 3, 4, 8, 16])
def test_shard_update_equals_single_device_step(R):
    numels = random_param_list(np.random.Generator(np.random.Philox(70 + R)), 40, 300_000)
    plan = dpg.dpg_plan_buckets(numels, 1 << 19, R)
    N, nb = plan.total_padded, plan.n_buckets
    assert nb >= 2
    segs = segments(plan.param_offset, numels)
    grads = [flat_grads_bf16(segs, N, 1e-3, stream_seed(70, KIND_GRAD, s), device="cuda")
             for s in range(R)]
    master0 = master_f32(N, stream_seed(70, KIND_MASTER), device="cuda")
    tok = [2900 + 31 * s for s in range(R)]
    hp = dpg.HParams(step=2)

    # the single-device step over every replica
    w, m, v = master0.clone(), torch.zeros(N, device="cuda"), torch.zeros(N, device="cuda")
    p = torch.empty(N, dtype=torch.bfloat16, device="cuda")
    sq = torch.empty(nb, device="cuda")
    dpg.dpg_step(plan, grads, tok, hp, w, m, v, [p], bucket_sqnorm=sq)
    torch.cuda.synchronize()
    # and the oracle's
    ow, om, ov = np_f32(master0).copy(), np.zeros(N, np.float32), np.zeros(N, np.float32)
    oviews, _, _ = oracle.step(plan.bucket_offset, plan.bucket_padded, [np_bf16(g) for g in grads],
                               np.asarray(tok, np.int64), ow, om, ov, t=2)

    shard_sq = []
    for r in range(R):
        st = ShardedStep(plan, r, R, "cuda")
        S = st.shard.total_padded
        ms = st.state_from_global(master0)
        mm, vv = torch.zeros(S, device="cuda"), torch.zeros(S, device="cuda")
        ssq = torch.full((nb,), float("nan"), device="cuda")
        loopback_receive(st, grads)
        st.update(tok, hp, ms, mm, vv, bucket_sqnorm=ssq)
        torch.cuda.synchronize()
        for b in range(nb):
            lo, hi = st.global_slice(b, r)
            a, z = st.shard_slice(b)
            for name, mine, ref, oref in (("master", ms, w, ow), ("m", mm, m, om), ("v", vv, v, ov)):
                got = np_f32(mine[a:z]).view(np.uint32)
                assert np.array_equal(got, np_f32(ref[lo:hi]).view(np.uint32)), (name, r, b)
                assert np.array_equal(got, oref[lo:hi].view(np.uint32)), (name, r, b)
            gp = np_bf16(st.param_shard[a:z])
            assert np.array_equal(gp, np_bf16(p[lo:hi])), ("param", r, b)
            assert np.array_equal(gp, oviews[0][lo:hi]), ("param", r, b)
        shard_sq.append(np_f32(ssq).astype(np.float64))
    total = np.sum(shard_sq, axis=0)
    ref = np_f32(sq).astype(np.float64)
    assert np.all(np.abs(total - ref) <= 1e-5 * ref)


@pytest.mark.parametrize("R,K", [(2, 3), (4, 4)])
def test_shard_update_of_accumulated_microbatches(R, K):
    # each rank adds its K microbatches into an fp32 buffer (dpg_accumulate),
    # the exchange carries fp32 slices: the single-device accumulation path's
    # bits (K - 1 fp32 passes, the last microbatch fused into the step)
    numels = random_param_list(np.random.Generator(np.random.Philox(90 + R)), 30, 200_000)
    plan = dpg.dpg_plan_buckets(numels, 1 << 19, R)
    N, nb = plan.total_padded, plan.n_buckets
    segs = segments(plan.param_offset, numels)
    micro = [[flat_grads_bf16(segs, N, 1e-3, stream_seed(91, KIND_GRAD, s, k), device="cuda")
              for k in range(K)] for s in range(R)]
    master0 = master_f32(N, stream_seed(91, KIND_MASTER), device="cuda")
    tok = [2000 + 17 * i for i in range(R * K)]
    hp = dpg.HParams(step=5)

    acc_k1 = [torch.empty(N, device="cuda") for _ in range(R)]      # K - 1 microbatches
    acc_all = [torch.empty(N, device="cuda") for _ in range(R)]     # all K
    for s in range(R):
        for k in range(K):
            if k < K - 1:
                dpg.dpg_accumulate(plan, micro[s][k], acc_k1[s], first=(k == 0))
            dpg.dpg_accumulate(plan, micro[s][k], acc_all[s], first=(k == 0))
    w, m, v = master0.clone(), torch.zeros(N, device="cuda"), torch.zeros(N, device="cuda")
    p = torch.empty(N, dtype=torch.bfloat16, device="cuda")
    dpg.dpg_step(plan, acc_k1, tok, hp, w, m, v, [p], last_micro=[micro[s][K - 1] for s in range(R)])
    torch.cuda.synchronize()

    for r in range(R):
        st = ShardedStep(plan, r, R, "cuda", grad_dtype=torch.float32)
        S = st.shard.total_padded
        ms = st.state_from_global(master0)
        mm, vv = torch.zeros(S, device="cuda"), torch.zeros(S, device="cuda")
        loopback_receive(st, acc_all)
        st.update(tok, hp, ms, mm, vv)
        torch.cuda.synchronize()
        for b in range(nb):
            lo, hi = st.global_slice(b, r)
            a, z = st.shard_slice(b)
            for name, mine, ref in (("master", ms, w), ("m", mm, m), ("v", vv, v)):
                assert torch.equal(mine[a:z].view(torch.int32), ref[lo:hi].view(torch.int32)), (name, r, b)
            assert torch.equal(st.param_shard[a:z].view(torch.int16), p[lo:hi].view(torch.int16))


@pytest.mark.parametrize("groups,K", [(1, 1), (3, 1), (3, 2)])
def test_whole_split_step_over_nccl_single_rank(groups, K):
    # the real collectives (token all-gather, exchange, all-gather of the
    # parameter shards) over a one-rank NCCL group on this GPU, plain and
    # pipelined: the single-device step's bits
    import socket

    import torch.distributed as dist
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        port = s.getsockname()[1]
    dist.init_process_group("nccl", init_method=f"tcp://127.0.0.1:{port}", rank=0, world_size=1,
                            device_id=torch.device("cuda", torch.cuda.current_device()))
    try:
        numels = random_param_list(np.random.Generator(np.random.Philox(95)), 30, 300_000)
        plan = dpg.dpg_plan_buckets(numels, 1 << 19, 1)
        N = plan.total_padded
        segs = segments(plan.param_offset, numels)
        micro = [flat_grads_bf16(segs, N, 1e-3, stream_seed(95, KIND_GRAD, 0, k), device="cuda")
                 for k in range(K)]
        master0 = master_f32(N, stream_seed(95, KIND_MASTER), device="cuda")
        hp = dpg.HParams(step=1)
        counts = [3333 + k for k in range(K)]
        w, m, v = master0.clone(), torch.zeros(N, device="cuda"), torch.zeros(N, device="cuda")
        p = torch.empty(N, dtype=torch.bfloat16, device="cuda")
        if K == 1:
            dpg.dpg_step(plan, micro, counts, hp, w, m, v, [p])
            src = micro[0]
        else:
            acc, src = torch.empty(N, device="cuda"), torch.empty(N, device="cuda")
            for k in range(K):
                if k < K - 1:
                    dpg.dpg_accumulate(plan, micro[k], acc, first=(k == 0))
                dpg.dpg_accumulate(plan, micro[k], src, first=(k == 0))
            dpg.dpg_step(plan, [acc], counts, hp, w, m, v, [p], last_micro=[micro[K - 1]])
        st = ShardedStep(plan, 0, 1, "cuda", grad_dtype=torch.bfloat16 if K == 1 else torch.float32)
        S = st.shard.total_padded
        ms = st.state_from_global(master0)
        mm, vv = torch.zeros(S, device="cuda"), torch.zeros(S, device="cuda")
        param = torch.full((N,), float("nan"), dtype=torch.bfloat16, device="cuda")
        tokens = st.step(src, counts, hp, ms, mm, vv, param, groups=groups)
        torch.cuda.synchronize()
        assert list(tokens) == counts
        assert torch.equal(param.view(torch.int16), p.view(torch.int16))
        for b in range(plan.n_buckets):
            lo, hi = st.global_slice(b, 0)
            a, z = st.shard_slice(b)
            assert torch.equal(ms[a:z].view(torch.int32), w[lo:hi].view(torch.int32))
    finally:
        dist.destroy_process_group()
