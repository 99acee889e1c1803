"""The ZeRO-2 split across ranks ("Parallelisms" -- ZeRO-2; "Parallelism
Starts With the Bottleneck" -- Allreduce equals reducescatter plus allgather)
run as real processes over gloo on CPU tensors, world sizes 2 and 4.

Each rank holds its own replica gradient (rank r = replica r of the seeded
workload), exchanges slices through zero_optimizer_step_gb300.sharded, and
updates its shard.  On the CPU the local update is the oracle's step over the
shard plan (the library's update is a CUDA kernel; tests/test_gpu_sharded.py
checks it against the single-device step on the GPU).  Checked on every rank:

* after the exchange, recv[s] holds, bit for bit, rank s's slice of this
  rank's shard of every bucket, as the plan's shard_numel defines it, and
  zeros in the shard plan's padding;
* the all-gathered token counts are every rank's, replica-major;
* the rank's master/m/v shard equals the single-process oracle step over all
  R replicas at the shard's positions, bit for bit;
* the all-gathered bf16 parameters equal the concatenated owned shards and
  the single-process oracle's parameters, bit for bit;
* exchanging and updating in two bucket ranges, or pipelined over three
  (ShardedStep.step with groups=3), gives the same bits;
* with K = 3 microbatches accumulated on each rank and fp32 slices exchanged,
  the same holds against the oracle's accumulation path.
"""
import os
import socket
import sys

import numpy as np
import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _u16(t):
    import torch
    return t.view(torch.int16).numpy().view(np.uint16)


def _host(t):
    """numpy view of a CPU tensor: uint16 bit patterns for bf16, else float32."""
    import torch
    return _u16(t) if t.dtype == torch.bfloat16 else t.numpy()


def _oracle_update(shard_plan, recv, tokens, hp, master, m, v, views, *, bucket_sqnorm=None,
                   bucket_nonfinite=None, b0=0, b1=None, stream=None):
    """The shard update on the CPU: the oracle's step over the shard plan's
    buckets [b0, b1) with the received slice buffers as its R replicas."""
    import torch

    import oracle
    b1 = shard_plan.n_buckets if b1 is None else b1
    bo = shard_plan.bucket_offset[b0:b1]
    bp = shard_plan.bucket_padded[b0:b1]
    out, _, sq = oracle.step(bo, bp, [_host(x) for x in recv], tokens, master.numpy(), m.numpy(),
                             v.numpy(), lr=hp.lr, beta1=hp.beta1, beta2=hp.beta2, eps=hp.eps,
                             wd=hp.weight_decay, t=hp.step)
    p = _u16(views[0])
    for o, n in zip(bo, bp):
        p[o:o + n] = out[0][o:o + n]
    if bucket_sqnorm is not None:
        bucket_sqnorm[b0:b1] = torch.from_numpy(sq.astype(np.float32))


def _case(world):
    from workloads import random_param_list
    numels = random_param_list(np.random.Generator(np.random.Philox(600 + world)), 30, 50_000)
    return numels, 1 << 16


def _worker(rank, world, port, split, K):
    sys.path.insert(0, ROOT)
    import torch
    import torch.distributed as dist

    import oracle
    import zero_optimizer_step_gb300 as dpg
    from zero_optimizer_step_gb300.sharded import ShardedStep
    from workloads import KIND_GRAD, KIND_MASTER, flat_grads_bf16, master_f32, segments, stream_seed

    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank,
                            world_size=world)
    numels, cap = _case(world)
    plan = dpg.dpg_plan_buckets(numels, cap, world)
    N, nb = plan.total_padded, plan.n_buckets
    assert nb >= 4
    segs = segments(plan.param_offset, numels)
    micro = [[flat_grads_bf16(segs, N, 1e-3, stream_seed(61, KIND_GRAD, s, k)) for k in range(K)]
             for s in range(world)]
    master0 = master_f32(N, stream_seed(61, KIND_MASTER))
    tokens_all = np.array([3001 + 97 * s + 13 * k for s in range(world) for k in range(K)],
                          np.int64)
    hp = dpg.HParams(step=3)
    if K == 1:
        grads = [mr[0] for mr in micro]
    else:
        # each rank adds all K microbatches into its fp32 buffer, then the
        # exchange carries fp32 slices
        grads = []
        for s in range(world):
            acc = np.empty(N, np.float32)
            for k in range(K):
                oracle.accumulate(_u16(micro[s][k]), acc, first=(k == 0))
            grads.append(torch.from_numpy(acc))

    st = ShardedStep(plan, rank, world, "cpu", update_fn=_oracle_update,
                     grad_dtype=torch.bfloat16 if K == 1 else torch.float32)
    S = st.shard.total_padded
    master = st.state_from_global(master0)
    m, v = torch.zeros(S), torch.zeros(S)
    param = torch.full((N,), float("nan"), dtype=torch.bfloat16)

    local = tokens_all[rank * K:(rank + 1) * K]
    if split == "pipelined":
        # three bucket ranges, each range's exchange in flight while the
        # previous one is updated
        assert len(st.bucket_groups(3)) == 3
        tokens = st.step(grads[rank], local, hp, master, m, v, param, groups=3)
    else:
        tokens = st.all_tokens(local)
        cuts = [(0, nb)] if not split else [(0, nb // 2), (nb // 2, nb)]
        for b0, b1 in cuts:
            st.exchange(grads[rank], b0, b1)
            st.update(tokens, hp, master, m, v, b0=b0, b1=b1)
            st.allgather(param, b0, b1)
    np.testing.assert_array_equal(tokens, tokens_all)

    # the exchange delivered exactly rank s's slice of this rank's shard
    for s in range(world):
        got = _host(st.recv[s]).view(np.uint16 if K == 1 else np.uint32)
        sent = _host(grads[s]).view(got.dtype)
        filled = np.zeros(S, bool)
        for b in range(nb):
            lo, hi = st.global_slice(b, rank)
            a, z = st.shard_slice(b)
            assert z - a == plan.shard_numel[b]
            np.testing.assert_array_equal(got[a:z], sent[lo:hi])
            filled[a:z] = True
        assert not got[~filled].any(), "padding of a receive buffer is not zero"

    # the single-process oracle over all R replicas: for K > 1 the
    # accumulation path (K - 1 microbatches in fp32, the last one fused)
    w, mm, vv = master0.numpy().copy(), np.zeros(N, np.float32), np.zeros(N, np.float32)
    if K == 1:
        ref_grads, last = [_u16(g) for g in grads], None
    else:
        ref_grads, last = [], [_u16(micro[s][K - 1]) for s in range(world)]
        for s in range(world):
            acc = np.empty(N, np.float32)
            for k in range(K - 1):
                oracle.accumulate(_u16(micro[s][k]), acc, first=(k == 0))
            ref_grads.append(acc)
    views, _, _ = oracle.step(plan.bucket_offset, plan.bucket_padded, ref_grads, tokens_all, w, mm,
                              vv, last=last, t=3)
    for b in range(nb):
        lo, hi = st.global_slice(b, rank)
        a, z = st.shard_slice(b)
        for name, mine, ref in (("master", master, w), ("m", m, mm), ("v", v, vv)):
            assert np.array_equal(mine.numpy()[a:z].view(np.uint32), ref[lo:hi].view(np.uint32)), name
    p = _u16(param)
    np.testing.assert_array_equal(p, views[0])
    # the gathered buffer is the concatenation of the owned shards
    mine = _u16(st.param_shard)
    for b in range(nb):
        lo, hi = st.global_slice(b, rank)
        a, z = st.shard_slice(b)
        np.testing.assert_array_equal(p[lo:hi], mine[a:z])
    dist.barrier()
    dist.destroy_process_group()


@pytest.mark.parametrize("world", [2, 4])
@pytest.mark.parametrize("split", [False, True, "pipelined"])
def test_sharded_exchange_matches_single_process_oracle(world, split):
    import oracle
    oracle.build()
    from zero_optimizer_step_gb300 import build
    build.build()
    mp.spawn(_worker, args=(world, _free_port(), split, 1), nprocs=world, join=True)


@pytest.mark.parametrize("world", [2, 4])
def test_sharded_exchange_of_accumulated_microbatches(world):
    # K = 3 microbatches accumulated in fp32 on each rank, fp32 slices
    # exchanged: the single-process accumulation path's bits
    import oracle
    oracle.build()
    from zero_optimizer_step_gb300 import build
    build.build()
    mp.spawn(_worker, args=(world, _free_port(), True, 3), nprocs=world, join=True)


def test_sharded_step_rejects_a_plan_for_another_world_size():
    sys.path.insert(0, ROOT)
    import zero_optimizer_step_gb300 as dpg
    from zero_optimizer_step_gb300.sharded import ShardedStep
    plan = dpg.dpg_plan_buckets([1000, 2000], 1 << 12, 4)
    with pytest.raises(ValueError):
        ShardedStep(plan, 0, 2, "cpu")
    with pytest.raises(ValueError):
        ShardedStep(plan, 4, 4, "cpu")


def test_sharded_step_checks_the_exchange_dtype():
    sys.path.insert(0, ROOT)
    import torch

    import zero_optimizer_step_gb300 as dpg
    from zero_optimizer_step_gb300.sharded import ShardedStep
    plan = dpg.dpg_plan_buckets([1000, 2000], 1 << 12, 2)
    with pytest.raises(ValueError):
        ShardedStep(plan, 0, 2, "cpu", grad_dtype=torch.float16)
    st = ShardedStep(plan, 0, 2, "cpu", grad_dtype=torch.float32)
    with pytest.raises(ValueError):
        st.exchange(torch.zeros(plan.total_padded, dtype=torch.bfloat16))


def test_bucket_groups_cover_the_plan_in_order():
    sys.path.insert(0, ROOT)
    import zero_optimizer_step_gb300 as dpg
    from workloads import CONFIGS
    from zero_optimizer_step_gb300.sharded import ShardedStep
    c = CONFIGS["llama1b"]
    st = ShardedStep(dpg.dpg_plan_buckets(c.numels, c.cap_bytes, 2), 0, 2, "cpu")
    for n in (1, 2, 4, 7, 83, 500):
        g = st.bucket_groups(n)
        assert g[0][0] == 0 and g[-1][1] == st.plan.n_buckets
        assert all(a < b for a, b in g) and all(g[i][1] == g[i + 1][0] for i in range(len(g) - 1))
        assert len(g) <= min(n, st.plan.n_buckets)
    sizes = [int(st.plan.bucket_padded[a:b].sum()) for a, b in st.bucket_groups(4)]
    assert max(sizes) < 2 * min(sizes)
