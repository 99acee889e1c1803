"""Paired accumulation and the two-microbatch fold, on the GPU, against the
oracle's one-microbatch-at-a-time accumulation ("Distributed Training and
Parallelism" -- Data parallelism and the global gradient: no_sync
accumulation, normalisation by the count over ranks and microbatches).

The paired schedule performs the same binary32 additions in the same order,
so every output is expected bit for bit (bars as elsewhere: 2 ulp fp32,
1 ulp bf16, norms rel 1e-5).
"""
import numpy as np
import pytest
import torch

import oracle
import zero_optimizer_step_gb300 as dpg
from parity_util import check_norms, np_bf16, np_f32, ulp_bf16, ulp_f32
from workloads import (KIND_GRAD, KIND_M, KIND_MASTER, KIND_V, flat_grads_bf16, master_f32,
                       random_param_list, segments, stream_seed, warm_moments)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    from zero_optimizer_step_gb300 import build
    build.build()
    oracle.build()


def _micro(R, K, seed, n=50, mx=120_000, cap=1 << 19):
    numels = random_param_list(np.random.Generator(np.random.Philox(seed)), n, mx)
    plan = dpg.dpg_plan_buckets(numels, cap, R)
    op = oracle.plan_buckets(numels, cap, R)
    N = op.total_padded
    segs = segments(op.param_offset, numels)
    micro = [[flat_grads_bf16(segs, N, 1e-3, stream_seed(seed, KIND_GRAD, r, k)) for k in range(K)]
             for r in range(R)]
    tok = [2500 + 17 * i for i in range(R * K)]
    return plan, op, micro, tok


@pytest.mark.parametrize("first", [True, False])
def test_accumulate_pair_matches_two_single_accumulations(first):
    plan, op, micro, _ = _micro(1, 3, seed=31)
    N = op.total_padded
    a, b, c = (x.cuda() for x in micro[0])
    acc = torch.empty(N, device="cuda")
    ref = np.empty(N, np.float32)
    if not first:
        dpg.dpg_accumulate(plan, c, acc, first=True)
        oracle.accumulate(np_bf16(micro[0][2]), ref, first=True)
    dpg.dpg_accumulate_pair(plan, a, b, acc, first=first)
    oracle.accumulate(np_bf16(micro[0][0]), ref, first=first)
    oracle.accumulate(np_bf16(micro[0][1]), ref, first=False)
    torch.cuda.synchronize()
    assert ulp_f32(np_f32(acc), ref) == 0
    # and against the library's own single accumulations
    acc2 = torch.empty(N, device="cuda")
    if not first:
        dpg.dpg_accumulate(plan, c, acc2, first=True)
    dpg.dpg_accumulate(plan, a, acc2, first=first)
    dpg.dpg_accumulate(plan, b, acc2, first=False)
    torch.cuda.synchronize()
    assert torch.equal(acc.view(torch.int32), acc2.view(torch.int32))


@pytest.mark.parametrize("R,K,warm", [(4, 4, False), (8, 4, True), (3, 6, False), (1, 2, False),
                                      (2, 3, True)])
def test_fold2_cycle_matches_oracle(R, K, warm):
    """Cycle: pairs of microbatches into the fp32 buffers (a single one when
    K - 2 is odd), then the fused step with the last two folded in."""
    plan, op, micro, tok = _micro(R, K, seed=40 + R * 10 + K)
    N = op.total_padded
    w0 = master_f32(N, stream_seed(41, KIND_MASTER))
    if warm:
        m0, v0 = warm_moments(N, 1e-3, stream_seed(41, KIND_M), stream_seed(41, KIND_V))
    else:
        m0, v0 = torch.zeros(N), torch.zeros(N)
    t = 3 if warm else 1
    dm = [[x.cuda() for x in row] for row in micro]
    acc = [torch.empty(N, device="cuda") for _ in range(R)]
    for r in range(R):
        k = 0
        while k + 1 < K - 2:
            dpg.dpg_accumulate_pair(plan, dm[r][k], dm[r][k + 1], acc[r], first=(k == 0))
            k += 2
        if k < K - 2:
            dpg.dpg_accumulate(plan, dm[r][k], acc[r], first=(k == 0))
    d = [w0.cuda(), m0.cuda(), v0.cuda()]
    view = torch.empty(N, dtype=torch.bfloat16, device="cuda")
    sq = torch.empty(op.n_buckets, device="cuda")
    nf = torch.empty(op.n_buckets, dtype=torch.int64, device="cuda")
    if K == 2:
        # no accumulation buffer yet: a zero buffer plus both microbatches
        for r in range(R):
            acc[r].zero_()
    dpg.dpg_step_fold2(plan, acc, [dm[r][K - 2] for r in range(R)], [dm[r][K - 1] for r in range(R)],
                       tok, dpg.HParams(step=t), *d, [view], bucket_sqnorm=sq, bucket_nonfinite=nf)
    torch.cuda.synchronize()

    # oracle: one microbatch at a time, the last passed to the reduction
    hm = [[np_bf16(x) for x in row] for row in micro]
    accs = [np.zeros(N, np.float32) for _ in range(R)]
    for r in range(R):
        for k in range(K - 1):
            if K == 2:
                oracle.accumulate(hm[r][k], accs[r], first=False)
            else:
                oracle.accumulate(hm[r][k], accs[r], first=(k == 0))
    w, m, v = np_f32(w0).copy(), np_f32(m0).copy(), np_f32(v0).copy()
    views, red, rsq = oracle.step(op.bucket_offset, op.bucket_padded, accs, tok, w, m, v,
                                  last=[hm[r][K - 1] for r in range(R)], n_views=1, t=t,
                                  want_reduced=True)
    for got, ref in zip(d, (w, m, v)):
        assert ulp_f32(np_f32(got), ref) == 0
    assert ulp_bf16(np_bf16(view), views[0]) == 0
    check_norms(np_f32(sq), rsq)
    nfr = [int(np.sum(~np.isfinite(red[o:o + p]))) for o, p in zip(op.bucket_offset, op.bucket_padded)]
    np.testing.assert_array_equal(nf.cpu().numpy(), nfr)


def test_fold2_equals_accumulate_then_step_on_device():
    R, K = 4, 3
    plan, op, micro, tok = _micro(R, K, seed=55)
    N = op.total_padded
    dm = [[x.cuda() for x in row] for row in micro]
    w0 = master_f32(N, stream_seed(55, KIND_MASTER), device="cuda")
    outs = []
    for fold in (True, False):
        acc = [torch.empty(N, device="cuda") for _ in range(R)]
        for r in range(R):
            dpg.dpg_accumulate(plan, dm[r][0], acc[r], first=True)
        d = [w0.clone(), torch.zeros(N, device="cuda"), torch.zeros(N, device="cuda")]
        p = torch.empty(N, dtype=torch.bfloat16, device="cuda")
        if fold:
            dpg.dpg_step_fold2(plan, acc, [dm[r][1] for r in range(R)], [dm[r][2] for r in range(R)],
                               tok, dpg.HParams(), *d, [p])
        else:
            for r in range(R):
                dpg.dpg_accumulate(plan, dm[r][1], acc[r], first=False)
            dpg.dpg_step(plan, acc, tok, dpg.HParams(), *d, [p],
                         last_micro=[dm[r][2] for r in range(R)])
        outs.append((*d, p))
    torch.cuda.synchronize()
    for a, b in zip(*outs):
        assert torch.equal(a.view(torch.uint8), b.view(torch.uint8))


def test_fold2_reads_pinned_host_microbatches():
    R, K = 2, 3
    plan, op, micro, tok = _micro(R, K, seed=57)
    N = op.total_padded
    acc = [torch.empty(N, device="cuda") for _ in range(R)]
    for r in range(R):
        dpg.dpg_accumulate(plan, micro[r][0].pin_memory(), acc[r], first=True)
    w0 = master_f32(N, stream_seed(57, KIND_MASTER), device="cuda")
    outs = []
    for src in ("device", "host"):
        conv = (lambda x: x.cuda()) if src == "device" else (lambda x: x.pin_memory())
        d = [w0.clone(), torch.zeros(N, device="cuda"), torch.zeros(N, device="cuda")]
        p = torch.empty(N, dtype=torch.bfloat16, device="cuda")
        dpg.dpg_step_fold2(plan, acc, [conv(micro[r][1]) for r in range(R)],
                           [conv(micro[r][2]) for r in range(R)], tok, dpg.HParams(), *d, [p])
        torch.cuda.synchronize()
        outs.append((*d, p))
    for a, b in zip(*outs):
        assert torch.equal(a.view(torch.uint8), b.view(torch.uint8))


# ---------------------------------------------------------------------------
# deferred accumulation: every microbatch kept in bf16, summed in the step
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("R,K,warm", [(4, 4, False), (8, 4, True), (3, 6, False), (1, 1, False),
                                      (2, 3, True), (4, 2, False), (16, 4, False)])
def test_deferred_cycle_matches_oracle(R, K, warm):
    """dpg_step_deferred on R x K bf16 microbatch buffers equals the oracle's
    K - 1 accumulations (one microbatch at a time) followed by its step with
    the last microbatch, bit for bit.  K = 4 runs the kernel with K fixed at
    compile time, the others the run-time K; R = 3 and 16 the generic
    replica loop."""
    plan, op, micro, tok = _micro(R, K, seed=70 + R * 10 + K, n=30, mx=60_000, cap=1 << 18)
    N = op.total_padded
    w0 = master_f32(N, stream_seed(71, KIND_MASTER))
    if warm:
        m0, v0 = warm_moments(N, 1e-3, stream_seed(71, KIND_M), stream_seed(71, KIND_V))
    else:
        m0, v0 = torch.zeros(N), torch.zeros(N)
    t = 5 if warm else 1
    dm = [[x.cuda() for x in row] for row in micro]
    d = [w0.cuda(), m0.cuda(), v0.cuda()]
    view = torch.empty(N, dtype=torch.bfloat16, device="cuda")
    sq = torch.empty(op.n_buckets, device="cuda")
    nf = torch.empty(op.n_buckets, dtype=torch.int64, device="cuda")
    dpg.dpg_step_deferred(plan, dm, tok, dpg.HParams(step=t), *d, [view], bucket_sqnorm=sq,
                          bucket_nonfinite=nf)
    torch.cuda.synchronize()

    hm = [[np_bf16(x) for x in row] for row in micro]
    w, m, v = np_f32(w0).copy(), np_f32(m0).copy(), np_f32(v0).copy()
    if K == 1:
        views, red, rsq = oracle.step(op.bucket_offset, op.bucket_padded, [hm[r][0] for r in range(R)],
                                      tok, w, m, v, n_views=1, t=t, want_reduced=True)
    else:
        accs = [np.empty(N, np.float32) for _ in range(R)]
        for r in range(R):
            for k in range(K - 1):
                oracle.accumulate(hm[r][k], accs[r], first=(k == 0))
        views, red, rsq = oracle.step(op.bucket_offset, op.bucket_padded, accs, tok, w, m, v,
                                      last=[hm[r][K - 1] for r in range(R)], n_views=1, t=t,
                                      want_reduced=True)
    for got, ref in zip(d, (w, m, v)):
        assert ulp_f32(np_f32(got), ref) == 0
    assert ulp_bf16(np_bf16(view), views[0]) == 0
    check_norms(np_f32(sq), rsq)
    nfr = [int(np.sum(~np.isfinite(red[o:o + p]))) for o, p in zip(op.bucket_offset, op.bucket_padded)]
    np.testing.assert_array_equal(nf.cpu().numpy(), nfr)


def test_deferred_equals_accumulate_then_step_on_device():
    """The same bits as the library's own accumulation path, and with the
    microbatches in page-locked host memory."""
    R, K = 4, 4
    plan, op, micro, tok = _micro(R, K, seed=77)
    N = op.total_padded
    w0 = master_f32(N, stream_seed(77, KIND_MASTER), device="cuda")
    dm = [[x.cuda() for x in row] for row in micro]
    outs = []
    for how in ("accumulate", "deferred", "deferred_pinned"):
        d = [w0.clone(), torch.zeros(N, device="cuda"), torch.zeros(N, device="cuda")]
        p = torch.empty(N, dtype=torch.bfloat16, device="cuda")
        sq = torch.empty(op.n_buckets, device="cuda")
        if how == "accumulate":
            acc = [torch.empty(N, device="cuda") for _ in range(R)]
            for r in range(R):
                for k in range(K - 1):
                    dpg.dpg_accumulate(plan, dm[r][k], acc[r], first=(k == 0))
            dpg.dpg_step(plan, acc, tok, dpg.HParams(), *d, [p],
                         last_micro=[dm[r][K - 1] for r in range(R)], bucket_sqnorm=sq)
        elif how == "deferred":
            dpg.dpg_step_deferred(plan, dm, tok, dpg.HParams(), *d, [p], bucket_sqnorm=sq)
        else:
            pinned = [[x.pin_memory() for x in row] for row in micro]
            dpg.dpg_step_deferred(plan, pinned, tok, dpg.HParams(), *d, [p], bucket_sqnorm=sq)
        torch.cuda.synchronize()
        outs.append((*d, p, sq))
    for other in outs[1:]:
        for a, b in zip(outs[0][:4], other[:4]):
            assert torch.equal(a.view(torch.uint8), b.view(torch.uint8))
        np.testing.assert_allclose(np_f32(other[4]), np_f32(outs[0][4]), rtol=1e-5)
