"""GPU parity: the sm_103a library (through its C ABI) against the CPU oracle on
identical seeded inputs, element by element, at sizes the oracle finishes in
seconds that still span many tiles (2048 elements each) and ragged tails.

Bars: accumulation and reduced gradients bit-exact; master/m/v within 2 ulp;
bf16 parameters within 1 ulp; per-bucket norms within 1e-5 relative; the
non-finite counts exact.  Every case also records whether the result was
bit-exact everywhere (it is expected to be).
"""
import numpy as np
import pytest
import torch

import oracle
import zero_optimizer_step_gb300 as dpg
from parity_util import (StepCase, assert_parity, exact_everywhere, np_bf16, np_f32, run_case,
                         ulp_bf16, ulp_f32)
from workloads import CONFIGS, KIND_GRAD, flat_grads_bf16, random_param_list, segments, stream_seed

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    from zero_optimizer_step_gb300 import build
    build.build()
    oracle.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"


def _ragged(seed, n, max_numel):
    rng = np.random.Generator(np.random.Philox(seed))
    return random_param_list(rng, n, max_numel)


def test_tiny_config_bit_exact():
    cfg = CONFIGS["tiny"]
    for n_views in (1, cfg.R):
        res = run_case(StepCase(cfg.numels, cfg.cap_bytes, cfg.R, grad_std=cfg.grad_std,
                                tokens=cfg.fixed_tokens, n_views=n_views, seed=cfg.seed))
        assert res.plan.n_buckets == 2 and res.plan.total_padded == 2400
        assert_parity(res)
        assert exact_everywhere(res)


CASES = {
    # name: StepCase kwargs
    "R8_bf16_many_tiles": dict(numels=_ragged(1, 40, 200_000), cap_bytes=1 << 20, R=8),
    "R4_acc_K4_warm_t7": dict(numels=_ragged(2, 30, 100_000), cap_bytes=1 << 19, R=4, K=4,
                              warm=True, t=7),
    "R3_generic_warm_wd": dict(numels=_ragged(3, 25, 50_000), cap_bytes=300_000, R=3, warm=True,
                               t=3, wd=0.1),
    "R5_f32_grads": dict(numels=_ragged(4, 20, 80_000), cap_bytes=1 << 18, R=5, f32_grads=True,
                         t=2, warm=True),
    "R16_generic": dict(numels=_ragged(5, 20, 30_000), cap_bytes=1 << 17, R=16, grad_std=1e-3),
    "R1_single_replica": dict(numels=_ragged(6, 30, 60_000), cap_bytes=1 << 18, R=1),
    "R2_acc_K2": dict(numels=_ragged(7, 20, 60_000), cap_bytes=1 << 18, R=2, K=2),
    "R64_max_replicas": dict(numels=_ragged(8, 10, 5_000), cap_bytes=1 << 14, R=64),
    "R8_split_launch": dict(numels=_ragged(9, 40, 100_000), cap_bytes=1 << 18, R=8, b_split=3),
    "R8_views_distinct": dict(numels=_ragged(10, 15, 40_000), cap_bytes=1 << 18, R=8, n_views=8),
    "R2_views_max": dict(numels=_ragged(19, 8, 6_000), cap_bytes=1 << 14, R=2, n_views=64),
    "R8_tiny_buckets": dict(numels=_ragged(11, 500, 64), cap_bytes=256, R=8),
    "R4_oversize_param": dict(numels=[5, 300_001, 7, 0, 12], cap_bytes=4096, R=4),
    "R8_nan": dict(numels=_ragged(12, 10, 10_000), cap_bytes=1 << 15, R=8, inject="nan"),
    "R8_inf": dict(numels=_ragged(13, 10, 10_000), cap_bytes=1 << 15, R=8, inject="inf"),
    "R4_denormal": dict(numels=_ragged(14, 10, 10_000), cap_bytes=1 << 15, R=4, inject="denormal",
                        grad_std=1e-37),
    "R8_acc_K3_nan": dict(numels=_ragged(15, 10, 10_000), cap_bytes=1 << 15, R=8, K=3,
                          inject="nan"),
    # other hyper-parameters: a large step (bias corrections near 1), a small
    # beta2 and eps where eps matters, AdamW with a large lr
    "R8_hp_late_step": dict(numels=_ragged(16, 20, 40_000), cap_bytes=1 << 18, R=8, warm=True,
                            t=100_000, lr=3e-4, beta1=0.95, beta2=0.98, eps=1e-6),
    "R4_hp_eps_dominant": dict(numels=_ragged(17, 20, 40_000), cap_bytes=1 << 18, R=4,
                               grad_std=1e-9, eps=1e-5, lr=1e-2),
    "R2_hp_adamw": dict(numels=_ragged(18, 20, 40_000), cap_bytes=1 << 18, R=2, warm=True, t=9,
                        lr=5e-2, wd=0.3, beta1=0.5, beta2=0.9),
}


@pytest.mark.parametrize("name", sorted(CASES))
def test_step_parity(name):
    res = run_case(StepCase(**CASES[name]))
    assert res.plan.total_padded > 0
    assert_parity(res)
    assert exact_everywhere(res)
    if CASES[name].get("inject") in ("nan", "inf"):
        assert res.gpu["nf"].sum() > 0


@pytest.mark.parametrize("cap_bytes", [4096, 1 << 20, 256 << 20])
def test_sweep_list_parity(cap_bytes):
    """The 10,000-tensor sweep list at its real size (about 4.9M parameters,
    1 to 4096 elements each): at 4 KiB caps 2595 buckets, most of them a
    single tile or less, up to one bucket holding everything."""
    cfg = CONFIGS["sweep"]
    res = run_case(StepCase(numels=cfg.numels, cap_bytes=cap_bytes, R=cfg.R, seed=cfg.seed,
                            grad_std=1e-3))
    assert res.plan.n_buckets == {4096: 2595, 1 << 20: 10, 256 << 20: 1}[cap_bytes]
    assert_parity(res)
    assert exact_everywhere(res)


def test_empty_plan_is_a_no_op():
    res = run_case(StepCase(numels=[], cap_bytes=1024, R=4))
    assert res.plan.n_buckets == 0 and res.plan.total_padded == 0


def test_zero_size_parameters_only():
    res = run_case(StepCase(numels=[0, 0, 0], cap_bytes=1024, R=2))
    assert res.plan.n_buckets == 1 and res.plan.total_padded == 0


def test_zero_tokens_rejected_and_nothing_written():
    plan = dpg.dpg_plan_buckets([100, 50], 4096, 2)
    N = plan.total_padded
    g = [torch.ones(N, dtype=torch.bfloat16, device="cuda") for _ in range(2)]
    w = torch.full((N,), 0.5, device="cuda")
    m, v = torch.zeros(N, device="cuda"), torch.zeros(N, device="cuda")
    p = torch.zeros(N, dtype=torch.bfloat16, device="cuda")
    before = dpg.dpg_launch_count()
    with pytest.raises(dpg.DpgError) as e:
        dpg.dpg_step(plan, g, [0, 0], dpg.HParams(), w, m, v, [p])
    assert e.value.status == dpg.DPG_ERR_ZERO_TOKENS
    torch.cuda.synchronize()
    assert dpg.dpg_launch_count() == before
    assert torch.all(w == 0.5) and torch.all(p == 0)


def test_multi_step_trajectory():
    """Five consecutive steps (t = 1..5) on fresh gradients stay bit-exact."""
    numels = _ragged(20, 20, 50_000)
    R = 4
    plan = dpg.dpg_plan_buckets(numels, 1 << 18, R)
    oplan = oracle.plan_buckets(numels, 1 << 18, R)
    N = oplan.total_padded
    segs = segments(oplan.param_offset, numels)
    w0 = torch.randn(N, generator=torch.Generator().manual_seed(1)) * 0.02
    d = dict(w=w0.cuda(), m=torch.zeros(N, device="cuda"), v=torch.zeros(N, device="cuda"))
    h = dict(w=w0.numpy().copy(), m=np.zeros(N, np.float32), v=np.zeros(N, np.float32))
    view = torch.empty(N, dtype=torch.bfloat16, device="cuda")
    for t in range(1, 6):
        gs = [flat_grads_bf16(segs, N, 1e-3, stream_seed(77, KIND_GRAD, r, t)) for r in range(R)]
        tok = [3000 + 17 * t + r for r in range(R)]
        dpg.dpg_step(plan, [g.cuda() for g in gs], tok, dpg.HParams(step=t), d["w"], d["m"],
                     d["v"], [view])
        views, _, _ = oracle.step(oplan.bucket_offset, oplan.bucket_padded,
                                  [np_bf16(g) for g in gs], tok, h["w"], h["m"], h["v"], t=t)
        torch.cuda.synchronize()
        for k in ("w", "m", "v"):
            assert ulp_f32(np_f32(d[k]), h[k]) == 0, (t, k)
        assert ulp_bf16(np_bf16(view), views[0]) == 0


@pytest.mark.parametrize("seed", range(4))
def test_pack_unpack_bit_exact(seed):
    rng = np.random.Generator(np.random.Philox(300 + seed))
    numels = random_param_list(rng, int(rng.integers(1, 300)), 20_000)
    numels[0] = 3 * 65536 + 5           # several pack items (65536 elements each) for one parameter
    R = int(rng.choice([1, 2, 4, 8]))
    cap = int(rng.integers(64, 1 << 17))
    plan = dpg.dpg_plan_buckets(numels, cap, R)
    # parameter gradients live inside one big buffer at odd 2-byte offsets, so
    # both the 16-byte and the unaligned copy paths run
    total = int(numels.sum()) + 2 * len(numels) + 8
    store = torch.randn(total, generator=torch.Generator().manual_seed(seed)).to(torch.bfloat16)
    d_store = store.cuda()
    grads, h_grads, off = [], [], 1
    for n in numels:
        grads.append(d_store[off:off + int(n)])
        h_grads.append(np_bf16(store[off:off + int(n)]))
        off += int(n) + int(rng.integers(0, 2))
    flat = torch.full((plan.total_padded,), float("nan"), dtype=torch.bfloat16, device="cuda")
    dpg.dpg_pack(plan, grads, flat)
    oplan = oracle.plan_buckets(numels, cap, R)
    np.testing.assert_array_equal(oplan.param_offset, plan.param_offset)
    ref = oracle.pack(oplan, h_grads)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(np_bf16(flat), ref)
    outs = [torch.full((int(n),), float("nan"), dtype=torch.bfloat16, device="cuda") for n in numels]
    dpg.dpg_unpack(plan, flat, outs)
    torch.cuda.synchronize()
    for o, h in zip(outs, h_grads):
        np.testing.assert_array_equal(np_bf16(o), h)


def test_pack_unpack_many_parameters():
    """2600 parameters: the pointer table travels 1024 parameters per launch,
    so pack and unpack run three launches over the item list."""
    rng = np.random.Generator(np.random.Philox(377))
    numels = rng.integers(1, 65, 2600)
    numels[1500] = 70_000               # one parameter split into several items mid-list
    R, cap = 4, 1 << 12
    plan = dpg.dpg_plan_buckets(numels, cap, R)
    store = torch.randn(int(numels.sum()), generator=torch.Generator().manual_seed(377)).to(torch.bfloat16)
    d_store = store.cuda()
    grads, h_grads, off = [], [], 0
    for n in numels:
        grads.append(d_store[off:off + int(n)])
        h_grads.append(np_bf16(store[off:off + int(n)]))
        off += int(n)
    flat = torch.full((plan.total_padded,), float("nan"), dtype=torch.bfloat16, device="cuda")
    before = dpg.dpg_launch_count()
    dpg.dpg_pack(plan, grads, flat)
    assert dpg.dpg_launch_count() - before == 3
    oplan = oracle.plan_buckets(numels, cap, R)
    ref = oracle.pack(oplan, h_grads)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(np_bf16(flat), ref)
    outs = [torch.full((int(n),), float("nan"), dtype=torch.bfloat16, device="cuda") for n in numels]
    dpg.dpg_unpack(plan, flat, outs)
    torch.cuda.synchronize()
    for o, h in zip(outs, h_grads):
        np.testing.assert_array_equal(np_bf16(o), h)


def test_pack_then_step_matches_oracle():
    cfg = CONFIGS["tiny"]
    plan = dpg.dpg_plan_buckets(cfg.numels, cfg.cap_bytes, cfg.R)
    oplan = oracle.plan_buckets(cfg.numels, cfg.cap_bytes, cfg.R)
    gen = torch.Generator().manual_seed(cfg.seed)
    per = [[(torch.randn(int(n), generator=gen) * cfg.grad_std).to(torch.bfloat16)
            for n in cfg.numels] for _ in range(cfg.R)]
    flats = []
    for r in range(cfg.R):
        f = torch.full((plan.total_padded,), 7.0, dtype=torch.bfloat16, device="cuda")
        dpg.dpg_pack(plan, [g.cuda() for g in per[r]], f)
        flats.append(f)
    h_flats = [oracle.pack(oplan, [np_bf16(g) for g in per[r]]) for r in range(cfg.R)]
    torch.cuda.synchronize()
    for f, hf in zip(flats, h_flats):
        np.testing.assert_array_equal(np_bf16(f), hf)
    w0 = torch.randn(plan.total_padded, generator=gen) * 0.02
    w, m, v = w0.cuda(), torch.zeros(plan.total_padded, device="cuda"), torch.zeros(plan.total_padded, device="cuda")
    view = torch.empty(plan.total_padded, dtype=torch.bfloat16, device="cuda")
    dpg.dpg_step(plan, flats, cfg.fixed_tokens, dpg.HParams(), w, m, v, [view])
    hw, hm, hv = w0.numpy().copy(), np.zeros(plan.total_padded, np.float32), np.zeros(plan.total_padded, np.float32)
    views, _, _ = oracle.step(oplan.bucket_offset, oplan.bucket_padded, h_flats, cfg.fixed_tokens,
                              hw, hm, hv)
    torch.cuda.synchronize()
    assert ulp_f32(np_f32(w), hw) == 0 and ulp_f32(np_f32(m), hm) == 0 and ulp_f32(np_f32(v), hv) == 0
    assert ulp_bf16(np_bf16(view), views[0]) == 0


def test_allgather_bit_exact_with_special_values():
    numels = [1000, 77, 4096, 3]
    plan = dpg.dpg_plan_buckets(numels, 2048, 2)
    N = plan.total_padded
    w = (torch.randn(N, generator=torch.Generator().manual_seed(5)) *
         torch.logspace(-40, 38, N)).float()
    specials = torch.tensor([0.0, -0.0, float("inf"), -float("inf"), float("nan"), 3.4e38,
                             -3.4e38, 1e-45, -1e-45, 1.00390625, 1.01171875])
    w[: specials.numel()] = specials
    views = [torch.empty(N, dtype=torch.bfloat16, device="cuda") for _ in range(3)]
    dpg.dpg_allgather_params(plan, w.cuda(), views)
    ref = oracle.allgather(w.numpy(), 1)[0]
    oplan = oracle.plan_buckets(numels, 2048, 2)
    torch.cuda.synchronize()
    for v in views:
        assert ulp_bf16(np_bf16(v), ref) == 0
    # a bucket sub-range writes only that range
    part = torch.zeros(N, dtype=torch.bfloat16, device="cuda")
    dpg.dpg_allgather_params(plan, w.cuda(), [part], b0=1, b1=2)
    lo, hi = oplan.bucket_offset[1], oplan.bucket_offset[1] + oplan.bucket_padded[1]
    got = np_bf16(part)
    assert ulp_bf16(got[lo:hi], ref[lo:hi]) == 0
    assert not got[:lo].any() and not got[hi:].any()


def test_norm_is_deterministic_across_runs():
    numels = _ragged(30, 30, 300_000)
    res = [run_case(StepCase(numels=numels, cap_bytes=1 << 20, R=8, seed=9)) for _ in range(2)]
    np.testing.assert_array_equal(res[0].gpu["sq"], res[1].gpu["sq"])


def test_multi_segment_bucket_norms_and_counter_reset():
    """A 20M-element parameter alone in its bucket (4883 tiles: three norm
    segments of at most 2048 tiles) next to a small bucket, launched whole and
    bucket by bucket; then one plan reused on other inputs: the per-bucket
    arrival counters reset themselves, so its norms equal a fresh plan's."""
    numels = [20_000_000, 3000, 777, 1_000_000]
    for b_split in (None, 1):
        res = run_case(StepCase(numels=numels, cap_bytes=16 << 20, R=2, seed=41, b_split=b_split))
        assert res.plan.n_buckets == 2
        assert_parity(res)

    plan = dpg.dpg_plan_buckets(numels, 16 << 20, 2)
    N = plan.total_padded
    segs = segments(plan.param_offset, numels)

    def norms(pl, seed):
        g = [flat_grads_bf16(segs, N, 1e-3, stream_seed(seed, KIND_GRAD, r), device="cuda")
             for r in range(2)]
        w, m, v = (torch.zeros(N, device="cuda") for _ in range(3))
        p = torch.empty(N, dtype=torch.bfloat16, device="cuda")
        sq = torch.full((pl.n_buckets,), float("nan"), device="cuda")
        nf = torch.full((pl.n_buckets,), -1, dtype=torch.int64, device="cuda")
        dpg.dpg_step(pl, g, [100, 200], dpg.HParams(), w, m, v, [p], bucket_sqnorm=sq,
                     bucket_nonfinite=nf)
        torch.cuda.synchronize()
        return sq, nf

    a, _ = norms(plan, 41)
    b, nfb = norms(plan, 42)
    b2, _ = norms(plan, 42)
    fresh = dpg.dpg_plan_buckets(numels, 16 << 20, 2)
    bf, _ = norms(fresh, 42)
    assert torch.isfinite(b).all() and not torch.equal(a, b)
    assert torch.equal(b, bf) and torch.equal(b2, bf)
    assert (nfb == 0).all()


def test_short_and_long_bucket_norms_in_one_finalize():
    """Buckets of at most 256 tiles (1,048,576 elements) are finalized by one
    warp each, longer ones by one CTA per segment, in the same launch; a
    bucket of exactly 256 tiles, one of 257, a two-segment bucket and small
    packed buckets side by side, launched whole and split at every bucket
    boundary: parity with the oracle, and the same norm bits in every split."""
    numels = [9_000_000, 1_052_672, 1_048_576, 5000, 70_000, 300_000, 1_048_568, 12_345, 777,
              2_000_000, 4096, 1]
    whole = run_case(StepCase(numels=numels, cap_bytes=2 << 20, R=2, seed=43))
    assert_parity(whole)
    tiles = -(-np.asarray(whole.plan.bucket_padded) // 4096)
    assert 256 in tiles and 257 in tiles and (tiles > 2048).any() and (tiles < 256).sum() >= 3
    for b in range(1, whole.plan.n_buckets):
        part = run_case(StepCase(numels=numels, cap_bytes=2 << 20, R=2, seed=43, b_split=b))
        assert_parity(part)
        assert np.array_equal(part.gpu["sq"].view(np.uint32), whole.gpu["sq"].view(np.uint32)), b
        np.testing.assert_array_equal(part.gpu["nf"], whole.gpu["nf"])


def test_launch_count_and_kernels():
    cfg = CONFIGS["tiny"]
    before = dpg.dpg_launch_count()
    run_case(StepCase(cfg.numels, cfg.cap_bytes, cfg.R, tokens=cfg.fixed_tokens))
    # fused pass + norm finalize
    assert dpg.dpg_launch_count() - before == 2
