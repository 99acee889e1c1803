"""Host-side checks of the C ABI (no GPU needed).

* libdpg.so loads and exports every function that include/dpg.h declares.
* The library's bucket planner (C++) equals the oracle's planner (C) bit for
  bit on the hand-worked cases, random ragged lists and every workload.
* Argument validation returns the documented status codes before any device
  work is issued.
"""
import ctypes
import os
import re
import subprocess

import numpy as np
import pytest

import zero_optimizer_step_gb300 as dpg
from workloads import CONFIGS, random_param_list

from test_oracle_plan import load_plan_cases

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "dpg.h")


@pytest.fixture(scope="module", autouse=True)
def built():
    from zero_optimizer_step_gb300 import build
    build.build()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(dpg_[a-z_0-9]+)\s*\(", text)))


def test_header_declares_the_binding_names():
    assert declared_functions() == sorted(dpg.EXPORTED)


def test_library_exports_every_declared_symbol():
    L = dpg.lib()
    for name in declared_functions():
        assert hasattr(L, name), name
    out = subprocess.run(["nm", "-D", "--defined-only", dpg.LIB_PATH], capture_output=True,
                         text=True, check=True).stdout
    exported = set(re.findall(r" T (dpg_\w+)", out))
    assert set(declared_functions()) <= exported


def test_abi_version_and_status_strings():
    assert dpg.dpg_abi_version() == 1
    L = dpg.lib()
    assert L.dpg_status_string(dpg.DPG_ERR_ZERO_TOKENS) == b"DPG_ERR_ZERO_TOKENS"
    assert L.dpg_status_string(12345) == b"DPG_ERR_UNKNOWN"


def _same_plan(a, o):
    assert a.n_buckets == o.n_buckets
    assert a.total_padded == o.total_padded
    np.testing.assert_array_equal(a.bucket_offset, o.bucket_offset)
    np.testing.assert_array_equal(a.bucket_padded, o.bucket_padded)
    np.testing.assert_array_equal(a.param_bucket, o.param_bucket)
    np.testing.assert_array_equal(a.param_offset, o.param_offset)


@pytest.mark.parametrize("case", load_plan_cases(), ids=lambda c: c["name"])
def test_plan_hand_worked(oracle_lib, case):
    a = dpg.dpg_plan_buckets(case["numels"], case["cap"], case["R"])
    _same_plan(a, oracle_lib.plan_buckets(case["numels"], case["cap"], case["R"]))
    for b, off, pad, shard in case["buckets"]:
        assert dpg.dpg_plan_bucket(a, b) == (off, pad, shard)
    for i, b, off in case["params"]:
        assert dpg.dpg_plan_param(a, i) == (b, off, case["numels"][i])


@pytest.mark.parametrize("seed", range(60))
def test_plan_matches_oracle_random(oracle_lib, seed):
    rng = np.random.Generator(np.random.Philox(1000 + seed))
    n = int(rng.integers(0, 400))
    numels = random_param_list(rng, n, int(rng.choice([10, 1000, 100_000])))
    R = int(rng.integers(1, 65))
    cap = int(rng.choice([1, 2, 16, 64, 4096, 1 << 20, int(rng.integers(1, 1 << 22))]))
    _same_plan(dpg.dpg_plan_buckets(numels, cap, R), oracle_lib.plan_buckets(numels, cap, R))


@pytest.mark.parametrize("name", sorted(CONFIGS))
def test_plan_matches_oracle_configs(oracle_lib, name):
    cfg = CONFIGS[name]
    caps = cfg.cap_sweep or (cfg.cap_bytes,)
    for cap in caps:
        _same_plan(dpg.dpg_plan_buckets(cfg.numels, cap, cfg.R),
                   oracle_lib.plan_buckets(cfg.numels, cap, cfg.R))


def test_plan_bucket_counts_of_workloads():
    # bucket counts of the synthetic workloads at their caps
    got = {name: dpg.dpg_plan_buckets(CONFIGS[name].numels, CONFIGS[name].cap_bytes,
                                      CONFIGS[name].R).n_buckets for name in CONFIGS}
    assert got["tiny"] == 2
    assert got["gpt2"] == 9
    assert got["llama1b"] == 83
    assert got["llama8b16l"] == 67
    cfg = CONFIGS["llama1b"]
    assert [dpg.dpg_plan_buckets(cfg.numels, c, cfg.R).n_buckets for c in cfg.cap_sweep] == [147, 83, 24]


def test_plan_invalid_arguments():
    for numels, cap, R in (([1, 2], 0, 2), ([1, -2], 64, 2), ([4], 64, 0), ([4], 64, 65)):
        with pytest.raises(dpg.DpgError) as e:
            dpg.dpg_plan_buckets(numels, cap, R)
        assert e.value.status == dpg.DPG_ERR_INVALID_ARG
    L = dpg.lib()
    assert L.dpg_plan_info(None, None, None, None, None) == dpg.DPG_ERR_INVALID_ARG
    assert b"NULL" in L.dpg_last_error()
    assert L.dpg_plan_buckets(None, 0, 64, 2, None) == dpg.DPG_ERR_INVALID_ARG
    with pytest.raises(dpg.DpgError):
        dpg.dpg_plan_bucket(dpg.dpg_plan_buckets([8], 64, 1), 1)


def test_empty_plan():
    p = dpg.dpg_plan_buckets([], 1024, 8)
    assert (p.n_buckets, p.total_padded, p.n_params) == (0, 0, 0)


# ---- validation paths that return before any CUDA call ---------------------
FAKE = 1 << 20          # 16- and 32-byte aligned fake device address


def _rs(plan, **over):
    L = dpg.lib()
    args = dict(grads=[FAKE] * plan.R, dtype=dpg.DPG_BF16, last=None, tokens=[10] * plan.R,
                hp=dpg.HParams(), master=FAKE, m=FAKE, v=FAKE, views=[FAKE], sq=None, nf=None,
                red=None, b0=0, b1=plan.n_buckets)
    args.update(over)
    tok = np.asarray(args["tokens"], np.int64)
    hp = args["hp"].c() if args["hp"] is not None else None
    return L.dpg_reduce_scatter_adam(
        plan.handle, dpg._ptrs(args["grads"]), args["dtype"],
        None if args["last"] is None else dpg._ptrs(args["last"]),
        tok.ctypes.data if tok.size else None, tok.size,
        ctypes.byref(hp) if hp is not None else None, args["master"], args["m"], args["v"],
        dpg._ptrs(args["views"]), len(args["views"]), args["sq"], args["nf"], args["red"],
        args["b0"], args["b1"], None)


def test_reduce_scatter_adam_validation():
    plan = dpg.dpg_plan_buckets([64, 32, 320], 2048, 4)
    E = dpg
    assert _rs(plan, tokens=[0, 0, 0, 0]) == E.DPG_ERR_ZERO_TOKENS
    assert _rs(plan, tokens=[5, -1, 0, 0]) == E.DPG_ERR_INVALID_ARG
    assert _rs(plan, tokens=[]) == E.DPG_ERR_INVALID_ARG
    assert _rs(plan, b0=1, b1=0) == E.DPG_ERR_INVALID_ARG
    assert _rs(plan, b1=plan.n_buckets + 1) == E.DPG_ERR_INVALID_ARG
    assert _rs(plan, dtype=7) == E.DPG_ERR_INVALID_ARG
    assert _rs(plan, last=[FAKE] * 4) == E.DPG_ERR_INVALID_ARG       # needs fp32 grads
    assert _rs(plan, hp=dpg.HParams(step=0)) == E.DPG_ERR_INVALID_ARG
    assert _rs(plan, hp=dpg.HParams(beta1=1.0)) == E.DPG_ERR_INVALID_ARG
    assert _rs(plan, hp=None) == E.DPG_ERR_INVALID_ARG
    assert _rs(plan, grads=[FAKE, FAKE, 0, FAKE]) == E.DPG_ERR_INVALID_ARG
    assert _rs(plan, grads=[FAKE, FAKE + 2, FAKE, FAKE]) == E.DPG_ERR_MISALIGNED
    assert _rs(plan, dtype=dpg.DPG_F32, grads=[FAKE, FAKE + 16, FAKE, FAKE]) == E.DPG_ERR_MISALIGNED
    assert _rs(plan, master=FAKE + 16) == E.DPG_ERR_MISALIGNED
    assert _rs(plan, views=[FAKE + 8]) == E.DPG_ERR_MISALIGNED
    assert _rs(plan, views=[0]) == E.DPG_ERR_INVALID_ARG
    assert _rs(plan, master=None) == E.DPG_ERR_INVALID_ARG
    # an empty bucket range is a valid no-op and issues no device work
    assert _rs(plan, b0=1, b1=1) == E.DPG_OK
    assert dpg.lib().dpg_last_error() == b""


def _rs_ready(plan, events, **over):
    L = dpg.lib()
    args = dict(grads=[FAKE] * plan.R, tokens=[10] * plan.R, hp=dpg.HParams(), master=FAKE,
                b0=0, b1=plan.n_buckets)
    args.update(over)
    tok = np.asarray(args["tokens"], np.int64)
    hp = args["hp"].c()
    evs = None if events is None else (ctypes.c_void_p * max(1, len(events)))(*events)
    return L.dpg_reduce_scatter_adam_when_ready(
        plan.handle, dpg._ptrs(args["grads"]), dpg.DPG_BF16, None, tok.ctypes.data, tok.size,
        ctypes.byref(hp), args["master"], FAKE, FAKE, dpg._ptrs([FAKE]), 1, None, None, None,
        args["b0"], args["b1"], evs, None)


def test_when_ready_validation():
    """The event-gated per-bucket update checks its events, then every other
    argument over the whole range, before it gives the stream any work."""
    plan = dpg.dpg_plan_buckets([64, 32, 320], 2048, 4)
    nb = plan.n_buckets
    E = dpg
    assert _rs_ready(plan, None) == E.DPG_ERR_INVALID_ARG
    assert _rs_ready(plan, [FAKE] * (nb - 1) + [0]) == E.DPG_ERR_INVALID_ARG
    assert _rs_ready(plan, [FAKE] * nb, tokens=[0] * 4) == E.DPG_ERR_ZERO_TOKENS
    assert _rs_ready(plan, [FAKE] * nb, master=FAKE + 16) == E.DPG_ERR_MISALIGNED
    assert _rs_ready(plan, [FAKE] * nb, grads=[FAKE, 0, FAKE, FAKE]) == E.DPG_ERR_INVALID_ARG
    assert _rs_ready(plan, [FAKE] * nb, b0=2, b1=1) == E.DPG_ERR_INVALID_ARG
    # an empty range needs no events and issues nothing
    assert _rs_ready(plan, None, b0=1, b1=1) == E.DPG_OK
    assert dpg.lib().dpg_reduce_scatter_adam_when_ready(
        None, None, 0, None, None, 0, None, None, None, None, None, 0, None, None, None, 0, 0,
        None, None) == E.DPG_ERR_INVALID_ARG


def test_step_deferred_validation():
    """Deferred accumulation checks K, R*K and every microbatch pointer before
    any device work."""
    plan = dpg.dpg_plan_buckets([64, 32, 320], 2048, 4)
    L = dpg.lib()
    hp = dpg.HParams().c()

    def call(micro, K, tokens=None):
        tok = np.asarray(tokens if tokens is not None else [10] * (4 * max(K, 1)), np.int64)
        return L.dpg_step_deferred(plan.handle, None if micro is None else dpg._ptrs(micro), K,
                                   tok.ctypes.data, tok.size, ctypes.byref(hp), FAKE, FAKE, FAKE,
                                   dpg._ptrs([FAKE]), 1, None, None, None)

    E = dpg
    assert call([FAKE] * 4, 0) == E.DPG_ERR_INVALID_ARG
    assert call([FAKE] * 68, 17) == E.DPG_ERR_INVALID_ARG          # R*K > 64
    assert call(None, 2) == E.DPG_ERR_INVALID_ARG
    assert call([FAKE] * 7 + [0], 2) == E.DPG_ERR_INVALID_ARG       # a later microbatch NULL
    assert call([FAKE] * 7 + [FAKE + 2], 2) == E.DPG_ERR_MISALIGNED
    assert call([FAKE] * 8, 2, tokens=[0] * 8) == E.DPG_ERR_ZERO_TOKENS
    assert L.dpg_step_deferred(None, None, 1, None, 0, None, None, None, None, None, 0, None,
                               None, None) == E.DPG_ERR_INVALID_ARG


def test_other_entry_points_validation():
    L = dpg.lib()
    plan = dpg.dpg_plan_buckets([64, 32, 320], 2048, 4)
    assert L.dpg_accumulate(plan.handle, None, FAKE, 1, None) == dpg.DPG_ERR_INVALID_ARG
    assert L.dpg_accumulate(plan.handle, FAKE + 2, FAKE, 1, None) == dpg.DPG_ERR_MISALIGNED
    assert L.dpg_accumulate(plan.handle, FAKE, FAKE + 16, 0, None) == dpg.DPG_ERR_MISALIGNED
    assert L.dpg_allgather_params(plan.handle, FAKE, dpg._ptrs([FAKE]), 1, 0, 3, None) == dpg.DPG_ERR_INVALID_ARG
    assert L.dpg_allgather_params(plan.handle, FAKE, dpg._ptrs([FAKE]), 65, 0, 1, None) == dpg.DPG_ERR_INVALID_ARG
    assert L.dpg_allgather_params(plan.handle, FAKE + 4, dpg._ptrs([FAKE]), 1, 0, 1, None) == dpg.DPG_ERR_MISALIGNED
    assert L.dpg_allgather_params(plan.handle, FAKE, dpg._ptrs([FAKE]), 1, 1, 1, None) == dpg.DPG_OK
    assert L.dpg_set_fused_max_ctas(-1) == dpg.DPG_ERR_INVALID_ARG
    assert L.dpg_set_fused_max_ctas(0) == dpg.DPG_OK
    assert L.dpg_set_programmatic_launch(2) == dpg.DPG_ERR_INVALID_ARG
    assert L.dpg_set_programmatic_launch(-1) == dpg.DPG_ERR_INVALID_ARG
    assert L.dpg_set_programmatic_launch(0) == dpg.DPG_OK
    assert L.dpg_set_programmatic_launch(1) == dpg.DPG_OK
    A2 = L.dpg_accumulate_pair
    assert A2(None, FAKE, FAKE, FAKE, 1, None) == dpg.DPG_ERR_INVALID_ARG
    assert A2(plan.handle, FAKE, None, FAKE, 1, None) == dpg.DPG_ERR_INVALID_ARG
    assert A2(plan.handle, FAKE, FAKE + 2, FAKE, 1, None) == dpg.DPG_ERR_MISALIGNED
    assert A2(plan.handle, FAKE, FAKE, FAKE + 16, 0, None) == dpg.DPG_ERR_MISALIGNED
    F2 = L.dpg_step_fold2
    tok = (ctypes.c_int64 * 4)(100, 80, 120, 60)
    hp = dpg.HParams().c()
    four = dpg._ptrs([FAKE] * 4)
    assert F2(plan.handle, four, None, four, tok, 4, ctypes.byref(hp), FAKE, FAKE, FAKE, None, 0,
              None, None, None) == dpg.DPG_ERR_INVALID_ARG
    assert F2(plan.handle, four, four, None, tok, 4, ctypes.byref(hp), FAKE, FAKE, FAKE, None, 0,
              None, None, None) == dpg.DPG_ERR_INVALID_ARG
    assert F2(plan.handle, four, four, dpg._ptrs([FAKE, FAKE, FAKE, FAKE + 2]), tok, 4,
              ctypes.byref(hp), FAKE, FAKE, FAKE, None, 0, None, None,
              None) == dpg.DPG_ERR_MISALIGNED
    assert F2(plan.handle, four, four, dpg._ptrs([FAKE, 0, FAKE, FAKE]), tok, 4,
              ctypes.byref(hp), FAKE, FAKE, FAKE, None, 0, None, None,
              None) == dpg.DPG_ERR_INVALID_ARG
    zero = (ctypes.c_int64 * 4)(0, 0, 0, 0)
    assert F2(plan.handle, four, four, four, zero, 4, ctypes.byref(hp), FAKE, FAKE, FAKE, None, 0,
              None, None, None) == dpg.DPG_ERR_ZERO_TOKENS
    G = L.dpg_gather_params_bf16
    assert G(None, FAKE, dpg._ptrs([FAKE]), 1, 0, 1, None) == dpg.DPG_ERR_INVALID_ARG
    assert G(plan.handle, FAKE, dpg._ptrs([FAKE]), 1, 0, 3, None) == dpg.DPG_ERR_INVALID_ARG
    assert G(plan.handle, FAKE, dpg._ptrs([FAKE]), 1, 1, 0, None) == dpg.DPG_ERR_INVALID_ARG
    assert G(plan.handle, FAKE, dpg._ptrs([FAKE]), 65, 0, 1, None) == dpg.DPG_ERR_INVALID_ARG
    assert G(plan.handle, None, dpg._ptrs([FAKE]), 1, 0, 1, None) == dpg.DPG_ERR_INVALID_ARG
    assert G(plan.handle, FAKE, dpg._ptrs([0]), 1, 0, 1, None) == dpg.DPG_ERR_INVALID_ARG
    assert G(plan.handle, FAKE + 2, dpg._ptrs([FAKE]), 1, 0, 1, None) == dpg.DPG_ERR_MISALIGNED
    assert G(plan.handle, FAKE, dpg._ptrs([FAKE, FAKE + 8]), 2, 0, 1, None) == dpg.DPG_ERR_MISALIGNED
    assert G(plan.handle, FAKE, dpg._ptrs([FAKE]), 1, 1, 1, None) == dpg.DPG_OK
    assert G(plan.handle, None, None, 0, 0, 1, None) == dpg.DPG_OK
    assert L.dpg_pack(plan.handle, dpg._ptrs([FAKE, 0, FAKE]), FAKE, None) == dpg.DPG_ERR_INVALID_ARG
    assert L.dpg_pack(plan.handle, dpg._ptrs([FAKE, FAKE + 1, FAKE]), FAKE, None) == dpg.DPG_ERR_MISALIGNED
    assert L.dpg_pack(plan.handle, dpg._ptrs([FAKE] * 3), FAKE + 8, None) == dpg.DPG_ERR_MISALIGNED
    assert L.dpg_step(None, None, 0, None, None, 0, None, None, None, None, None, 0, None, None,
                      None) == dpg.DPG_ERR_INVALID_ARG


def test_state_export_import_validation():
    L = dpg.lib()
    plan = dpg.dpg_plan_buckets([64, 32, 320], 2048, 4)
    two = dpg._ptrs([FAKE, FAKE])
    assert L.dpg_export_state(plan.handle, two, two, 0, None) == dpg.DPG_ERR_INVALID_ARG
    assert L.dpg_export_state(plan.handle, two, two, 9, None) == dpg.DPG_ERR_INVALID_ARG
    assert L.dpg_export_state(plan.handle, None, two, 1, None) == dpg.DPG_ERR_INVALID_ARG
    assert L.dpg_export_state(plan.handle, dpg._ptrs([0]), two, 1, None) == dpg.DPG_ERR_INVALID_ARG
    assert L.dpg_export_state(plan.handle, dpg._ptrs([FAKE + 16]), two, 1, None) == dpg.DPG_ERR_MISALIGNED
    assert L.dpg_import_state(plan.handle, dpg._ptrs([FAKE + 2]), two, 1, None) == dpg.DPG_ERR_MISALIGNED
    assert plan.canon_total == 416
    # an empty plan has nothing to copy
    empty = dpg.dpg_plan_buckets([], 1024, 2)
    assert L.dpg_import_state(empty.handle, dpg._ptrs([0]), dpg._ptrs([0]), 1, None) == dpg.DPG_OK


def test_staged_fault_hook_needs_opt_in(monkeypatch):
    # a production process (no DPG_TEST_HOOKS=1) cannot arm the test hook
    for val in (None, "0", "yes"):
        if val is None:
            monkeypatch.delenv("DPG_TEST_HOOKS", raising=False)
        else:
            monkeypatch.setenv("DPG_TEST_HOOKS", val)
        with pytest.raises(dpg.DpgError) as e:
            dpg.dpg_set_staged_fault(skip_unit=3, timeout_ns=1)
        assert e.value.status == dpg.DPG_ERR_INVALID_ARG
        assert "DPG_TEST_HOOKS" in str(e.value)
    monkeypatch.setenv("DPG_TEST_HOOKS", "1")
    dpg.dpg_set_staged_fault(skip_unit=3, timeout_ns=1)
    dpg.dpg_set_staged_fault(skip_unit=-1, timeout_ns=0)   # disarm again


def test_shard_plan_layout():
    # one bucket per bucket of the global plan, holding its shard, padded to 8R
    for name in ("tiny", "gpt2", "sweep"):
        c = CONFIGS[name]
        g = dpg.dpg_plan_buckets(c.numels, c.cap_bytes, c.R)
        s = dpg.dpg_plan_shards(g)
        assert (s.n_buckets, s.R, s.n_params) == (g.n_buckets, g.R, g.n_buckets)
        np.testing.assert_array_equal(s.numels[::-1], g.shard_numel)
        np.testing.assert_array_equal(s.param_bucket, np.arange(g.n_buckets)[::-1])
        np.testing.assert_array_equal(s.param_offset[::-1], s.bucket_offset)
        assert np.all(s.bucket_padded % (8 * g.R) == 0)
        assert np.all((s.bucket_padded >= g.shard_numel) & (s.bucket_padded - g.shard_numel < 8 * g.R))
        assert s.total_padded == int(s.bucket_padded.sum())
    # the tiny case worked by hand: shards of 88 and 512 elements, R = 4
    t = CONFIGS["tiny"]
    s = dpg.dpg_plan_shards(dpg.dpg_plan_buckets(t.numels, t.cap_bytes, t.R))
    np.testing.assert_array_equal(s.bucket_offset, [0, 96])
    np.testing.assert_array_equal(s.bucket_padded, [96, 512])
    # an empty plan has an empty shard plan
    e = dpg.dpg_plan_shards(dpg.dpg_plan_buckets([], 1024, 2))
    assert e.n_buckets == 0 and e.total_padded == 0


def test_shard_plan_validation():
    L = dpg.lib()
    out = ctypes.c_void_p()
    assert L.dpg_plan_shards(None, ctypes.byref(out)) == dpg.DPG_ERR_INVALID_ARG
    g = dpg.dpg_plan_buckets([100], 1024, 2)
    assert L.dpg_plan_shards(g.handle, None) == dpg.DPG_ERR_INVALID_ARG
    # zero-size parameters only: one empty bucket, and one empty shard
    z = dpg.dpg_plan_buckets([0, 0], 1024, 2)
    assert z.n_buckets == 1 and z.total_padded == 0
    zs = dpg.dpg_plan_shards(z)
    assert zs.n_buckets == 1 and zs.total_padded == 0


def test_release_library_has_no_index_checks(monkeypatch):
    plan = dpg.dpg_plan_buckets([1000], 4096, 2)
    assert dpg.dpg_debug_checks(plan) == (False, 0)
    monkeypatch.setenv("DPG_TEST_HOOKS", "1")
    with pytest.raises(dpg.DpgError) as e:
        dpg.dpg_debug_set_limit(8)
    assert e.value.status == dpg.DPG_ERR_INVALID_ARG and "--debug" in str(e.value)
    L = dpg.lib()
    assert L.dpg_debug_checks(None, None, None) == dpg.DPG_ERR_INVALID_ARG
