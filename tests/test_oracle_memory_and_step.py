"""Pins for the oracle's model-state accounting (numbers printed on the pages,
tests/golden/memory_accounting.txt) and for the composition of the whole step
(the oracle's step equals its own pieces run in the order the pages give:
reduce-scatter, owner-local Adam, all-gather)."""
import os
import shlex

import numpy as np
import pytest

from workloads import CONFIGS

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "memory_accounting.txt")


def golden():
    out = {}
    for line in open(GOLDEN):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        tok = shlex.split(line)
        out[tok[0]] = float(tok[1])
    return out


def test_sixteen_bytes_per_parameter(oracle_lib):
    g = golden()
    assert g["bytes_param"] + g["bytes_grad"] + g["bytes_master_m_v"] == g["bytes_per_param_ddp"]
    assert g["bytes_master_m_v"] - 4 == g["bytes_moments_only"]
    assert oracle_lib.model_state_bytes(0, 1.0, 1) == g["bytes_per_param_ddp"]
    for N in (1, 2, 8, 64):
        assert oracle_lib.model_state_bytes(0, 1.0, N) == g["bytes_per_param_ddp"]


def test_seven_and_a_half_billion_needs_120_gb(oracle_lib):
    g = golden()
    assert oracle_lib.model_state_bytes(0, 7.5e9, 64) / 1e9 == pytest.approx(g["ddp_7p5b_gb"])


def test_zero_stage_reductions_tend_to_page_factors(oracle_lib):
    g = golden()
    psi = 7.5e9
    ddp = oracle_lib.model_state_bytes(0, psi, 1)
    big = 1 << 20
    assert ddp / oracle_lib.model_state_bytes(1, psi, big) == pytest.approx(g["zero1_reduction"], rel=1e-4)
    assert ddp / oracle_lib.model_state_bytes(2, psi, big) == pytest.approx(g["zero2_reduction"], rel=1e-4)
    # ZeRO-3 falls linearly with N
    for N in (2, 8, 64):
        assert oracle_lib.model_state_bytes(3, psi, N) * N == pytest.approx(ddp)
    # stages never increase memory; N = 1 is plain DP for every stage
    for N in (1, 2, 4, 64):
        vals = [oracle_lib.model_state_bytes(s, psi, N) for s in range(4)]
        assert vals == sorted(vals, reverse=True)
    for s in range(4):
        assert oracle_lib.model_state_bytes(s, psi, 1) == ddp


def test_step_equals_its_pieces(oracle_lib):
    cfg = CONFIGS["tiny"]
    rng = np.random.Generator(np.random.Philox(8))
    p = oracle_lib.plan_buckets(cfg.numels, cfg.cap_bytes, cfg.R)
    grads = [oracle_lib.pack(p, [oracle_lib.f32_to_bf16((rng.standard_normal(int(k)) * 1e-2)
                                                        .astype(np.float32)) for k in cfg.numels])
             for _ in range(cfg.R)]
    tokens = list(cfg.fixed_tokens)
    w0 = (rng.standard_normal(p.total_padded) * 0.02).astype(np.float32)
    w, m, v = w0.copy(), np.zeros_like(w0), np.zeros_like(w0)
    views, red, sq = oracle_lib.step(p.bucket_offset, p.bucket_padded, grads, tokens, w, m, v,
                                     n_views=cfg.R, want_reduced=True)
    c = oracle_lib.grad_scale(tokens)
    g = oracle_lib.reduce(grads, c)
    np.testing.assert_array_equal(red.view(np.uint32), g.view(np.uint32))
    w2, m2, v2 = w0.copy(), np.zeros_like(w0), np.zeros_like(w0)
    oracle_lib.adam(g, w2, m2, v2, t=1)
    np.testing.assert_array_equal(w.view(np.uint32), w2.view(np.uint32))
    for vw in views:
        np.testing.assert_array_equal(vw, oracle_lib.f32_to_bf16(w2))
    for b in range(p.n_buckets):
        lo, hi = p.bucket_offset[b], p.bucket_offset[b] + p.bucket_padded[b]
        assert sq[b] == pytest.approx(float(np.sum(g[lo:hi].astype(np.float64) ** 2)), rel=1e-12)
    # the all-gather alone writes the same views
    for vw in oracle_lib.allgather(w2, 2):
        np.testing.assert_array_equal(vw, views[0])


def test_step_zero_tokens_is_an_error(oracle_lib):
    z = np.zeros(16, np.uint16)
    w = np.zeros(16, np.float32)
    with pytest.raises(oracle_lib.OracleError) as e:
        oracle_lib.step([0], [16], [z, z], [0, 0], w, w.copy(), w.copy())
    assert e.value.status == oracle_lib.EZERO_TOKENS
