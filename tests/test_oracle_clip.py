"""Pins for the oracle's global gradient-norm clipping ("Parallelisms",
section ZeRO-2: the norm over all gradient shards is needed before any weight
is updated).  Library routine: torch.nn.utils.clip_grad_norm_ in binary64 on
the same values (same coefficient convention, max_norm / (norm + 1e-6)
clamped to 1); closed forms: no change below the threshold, clipped norm
equal to max_norm, direction preserved; non-finite norms."""
import numpy as np
import pytest
import torch


def torch_clip(g64, max_norm):
    t = torch.nn.Parameter(torch.zeros(g64.size, dtype=torch.float64))
    t.grad = torch.from_numpy(g64.copy())
    norm = torch.nn.utils.clip_grad_norm_([t], max_norm, foreach=False)
    return float(norm), t.grad.numpy()


@pytest.mark.parametrize("max_norm", [1e-6, 1e-3, 0.05, 1.0, 1e6])
def test_matches_torch_clip_grad_norm(oracle_lib, max_norm):
    rng = np.random.Generator(np.random.Philox(17))
    g = (rng.standard_normal(200_000) * 10.0 ** rng.uniform(-5, -2, 200_000)).astype(np.float32)
    norm, coef = oracle_lib.clip_coef(g, max_norm)
    t_norm, t_grad = torch_clip(g.astype(np.float64), max_norm)
    assert norm == pytest.approx(t_norm, rel=1e-12)
    ours = oracle_lib.scale(g, coef).astype(np.float64)
    # fp32 coefficient (half an ulp) and one fp32 multiply (half an ulp)
    assert np.all(np.abs(ours - t_grad) <= 2.0 ** -23 * np.abs(t_grad) + 1e-45)


def test_below_threshold_is_the_identity(oracle_lib):
    g = np.array([3e-3, -4e-3, 0.0, 1e-9], np.float32)      # norm 5e-3
    norm, coef = oracle_lib.clip_coef(g, 0.0051)
    assert coef == np.float32(1.0)
    np.testing.assert_array_equal(oracle_lib.scale(g, coef), g)
    assert norm == pytest.approx(5e-3, rel=1e-7)


def test_clipped_norm_and_direction(oracle_lib):
    rng = np.random.Generator(np.random.Philox(3))
    g = rng.standard_normal(10_000).astype(np.float32)
    norm, coef = oracle_lib.clip_coef(g, 2.5)
    assert norm == pytest.approx(float(np.linalg.norm(g.astype(np.float64))), rel=1e-12)
    c = oracle_lib.scale(g, coef)
    assert float(np.linalg.norm(c.astype(np.float64))) == pytest.approx(2.5, rel=1e-6)
    np.testing.assert_array_equal(np.sign(c), np.sign(g))


def test_non_finite_norms(oracle_lib):
    _, coef = oracle_lib.clip_coef(np.array([1.0, np.inf], np.float32), 1.0)
    assert coef == 0.0
    _, coef = oracle_lib.clip_coef(np.array([1.0, np.nan], np.float32), 1.0)
    assert np.isnan(coef)
    norm, coef = oracle_lib.clip_coef(np.zeros(8, np.float32), 1.0)
    assert norm == 0.0 and coef == 1.0
