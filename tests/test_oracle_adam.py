"""Pins for the oracle's mixed-precision Adam (Kingma & Ba 2015, Algorithm 1;
the pages name Adam with its first/second moments, step counter and fp32
master weight -- "Parallelisms", section "ZeRO-1" -- but print no formula).

* Library routine: torch.optim.Adam / AdamW in binary64 on the same inputs,
  t = 1..10; the binary32 oracle must stay within a derived error bound.
* Closed forms: from m = v = 0 with a constant gradient g, the bias-corrected
  moments are exactly g and g^2 at every t, so each step moves the weight by
  -lr*g/(|g|+eps); for |g| << eps the step is -lr*g/eps (eps outside the
  square root).
* Exact invariants: with eps = 0, scaling g by a power of two leaves every
  update bit-identical; negating g (from a zero weight) negates the result.
"""
import numpy as np
import pytest
import torch

HP = dict(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8)


def torch_adam_trajectory(w0, grads, wd=0.0, **hp):
    w = torch.nn.Parameter(torch.from_numpy(w0.astype(np.float64)))
    cls = torch.optim.AdamW if wd else torch.optim.Adam
    opt = cls([w], lr=hp["lr"], betas=(hp["beta1"], hp["beta2"]), eps=hp["eps"],
              weight_decay=wd, foreach=False)
    out = []
    for g in grads:
        w.grad = torch.from_numpy(g.astype(np.float64))
        opt.step()
        st = opt.state[w]
        out.append((w.detach().numpy().copy(), st["exp_avg"].numpy().copy(),
                    st["exp_avg_sq"].numpy().copy()))
    return out


HP_SETS = {
    "default": HP,
    "small_betas_large_lr": dict(lr=5e-2, beta1=0.5, beta2=0.9, eps=1e-6),
    "high_beta1": dict(lr=3e-4, beta1=0.95, beta2=0.98, eps=1e-6),
}


@pytest.mark.parametrize("hp_name", sorted(HP_SETS))
@pytest.mark.parametrize("wd", [0.0, 0.1])
def test_matches_torch_adam_binary64(oracle_lib, wd, hp_name):
    hp = HP_SETS[hp_name]
    rng = np.random.Generator(np.random.Philox(42))
    n, T = 20_000, 10
    w0 = (rng.standard_normal(n) * 0.02).astype(np.float32)
    # magnitudes from 1e-9 (around eps) to 1e-1
    mag = 10.0 ** rng.uniform(-9, -1, n)
    grads = [(rng.standard_normal(n) * mag).astype(np.float32) for _ in range(T)]
    ref = torch_adam_trajectory(w0, grads, wd=wd, **hp)
    w, m, v = w0.copy(), np.zeros(n, np.float32), np.zeros(n, np.float32)
    m_mag = np.zeros(n)      # sum of |terms| of the m recurrence (cancellation-free)
    # |u| = |m_hat| / (sqrt(v_hat) + eps) <= (1-b1)/sqrt(1-b2) when b1^2 < b2
    # (Kingma & Ba, the bound on the effective step)
    assert hp["beta1"] ** 2 < hp["beta2"]
    ub = (1 - hp["beta1"]) / np.sqrt(1 - hp["beta2"])
    for t, g in enumerate(grads, start=1):
        oracle_lib.adam(g, w, m, v, wd=wd, t=t, **hp)
        rw, rm, rv = ref[t - 1]
        m_mag = hp["beta1"] * m_mag + (1 - hp["beta1"]) * np.abs(g.astype(np.float64))
        # m, v: chains of binary32 multiply-adds; error a few t * 2^-24 of the
        # magnitude of the terms (v has only non-negative terms)
        assert np.all(np.abs(m - rm) <= 4 * t * 2.0 ** -24 * m_mag + 1e-45)
        np.testing.assert_allclose(v, rv, rtol=4 * t * 2.0 ** -24, atol=1e-45)
        # weight: one rounding of the weight per step (half an ulp of the
        # largest |w| reached; two with decoupled decay, whose subtraction
        # rounds w once more) plus lr * |u| * (relative error of u)
        wmax = np.float32(np.max(np.abs(w0)) + t * hp["lr"] * ub)
        roundings = 2 if wd else 1
        bound = t * (0.5 * roundings * np.spacing(wmax) + hp["lr"] * ub * 64 * t * 2.0 ** -24)
        assert np.max(np.abs(w.astype(np.float64) - rw)) <= bound


def test_first_step_closed_form(oracle_lib):
    rng = np.random.Generator(np.random.Philox(1))
    g = (rng.standard_normal(10_000) * 10.0 ** rng.uniform(-6, 0, 10_000)).astype(np.float32)
    w = np.zeros_like(g)
    m, v = np.zeros_like(g), np.zeros_like(g)
    oracle_lib.adam(g, w, m, v, t=1, **HP)
    gd = g.astype(np.float64)
    expect = -HP["lr"] * gd / (np.abs(gd) + HP["eps"])
    np.testing.assert_allclose(w, expect, rtol=1e-5)
    np.testing.assert_allclose(m, 0.1 * gd, rtol=1e-6)
    np.testing.assert_allclose(v, 0.001 * gd * gd, rtol=1e-6)


def test_constant_gradient_closed_form(oracle_lib):
    # bias correction makes m_hat = g and v_hat = g^2 at every step
    g = np.array([1e-3, -2e-3, 5e-5, 0.3, -7e-7], np.float32)
    w0 = np.array([0.01, -0.02, 0.0, 0.5, 0.03], np.float32)
    w, m, v = w0.copy(), np.zeros_like(g), np.zeros_like(g)
    T = 50
    for t in range(1, T + 1):
        oracle_lib.adam(g, w, m, v, t=t, **HP)
        gd = g.astype(np.float64)
        expect = w0.astype(np.float64) - t * HP["lr"] * gd / (np.abs(gd) + HP["eps"])
        np.testing.assert_allclose(w, expect, rtol=0, atol=t * 2e-8 + 1e-6 * t * HP["lr"])


def test_eps_sits_outside_the_square_root(oracle_lib):
    g = np.array([1e-12, -3e-13], np.float32)
    w, m, v = np.zeros_like(g), np.zeros_like(g), np.zeros_like(g)
    oracle_lib.adam(g, w, m, v, t=1, **HP)
    gd = g.astype(np.float64)
    expect = -HP["lr"] * gd / (np.abs(gd) + HP["eps"])       # ~ -lr * g / eps
    np.testing.assert_allclose(w, expect, rtol=1e-5)
    inside = -HP["lr"] * gd / np.sqrt(gd * gd + HP["eps"])    # the other reading
    assert np.all(np.abs(w - inside) > 100 * np.abs(expect - inside) * 1e-5)


@pytest.mark.parametrize("k", [-20, -3, 1, 7])
def test_power_of_two_scale_invariance_without_eps(oracle_lib, k):
    rng = np.random.Generator(np.random.Philox(2))
    n = 5000
    g1s = [(rng.standard_normal(n) * 1e-3).astype(np.float32) for _ in range(4)]
    hp = dict(HP, eps=0.0)
    w0 = (rng.standard_normal(n) * 0.02).astype(np.float32)
    outs = []
    for s in (1.0, 2.0 ** k):
        w, m, v = w0.copy(), np.zeros(n, np.float32), np.zeros(n, np.float32)
        for t, g in enumerate(g1s, start=1):
            oracle_lib.adam((g * np.float32(s)).astype(np.float32), w, m, v, t=t, **hp)
        outs.append(w)
    np.testing.assert_array_equal(outs[0].view(np.uint32), outs[1].view(np.uint32))


def test_sign_symmetry(oracle_lib):
    rng = np.random.Generator(np.random.Philox(3))
    g = (rng.standard_normal(3000) * 1e-3).astype(np.float32)
    res = []
    for s in (1, -1):
        w, m, v = np.zeros_like(g), np.zeros_like(g), np.zeros_like(g)
        for t in range(1, 4):
            oracle_lib.adam(g * np.float32(s), w, m, v, t=t, **HP)
        res.append(w)
    np.testing.assert_array_equal(res[0], -res[1])


def test_zero_gradient_leaves_state(oracle_lib):
    w0 = np.array([0.5, -0.25, 0.0], np.float32)
    w, m, v = w0.copy(), np.zeros(3, np.float32), np.zeros(3, np.float32)
    oracle_lib.adam(np.zeros(3, np.float32), w, m, v, t=1, **HP)
    np.testing.assert_array_equal(w, w0)
    assert not m.any() and not v.any()


def test_invalid_step_and_betas(oracle_lib):
    z = np.zeros(1, np.float32)
    with pytest.raises(oracle_lib.OracleError):
        oracle_lib.adam(z, z.copy(), z.copy(), z.copy(), t=0, **HP)
    with pytest.raises(oracle_lib.OracleError):
        oracle_lib.adam(z, z.copy(), z.copy(), z.copy(), t=1, lr=1e-3, beta1=1.0,
                        beta2=0.999, eps=1e-8)
