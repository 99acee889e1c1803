"""Pin for the token normalisation: a data-parallel step that scales each
rank's local SUMMED loss by R/G and averages over R ranks must give the
gradient of the single-device MEAN loss over all G valid tokens
("Distributed Training and Parallelism", section "Data parallelism and the
global gradient": unequal valid-token counts need an explicit normalisation;
matching a single-device update needs matching loss normalisation).

Toy model: linear least squares in binary64 with per-token losses
l_i = 0.5 (w.x_i - y_i)^2 on R = 4 ranks holding 100, 80, 120 and 60 tokens.
The oracle's reduce + scale, fed each rank's summed-loss gradient, must match
the single-device mean-loss gradient; averaging per-rank MEAN gradients (the
naive rule) must not.
"""
import numpy as np
import pytest


def toy_problem(seed=3, d=64, tokens=(100, 80, 120, 60)):
    rng = np.random.Generator(np.random.Philox(seed))
    w = rng.standard_normal(d)
    xs = [rng.standard_normal((t, d)) for t in tokens]
    ys = [x @ rng.standard_normal(d) + 0.1 * rng.standard_normal(len(x)) for x in xs]
    return w, xs, ys


def summed_loss_grad(w, x, y):
    return x.T @ (x @ w - y)            # d/dw sum_i 0.5 (w.x_i - y_i)^2


def test_dp_normalisation_equals_single_device_mean(oracle_lib):
    tokens = (100, 80, 120, 60)
    w, xs, ys = toy_problem(tokens=tokens)
    G = sum(tokens)
    x_all, y_all = np.concatenate(xs), np.concatenate(ys)
    single = summed_loss_grad(w, x_all, y_all) / G        # mean over all tokens

    local = [summed_loss_grad(w, x, y) for x, y in zip(xs, ys)]
    c = oracle_lib.grad_scale(list(tokens))
    dp = oracle_lib.reduce([g.astype(np.float32) for g in local], c).astype(np.float64)
    # fp32 inputs, R-1 additions and one multiply: relative error a few 2^-24
    # of the summed magnitudes
    mag = np.sum([np.abs(g) for g in local], axis=0) / G
    assert np.all(np.abs(dp - single) <= 8 * 2.0 ** -24 * mag + 1e-30)

    # negative control: averaging each rank's mean gradient is NOT the same
    naive = np.mean([g / t for g, t in zip(local, tokens)], axis=0)
    assert np.max(np.abs(naive - single)) > 1e3 * np.max(8 * 2.0 ** -24 * mag)


def test_accumulated_microbatches_count_every_token(oracle_lib):
    # two microbatches per rank: G is the sum over ranks AND microbatches
    tokens = (100, 80, 120, 60, 90, 70, 110, 50)   # rank-major, K = 2
    w, xs, ys = toy_problem(seed=4, tokens=tokens)
    single = summed_loss_grad(w, np.concatenate(xs), np.concatenate(ys)) / sum(tokens)
    R, K = 4, 2
    accs = []
    for r in range(R):
        acc = sum(summed_loss_grad(w, xs[r * K + k], ys[r * K + k]) for k in range(K))
        accs.append(acc.astype(np.float32))
    c = oracle_lib.grad_scale(list(tokens))
    dp = oracle_lib.reduce(accs, c).astype(np.float64)
    mag = np.sum([np.abs(a.astype(np.float64)) for a in accs], axis=0) / sum(tokens)
    assert np.all(np.abs(dp - single) <= 8 * 2.0 ** -24 * mag + 1e-30)
    # scaling each microbatch by its own count would be wrong
    wrong = sum(summed_loss_grad(w, xs[i], ys[i]) / tokens[i] for i in range(R * K)) / (R * K)
    assert np.max(np.abs(wrong - single)) > 1e-4 * np.max(np.abs(single))
