"""Pins for the oracle's reduction, normalisation scale and accumulation.

* Reduce-scatter followed by all-gather equals all-reduce, bit for bit
  ("Parallelism Starts With the Bottleneck", section "Allreduce equals
  reducescatter plus allgather"; "Parallelisms", section "ZeRO-1").
* The rank-ordered fp32 sum stays within the forward-error bound of recursive
  summation of the exact sum (the bf16 inputs sum exactly in binary64).
* For two replicas the fp32 sum is the correctly rounded exact sum: numpy's
  binary64 -> binary32 conversion (IEEE round-to-nearest) is the library pin.
* The scale is fp32(1/G), checked against exact rational arithmetic.
* Accumulation over microbatches equals sequential binary32 addition, checked
  against the exact sum and the recursive-summation error bound.
"""
from fractions import Fraction

import numpy as np
import pytest
import torch


def rand_bf16(rng, n, std, oracle_lib):
    x = (rng.standard_normal(n) * std).astype(np.float32)
    return oracle_lib.f32_to_bf16(x)


@pytest.mark.parametrize("R", [1, 2, 3, 4, 8, 16])
def test_reduce_scatter_then_allgather_equals_allreduce(oracle_lib, R):
    rng = np.random.Generator(np.random.Philox(R))
    numels = [1000, 37, 4096, 5, 700]
    p = oracle_lib.plan_buckets(numels, 6000, R)
    grads = [oracle_lib.pack(p, [rand_bf16(rng, k, 1e-2, oracle_lib) for k in numels])
             for _ in range(R)]
    scale = oracle_lib.grad_scale([int(x) for x in rng.integers(1, 5000, R)])
    ar = oracle_lib.allreduce(grads, scale)
    # reduce-scatter: owner r reduces only its shard of each bucket ...
    owned = {}
    for b in range(p.n_buckets):
        sh = p.bucket_padded[b] // R
        for r in range(R):
            lo = p.bucket_offset[b] + r * sh
            owned[(b, r)] = oracle_lib.reduce(grads, scale, lo=lo, hi=lo + sh)
    # ... and all-gather concatenates every owner's shard on every rank
    gathered = np.concatenate([owned[(b, r)] for b in range(p.n_buckets) for r in range(R)])
    for r in range(R):
        np.testing.assert_array_equal(gathered.view(np.uint32), ar[r].view(np.uint32))
    # every rank's all-reduce copy is identical
    for r in range(1, R):
        np.testing.assert_array_equal(ar[0].view(np.uint32), ar[r].view(np.uint32))


@pytest.mark.parametrize("R", [2, 3, 4, 8, 16])
def test_reduce_error_bound_vs_exact_sum(oracle_lib, R):
    rng = np.random.Generator(np.random.Philox(10 + R))
    n = 50_000
    xs = [rand_bf16(rng, n, 10.0 ** rng.uniform(-4, 1), oracle_lib) for _ in range(R)]
    s = oracle_lib.reduce(xs, np.float32(1.0)).astype(np.float64)
    vals = np.stack([oracle_lib.bf16_to_f32(x).astype(np.float64) for x in xs])
    exact = vals.sum(axis=0)       # exact: bf16 values, few terms, binary64
    u = 2.0 ** -24
    bound = (R - 1) * u / (1 - (R - 1) * u) * np.abs(vals).sum(axis=0)
    assert np.all(np.abs(s - exact) <= bound)


def test_two_replicas_is_correctly_rounded_sum(oracle_lib):
    rng = np.random.Generator(np.random.Philox(99))
    n = 200_000
    a = rand_bf16(rng, n, 1.0, oracle_lib)
    # second addend spans many magnitudes so rounding actually happens
    b = oracle_lib.f32_to_bf16((rng.standard_normal(n) * 10.0 ** rng.integers(-6, 6, n))
                               .astype(np.float32))
    s = oracle_lib.reduce([a, b], np.float32(1.0))
    exact = (oracle_lib.bf16_to_f32(a).astype(np.float64)
             + oracle_lib.bf16_to_f32(b).astype(np.float64))
    np.testing.assert_array_equal(s.view(np.uint32), exact.astype(np.float32).view(np.uint32))


def test_reduce_order_is_rank_order(oracle_lib):
    # (1 + 2^-24) + ... : rank order 0..R-1 is observable in binary32
    one = np.float32(1.0)
    tiny = np.float32(2.0 ** -24)
    xs = [np.array([tiny], np.float32), np.array([tiny], np.float32),
          np.array([one], np.float32)]
    s = oracle_lib.reduce(xs, np.float32(1.0))
    # ((2^-24 + 2^-24) + 1) = 1 + 2^-23 exactly; (1 + 2^-24) + 2^-24 would be 1
    assert s[0] == np.float32(1.0 + 2.0 ** -23)
    s2 = oracle_lib.reduce(xs[::-1], np.float32(1.0))
    assert s2[0] == np.float32(1.0)


def test_negative_zero_survives_single_replica_and_sum(oracle_lib):
    nz = oracle_lib.f32_to_bf16(np.array([-0.0], np.float32))
    s = oracle_lib.reduce([nz], np.float32(1.0))
    assert np.signbit(s[0])
    s = oracle_lib.reduce([nz, nz], np.float32(1.0))
    assert np.signbit(s[0])


@pytest.mark.parametrize("tokens", [[100, 80, 120, 60], [1], [3], [7, 7, 7],
                                    [3000, 4096, 3500, 3999, 4001, 3333, 3777, 4000],
                                    [123456789]])
def test_grad_scale_is_rounded_reciprocal(oracle_lib, tokens):
    c = oracle_lib.grad_scale(tokens)
    G = sum(tokens)
    exact = Fraction(1, G)
    cf = Fraction(float(c))
    # c is within half an ulp of 1/G (binary32 round to nearest)
    m, e = np.frexp(np.float32(c))
    ulp = Fraction(2) ** (int(e) - 24)
    assert abs(cf - exact) <= ulp / 2


def test_grad_scale_errors(oracle_lib):
    with pytest.raises(oracle_lib.OracleError) as e:
        oracle_lib.grad_scale([0, 0, 0])
    assert e.value.status == oracle_lib.EZERO_TOKENS
    with pytest.raises(oracle_lib.OracleError):
        oracle_lib.grad_scale([5, -1])
    with pytest.raises(oracle_lib.OracleError):
        oracle_lib.grad_scale([])


@pytest.mark.parametrize("K", [1, 2, 4, 7])
def test_accumulation_bound_and_first(oracle_lib, K):
    rng = np.random.Generator(np.random.Philox(500 + K))
    n = 40_000
    micro = [rand_bf16(rng, n, 10.0 ** rng.uniform(-4, 0), oracle_lib) for _ in range(K)]
    acc = np.full(n, np.nan, dtype=np.float32)
    oracle_lib.accumulate(micro[0], acc, first=True)
    np.testing.assert_array_equal(acc, oracle_lib.bf16_to_f32(micro[0]))
    for k in range(1, K):
        oracle_lib.accumulate(micro[k], acc, first=False)
    vals = np.stack([oracle_lib.bf16_to_f32(x).astype(np.float64) for x in micro])
    exact = vals.sum(axis=0)
    u = 2.0 ** -24
    bound = (K - 1) * u / (1 - (K - 1) * u) * np.abs(vals).sum(axis=0)
    assert np.all(np.abs(acc.astype(np.float64) - exact) <= bound)
    if K == 2:
        np.testing.assert_array_equal(acc, exact.astype(np.float32))


def test_last_microbatch_folds_into_reduce(oracle_lib):
    # reducing (acc_r + last_r) equals reducing the fully accumulated buffers
    rng = np.random.Generator(np.random.Philox(77))
    R, K, n = 4, 3, 5000
    micro = [[rand_bf16(rng, n, 1e-2, oracle_lib) for _ in range(K)] for _ in range(R)]
    accs_partial, accs_full = [], []
    for r in range(R):
        a = np.empty(n, np.float32)
        oracle_lib.accumulate(micro[r][0], a, True)
        for k in range(1, K - 1):
            oracle_lib.accumulate(micro[r][k], a, False)
        accs_partial.append(a.copy())
        oracle_lib.accumulate(micro[r][K - 1], a, False)
        accs_full.append(a)
    c = np.float32(1.0 / 12345)
    fused = oracle_lib.reduce(accs_partial, c, last=[micro[r][K - 1] for r in range(R)])
    plain = oracle_lib.reduce(accs_full, c)
    np.testing.assert_array_equal(fused.view(np.uint32), plain.view(np.uint32))


def test_scale_is_one_multiply(oracle_lib):
    # the scaled sum equals fp32(sum) * fp32(c) rounded once (numpy binary32 multiply)
    rng = np.random.Generator(np.random.Philox(5))
    xs = [rand_bf16(rng, 10_000, 1e-2, oracle_lib) for _ in range(4)]
    c = oracle_lib.grad_scale([100, 80, 120, 60])
    s1 = oracle_lib.reduce(xs, np.float32(1.0))
    sc = oracle_lib.reduce(xs, c)
    with np.errstate(all="ignore"):
        np.testing.assert_array_equal(sc.view(np.uint32), (s1 * np.float32(c)).view(np.uint32))
