"""Pins for the oracle's fp32 <-> bf16 conversions.

The rounding rule is IEEE-754 round-to-nearest-even onto the bfloat16 format
(the upper half of binary32).  Pinned by (a) hand-worked encodings in
tests/golden/bf16_cast.txt, (b) torch's CPU float32 -> bfloat16 conversion (a
library routine that implements the same IEEE rounding) on structured and
random bit patterns, (c) the exactness of the bf16 -> fp32 widening.
"""
import os

import numpy as np
import pytest
import torch

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "bf16_cast.txt")


def _golden():
    rows = []
    for line in open(GOLDEN):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        a, b, *_ = line.split()
        rows.append((int(a, 16), b))
    return rows


def _bits_to_f32(bits):
    return np.array(bits, dtype=np.uint32).view(np.float32)


def test_golden_hand_worked_cases(oracle_lib):
    rows = _golden()
    assert len(rows) >= 20
    x = _bits_to_f32([a for a, _ in rows])
    y = oracle_lib.f32_to_bf16(x)
    for (a, want), got in zip(rows, y):
        got = int(got)
        if want.startswith("nan"):
            assert (got & 0x7F80) == 0x7F80 and (got & 0x007F) != 0, hex(a)
            assert (got & 0x0040) != 0, f"{a:08x}: NaN must be quiet"
            assert (got >> 15) == (1 if want == "nan-" else 0), hex(a)
        else:
            assert got == int(want, 16), f"{a:08x}: got {got:04x} want {want}"


def _torch_bf16_bits(x_f32: np.ndarray) -> np.ndarray:
    t = torch.from_numpy(x_f32.copy()).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def _structured_patterns():
    # every exponent, both signs, and dropped-half patterns around the tie
    # point, with both parities of the kept significand
    exps = np.arange(256, dtype=np.uint32) << 23
    kept_lsb = np.array([0, 1 << 16, 0x7F << 16, 0x7E << 16], dtype=np.uint32)
    dropped = np.array([0, 1, 0x7FFF, 0x8000, 0x8001, 0xFFFF, 0x4000, 0xC000], dtype=np.uint32)
    sign = np.array([0, 0x80000000], dtype=np.uint32)
    pats = (sign[:, None, None, None] | exps[None, :, None, None]
            | kept_lsb[None, None, :, None] | dropped[None, None, None, :]).reshape(-1)
    return pats


def test_matches_torch_on_structured_patterns(oracle_lib):
    pats = _structured_patterns()
    x = pats.view(np.float32)
    ours = oracle_lib.f32_to_bf16(x)
    ref = _torch_bf16_bits(x)
    finite = np.isfinite(x)
    np.testing.assert_array_equal(ours[finite], ref[finite])
    # non-finite: infinities exact, NaNs stay NaN with their sign
    inf = np.isinf(x)
    np.testing.assert_array_equal(ours[inf], ref[inf])
    nan = np.isnan(x)
    assert np.all((ours[nan] & 0x7F80) == 0x7F80) and np.all((ours[nan] & 0x7F) != 0)
    np.testing.assert_array_equal(ours[nan] >> 15, pats[nan] >> 31)


def test_matches_torch_on_random_patterns(oracle_lib):
    rng = np.random.Generator(np.random.Philox(1234))
    pats = rng.integers(0, 2 ** 32, size=4_000_000, dtype=np.uint64).astype(np.uint32)
    x = pats.view(np.float32)
    ours = oracle_lib.f32_to_bf16(x)
    ref = _torch_bf16_bits(x)
    ok = ~np.isnan(x)
    np.testing.assert_array_equal(ours[ok], ref[ok])


def test_widening_is_exact(oracle_lib):
    h = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    f = oracle_lib.bf16_to_f32(h)
    np.testing.assert_array_equal(f.view(np.uint32), h.astype(np.uint32) << 16)
    # round trip of every non-NaN bf16 value is the identity
    back = oracle_lib.f32_to_bf16(f)
    notnan = ~np.isnan(f)
    np.testing.assert_array_equal(back[notnan], h[notnan])


def test_rounding_error_bound(oracle_lib):
    # |bf16(x) - x| <= half an ulp of bf16 for finite results (2^-8 relative)
    rng = np.random.Generator(np.random.Philox(7))
    x = (rng.standard_normal(200_000) * 10.0 ** rng.integers(-30, 30, 200_000)).astype(np.float32)
    y = oracle_lib.bf16_to_f32(oracle_lib.f32_to_bf16(x)).astype(np.float64)
    err = np.abs(y - x.astype(np.float64))
    assert np.all(err <= np.abs(x.astype(np.float64)) * 2.0 ** -8 + 1e-45)
