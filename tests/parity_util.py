"""Shared helpers of the GPU parity tests: run one step through the C ABI on
the device and the same step through the CPU oracle on host copies of the
same inputs, then compare element by element.

Bars (from the method statement): layouts and reduced gradients bit-exact,
fp32 master/m/v within 2 ulp, bf16 parameters within 1 ulp, per-bucket norms
within 1e-5 relative of the oracle's binary64 sum.  Both sides use the same
correctly rounded operations in the same order, so the expected difference is
zero everywhere; the tolerances are the stated ceilings.
"""
from __future__ import annotations

from dataclasses import dataclass, field
from typing import List, Optional, Sequence

import numpy as np
import torch

import oracle
import zero_optimizer_step_gb300 as dpg
from workloads import (KIND_GRAD, KIND_M, KIND_MASTER, KIND_V, flat_grads_bf16,
                       flat_values_f32, master_f32, normal_f32, segments, stream_seed,
                       warm_moments)

F32_ULP = 2
BF16_ULP = 1
NORM_RTOL = 1e-5


def np_bf16(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def np_f32(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().contiguous().numpy()


def _ordered(bits: np.ndarray, width: int) -> np.ndarray:
    x = bits.astype(np.int64)
    sign = np.int64(1) << (width - 1)
    return np.where(x >= sign, sign - x, x)   # -0 and +0 both map to 0


def ulp_f32(a: np.ndarray, b: np.ndarray) -> int:
    """Max distance in binary32 ulps (NaN == NaN counts as 0)."""
    a = np.asarray(a, np.float32).reshape(-1)
    b = np.asarray(b, np.float32).reshape(-1)
    if a.size == 0:
        return 0
    both_nan = np.isnan(a) & np.isnan(b)
    ia = _ordered(a.view(np.uint32).astype(np.int64), 32)
    ib = _ordered(b.view(np.uint32).astype(np.int64), 32)
    d = np.abs(ia - ib)
    d[both_nan] = 0
    one_nan = np.isnan(a) ^ np.isnan(b)
    d[one_nan] = 1 << 40
    return int(d.max())


def ulp_bf16(a: np.ndarray, b: np.ndarray) -> int:
    a = np.asarray(a, np.uint16).reshape(-1)
    b = np.asarray(b, np.uint16).reshape(-1)
    if a.size == 0:
        return 0
    nan_a = ((a & 0x7F80) == 0x7F80) & ((a & 0x7F) != 0)
    nan_b = ((b & 0x7F80) == 0x7F80) & ((b & 0x7F) != 0)
    ia = _ordered(a.astype(np.int64), 16)
    ib = _ordered(b.astype(np.int64), 16)
    d = np.abs(ia - ib)
    d[nan_a & nan_b] = 0
    d[nan_a ^ nan_b] = 1 << 40
    return int(d.max())


def check_norms(gpu_sq: np.ndarray, ref_sq: np.ndarray):
    gpu_sq = gpu_sq.astype(np.float64)
    fin = np.isfinite(ref_sq)
    assert np.array_equal(np.isfinite(gpu_sq), fin)
    assert np.all(np.abs(gpu_sq[fin] - ref_sq[fin]) <= NORM_RTOL * np.abs(ref_sq[fin]) + 1e-30)


@dataclass
class StepCase:
    numels: Sequence[int]
    cap_bytes: int
    R: int
    K: int = 1                   # microbatches (K > 1: fp32 accumulation + last bf16)
    f32_grads: bool = False      # K == 1 with fp32 gradient buffers
    warm: bool = False           # non-zero m, v
    t: int = 1
    wd: float = 0.0
    lr: float = 1e-3
    beta1: float = 0.9
    beta2: float = 0.999
    eps: float = 1e-8
    n_views: int = 1
    grad_std: float = 1e-2
    seed: int = 1234
    tokens: Optional[Sequence[int]] = None
    b_split: Optional[int] = None   # run buckets [0, b) and [b, nb) as two calls
    inject: Optional[str] = None    # "nan", "inf", "denormal"


@dataclass
class StepResult:
    plan: object = None
    host: dict = field(default_factory=dict)
    gpu: dict = field(default_factory=dict)
    ref: dict = field(default_factory=dict)


def run_case(c: StepCase) -> StepResult:
    """Build inputs on the host, run device and oracle, return both."""
    res = StepResult()
    plan = dpg.dpg_plan_buckets(c.numels, c.cap_bytes, c.R)
    res.plan = plan
    # the oracle lays out its own buffers; the library's layout must be identical
    oplan = oracle.plan_buckets(c.numels, c.cap_bytes, c.R)
    assert (oplan.n_buckets, oplan.total_padded) == (plan.n_buckets, plan.total_padded)
    np.testing.assert_array_equal(oplan.param_offset, plan.param_offset)
    np.testing.assert_array_equal(oplan.bucket_offset, plan.bucket_offset)
    np.testing.assert_array_equal(oplan.bucket_padded, plan.bucket_padded)
    N = oplan.total_padded
    segs = segments(oplan.param_offset, c.numels)
    R, K = c.R, c.K
    rng = np.random.Generator(np.random.Philox(c.seed))
    tokens = (np.asarray(c.tokens, np.int64) if c.tokens is not None
              else rng.integers(3000, 4097, size=R * K).astype(np.int64))

    # ---- inputs (host, torch CPU generators) --------------------------------
    micro = [[None] * K for _ in range(R)]
    for r in range(R):
        for k in range(K):
            if c.f32_grads:
                micro[r][k] = flat_values_f32(segs, N, c.grad_std, stream_seed(c.seed, KIND_GRAD, r, k))
            else:
                micro[r][k] = flat_grads_bf16(segs, N, c.grad_std, stream_seed(c.seed, KIND_GRAD, r, k))
    if c.inject and N and segs:
        o, n = segs[len(segs) // 2]
        idx = o + np.arange(min(n, 64))
        val = {"nan": float("nan"), "inf": float("inf"), "denormal": 3e-39}[c.inject]
        for r in range(R):
            micro[r][K - 1][idx[: 1 + r]] = val
    master0 = master_f32(N, stream_seed(c.seed, KIND_MASTER))
    if c.warm:
        m0, v0 = warm_moments(N, c.grad_std, stream_seed(c.seed, KIND_M), stream_seed(c.seed, KIND_V))
    else:
        m0, v0 = torch.zeros(N), torch.zeros(N)
    res.host = dict(micro=micro, master=master0, m=m0, v=v0, tokens=tokens)

    # ---- device run -----------------------------------------------------------
    dev = torch.device("cuda")
    d_master, d_m, d_v = master0.to(dev), m0.to(dev), v0.to(dev)
    d_views = [torch.full((N,), float("nan"), dtype=torch.bfloat16, device=dev)
               for _ in range(c.n_views)]
    d_sq = torch.full((max(1, plan.n_buckets),), -1.0, device=dev)
    d_nf = torch.full((max(1, plan.n_buckets),), -1, dtype=torch.int64, device=dev)
    d_red = torch.full((N,), float("nan"), device=dev)
    d_micro = [[micro[r][k].to(dev) for k in range(K)] for r in range(R)]
    hp = dpg.HParams(step=c.t, weight_decay=c.wd, lr=c.lr, beta1=c.beta1, beta2=c.beta2, eps=c.eps)
    acc_after = []
    if K > 1:
        d_acc = [torch.full((N,), float("nan"), device=dev) for _ in range(R)]
        for k in range(K - 1):
            for r in range(R):
                dpg.dpg_accumulate(plan, d_micro[r][k], d_acc[r], first=(k == 0))
            acc_after.append([np_f32(a) for a in d_acc])
        grads, last = d_acc, [d_micro[r][K - 1] for r in range(R)]
    else:
        grads, last = [d_micro[r][0] for r in range(R)], None
    splits = [(0, plan.n_buckets)]
    if c.b_split is not None:
        splits = [(0, c.b_split), (c.b_split, plan.n_buckets)]
    for b0, b1 in splits:
        dpg.dpg_reduce_scatter_adam(plan, grads, tokens, hp, d_master, d_m, d_v, d_views,
                                    last_micro=last, bucket_sqnorm=d_sq, bucket_nonfinite=d_nf,
                                    reduced_grad=d_red, b0=b0, b1=b1)
    torch.cuda.synchronize()
    res.gpu = dict(master=np_f32(d_master), m=np_f32(d_m), v=np_f32(d_v),
                   views=[np_bf16(x) for x in d_views], sq=np_f32(d_sq)[: plan.n_buckets],
                   nf=d_nf.cpu().numpy()[: plan.n_buckets], reduced=np_f32(d_red),
                   acc_after=acc_after)

    # ---- oracle run -------------------------------------------------------------
    if c.f32_grads:
        h_micro = [[np_f32(micro[r][k]) for k in range(K)] for r in range(R)]
    else:
        h_micro = [[np_bf16(micro[r][k]) for k in range(K)] for r in range(R)]
    w, m, v = np_f32(master0).copy(), np_f32(m0).copy(), np_f32(v0).copy()
    ref_acc_after = []
    if K > 1:
        accs = [np.empty(N, np.float32) for _ in range(R)]
        for k in range(K - 1):
            for r in range(R):
                oracle.accumulate(h_micro[r][k], accs[r], first=(k == 0))
            ref_acc_after.append([a.copy() for a in accs])
        ograds, olast = accs, [h_micro[r][K - 1] for r in range(R)]
    else:
        ograds, olast = [h_micro[r][0] for r in range(R)], None
    views, red, sq = oracle.step(oplan.bucket_offset, oplan.bucket_padded, ograds, tokens, w, m, v,
                                 last=olast, n_views=c.n_views, wd=c.wd, t=c.t, lr=c.lr,
                                 beta1=c.beta1, beta2=c.beta2, eps=c.eps, want_reduced=True)
    nf = np.array([int(np.sum(~np.isfinite(red[o:o + p])))
                   for o, p in zip(oplan.bucket_offset, oplan.bucket_padded)], np.int64)
    res.ref = dict(master=w, m=m, v=v, views=views, sq=sq, nf=nf, reduced=red,
                   acc_after=ref_acc_after)
    return res


def assert_parity(res: StepResult):
    g, r = res.gpu, res.ref
    for k, (ga, ra) in enumerate(zip(g["acc_after"], r["acc_after"])):
        for x, y in zip(ga, ra):
            assert ulp_f32(x, y) == 0, f"accumulation after microbatch {k} not bit-exact"
    # reduced gradients: bit-exact (NaN positions must agree)
    assert ulp_f32(g["reduced"], r["reduced"]) == 0, "reduced gradient not bit-exact"
    for name in ("master", "m", "v"):
        assert ulp_f32(g[name], r[name]) <= F32_ULP, f"{name} beyond {F32_ULP} ulp"
    for gv, rv in zip(g["views"], r["views"]):
        assert ulp_bf16(gv, rv) <= BF16_ULP, "bf16 parameters beyond 1 ulp"
    check_norms(g["sq"], r["sq"])
    np.testing.assert_array_equal(g["nf"], r["nf"])


def exact_everywhere(res: StepResult) -> bool:
    g, r = res.gpu, res.ref
    return (all(ulp_f32(g[n], r[n]) == 0 for n in ("master", "m", "v"))
            and all(ulp_bf16(a, b) == 0 for a, b in zip(g["views"], r["views"])))
