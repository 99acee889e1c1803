"""GPU parity of dpg_step_clipped (global gradient-norm clipping) against the
oracle: g = rank-ordered sum x fp32(1/G); norm over ALL buckets; coef =
fp32(min(1, max_norm / (norm + 1e-6))); Adam on g * coef.  Both sides sum the
exact binary64 squares, so the coefficient is expected to agree bit for bit,
and with it every output (bars as elsewhere: 2 ulp fp32, 1 ulp bf16)."""
import numpy as np
import pytest
import torch

import oracle
import zero_optimizer_step_gb300 as dpg
from parity_util import BF16_ULP, F32_ULP, check_norms, np_bf16, np_f32, ulp_bf16, ulp_f32
from workloads import (KIND_GRAD, KIND_M, KIND_MASTER, KIND_V, flat_grads_bf16, master_f32,
                       random_param_list, segments, stream_seed, warm_moments)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    from zero_optimizer_step_gb300 import build
    build.build()
    oracle.build()


def _numels(seed, n, mx):
    return random_param_list(np.random.Generator(np.random.Philox(seed)), n, mx)


CASES = {
    "R8_clip_stored_g": dict(numels=_numels(1, 40, 150_000), cap=1 << 20, R=8, K=1, max_norm=1e-6,
                             stored=True, clips=True),
    "R8_clip_recompute": dict(numels=_numels(1, 40, 150_000), cap=1 << 20, R=8, K=1,
                              max_norm=1e-6, stored=False, clips=True),
    "R4_acc_K3_clip_warm": dict(numels=_numels(2, 30, 80_000), cap=1 << 19, R=4, K=3,
                                max_norm=1e-6, stored=True, warm=True, t=4, clips=True),
    "R3_generic_no_clip": dict(numels=_numels(3, 20, 50_000), cap=300_000, R=3, K=1,
                               max_norm=1e6, stored=False, clips=False),
    "R8_nan": dict(numels=_numels(4, 10, 20_000), cap=1 << 15, R=8, K=1, max_norm=1e-3,
                   stored=True, inject=True),
}


def _run(c, device_fn="clipped"):
    numels, R, K = c["numels"], c["R"], c["K"]
    plan = dpg.dpg_plan_buckets(numels, c["cap"], R)
    op = oracle.plan_buckets(numels, c["cap"], R)
    N = op.total_padded
    segs = segments(op.param_offset, numels)
    micro = [[flat_grads_bf16(segs, N, 1e-3, stream_seed(9, KIND_GRAD, r, k)) for k in range(K)]
             for r in range(R)]
    if c.get("inject"):
        o, _ = segs[len(segs) // 2]
        micro[0][K - 1][o] = float("nan")
    tok = [3000 + 37 * i for i in range(R * K)]
    w0 = master_f32(N, stream_seed(9, KIND_MASTER))
    if c.get("warm"):
        m0, v0 = warm_moments(N, 1e-3, stream_seed(9, KIND_M), stream_seed(9, KIND_V))
    else:
        m0, v0 = torch.zeros(N), torch.zeros(N)
    t = c.get("t", 1)
    dev = "cuda"
    d = dict(w=w0.to(dev), m=m0.to(dev), v=v0.to(dev))
    view = torch.empty(N, dtype=torch.bfloat16, device=dev)
    sq = torch.empty(op.n_buckets, device=dev)
    nf = torch.empty(op.n_buckets, dtype=torch.int64, device=dev)
    red = torch.full((N,), float("nan"), device=dev) if c["stored"] else None
    clip = torch.zeros(2, device=dev)
    dm = [[x.to(dev) for x in row] for row in micro]
    if K > 1:
        acc = [torch.empty(N, device=dev) for _ in range(R)]
        for k in range(K - 1):
            for r in range(R):
                dpg.dpg_accumulate(plan, dm[r][k], acc[r], first=(k == 0))
        grads, last = acc, [dm[r][K - 1] for r in range(R)]
    else:
        grads, last = [dm[r][0] for r in range(R)], None
    hp = dpg.HParams(step=t)
    if device_fn == "clipped":
        dpg.dpg_step_clipped(plan, grads, tok, hp, c["max_norm"], d["w"], d["m"], d["v"], [view],
                             last_micro=last, bucket_sqnorm=sq, bucket_nonfinite=nf,
                             reduced_grad=red, clip_out=clip)
    else:
        dpg.dpg_step(plan, grads, tok, hp, d["w"], d["m"], d["v"], [view], last_micro=last)
    torch.cuda.synchronize()
    got = dict(w=np_f32(d["w"]), m=np_f32(d["m"]), v=np_f32(d["v"]), p=np_bf16(view),
               sq=np_f32(sq), nf=nf.cpu().numpy(), clip=np_f32(clip),
               red=None if red is None else np_f32(red))
    # oracle
    hm = [[np_bf16(x) for x in row] for row in micro]
    if K > 1:
        accs = [np.empty(N, np.float32) for _ in range(R)]
        for k in range(K - 1):
            for r in range(R):
                oracle.accumulate(hm[r][k], accs[r], first=(k == 0))
        g = oracle.reduce(accs, oracle.grad_scale(tok), last=[hm[r][K - 1] for r in range(R)])
    else:
        g = oracle.reduce([hm[r][0] for r in range(R)], oracle.grad_scale(tok))
    norm, coef = oracle.clip_coef(g, c["max_norm"])
    g2 = oracle.scale(g, coef)
    w, m, v = np_f32(w0).copy(), np_f32(m0).copy(), np_f32(v0).copy()
    oracle.adam(g2, w, m, v, t=t)
    bsq = np.array([np.sum(g[o:o + p].astype(np.float64) ** 2)
                    for o, p in zip(op.bucket_offset, op.bucket_padded)])
    ref = dict(w=w, m=m, v=v, p=oracle.f32_to_bf16(w), g=g, norm=norm, coef=coef, sq=bsq)
    return got, ref


@pytest.mark.parametrize("name", sorted(CASES))
def test_clipped_step_parity(name):
    c = CASES[name]
    got, ref = _run(c)
    if c.get("inject"):
        assert np.isnan(got["clip"][1]) and np.isnan(ref["coef"])
    else:
        assert got["clip"][1] == ref["coef"], (got["clip"][1], ref["coef"])
        assert got["clip"][0] == np.float32(ref["norm"])
        assert (ref["coef"] < 1.0) == c["clips"]
    for k in ("w", "m", "v"):
        assert ulp_f32(got[k], ref[k]) <= F32_ULP, k
    assert ulp_bf16(got["p"], ref["p"]) <= BF16_ULP
    check_norms(got["sq"], ref["sq"])
    if got["red"] is not None:
        assert ulp_f32(got["red"], ref["g"]) == 0


def test_no_clip_equals_dpg_step():
    c = CASES["R3_generic_no_clip"]
    a, _ = _run(c, "clipped")
    b, _ = _run(c, "step")
    for k in ("w", "m", "v"):
        np.testing.assert_array_equal(a[k].view(np.uint32), b[k].view(np.uint32))
    np.testing.assert_array_equal(a["p"], b["p"])


@pytest.mark.parametrize("name", ["R8_clip_stored_g", "R4_acc_K3_clip_warm"])
def test_clipped_step_parity_on_the_persistent_grid(name):
    """With a grid cap the clipped step runs its persistent norm and update
    passes; the coefficient and every output are the oracle's as before."""
    c = CASES[name]
    dpg.dpg_set_fused_max_ctas(40)
    try:
        got, ref = _run(c)
    finally:
        dpg.dpg_set_fused_max_ctas(0)
    assert got["clip"][1] == ref["coef"]
    for k in ("w", "m", "v"):
        assert ulp_f32(got[k], ref[k]) <= F32_ULP, k
    assert ulp_bf16(got["p"], ref["p"]) <= BF16_ULP
    check_norms(got["sq"], ref["sq"])
