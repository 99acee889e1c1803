"""Guard regions around every buffer an entry point touches.

Each device buffer is carved out of a larger allocation whose head and tail
(GUARD elements each) hold a byte pattern.  After every call:

* no guard byte has changed (no write before or after any buffer);
* every input (replica gradients, last microbatch, reduced gradient, master
  for the all-gathers) is bit-identical to what was passed in;
* calls restricted to buckets [b0, b1) leave every element outside that
  range, and every per-bucket output outside [b0, b1), unchanged.

These are the canary checks that stand in for a memory checker on the path.
"""
import numpy as np
import pytest
import torch

import zero_optimizer_step_gb300 as dpg
from workloads import (KIND_GRAD, KIND_MASTER, flat_grads_bf16, flat_values_f32, master_f32,
                       random_param_list, segments, stream_seed)

pytestmark = pytest.mark.gpu

GUARD = 2048
PATTERN = 0xA7


@pytest.fixture(scope="module", autouse=True)
def built():
    from zero_optimizer_step_gb300 import build
    build.build()


class Buf:
    """A device tensor of n elements with GUARD poisoned elements on each side."""

    def __init__(self, n, dtype, init=None):
        self.n = n
        self.whole = torch.empty(n + 2 * GUARD, dtype=dtype, device="cuda")
        self.whole.view(torch.uint8).fill_(PATTERN)
        self.t = self.whole[GUARD:GUARD + n]
        if init is not None:
            self.t.copy_(init)
        else:
            self.t.view(torch.uint8).fill_(0x3C)
        self.esz = self.whole.element_size()

    def guards_intact(self):
        b = self.whole.view(torch.uint8)
        head, tail = b[: GUARD * self.esz], b[(GUARD + self.n) * self.esz:]
        return bool((head == PATTERN).all()) and bool((tail == PATTERN).all())

    def snapshot(self):
        return self.whole.view(torch.uint8).clone()

    def same_as(self, snap):
        return torch.equal(self.whole.view(torch.uint8), snap)

    def same_outside(self, snap, lo, hi):
        """Elements [0, lo) and [hi, n) unchanged (byte compare)."""
        b = self.whole.view(torch.uint8)
        a0, a1 = (GUARD + lo) * self.esz, (GUARD + hi) * self.esz
        return torch.equal(b[:a0], snap[:a0]) and torch.equal(b[a1:], snap[a1:])


def _case(R=4, seed=21, cap=1 << 18):
    numels = random_param_list(np.random.Generator(np.random.Philox(seed)), 40, 90_000)
    plan = dpg.dpg_plan_buckets(numels, cap, R)
    N = plan.total_padded
    segs = segments(plan.param_offset, numels)
    grads = [Buf(N, torch.bfloat16, flat_grads_bf16(segs, N, 1e-3, stream_seed(seed, KIND_GRAD, r)))
             for r in range(R)]
    tok = [2000 + 13 * r for r in range(R)]
    return numels, plan, grads, tok


def _state(plan, seed=21):
    N = plan.total_padded
    return (Buf(N, torch.float32, master_f32(N, stream_seed(seed, KIND_MASTER))),
            Buf(N, torch.float32, torch.zeros(N)), Buf(N, torch.float32, torch.zeros(N)))


def _check(outs, ins_with_snaps):
    torch.cuda.synchronize()
    for b in outs:
        assert b.guards_intact()
    for b, snap in ins_with_snaps:
        assert b.same_as(snap)


def test_step_stays_inside_its_buffers():
    _, plan, grads, tok = _case()
    N, nb = plan.total_padded, plan.n_buckets
    w, m, v = _state(plan)
    views = [Buf(N, torch.bfloat16) for _ in range(2)]
    sq, nf = Buf(nb, torch.float32), Buf(nb, torch.int64)
    snaps = [(g, g.snapshot()) for g in grads]
    dpg.dpg_step(plan, [g.t for g in grads], tok, dpg.HParams(), w.t, m.t, v.t,
                 [x.t for x in views], bucket_sqnorm=sq.t, bucket_nonfinite=nf.t)
    _check([w, m, v, sq, nf, *views], snaps)


def test_accumulation_path_and_accumulate_stay_inside():
    numels, plan, last, tok = _case(R=2, seed=22)
    N, nb = plan.total_padded, plan.n_buckets
    segs = segments(plan.param_offset, numels)
    acc = [Buf(N, torch.float32) for _ in range(2)]
    for r in range(2):
        dpg.dpg_accumulate(plan, last[r].t, acc[r].t, first=True)
        dpg.dpg_accumulate(plan, last[r].t, acc[r].t, first=False)
    snaps = [(b, b.snapshot()) for b in (*last, *acc)]
    _check(acc, [(b, s) for b, s in snaps if b in last])
    w, m, v = _state(plan, seed=22)
    view = Buf(N, torch.bfloat16)
    sq = Buf(nb, torch.float32)
    dpg.dpg_step(plan, [a.t for a in acc], tok * 2, dpg.HParams(), w.t, m.t, v.t, [view.t],
                 last_micro=[x.t for x in last], bucket_sqnorm=sq.t)
    _check([w, m, v, view, sq], snaps)
    # fp32 replica gradients alone
    f32 = [Buf(N, torch.float32, flat_values_f32(segs, N, 1e-3, stream_seed(22, KIND_GRAD, r)))
           for r in range(2)]
    snaps = [(b, b.snapshot()) for b in f32]
    dpg.dpg_step(plan, [x.t for x in f32], tok, dpg.HParams(), w.t, m.t, v.t, [view.t])
    _check([w, m, v, view], snaps)


def test_bucket_range_calls_touch_only_their_range():
    _, plan, grads, tok = _case(seed=23, cap=1 << 16)
    N, nb = plan.total_padded, plan.n_buckets
    assert nb >= 4
    b0, b1 = 1, nb - 1
    lo, hi = int(plan.bucket_offset[b0]), int(plan.bucket_offset[b1 - 1] + plan.bucket_padded[b1 - 1])
    gsn = [(g, g.snapshot()) for g in grads]
    w, m, v = _state(plan, seed=23)
    views = [Buf(N, torch.bfloat16) for _ in range(2)]
    red = Buf(N, torch.float32)
    sq, nf = Buf(nb, torch.float32), Buf(nb, torch.int64)
    outs = [w, m, v, red, *views]
    before = [b.snapshot() for b in outs]
    per_bucket = [sq.snapshot(), nf.snapshot()]
    dpg.dpg_reduce_scatter_adam(plan, [g.t for g in grads], tok, dpg.HParams(), w.t, m.t, v.t,
                                [x.t for x in views], bucket_sqnorm=sq.t, bucket_nonfinite=nf.t,
                                reduced_grad=red.t, b0=b0, b1=b1)
    _check([*outs, sq, nf], gsn)
    for b, s in zip(outs, before):
        assert b.same_outside(s, lo, hi)
    assert sq.same_outside(per_bucket[0], b0, b1) and nf.same_outside(per_bucket[1], b0, b1)

    # DDP pieces over the same range
    red2 = Buf(N, torch.float32)
    s_red2 = red2.snapshot()
    dpg.dpg_allreduce_grads(plan, [g.t for g in grads], tok, red2.t, b0=b0, b1=b1)
    _check([red2], gsn)
    assert red2.same_outside(s_red2, lo, hi)
    rsn = red2.snapshot()
    before = [b.snapshot() for b in (w, m, v, views[0])]
    dpg.dpg_adam_from_reduced(plan, red2.t, dpg.HParams(step=2), w.t, m.t, v.t, [views[0].t],
                              b0=b0, b1=b1)
    _check([w, m, v, views[0]], [(red2, rsn)])
    for b, s in zip((w, m, v, views[0]), before):
        assert b.same_outside(s, lo, hi)

    # all-gather (fp32 master -> bf16) and the ZeRO-3 gather (bf16 -> bf16)
    wsn = w.snapshot()
    s_v = views[1].snapshot()
    dpg.dpg_allgather_params(plan, w.t, [views[1].t], b0=b0, b1=b1)
    _check([views[1]], [(w, wsn)])
    assert views[1].same_outside(s_v, lo, hi)
    psn = views[1].snapshot()
    dst = [Buf(N, torch.bfloat16) for _ in range(3)]
    s_d = [d.snapshot() for d in dst]
    dpg.dpg_gather_params_bf16(plan, views[1].t, [d.t for d in dst], b0=b0, b1=b1)
    _check(dst, [(views[1], psn)])
    for d, s in zip(dst, s_d):
        assert d.same_outside(s, lo, hi)


def test_clipped_and_staged_stay_inside():
    _, plan, grads, tok = _case(seed=24)
    N, nb = plan.total_padded, plan.n_buckets
    snaps = [(g, g.snapshot()) for g in grads]
    for stored in (True, False):
        w, m, v = _state(plan, seed=24)
        view = Buf(N, torch.bfloat16)
        sq, nf = Buf(nb, torch.float32), Buf(nb, torch.int64)
        red = Buf(N, torch.float32) if stored else None
        clip = Buf(2, torch.float32)
        dpg.dpg_step_clipped(plan, [g.t for g in grads], tok, dpg.HParams(), 1e-6, w.t, m.t, v.t,
                             [view.t], bucket_sqnorm=sq.t, bucket_nonfinite=nf.t,
                             reduced_grad=None if red is None else red.t, clip_out=clip.t)
        _check([w, m, v, view, sq, nf, clip] + ([red] if red else []), snaps)
    w, m, v = _state(plan, seed=24)
    view = Buf(N, torch.bfloat16)
    sq, nf = Buf(nb, torch.float32), Buf(nb, torch.int64)
    dpg.dpg_step_staged(plan, [g.t for g in grads], tok, dpg.HParams(), w.t, m.t, v.t, [view.t],
                        bucket_sqnorm=sq.t, bucket_nonfinite=nf.t)
    dpg.dpg_check_device_status(plan)
    _check([w, m, v, view, sq, nf], snaps)


def test_pack_unpack_and_state_copies_stay_inside():
    numels, plan, _, _ = _case(R=3, seed=25)
    N = plan.total_padded
    gen = torch.Generator().manual_seed(25)
    params = [Buf(n, torch.bfloat16, torch.randn(n, generator=gen).to(torch.bfloat16))
              for n in numels]
    flat = Buf(N, torch.bfloat16)
    psn = [(p, p.snapshot()) for p in params]
    dpg.dpg_pack(plan, [p.t for p in params], flat.t)
    _check([flat], psn)
    fsn = flat.snapshot()
    outp = [Buf(n, torch.bfloat16) for n in numels]
    dpg.dpg_unpack(plan, flat.t, [p.t for p in outp])
    _check(outp, [(flat, fsn)])
    for a, b in zip(outp, params):
        assert torch.equal(a.t.view(torch.int16), b.t.view(torch.int16))
    # checkpoint layout conversions, both directions, two arrays
    st = [Buf(N, torch.float32, torch.randn(N, generator=gen)) for _ in range(2)]
    canon = [Buf(plan.canon_total, torch.float32) for _ in range(2)]
    ssn = [(s, s.snapshot()) for s in st]
    dpg.dpg_export_state(plan, [s.t for s in st], [c.t for c in canon])
    _check(canon, ssn)
    csn = [(c, c.snapshot()) for c in canon]
    back = [Buf(N, torch.float32) for _ in range(2)]
    dpg.dpg_import_state(plan, [c.t for c in canon], [b.t for b in back])
    _check(back, csn)


@pytest.mark.parametrize("K", [4, 3])
def test_deferred_step_stays_inside(K):
    # K = 4 runs the kernel compiled for four microbatches, K = 3 the
    # run-time-K loop; both read R*K microbatch buffers per element
    numels, plan, _, tok = _case(R=2, seed=26)
    N, nb = plan.total_padded, plan.n_buckets
    segs = segments(plan.param_offset, numels)
    micro = [[Buf(N, torch.bfloat16,
                  flat_grads_bf16(segs, N, 1e-3, stream_seed(26, KIND_GRAD, r, k)))
              for k in range(K)] for r in range(2)]
    snaps = [(b, b.snapshot()) for mr in micro for b in mr]
    w, m, v = _state(plan, seed=26)
    views = [Buf(N, torch.bfloat16) for _ in range(2)]
    sq, nf = Buf(nb, torch.float32), Buf(nb, torch.int64)
    dpg.dpg_step_deferred(plan, [[b.t for b in mr] for mr in micro], [3000 + k for k in range(2 * K)],
                          dpg.HParams(), w.t, m.t, v.t, [x.t for x in views],
                          bucket_sqnorm=sq.t, bucket_nonfinite=nf.t)
    _check([w, m, v, sq, nf, *views], snaps)


def test_noalloc_step_stays_inside():
    _, plan, grads, tok = _case(seed=27)
    N, nb = plan.total_padded, plan.n_buckets
    snaps = [(g, g.snapshot()) for g in grads]
    for _ in range(2):
        w, m, v = _state(plan, seed=27)
        view = Buf(N, torch.bfloat16)
        sq, nf = Buf(nb, torch.float32), Buf(nb, torch.int64)
        dpg.dpg_step_noalloc(plan, [g.t for g in grads], tok, dpg.HParams(), w.t, m.t, v.t,
                             [view.t], bucket_sqnorm=sq.t, bucket_nonfinite=nf.t)
        _check([w, m, v, view, sq, nf], snaps)
