"""Pins for the oracle's bucket planner and pack/unpack.

Pinned by hand-worked plans (tests/golden/plan_cases.txt), by invariants that
any plan obeying the rules must satisfy (reverse backward-ready order,
alignment, equal shards, cap respected unless a parameter is alone), by an
independent brute-force characterisation of the greedy rule (every bucket is
the LONGEST run of consecutive parameters, in reverse order, that fits under
the cap), and by the pack/unpack bijection ("Parallelisms", section "Flat
parameter": the originals are views into slices of one flat buffer).
"""
import os

import numpy as np
import pytest

from workloads import CONFIGS, random_param_list

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "plan_cases.txt")


def load_plan_cases():
    cases, cur = [], None
    for line in open(GOLDEN):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        tok = line.split()
        if tok[0] == "case":
            kv = dict(t.split("=", 1) for t in tok[2:])
            numels = [int(x) for x in kv["numels"].split(",") if x]
            cur = dict(name=tok[1], R=int(kv["R"]), cap=int(kv["cap_bytes"]), numels=numels,
                       buckets=[], params=[], total=None)
            cases.append(cur)
        elif tok[0] == "bucket":
            kv = dict(t.split("=") for t in tok[2:])
            cur["buckets"].append((int(tok[1]), int(kv["offset"]), int(kv["padded"]),
                                   int(kv["shard"])))
        elif tok[0] == "param":
            kv = dict(t.split("=") for t in tok[2:])
            cur["params"].append((int(tok[1]), int(kv["bucket"]), int(kv["offset"])))
        elif tok[0] == "total":
            cur["total"] = int(tok[1])
    return cases


@pytest.mark.parametrize("case", load_plan_cases(), ids=lambda c: c["name"])
def test_hand_worked_plans(oracle_lib, case):
    p = oracle_lib.plan_buckets(case["numels"], case["cap"], case["R"])
    assert p.n_buckets == len(case["buckets"])
    assert p.total_padded == case["total"]
    for b, off, pad, shard in case["buckets"]:
        assert (p.bucket_offset[b], p.bucket_padded[b], p.shard_numel[b]) == (off, pad, shard)
    for i, b, off in case["params"]:
        assert (p.param_bucket[i], p.param_offset[i]) == (b, off)


def check_invariants(p, numels, cap, R):
    n = len(numels)
    # buckets tile the flat buffer
    assert p.bucket_offset[0] == 0 if p.n_buckets else p.total_padded == 0
    for b in range(p.n_buckets):
        end = p.bucket_offset[b] + p.bucket_padded[b]
        nxt = p.bucket_offset[b + 1] if b + 1 < p.n_buckets else p.total_padded
        assert end == nxt
        assert p.bucket_padded[b] % (8 * R) == 0
        assert p.bucket_padded[b] // R % 8 == 0
    # reverse backward-ready order: bucket index never decreases as p goes down
    if n:
        assert np.all(np.diff(p.param_bucket[::-1]) >= 0)
        assert np.all(p.param_offset % 8 == 0)
    for b in range(p.n_buckets):
        members = [i for i in range(n) if p.param_bucket[i] == b]
        assert members, "no empty buckets"
        lo, hi = p.bucket_offset[b], p.bucket_offset[b] + p.bucket_padded[b]
        used = 0
        # inside the bucket: later params first, in ascending offsets, no overlap
        prev_end = lo
        for i in sorted(members, reverse=True):
            assert p.param_offset[i] >= prev_end
            assert p.param_offset[i] - prev_end < 8 or numels[i] == 0
            prev_end = p.param_offset[i] + numels[i]
            assert prev_end <= hi
            used = prev_end - lo
        nonzero = [i for i in members if numels[i] > 0]
        if len(nonzero) > 1:
            assert used * 2 <= cap, "cap exceeded by a bucket with several parameters"
        assert p.bucket_padded[b] - used < 8 * R + 8


def brute_force_plan(numels, cap, R):
    """Independent statement of the greedy rule: walk the reversed list and
    make each bucket the longest prefix of the remaining parameters whose
    aligned end fits under the cap (a first parameter with elements is always
    taken; zero-size parameters join the current run)."""
    order = list(range(len(numels)))[::-1]
    runs, i = [], 0
    while i < len(order):
        best = i + 1
        for j in range(i + 1, len(order) + 1):
            end = 0
            fits = True
            has_elems = False
            for q in order[i:j]:
                start = (end + 7) // 8 * 8
                e = start + numels[q]
                if has_elems and numels[q] > 0 and e * 2 > cap:
                    fits = False
                    break
                if numels[q] > 0:
                    has_elems = True
                end = e
            if fits:
                best = j
            else:
                break
        runs.append(order[i:best])
        i = best
    return runs


@pytest.mark.parametrize("seed", range(40))
def test_random_plans_invariants_and_brute_force(oracle_lib, seed):
    rng = np.random.Generator(np.random.Philox(seed))
    n = int(rng.integers(0, 9))
    numels = random_param_list(rng, n, 300)
    R = int(rng.choice([1, 2, 3, 4, 8]))
    cap = int(rng.integers(2, 1200))
    p = oracle_lib.plan_buckets(numels, cap, R)
    check_invariants(p, numels, cap, R)
    runs = brute_force_plan(list(numels), cap, R)
    assert p.n_buckets == len(runs)
    for b, run in enumerate(runs):
        for q in run:
            assert p.param_bucket[q] == b


@pytest.mark.parametrize("name", ["tiny", "gpt2", "llama1b", "llama8b16l", "sweep"])
def test_config_plans(oracle_lib, name):
    cfg = CONFIGS[name]
    p = oracle_lib.plan_buckets(cfg.numels, cfg.cap_bytes, cfg.R)
    check_invariants(p, cfg.numels, cfg.cap_bytes, cfg.R)
    assert p.total_padded >= cfg.psi


def test_realised_parameter_counts():
    # parameter counts of the synthetic model lists (sums of the listed shapes)
    assert CONFIGS["tiny"].psi == 2_400
    assert CONFIGS["gpt2"].psi == 124_439_808
    assert CONFIGS["llama1b"].psi == 1_204_881_408
    assert CONFIGS["llama8b16l"].psi == 4_540_469_248
    assert len(CONFIGS["sweep"].shapes) == 10_000


def test_invalid_arguments(oracle_lib):
    with pytest.raises(oracle_lib.OracleError):
        oracle_lib.plan_buckets([4, 4], 0, 2)
    with pytest.raises(oracle_lib.OracleError):
        oracle_lib.plan_buckets([4, -1], 64, 2)
    with pytest.raises(oracle_lib.OracleError):
        oracle_lib.plan_buckets([4], 64, 0)


@pytest.mark.parametrize("seed", range(12))
def test_pack_unpack_bijection(oracle_lib, seed):
    rng = np.random.Generator(np.random.Philox(100 + seed))
    n = int(rng.integers(1, 60))
    numels = random_param_list(rng, n, 5000)
    R = int(rng.choice([1, 2, 4, 8]))
    cap = int(rng.integers(16, 40000))
    p = oracle_lib.plan_buckets(numels, cap, R)
    # index-coded payload: every element of every parameter is distinct
    # (values 1..65535 wrap, so use a per-element code plus a parameter tag check)
    grads = [rng.integers(1, 1 << 16, size=int(k), dtype=np.uint64).astype(np.uint16)
             for k in numels]
    flat = oracle_lib.pack(p, grads)
    assert flat.size == p.total_padded
    back = oracle_lib.unpack(p, flat)
    for a, b in zip(grads, back):
        np.testing.assert_array_equal(a, b)
    # every non-padding slot is hit exactly once; padding stays zero
    hit = np.zeros(p.total_padded, dtype=np.int64)
    for i, k in enumerate(numels):
        hit[p.param_offset[i]:p.param_offset[i] + k] += 1
    assert hit.max(initial=0) <= 1
    assert np.all(flat[hit == 0] == 0)
    assert np.all(flat[hit == 1] != 0)


@pytest.mark.parametrize("seed", range(8))
def test_checkpoint_layout_bijection_and_reshard(oracle_lib, seed):
    """Export/import of a state array ("Distributed Training and Parallelism",
    Reproduction and debugging: resumability and mesh reconfiguration): the
    canonical layout is the parameters back to back in registration order;
    import after export restores every parameter slot and zeroes padding;
    a state exported under one plan and imported under another (other R,
    other cap) carries every parameter's values across unchanged."""
    rng = np.random.Generator(np.random.Philox(700 + seed))
    numels = random_param_list(rng, int(rng.integers(1, 80)), 3000)
    pa = oracle_lib.plan_buckets(numels, int(rng.integers(16, 20000)), int(rng.choice([1, 2, 4, 8])))
    pb = oracle_lib.plan_buckets(numels, int(rng.integers(16, 20000)), int(rng.choice([1, 3, 8, 16])))
    flat = rng.standard_normal(pa.total_padded).astype(np.float32)
    canon = oracle_lib.export_state(pa, flat)
    assert canon.size == int(numels.sum())
    # canonical order is registration order: parameter p's values start at sum(numels[:p])
    c = 0
    for p_, n in enumerate(numels):
        np.testing.assert_array_equal(canon[c:c + n], flat[pa.param_offset[p_]:pa.param_offset[p_] + n])
        c += int(n)
    back = oracle_lib.import_state(pa, canon)
    hit = np.zeros(pa.total_padded, bool)
    for p_, n in enumerate(numels):
        hit[pa.param_offset[p_]:pa.param_offset[p_] + n] = True
    np.testing.assert_array_equal(back[hit], flat[hit])
    assert not back[~hit].any()
    # reshard: A -> canonical -> B -> canonical is the identity
    flat_b = oracle_lib.import_state(pb, canon)
    np.testing.assert_array_equal(oracle_lib.export_state(pb, flat_b), canon)
