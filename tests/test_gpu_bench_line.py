"""The benchmark's default JSON line on the GPU: every key the line promises
is there and its figures can be recomputed from its own fields.

* value = psi / step time (one GPU); hbm_gbs_step = (2R + 26) psi / step time;
* roofline: achieved = algorithmic bytes per launch / mean fused-launch time,
  frac = achieved / peak, the kernel's share of the step;
* the 4.5B leg: cycle_frac from (10K - 8)R + 26 = 154 B/param, the fused
  launch from 6R + 26 = 50, the deferred cycle from 2KR + 26 = 58;
* the GPT-2 list's step and fused launch (42 B/param);
* the Hockney records, clocks, the end-to-end leg with its copied bytes, the
  CPU baseline, and the launch count (two per step: fused pass + finalize).
"""
import json
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_default_line_keys_and_arithmetic():
    steps, warm = 4, 3
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--gpus", "1",
                        "--steps", str(steps), "--warmup", str(warm)],
                       cwd=ROOT, capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, r.stderr[-3000:]
    line = json.loads(r.stdout.strip().splitlines()[-1])
    for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
              "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config", "roofline",
              "gpu_launches", "clocks", "e2e", "cpu_baseline", "hockney", "secondary"):
        assert k in line, k
    c = line["config"]
    psi, R = c["psi"], c["R"]
    assert (line["n_gpus"], line["steps"], line["warmup"]) == (1, steps, warm)
    assert c["workload"].startswith("llama1b") and R == 8 and c["K"] == 1
    ms = line["ms_per_step"]
    assert line["value"] == pytest.approx(psi / (ms * 1e-3), rel=1e-9)
    assert line["hbm_gbs_step"] == pytest.approx((2 * R + 26) * psi / (ms * 1e-3) / 1e9, rel=1e-9)

    rf = line["roofline"]
    assert rf["bound"] == "hbm" and rf["unit"] == "GB/s"
    assert rf["algorithmic_bytes_per_launch"] == (2 * R + 26) * psi
    assert rf["achieved"] == pytest.approx(rf["algorithmic_bytes_per_launch"] /
                                           (rf["kernel_ms"] * 1e-3) / 1e9, rel=1e-9)
    assert rf["frac"] == pytest.approx(rf["achieved"] / rf["peak"], rel=1e-9)
    assert 0.8 < rf["frac"] < 1.3                      # at the HBM roofline, not past it
    assert rf["kernel_ms"] <= ms                       # the fused launch sits inside the step
    assert line["gpu_launches"] == 2 * steps
    assert set(line["clocks"]) >= {"sm_mhz", "sm_max_mhz", "reasons"}

    e = line["e2e"]
    assert e["unit"] == "params/s" and e["h2d_bytes_per_step"] >= R * psi * 2
    assert e["d2h_bytes_per_step"] > 0
    assert e["value"] == pytest.approx(psi / (e["ms_per_step"] * 1e-3), rel=1e-9)
    cb = line["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] == 1 and cb["value"] > 0

    h = line["hockney"]
    assert len(h["points"]) == 3 and h["fit"]["alpha_us"] > 0 and h["fit"]["inv_beta_gbs"] > 0
    hs = line["hockney_sweep"]
    assert [q["n_buckets"] for q in hs["points"]] == [2595, 149, 10, 1]
    assert hs["fit"]["alpha_us"] > 0

    g2 = line["gpt2"]
    assert g2["config"]["workload"].startswith("gpt2") and g2["config"]["R"] == 8
    assert g2["roofline"]["algorithmic_bytes_per_launch"] == 42 * g2["config"]["psi"]
    assert g2["value"] == pytest.approx(g2["config"]["psi"] / (g2["ms_per_step"] * 1e-3), rel=1e-9)
    assert 0.8 < g2["roofline"]["frac"] < 1.3

    s = line["secondary"]
    if "skipped" in s:
        pytest.skip("the 4.5B leg did not fit on this device: " + s["skipped"])
    sc = s["config"]
    psi4, R4, K4 = sc["psi"], sc["R"], sc["K"]
    assert (R4, K4) == (4, 4)
    assert s["cycle_frac"] == pytest.approx(((10 * K4 - 8) * R4 + 26) * psi4 /
                                            (s["ms_per_step"] * 1e-3) / 1e9 / s["roofline"]["peak"],
                                            rel=1e-9)
    sr = s["roofline"]
    assert sr["algorithmic_bytes_per_launch"] == (6 * R4 + 26) * psi4
    assert sr["frac"] == pytest.approx(sr["algorithmic_bytes_per_launch"] /
                                       (sr["kernel_ms"] * 1e-3) / 1e9 / sr["peak"], rel=1e-9)
    d = s["deferred"]
    if "skipped" not in d:
        assert d["roofline"]["algorithmic_bytes_per_launch"] == (2 * K4 * R4 + 26) * psi4
        assert d["cycle_frac"] == pytest.approx((2 * K4 * R4 + 26) * psi4 /
                                                (d["ms_per_step"] * 1e-3) / 1e9 /
                                                d["roofline"]["peak"], rel=1e-9)
