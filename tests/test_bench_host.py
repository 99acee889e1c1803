"""Host logic of bench.py that the reported numbers depend on (no GPU).

* algorithmic bytes per parameter of every schedule: (2R + 26) for the step,
  the K-microbatch cycle (10K - 8)R + 26, the paired schedule, and the
  deferred one (2KR + 26);
* the paired accumulation schedule covers microbatches 0..K-3 in order;
* the ncu launch-list parser behind `roofline.traffic` averages the fused
  kernel's DRAM bytes over its launches and ignores every other kernel;
* the stored traffic is used only while the kernel code hashes the same, and
  the hash ignores comments and whitespace.
"""
import json
import os
import types

import pytest

import bench
from workloads import CONFIGS


def test_algorithmic_bytes_of_the_workloads():
    assert bench.algorithmic_bytes_per_param(CONFIGS["llama1b"]) == {"fused": 42, "step": 42}
    assert bench.algorithmic_bytes_per_param(CONFIGS["gpt2"]) == {"fused": 42, "step": 42}
    # 4.5B, R = 4, K = 4: 6R+26 fused, (10K - 8)R + 26 per cycle
    c = CONFIGS["llama8b16l"]
    assert (c.R, c.K) == (4, 4)
    assert bench.algorithmic_bytes_per_param(c) == {"fused": 50, "step": 154}
    # paired: one first pair (8R) + the fused step with two microbatches (8R + 26)
    assert bench.algorithmic_bytes_per_param(c, fold2=True) == {"fused": 58, "step": 90}
    # deferred: one pass reading all K bf16 microbatches of every replica
    assert bench.algorithmic_bytes_per_param(c, deferred=True) == {"fused": 58, "step": 58}
    assert bench.algorithmic_bytes_per_param(_cfg(8, 3), deferred=True)["step"] == 2 * 3 * 8 + 26


def _cfg(R, K):
    return types.SimpleNamespace(R=R, K=K)


@pytest.mark.parametrize("K", range(3, 11))
def test_fold2_schedule_covers_the_microbatches_in_order(K):
    seen = []
    for k, pair in bench.fold2_schedule(K):
        seen += [k, k + 1] if pair else [k]
    assert seen == list(range(K - 2))
    # bytes agree with a by-hand count: first pass 8R / 6R, later 12R / 10R
    R = 3
    acc = 0
    for k, pair in bench.fold2_schedule(K):
        acc += (8 if pair else 6) * R if k == 0 else (12 if pair else 10) * R
    assert bench.algorithmic_bytes_per_param(_cfg(R, K), fold2=True)["step"] == 8 * R + 26 + acc


def _csv_row(i, name, metric, value):
    return ",".join(f'"{x}"' for x in [i, "1", "python3", "host", name, "1", "7", "(128, 1, 1)",
                                       "(10, 1, 1)", "0", "10.3", "sec", metric, "byte", value])


def test_traffic_parser_averages_the_fused_kernel_only(tmp_path, monkeypatch):
    lines = ["==PROF== banner", '"ID","Process ID"']
    rows = [("0", "void dpg::k_rs_adam_chunk<8, 0, 0>(dpg::RsAdamArgs)", 100, 40),
            ("1", "dpg::k_chunk_finalize(dpg::FinalizeArgs)", 5, 0),
            ("2", "void dpg::k_rs_adam_chunk<8, 0, 0>(dpg::RsAdamArgs)", 300, 60),
            ("3", "void dpg::k_rs_adam_staged<8>(dpg::StagedArgs)", 999, 999),
            ("4", "vectorized_elementwise_kernel", 7, 7)]
    for i, name, rd, wr in rows:
        lines.append(_csv_row(i, name, "dram__bytes_read.sum", f"{rd:,}"))
        lines.append(_csv_row(i, name, "dram__bytes_write.sum", f"{wr:,}"))
        lines.append(_csv_row(i, name, "gpu__time_duration.sum", "1000"))
    csv_path = tmp_path / "launches.csv"
    csv_path.write_text("\n".join(lines) + "\n")
    out = tmp_path / "traffic.json"
    monkeypatch.setattr(bench, "TRAFFIC_FILE", str(out))
    a = types.SimpleNamespace(config="gpt2", traffic_from=str(csv_path), cap_mib=None,
                              replicas=None, microbatches=None, fold2=False, deferred=False)
    bench.write_traffic(a)
    small = CONFIGS["gpt2"]
    t = json.loads(out.read_text())["entries"][bench.traffic_key(small)]
    assert t["launches"] == 2
    assert t["dram_bytes_read"] == 200 and t["dram_bytes_write"] == 50
    assert t["dram_bytes_per_launch"] == 250
    assert t["source_sha256"] == bench.kernel_source_sha256()
    # a second variant lands in its own entry, the first one stays
    a2 = types.SimpleNamespace(**{**vars(a), "replicas": 4, "microbatches": 4})
    bench.write_traffic(a2)
    entries = json.loads(out.read_text())["entries"]
    assert set(entries) == {"k_rs_adam_chunk R=8 K=1 bf16", "k_rs_adam_chunk R=4 K=4 acc_fp32_last_bf16"}
    # read back while the code hash matches, scaled by elements to a larger
    # workload of the same variant; another variant has no entry
    big = CONFIGS["llama1b"]
    n_small = t["elements"]
    assert bench.traffic_per_launch(big, big.cap_bytes, 10 * n_small) == pytest.approx(2500)
    acc = types.SimpleNamespace(R=4, K=4)
    assert bench.traffic_per_launch(acc, 0, n_small) == pytest.approx(250)
    assert bench.traffic_per_launch(acc, 0, n_small, deferred=True) is None
    assert bench.traffic_per_launch(types.SimpleNamespace(R=2, K=1), 0, n_small) is None
    whole = json.loads(out.read_text())
    whole["entries"]["k_rs_adam_chunk R=8 K=1 bf16"]["source_sha256"] = "0" * 64
    out.write_text(json.dumps(whole))
    assert bench.traffic_per_launch(big, big.cap_bytes, n_small) is None


def test_code_hash_ignores_comments_and_whitespace(tmp_path, monkeypatch):
    code = "int f(int x) {\n    return x + 1;   // add one\n}\n/* block */\n"
    a = tmp_path / "a.cu"
    a.write_text(code)
    monkeypatch.setattr(bench, "KERNEL_SRCS", [str(a)])
    h0 = bench.kernel_source_sha256()
    a.write_text("// header\nint f(int x) {\n\n  return x + 1;\n}\n")
    assert bench.kernel_source_sha256() == h0
    a.write_text("int f(int x) {\n    return x + 2;\n}\n")
    assert bench.kernel_source_sha256() != h0


def test_kernel_sources_exist():
    for f in bench.KERNEL_SRCS:
        assert os.path.exists(f), f


def test_replicas_override():
    a = types.SimpleNamespace(config="llama1b", replicas=16, microbatches=None)
    c = bench.config_of(a)
    assert c.R == 16 and c.psi == CONFIGS["llama1b"].psi
    assert bench.algorithmic_bytes_per_param(c)["fused"] == 2 * 16 + 26
    assert bench.config_of(types.SimpleNamespace(config="gpt2", replicas=None)) is CONFIGS["gpt2"]
    with pytest.raises(SystemExit):
        bench.config_of(types.SimpleNamespace(config="gpt2", replicas=65))
    c = bench.config_of(types.SimpleNamespace(config="gpt2", replicas=4, microbatches=4))
    assert (c.R, c.K) == (4, 4)
    assert bench.algorithmic_bytes_per_param(c) == {"fused": 50, "step": 154}
    with pytest.raises(SystemExit):
        bench.config_of(types.SimpleNamespace(config="gpt2", replicas=None, microbatches=0))


def test_reference_line_states_what_it_timed():
    # the reference arm times a sample per step; its line must say so, and
    # its full-workload step time must agree with its rate
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    out = subprocess.run([sys.executable, os.path.join(root, "bench.py"), "--impl", "reference",
                          "--config", "gpt2", "--steps", "3", "--warmup", "3",
                          "--cpu-sample-elems", "32768"],
                         capture_output=True, text=True, timeout=600, check=True).stdout
    line = json.loads(out.strip().splitlines()[-1])
    c = line["config"]
    assert line["impl"] == "reference"
    assert c["psi"] == CONFIGS["gpt2"].psi
    assert c["sample_elems_per_step"] == 32768
    assert c["sample_share_of_psi"] == pytest.approx(32768 / c["psi"])
    assert c["psi"] / (line["ms_per_step"] * 1e-3) == pytest.approx(line["value"], rel=1e-9)
    assert 32768 / (line["sample_ms_per_step"] * 1e-3) == pytest.approx(line["value"], rel=1e-9)
    assert line["cpu_baseline"]["value"] == line["value"]
    assert line["e2e"]["h2d_bytes_per_step"] == 0


def test_fused_roofline_arithmetic():
    # achieved = algorithmic bytes per launch / mean launch time; frac = achieved / peak
    k = [7.0, 7.1, 7.2, 7.3, 7.4]
    r = bench.fused_roofline("k", 42, 1_000_000_000, k, 6761.6, "measured", None)
    mean_ms = sum(k) / len(k)
    assert r["algorithmic_bytes_per_launch"] == 42_000_000_000
    assert r["achieved"] == pytest.approx(42e9 / (mean_ms * 1e-3) / 1e9)
    assert r["frac"] == pytest.approx(r["achieved"] / 6761.6)
    assert r["kernel_ms_p10_p50_p90"] == [7.0, 7.2, 7.4]
    assert r["bound"] == "hbm" and r["unit"] == "GB/s"


def test_secondary_workload_bytes():
    # the 4.5B line: fused step 6R+26, cycle (10K-8)R+26, deferred 2KR+26
    c = CONFIGS["llama8b16l"]
    assert (c.R, c.K, c.cap_bytes) == (4, 4, 100 << 20)
    assert bench.algorithmic_bytes_per_param(c) == {"fused": 50, "step": 154}
    assert bench.algorithmic_bytes_per_param(c, deferred=True)["step"] == 58
    assert bench.traffic_key(c) == "k_rs_adam_chunk R=4 K=4 acc_fp32_last_bf16"
    assert bench.traffic_key(c, deferred=True) == "k_rs_adam_chunk R=4 K=4 deferred"
    assert bench.traffic_key(CONFIGS["llama1b"]) == "k_rs_adam_chunk R=8 K=1 bf16"


def test_hockney_fit_recovers_alpha_and_beta():
    # K launches moving M bytes: T = K*alpha + M/B; exact data gives exact parameters
    alpha, bw = 4.5e-6, 7.1e12
    pts = [{"n_buckets": k, "bytes": m, "per_bucket_ms": (k * alpha + m / bw) * 1e3}
           for k, m in ((147, 5.06e10), (83, 5.06e10), (24, 5.06e10), (2595, 2.0e8))]
    fit = bench.hockney_fit(pts)
    assert fit["alpha_us"] == pytest.approx(4.5, rel=1e-9)
    assert fit["inv_beta_gbs"] == pytest.approx(7100.0, rel=1e-9)


def test_resident_bytes_decide_the_l2_flush():
    # only the 10,000-tensor list is small enough to be flushed between steps
    c = CONFIGS["llama1b"]
    assert bench.resident_bytes(c, c.psi) == (2 * 8 + 12 + 2) * c.psi
    c4 = CONFIGS["llama8b16l"]
    assert bench.resident_bytes(c4, c4.psi) == (2 * 4 + 4 * 4 + 14) * c4.psi
    assert bench.resident_bytes(c4, c4.psi, deferred=True) == (2 * 4 * 4 + 14) * c4.psi
    assert bench.resident_bytes(c4, c4.psi, fold2=True) == (2 * 4 * 2 + 4 * 4 + 14) * c4.psi
    small = [n for n, c in CONFIGS.items() if n != "tiny"
             and bench.resident_bytes(c, c.psi) < bench.L2_FLUSH_BELOW]
    assert small == ["sweep"]


def test_optional_leg_records_out_of_memory():
    import torch

    def boom():
        raise torch.cuda.OutOfMemoryError("CUDA out of memory. Tried to allocate 9 GiB")
    out = bench.optional_leg(boom, 1)
    assert out["skipped"].startswith("out of device memory: CUDA out of memory")
    assert bench.optional_leg(lambda: {"ok": 1}, 1) == {"ok": 1}
    with pytest.raises(torch.cuda.OutOfMemoryError):
        bench.optional_leg(boom, 2)        # several ranks: fail together, not apart
    assert bench.all_ranks_agree(True, 1, "cpu") and not bench.all_ranks_agree(False, 1, "cpu")
