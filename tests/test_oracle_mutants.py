"""Mutation check of the oracle's pins: each entry plants one plausible
mistake (a dropped term, a wrong sign, index, constant or rounding rule) in a
copy of oracle.c, builds it on the CPU, and runs the pin tests against it; at
least one pin must fail for every mutant.  Nothing here touches a GPU."""
import concurrent.futures as cf
import os
import subprocess
import sys
import tempfile

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "oracle.c")

# (name, original text, mutated text, pin test files expected to catch it)
MUTANTS = [
    ("tie_rounds_up", "if (kept & 1u) kept += 1u;", "kept += 1u;", ["test_oracle_cast.py"]),
    ("nan_not_quieted", "return (uint16_t)(kept | 0x0040u);", "return (uint16_t)kept;",
     ["test_oracle_cast.py"]),
    ("round_toward_zero", "if (dropped > 0x8000u) {", "if (dropped > 0xFFFFu) {",
     ["test_oracle_cast.py"]),
    ("no_alignment", "int64_t start = (used + 7) / 8 * 8;", "int64_t start = used;",
     ["test_oracle_plan.py"]),
    ("cap_inclusive", "end * 2 > cap_bytes", "end * 2 >= cap_bytes", ["test_oracle_plan.py"]),
    ("forward_order", "for (int32_t p = n - 1; p >= 0; --p) {",
     "for (int32_t p = 0; p < n; ++p) {", ["test_oracle_plan.py"]),
    ("pad_without_R", "int64_t unit = 8 * (int64_t)R;\n            int64_t padded",
     "int64_t unit = 8;\n            int64_t padded", ["test_oracle_plan.py"]),
    ("unpack_wrong_index", "grads[p][i] = flat[param_offset[p] + i];",
     "grads[p][i] = flat[param_offset[p]];", ["test_oracle_plan.py"]),
    ("reduce_subtracts", "s = s + x;", "s = s - x;", ["test_oracle_reduce.py"]),
    ("reduce_drops_last_rank", "for (int32_t r = 1; r < R; ++r) {\n            float x = replica_value",
     "for (int32_t r = 1; r < R - 1; ++r) {\n            float x = replica_value",
     ["test_oracle_reduce.py"]),
    ("reduce_from_plus_zero", "float s = replica_value(grads, dtype, last, 0, i);",
     "float s = 0.0f + replica_value(grads, dtype, last, 0, i);", ["test_oracle_reduce.py"]),
    ("scale_off_by_one", "double inv = 1.0 / (double)G;", "double inv = 1.0 / (double)(G + 1);",
     ["test_oracle_reduce.py", "test_oracle_normalization.py"]),
    ("scale_by_R_over_G", "double inv = 1.0 / (double)G;",
     "double inv = (double)n_counts / (double)G;",
     ["test_oracle_reduce.py", "test_oracle_normalization.py"]),
    ("accumulate_overwrites", "float s = acc[i] + x;", "float s = x;", ["test_oracle_reduce.py"]),
    ("last_micro_replaces", "x = x + y;", "x = y;", ["test_oracle_reduce.py"]),
    ("no_bias_correction_m", "float m_hat = mi / c.bias1;", "float m_hat = mi;",
     ["test_oracle_adam.py"]),
    ("eps_inside_sqrt", "float root = sqrtf(v_hat);\n        float denom = root + c.eps;",
     "float root = sqrtf(v_hat + c.eps);\n        float denom = root;", ["test_oracle_adam.py"]),
    ("bias2_off_by_one", "c->bias2 = (float)(1.0 - pow(beta2, (double)t));",
     "c->bias2 = (float)(1.0 - pow(beta2, (double)(t + 1)));", ["test_oracle_adam.py"]),
    ("v_uses_beta1", "float v_new_term = c.one_minus_beta2 * g2;",
     "float v_new_term = c.one_minus_beta1 * g2;", ["test_oracle_adam.py"]),
    ("v_uses_g_not_g2", "float v_new_term = c.one_minus_beta2 * g2;",
     "float v_new_term = c.one_minus_beta2 * gi;", ["test_oracle_adam.py"]),
    ("ascent", "w = w - step;", "w = w + step;", ["test_oracle_adam.py"]),
    ("decay_sign", "w = w - d;", "w = w + d;", ["test_oracle_adam.py"]),
    ("zero2_is_zero1", "case 2: return param * psi + (grad + optim) * psi / n;",
     "case 2: return (param + grad) * psi + optim * psi / n;",
     ["test_oracle_memory_and_step.py"]),
    ("norm_not_squared", "acc += gi * gi;", "acc += gi;", ["test_oracle_memory_and_step.py"]),
    ("shard_loop_ignores_owner", "int64_t lo = bucket_offset[b] + owner * shard;",
     "int64_t lo = bucket_offset[b];", ["test_oracle_memory_and_step.py"]),
    ("export_wrong_slot", "for (int64_t i = 0; i < numels[p]; ++i) canon[c + i] = flat[param_offset[p] + i];",
     "for (int64_t i = 0; i < numels[p]; ++i) canon[c + i] = flat[param_offset[p] + numels[p] - 1 - i];",
     ["test_oracle_plan.py"]),
    ("import_keeps_padding", "for (int64_t i = 0; i < total; ++i) flat[i] = 0.0f;",
     "for (int64_t i = 0; i < total; ++i) flat[i] = flat[i];", ["test_oracle_plan.py"]),
    ("clip_unclamped", "if (c > 1.0) c = 1.0;\n    *norm_out", "*norm_out", ["test_oracle_clip.py"]),
    ("clip_norm_squared", "double norm = sqrt(total);", "double norm = total;",
     ["test_oracle_clip.py"]),
    ("gather_truncates", "views[k][i] = oracle_f32_to_bf16(master[i]);\n    if (reduced)",
     "views[k][i] = (uint16_t)(f32_bits(master[i]) >> 16);\n    if (reduced)",
     ["test_oracle_memory_and_step.py"]),
    ("clip_no_eps", "double c = max_norm / (norm + 1e-6);", "double c = max_norm / norm;",
     ["test_oracle_clip.py"]),
    ("m_uses_beta2", "float m_old = c.beta1 * m[i];", "float m_old = c.beta2 * m[i];",
     ["test_oracle_adam.py"]),
    ("allreduce_rank0_only", "for (int32_t dst = 0; dst < R; ++dst)\n        oracle_reduce_range(",
     "for (int32_t dst = 0; dst < 1; ++dst)\n        oracle_reduce_range(", ["test_oracle_reduce.py"]),
]


def _run_mutant(args):
    name, old, new, files, tmp = args
    src = open(SRC).read()
    assert src.count(old) >= 1, f"{name}: pattern not found"
    mutated = src.replace(old, new, 1)
    c_path = os.path.join(tmp, f"{name}.c")
    so_path = os.path.join(tmp, f"{name}.so")
    open(c_path, "w").write(mutated)
    import oracle
    subprocess.run(["gcc", *oracle.CFLAGS, "-o", so_path, c_path, "-lm"], check=True)
    env = dict(os.environ, ORACLE_LIB=so_path)
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
                        *[os.path.join(ROOT, "tests", f) for f in files]],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    return name, r.returncode


def test_every_mutant_is_caught():
    with tempfile.TemporaryDirectory() as tmp:
        jobs = [(n, o, m, f, tmp) for n, o, m, f in MUTANTS]
        with cf.ThreadPoolExecutor(max_workers=min(8, os.cpu_count() or 1)) as ex:
            results = list(ex.map(_run_mutant, jobs))
    survivors = [n for n, rc in results if rc == 0]
    assert not survivors, f"pins missed these planted mistakes: {survivors}"
    # a mutant that breaks collection/build would also be "caught"; make sure
    # the failures are test failures (pytest exit code 1)
    assert all(rc == 1 for _, rc in results), results
