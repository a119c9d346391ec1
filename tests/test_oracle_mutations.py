"""Plant plausible mistakes in a copy of the oracle and check that its pins fail.

Each mutation edits the C source text of a temporary copy of oracle.c (on the
CPU; the real oracle is untouched), compiles it, and runs the oracle's pin
tests against the broken library in a subprocess. A pin suite that still
passes would mean that kind of mistake could go unnoticed.

The nibble order inside a packed E2M1 byte is deliberately not mutated: the
same swap applied to both operands permutes K identically inside one scale
block, so no output changes (test_oracle.py checks that invariance).
"""
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "oracle.c")

MUTATIONS = {
    "dropped_last_k_term": ("for (int64_t k = 0; k < K; ++k)\n                s += a[k] * b[k];",
                            "for (int64_t k = 0; k < K - 1; ++k)\n                s += a[k] * b[k];"),
    "transposed_b_operand": ("            const double* b = Bd + j * K;\n            double s = 0.0;\n            for (int64_t k = 0; k < K; ++k)\n                s += a[k] * b[k];\n            C[i * N + j] = s;\n        }\n    }\n    free(Ad);\n    free(Bd);\n    return 0;\n}\n\n/* Selected",
                             "            double s = 0.0;\n            for (int64_t k = 0; k < K; ++k)\n                s += a[k] * Bd[(k % N) * K + (j % K)];\n            C[i * N + j] = s;\n        }\n    }\n    free(Ad);\n    free(Bd);\n    return 0;\n}\n\n/* Selected"),
    "e2m1_sign_dropped": ("double v = (e == 0) ? 0.5 * (double)m : ldexp(1.0 + 0.5 * (double)m, (int)e - 1);\n    return s ? -v : v;",
                          "double v = (e == 0) ? 0.5 * (double)m : ldexp(1.0 + 0.5 * (double)m, (int)e - 1);\n    return v;"),
    "e2m1_subnormal_scale": ("(e == 0) ? 0.5 * (double)m", "(e == 0) ? 1.0 * (double)m"),
    "e4m3_wrong_bias": ("ldexp(1.0 + (double)m / 8.0, (int)e - 7)", "ldexp(1.0 + (double)m / 8.0, (int)e - 8)"),
    "scale_block_index_dropped": ("oracle_dec_e4m3(scales_row[k >> 4])", "oracle_dec_e4m3(scales_row[0])"),
    "ties_away_from_zero": ("if (r > 0.5 || (r == 0.5 && fmod(n, 2.0) != 0.0))", "if (r >= 0.5)"),
    "sampled_uses_row_for_b": ("const uint16_t* b = B + cols[t] * K;", "const uint16_t* b = B + rows[t] * K;"),
}


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_pins_catch_planted_mistake(name, tmp_path):
    old, new = MUTATIONS[name]
    src = open(SRC).read()
    assert src.count(old) >= 1, f"mutation {name} no longer applies to oracle.c"
    mutated = src.replace(old, new, 1)
    c_path = tmp_path / "oracle_mut.c"
    so_path = tmp_path / "liboracle_mut.so"
    c_path.write_text(mutated)
    subprocess.run(["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fPIC", "-shared", str(c_path),
                    "-o", str(so_path), "-lm"], check=True, capture_output=True)
    env = dict(os.environ, ORACLE_LIB_OVERRIDE=str(so_path))
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
                        os.path.join(ROOT, "tests", "test_oracle.py")],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode != 0, f"pins did not catch mutation {name}:\n{r.stdout[-2000:]}"


# The fused epilogue is numpy code in oracle/__init__.py: its mutations edit a copy of the
# package, which the pin run imports ahead of the real one.
PY_MUTATIONS = {
    "bias_indexed_by_row": ("bf16_bits_to_f64(bias)[None, :]", "bf16_bits_to_f64(bias)[:, None]"),
    "alpha_dropped": ("x = alpha * np.asarray(acc, dtype=np.float64)", "x = np.asarray(acc, dtype=np.float64)"),
    "beta_sign_flipped": ("x = x + beta * bf16_bits_to_f64(c_old)", "x = x - beta * bf16_bits_to_f64(c_old)"),
    "relu_ignored": ("x = np.maximum(x, 0.0)", "x = x"),
    "gelu_cubic_coefficient": ("(x + 0.044715 * x * x * x)", "(x + 0.04715 * x * x * x)"),
    "gelu_sqrt_two_pi": ("np.sqrt(2.0 / np.pi)", "np.sqrt(2.0 * np.pi)"),
    "gelu_half_dropped": ("return 0.5 * x * (1.0 + np.tanh(", "return x * (1.0 + np.tanh("),
}


@pytest.mark.parametrize("name", sorted(PY_MUTATIONS))
def test_epilogue_pins_catch_planted_mistake(name, tmp_path):
    import shutil
    old, new = PY_MUTATIONS[name]
    pkg = tmp_path / "oracle"
    shutil.copytree(os.path.join(ROOT, "oracle"), pkg, ignore=shutil.ignore_patterns("_build", "__pycache__"))
    src = (pkg / "__init__.py").read_text()
    assert src.count(old) == 1, f"mutation {name} no longer applies to oracle/__init__.py"
    (pkg / "__init__.py").write_text(src.replace(old, new))
    sys.path.insert(0, ROOT)
    import oracle
    env = dict(os.environ, ORACLE_LIB_OVERRIDE=oracle.build(),
               PYTHONPATH=os.pathsep.join([str(tmp_path), ROOT, os.environ.get("PYTHONPATH", "")]))
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider", "-k", "epilogue or gelu",
                        os.path.join(ROOT, "tests", "test_oracle.py")],
                       cwd=str(tmp_path), env=env, capture_output=True, text=True, timeout=600)
    # the copy must be the one imported (python -m puts the working directory first on sys.path)
    probe = subprocess.run([sys.executable, "-c", "import oracle; print(oracle.__file__)"], cwd=str(tmp_path), env=env,
                           capture_output=True, text=True, timeout=120)
    assert probe.stdout.strip().startswith(str(tmp_path)), probe.stdout + probe.stderr
    assert r.returncode != 0, f"pins did not catch mutation {name}:\n{r.stdout[-2000:]}"
