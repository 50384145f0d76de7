"""The oracle's pins have power: each plausible mistake planted in a scratch
copy of oracle.c (compiled on the CPU, never the real oracle) makes at least
one pin fail.  Each mutation names the test file expected to catch it."""
import os
import shutil
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

MUTATIONS = {
    "residual sign": ("double d = Pt[v] - Pd[v];", "double d = Pd[v] - Pt[v];",
                      "test_oracle_rules.py"),
    "residual without max(0, .)": ("R[v] = d > 0.0 ? d : 0.0;", "R[v] = d;",
                                   "test_oracle_rules.py"),
    "top-k tie rule reversed": ("return (x->v < y->v) ? -1 : (x->v > y->v);",
                                "return (x->v > y->v) ? -1 : (x->v < y->v);",
                                "test_oracle_rules.py"),
    "top-p prefix rule not strict": ("if (prefix < top_p) {", "if (prefix <= top_p) {",
                                     "test_oracle_rules.py"),
    "temperature dropped": ("e[v] = keep[v] ? exp(l[v] / T - M) : 0.0;",
                            "e[v] = keep[v] ? exp(l[v] - M) : 0.0;", "test_oracle_rules.py"),
    "inverse CDF with >=": ("if (C > t) {", "if (C >= t) {", "test_oracle_rules.py"),
    "LM head operand transposed": ("o[n] += h * widen(wrow, ORC_BF16, n);",
                                   "o[n] += h * widen(W, ORC_BF16, (int64_t)n * K + k);",
                                   "test_oracle_rules.py"),
    "Philox counter words 1/3 swapped": ("uint32_t n0 = hi1 ^ c1 ^ k0;",
                                         "uint32_t n0 = hi1 ^ c3 ^ k0;",
                                         "test_oracle_philox.py"),
    "Philox key increment": ("k1 += 0xBB67AE85u;", "k1 += 0xBB67AE86u;",
                             "test_oracle_philox.py"),
    "24-bit uniform shift": ("return (double)(w >> 8) * (1.0 / 16777216.0);",
                             "return (double)(w >> 9) * (1.0 / 16777216.0);",
                             "test_oracle_philox.py"),
    "bonus row off by one": ("const int64_t trow = (int64_t)b * (Kmax + 1) + Kb;",
                             "const int64_t trow = (int64_t)b * (Kmax + 1) + (Kb > 0 ? Kb - 1 : 0);",
                             "test_oracle_verify.py"),
    "accept ratio inverted": ("const double ratio = p / q;", "const double ratio = q / p;",
                              "test_oracle_verify.py"),
    "uniform words swapped": ("if (u0) *u0 = orc_u24(w[0]);", "if (u0) *u0 = orc_u24(w[1]);",
                              "test_oracle_verify.py"),
    "greedy argmax keeps the last maximum": ("if (isfinite(l[v]) && (a < 0 || l[v] > l[a])) a = v;",
                                             "if (isfinite(l[v]) && (a < 0 || l[v] >= l[a])) a = v;",
                                             "test_oracle_greedy.py"),
    "greedy emits the drafted token at the mismatch": ("                tok = a;\n            }\n        } else if",
                                                       "                tok = x;\n            }\n        } else if",
                                                       "test_oracle_greedy.py"),
    "resample uniform from another slot": (
        "u_smp_star = u_smp;",
        "verify_uniforms(s->seed, s->round, b, j + 1, 0u, NULL, &u_smp_star);",
        "test_oracle_verify.py"),
}


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_planted_mistake_is_caught(name, tmp_path):
    before, after, test_file = MUTATIONS[name]
    for sub in ("oracle", "tests", "workloads"):
        shutil.copytree(os.path.join(ROOT, sub), tmp_path / sub,
                        ignore=shutil.ignore_patterns("*.so", "*.so.tmp*", "__pycache__"))
    src_path = tmp_path / "oracle" / "oracle.c"
    src = src_path.read_text()
    assert src.count(before) == 1, f"mutation site for {name!r} not found once"
    src_path.write_text(src.replace(before, after))
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
                        os.path.join("tests", test_file)], cwd=tmp_path,
                       capture_output=True, text=True, timeout=600)
    assert r.returncode == 1, f"{name!r} not caught:\n{r.stdout[-2000:]}{r.stderr[-2000:]}"
