"""The oracle's pins have teeth: plant one plausible mistake at a time in a
copy of the oracle's C source (in a temporary directory, on the CPU), rebuild
it, and check that the pin suite fails.  The committed oracle is not touched."""
import os
import shutil
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

MUTATIONS = {
    "relu dropped": ("double relu = dot > 0.0 ? dot : 0.0;", "double relu = dot;"),
    "weight of the wrong head": ("s += (double)w[(int64_t)q * n_head + h] * relu;",
                                 "s += (double)w[(int64_t)q * n_head + (h ^ 1)] * relu;"),
    "ties favour the higher row": ("return (x->r > y->r) - (x->r < y->r);",
                                   "return (x->r < y->r) - (x->r > y->r);"),
    "row at the query position hidden": ("visible = row_pos[r] <= q_pos[q];",
                                         "visible = row_pos[r] < q_pos[q];"),
    "lse sign": ("lse[h] = mx + log(z);", "lse[h] = mx - log(z);"),
    "softmax scale dropped": ("l[j] = scale * dot;", "l[j] = dot;"),
    "bf16 exponent bias": ("v = ldexp((double)(m | 0x80), e - 127 - 7);",
                           "v = ldexp((double)(m | 0x80), e - 126 - 7);"),
    "f16 ties rounded up": ("n = (fmod(fl, 2.0) == 0.0) ? fl : fl + 1.0;", "n = fl + 1.0;"),
    "k-th score taken from the top": ("*kth = m > 0 ? v[m - 1].s : -INFINITY;",
                                      "*kth = m > 0 ? v[0].s : -INFINITY;"),
    "raw row decoded as bf16": ("x[(int64_t)(n_sel + j) * dim + d] = oracle_f16_to_double(",
                                "x[(int64_t)(n_sel + j) * dim + d] = oracle_bf16_to_double("),
    "pooling not normalised": ("out[j] = den > 0.0 ? num / den : 0.0;", "out[j] = den > 0.0 ? num : 0.0;"),
    "pooling max taken as a min": ("if (s > m) m = s;", "if (s < m) m = s;"),
    "pooling reads the next column's score": (
        "const double e = exp((double)score[(int64_t)r * width + j] - m);",
        "const double e = exp((double)score[(int64_t)r * width + (j + 1) % width] - m);"),
    "push slides by two rows": ("ring[(int64_t)(s - 1) * dim + d] = ring[(int64_t)s * dim + d];",
                                "ring[(int64_t)(s - 1) * dim + d] = ring[(int64_t)(s < cap - 1 ? s + 1 : s) * dim + d];"),
    "push keeps the full window one row short": ("        *n_raw = cap - 1;\n", "        *n_raw = cap - 2;\n"),
    "e4m3 exponent bias": ("v = ldexp((double)(8 + m), e - 7 - 3);", "v = ldexp((double)(8 + m), e - 8 - 3);"),
    "e4m3 subnormal step": ("v = ldexp((double)m, -9);", "v = ldexp((double)m, -10);"),
    "e4m3 ties rounded up": ("n = fmod(fl, 2.0) == 0.0 ? fl : fl + 1.0;", "n = fl + 1.0;"),
    "e4m3 saturates one step low": ("        return sign | 0x7E;\n    if (x == 0.0)", "        return sign | 0x7D;\n    if (x == 0.0)"),
    "fp8 row scale one power too small": ("while (e > -126 && amax <= 448.0 * ldexp(1.0, e - 1))",
                                          "while (e > -126 && amax <= 448.0 * ldexp(1.0, e))"),
    "fp8 codes not divided by the row scale": ("oracle_double_to_e4m3((double)xr[d] / s);",
                                               "oracle_double_to_e4m3((double)xr[d]);"),
    "fp8 attention ignores the row scale": ("x[(int64_t)j * dim + d] = oracle_e4m3_to_double(codes[(int64_t)sel[j] * dim + d]) * s;",
                                            "x[(int64_t)j * dim + d] = oracle_e4m3_to_double(codes[(int64_t)sel[j] * dim + d]);"),
}


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_planted_oracle_mistake_is_caught(name, tmp_path):
    before, after = MUTATIONS[name]
    src = open(os.path.join(ROOT, "oracle", "ds4a_oracle.c")).read()
    assert src.count(before) == 1, "mutation site moved; update the mutation"
    shutil.copytree(os.path.join(ROOT, "oracle"), tmp_path / "oracle",
                    ignore=shutil.ignore_patterns("_build", "__pycache__"))
    shutil.copytree(os.path.join(ROOT, "tests"), tmp_path / "tests",
                    ignore=shutil.ignore_patterns("__pycache__"))
    (tmp_path / "oracle" / "ds4a_oracle.c").write_text(src.replace(before, after))
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
                        "tests/test_oracle_pins.py"], cwd=tmp_path, capture_output=True, text=True,
                       timeout=600)
    assert r.returncode != 0, f"pins did not catch: {name}\n{r.stdout[-2000:]}"
