"""The pins have teeth: each test plants one plausible mistake in a copy of
the oracle's C source (on the CPU), builds it, and checks that the oracle pin
tests fail against it.  The oracle itself is never modified."""
import os
import subprocess
import sys

import pytest

from conftest import ROOT

SRC = os.path.join(ROOT, "oracle", "fp8q_oracle.c")
PINS = ["tests/test_oracle_codec.py", "tests/test_oracle_quant.py", "tests/test_oracle_gemm.py",
        "tests/test_oracle_mx.py"]

MUTATIONS = {
    "ties_away_from_zero": ("r = nearbyint(a / quantum) * quantum;",
                            "r = round(a / quantum) * quantum;"),
    "no_saturation": ("    if (r > 448.0)\n        r = 448.0;", ""),
    "inverted_scale": ("*s = a / 448.0f;", "*s = 448.0f / a;"),
    "cols_read_transposed": ("float v = fabsf(load_x(x, dtype, (mb * GROUP + j) * K + k));",
                             "float v = fabsf(load_x(x, dtype, k * M + mb * GROUP + j));"),
    "weight_scale_index_swapped": ("s_blk[nb * KB + kb] = s;", "s_blk[kb * NB + nb] = s;"),
    "gemm_dropped_sB": ("ex += ((double)sa * (double)sb) * p;", "ex += (double)sa * p;"),
    "gemm_B_transposed": ("int64_t k = kb * GROUP + j;\n            double prod = g_decode[Aq[m * K + k]] * g_decode[Bq[n * K + k]];",
                          "int64_t k = kb * GROUP + j;\n            double prod = g_decode[Aq[m * K + k]] * g_decode[Bq[k * N + n]];"),
    "gemm_sA_index": ("float sa = sA[kb * lds_a + m];", "float sa = sA[m * KB + kb];"),
    "gemm_pages_order_drops_scale": ("volatile float t = pf * s;", "volatile float t = pf;"),
    "mx_ceil_exponent": ("se = (e - 1) - E4M3_EMAX;", "se = e - E4M3_EMAX;"),
    "mx_no_lower_clamp": ("    if (se < -127)\n        se = -127;\n", ""),
    "mx_multiplies_by_scale": ("load_x(x, dtype, i) / X;", "load_x(x, dtype, i) * X;"),
    "mx_group_of_16_in_amax": ("for (int64_t j = 0; j < MX_GROUP; ++j) {\n                float v = fabsf(",
                               "for (int64_t j = 0; j < MX_GROUP / 2; ++j) {\n                float v = fabsf("),
    "mx_gemm_drops_eb": ("(int)ea[m * G + g] - 127 + (int)eb[n * G + g] - 127", "(int)ea[m * G + g] - 127"),
    "mx_gemm_b_scale_index": ("(int)eb[n * G + g]", "(int)eb[g * G + n]"),
}


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_pins_catch_planted_mistake(name, tmp_path):
    sys.path.insert(0, os.path.join(ROOT, "oracle"))
    import build as obuild
    old, new = MUTATIONS[name]
    src = open(SRC).read()
    assert src.count(old) == 1, "mutation anchor not found: " + name
    mutated = tmp_path / "mutant.c"
    mutated.write_text(src.replace(old, new))
    lib = obuild.build(src=str(mutated), out=str(tmp_path / "libmutant.so"), force=True)
    env = dict(os.environ, FP8Q_ORACLE_LIB=lib)
    res = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider", *PINS],
                         cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert res.returncode == 1, "pins did not catch mutation %s:\n%s" % (name, res.stdout[-2000:])
