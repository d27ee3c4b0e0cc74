"""Plants plausible mistakes in a temporary copy of the oracle and checks that the pins in
test_oracle_pins.py catch each one (the oracle under oracle/ is never modified)."""
import os
import shutil
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

MUTATIONS = {
    "nibble order": ("int q = (col & 1) ? (byte >> 4) : (byte & 15);",
                     "int q = (col & 1) ? (byte & 15) : (byte >> 4);"),
    "tie to higher id": ("return ia < ib;", "return ia > ib;"),
    "combine drops routing weight": ("float p = ws * eo[j];", "float p = eo[j];"),
    "gelu constant": ("0.044715 * g * g * g", "0.04471 * g * g * g"),
    "bias not before top-k": ("key[e] = bias ? l[e] + bias[e] : l[e];", "key[e] = l[e];"),
    "up bias dropped": ("if (X->up_b) u += or_bf16_to_double(X->up_b[(size_t)e * I + i]);\n        double h",
                        "if (0) u += or_bf16_to_double(X->up_b[(size_t)e * I + i]);\n        double h"),
    "swiglu lower clamp sign": ("if (u < -L) u = -L;", "if (u < -L) u = L;"),
    "int4 min dropped": ("return (double)q * scale + mn;", "return (double)q * scale;"),
    "e8m0 bias": ("return ldexp(1.0, byte - 127);", "return ldexp(1.0, byte - 128);"),
    "route list not stable": ("for (int r = 0; r < n; ++r)\n            if (idx[r] == e)",
                              "for (int r = n - 1; r >= 0; --r)\n            if (idx[r] == e)"),
    "h not rounded to 16 bits": ("h_out[i] = adt_to_double(double_to_adt(h, adt), adt);",
                                 "h_out[i] = h;"),
    "tail drops the layer scalar": ("float m = (float)adt_to_double(xs, adt) * layer_scalar;",
                                    "float m = (float)adt_to_double(xs, adt);"),
    "tail skips the dense branch": ("float s = (float)adt_to_double(ht[j], adt) + (float)adt_to_double(yt[j], adt);",
                                    "float s = (float)adt_to_double(yt[j], adt);"),
}


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_pins_catch_planted_mistake(name, tmp_path):
    if shutil.which("gcc") is None:
        pytest.skip("gcc not available")
    src = open(os.path.join(ROOT, "oracle", "ts_oracle.c")).read()
    old, new = MUTATIONS[name]
    assert src.count(old) == 1, f"mutation anchor not found: {old!r}"
    d = tmp_path / "mut"
    d.mkdir()
    (d / "ts_oracle.c").write_text(src.replace(old, new))
    shutil.copy(os.path.join(ROOT, "oracle", "ts_oracle.h"), d / "ts_oracle.h")
    so = d / "libmut.so"
    subprocess.check_call(["gcc", "-std=c11", "-O2", "-ffp-contract=off", "-fopenmp", "-shared",
                           "-fPIC", "-o", str(so), str(d / "ts_oracle.c"), "-lm"])
    env = dict(os.environ, TS_ORACLE_LIB_OVERRIDE=str(so))
    r = subprocess.run([sys.executable, "-m", "pytest", "-q", "-x", "-p", "no:cacheprovider",
                        os.path.join(ROOT, "tests", "test_oracle_pins.py")],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode != 0, f"pins did not catch mutation '{name}':\n{r.stdout[-2000:]}"
