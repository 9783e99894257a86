"""The oracle's pins catch plausible mistakes (CPU only).

Each case copies oracle/, synth/ and the pin tests into a temporary directory,
plants one mistake in the copied oracle source (a dropped term, a wrong sign,
a wrong index, a transposed operand, a broken tie rule), rebuilds it there and
runs the pins against it: at least one pin must fail.  The real oracle is
never modified.
"""
import os
import shutil
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

# (name, file, original text, planted text)
MUTATIONS = [
    ("silu_sign", "moe_oracle_body.h",
     "return v / (1.0 + exp(-v));", "return v / (1.0 + exp(v));"),
    ("gate_up_swapped", "moe_oracle_body.h",
     "g[i] += ah * LA(row, i);\n      u[i] += ah * LA(row, I + i);",
     "g[i] += ah * LA(row, I + i);\n      u[i] += ah * LA(row, i);"),
    ("down_transposed", "moe_oracle_body.h",
     "f_out[c] += hv[i] * LA(row, c);", "f_out[c] += hv[i] * LA(dn_e, c * I + i);"),
    ("tie_to_higher_index", "moe_oracle_body.h",
     "(best < 0 || p[e] > p[best])", "(best < 0 || p[e] >= p[best])"),
    ("renormalisation_dropped", "moe_oracle_body.h",
     "w[t * k + j] = p[ids[t * k + j]] / psum;", "w[t * k + j] = p[ids[t * k + j]];"),
    ("router_bias_dropped", "moe_oracle_body.h",
     "z[e] += LR(bias, e);", "z[e] += 0.0 * LR(bias, e);"),
    ("permute_unstable", "moe_oracle.c",
     "const int32_t row = offsets[e] + fill[e];", "const int32_t row = offsets[e + 1] - 1 - fill[e];"),
    ("combine_slot_swapped", "moe_oracle.c",
     "y[t * H + c] += w[t * k + j] * y_perm[row * H + c];",
     "y[t * H + c] += w[t * k + (k - 1 - j)] * y_perm[row * H + c];"),
    ("logit_grad_sign", "moe_oracle_body.h",
     "dz[ids[t * k + j]] = w[t * k + j] * (dw[j] - mean);",
     "dz[ids[t * k + j]] = w[t * k + j] * (mean - dw[j]);"),
    ("silu_grad_term", "moe_oracle_body.h",
     "dg[i] = dh * u[i] * sg * (1.0 + g[i] * (1.0 - sg));      /* dh * u * silu'(g) */",
     "dg[i] = dh * u[i] * sg;"),
    ("router_term_dropped_from_dx", "moe_oracle_body.h",
     "    dX[c] += acc;\n  }", "    dX[c] += 0.0 * acc;\n  }"),
    ("d_down_missing_gate_weight", "moe_oracle_body.h",
     "const double s = hv[r * I + i] * rw[r];", "const double s = hv[r * I + i];"),
    ("shared_expert_dropped", "moe_oracle_body.h",
     "  oracle_unpermute_combine(T, k, H, yp, row_map, w, ysh, y);",
     "  oracle_unpermute_combine(T, k, H, yp, row_map, w, NULL, y);"),
]


@pytest.mark.parametrize("name,fname,orig,planted", MUTATIONS, ids=[m[0] for m in MUTATIONS])
def test_pins_catch_planted_mistake(tmp_path, name, fname, orig, planted):
    for d in ("oracle", "synth"):
        shutil.copytree(os.path.join(ROOT, d), tmp_path / d,
                        ignore=shutil.ignore_patterns("*.so", "__pycache__"))
    (tmp_path / "tests").mkdir()
    for f in ("conftest.py", "test_oracle_pins.py"):
        shutil.copy(os.path.join(ROOT, "tests", f), tmp_path / "tests" / f)
    shutil.copytree(os.path.join(ROOT, "tests", "golden"), tmp_path / "tests" / "golden")
    src = tmp_path / "oracle" / fname
    text = src.read_text()
    assert text.count(orig) == 1, "mutation anchor must match exactly once: %s" % name
    src.write_text(text.replace(orig, planted))
    r = subprocess.run([sys.executable, "-m", "pytest", "-q", "-x", "-p", "no:cacheprovider",
                        "tests/test_oracle_pins.py"], cwd=tmp_path, capture_output=True, text=True,
                       timeout=600)
    assert r.returncode == 1, "planted mistake %r was not caught:\n%s" % (name, r.stdout[-2000:])
