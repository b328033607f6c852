"""The oracle's pins catch plausible slips.

Each mutant plants one mistake in a copy of the oracle's C source -- a dropped term, a wrong
sign, bound or index, a transposed operand -- and runs the pin tests (the oracle against the
pages' closed forms, brute force, library reductions and finite differences) on that copy
through the loader's PI_ORACLE_SRC override.  Every mutant must fail at least one pin, and the
unchanged copy must pass them all.  CPU only; nothing here touches the CUDA library.
"""
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
ORACLE_C = os.path.join(ROOT, "oracle", "oracle.c")
PIN_FILES = ["tests/test_oracle_pins.py", "tests/test_oracle_pins_bidir.py", "tests/test_oracle_pins_gate.py"]

# (name, text in oracle.c, its replacement): each text occurs exactly once
MUTANTS = [
    ("skip prior dropped",
     "prior = (tag[t] == 0) ? log(a) : log1p(-a);", "prior = (tag[t] == 0) ? log(a) : 0.0;"),
    ("band prior on skip keys",
     "prior = (tag[t] == 0) ? log(a) : log1p(-a);", "prior = log(a);"),
    ("skip at m*pi = k kept beside the band key",
     "if (back <= k_local) continue;   /* inside the band already */",
     "if (back < k_local) continue;"),
    ("band one key short",
     "for (j = lo; j <= i; ++j) { idx[n] = j; tag[n] = 0; ++n; }\n        for (int m = 1; m <= S; ++m) {\n            long back",
     "for (j = lo; j < i; ++j) { idx[n] = j; tag[n] = 0; ++n; }\n        for (int m = 1; m <= S; ++m) {\n            long back"),
    ("ECP window starts one half-segment late", "lo = (s - 1) * k_local;", "lo = s * k_local;"),
    ("bidirectional forward skips dropped",
     "if (i + off < N) { idx[n] = i + off; tag[n] = 1; ++n; }", ""),
    ("scale dropped in the logits", "z[t] = dot * scale + prior;", "z[t] = dot + prior;"),
    ("lse without the maximum", "return M + log(l);", "return log(l);"),
    ("GQA map h mod Hkv", "long g = h / (H / Hkv);", "long g = h % Hkv;"),
    ("scale dropped in dK", "dkg[koff + c] += dz * qrow[c] * scale;", "dkg[koff + c] += dz * qrow[c];"),
    ("dV from q instead of dout", "dvg[koff + c] += p[t] * grow[c];", "dvg[koff + c] += p[t] * qrow[c];"),
    ("D_i dropped from dz", "double dz = p[t] * (dp - D);", "double dz = p[t] * dp;"),
    ("sign of dalpha's skip term",
     "g_a = sum_local / a - sum_skip / (1.0 - a);", "g_a = sum_local / a + sum_skip / (1.0 - a);"),
    ("gate weights read transposed", "w1[(h * F + f) * d + t]", "w1[(h * d + t) * F + f]"),
    ("gate ReLU dropped", "if (pre > 0.0) z += w2[h * F + f] * pre;", "z += w2[h * F + f] * pre;"),
    ("gate hidden bias dropped", "double pre = b1[h * F + f];", "double pre = 0.0;"),
    ("gate logit doubled", "alpha[row] = 1.0 / (1.0 + exp(-z));", "alpha[row] = 1.0 / (1.0 + exp(-2.0 * z));"),
    ("GQA group sum of dK/dV cut to one head",
     "for (long h = g * G; h < (g + 1) * G; ++h) {", "for (long h = g * G; h < g * G + 1; ++h) {"),
    ("scale dropped in dQ", "dqrow[c] += dz * kg[koff + c] * scale;", "dqrow[c] += dz * kg[koff + c];"),
    ("gate output weights of head 0", "if (pre > 0.0) z += w2[h * F + f] * pre;", "if (pre > 0.0) z += w2[f] * pre;"),
    ("gate output bias of head 0", "double z = b2[h];", "double z = b2[0];"),
    ("ECP first segment's window clamped wrongly",
     "        lo = (s - 1) * k_local;\n        if (lo < 0) lo = 0;",
     "        lo = (s - 1) * k_local;\n        if (lo < 0) lo = k_local;"),
    ("bidirectional band one key short on the right", "hi = i + k_local;", "hi = i + k_local - 1;"),
    ("first skip multiple dropped",
     "for (int m = 1; m <= S; ++m) {\n            long back", "for (int m = 2; m <= S; ++m) {\n            long back"),
]


def run_pins(src_path):
    env = dict(os.environ, PI_ORACLE_SRC=src_path)
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider", *PIN_FILES],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=900)
    return r.returncode, (r.stdout + r.stderr)[-3000:]


def test_pins_pass_on_an_unchanged_copy(tmp_path):
    p = tmp_path / "oracle.c"
    p.write_text(open(ORACLE_C).read())
    rc, out = run_pins(str(p))
    assert rc == 0, out


@pytest.mark.parametrize("old,new", [(m[1], m[2]) for m in MUTANTS], ids=[m[0] for m in MUTANTS])
def test_each_planted_slip_fails_a_pin(tmp_path, old, new):
    src = open(ORACLE_C).read()
    assert src.count(old) == 1, "the mutant's text must occur once in oracle.c"
    p = tmp_path / "oracle.c"
    p.write_text(src.replace(old, new))
    rc, out = run_pins(str(p))
    assert rc == 1, f"pytest exit code {rc} (1 = a pin failed):\n{out}"
