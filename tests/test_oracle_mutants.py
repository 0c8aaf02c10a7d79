"""The pins catch plausible mistakes: each case plants one mistake in a copy of
the oracle's C source (on the CPU, in a temporary directory), builds it, and
runs the pin suite against that build, which must fail.  The unmodified
oracle passes the same suite (tests/test_oracle_pins.py in the normal run)."""
import os
import subprocess
import sys

import pytest

from conftest import ROOT

SRC = os.path.join(ROOT, "oracle", "csa2_oracle.c")

# (name, exact text in the oracle, the planted replacement)
MUTANTS = [
    ("fp4 tie to the odd code", "(d == bd && i % 2 == 0)", "(d == bd && i % 2 == 1)"),
    ("fp4 scale strictly above amax / 6", "if (6.0 * or_e4m3_value(b) >= amax) return b;",
     "if (6.0 * or_e4m3_value(b) > amax) return b;"),
    ("nibble order swapped", "codes[i] = (uint8_t)(nib[2 * i] | (nib[2 * i + 1] << 4));",
     "codes[i] = (uint8_t)(nib[2 * i + 1] | (nib[2 * i] << 4));"),
    ("fp8 scale one step early", "while (ldexp(448.0, e) < amax) ++e;",
     "while (ldexp(448.0, e) <= amax) ++e;"),
    ("softmax(Z) sign", "double e = exp((double)Z[i * OR_D + c] - zmax);",
     "double e = exp(zmax - (double)Z[i * OR_D + c]);"),
    ("missing ReLU", "s += (double)w[h] * (dot > 0.0 ? dot : 0.0);", "s += (double)w[h] * dot;"),
    ("top-k ties to the higher position", "return (x->p < y->p) ? -1 : (x->p > y->p);",
     "return (x->p > y->p) ? -1 : (x->p < y->p);"),
    ("partial pool block counted whole", "hi = lo + 8 < n ? lo + 8 : n;", "hi = lo + 8;"),
    ("window one row longer", "int64_t lo = t - n_win + 1;", "int64_t lo = t - n_win;"),
    ("visibility counts the open block", "int64_t nt = (t + 1) / a->m;", "int64_t nt = t / a->m + 1;"),
    ("projection with W_IK transposed", "or_bf16_value(w_ik[c * d_idx + d])",
     "or_bf16_value(w_ik[d * OR_D + c])"),
]


@pytest.mark.parametrize("name,orig,planted", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_pins_catch_planted_mistake(name, orig, planted, tmp_path):
    src = open(SRC).read()
    assert src.count(orig) == 1, name
    mut = tmp_path / "csa2_oracle.c"
    mut.write_text(src.replace(orig, planted))
    so = tmp_path / "liboracle_mutant.so"
    subprocess.run(["gcc", "-O2", "-std=c11", "-shared", "-fPIC", "-o", str(so), str(mut), "-lm"],
                   check=True, capture_output=True)
    env = dict(os.environ, CSA2_ORACLE_LIB=str(so))
    r = subprocess.run([sys.executable, "-m", "pytest", os.path.join(ROOT, "tests", "test_oracle_pins.py"),
                        "-x", "-q", "-p", "no:cacheprovider"], cwd=ROOT, env=env,
                       capture_output=True, text=True, timeout=600)
    assert r.returncode == 1 and " failed" in r.stdout, (name, r.stdout[-2000:])
