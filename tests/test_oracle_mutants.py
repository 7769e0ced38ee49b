"""Plant plausible mistakes in a copy of the oracle's C source (on the CPU) and
check that the pins in ``test_oracle_pins.py`` catch every one of them.

Each mutant is compiled to a temporary library and the pin suite runs against
it in a child process (``ORACLE_LIB`` selects the library); the child must
fail.  A mutant that crashes the child counts as caught too.  The committed
oracle source itself is never modified.
"""
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "oracle.c")

# (name, text in oracle.c, replacement)
MUTANTS = [
    ("dropped_last_term", "for (int64_t k = 0; k < j->K; ++k) acc += a[k] * b[k];",
     "for (int64_t k = 0; k + 1 < j->K; ++k) acc += a[k] * b[k];"),
    ("entries_dropped_first_term",
     "for (int64_t k = 0; k < K; ++k) acc += oracle_f16_to_f64(a[k])",
     "for (int64_t k = 1; k < K; ++k) acc += oracle_f16_to_f64(a[k])"),
    ("transposed_b", "const double *b = j->B + n * j->K;",
     "const double *b = j->B + n;"),
    ("subtract_instead_of_add", "acc += a[k] * b[k];", "acc -= a[k] * b[k];"),
    ("row_col_swap_in_c", "j->C[(m - j->m_begin) * j->N + n] = acc;",
     "j->C[n * (j->m_end - j->m_begin) + (m - j->m_begin)] = acc;"),
    ("decode_drops_sign", "return sign ? -v : v;", "return v;"),
    ("decode_bias_off_by_one", "v = ldexp((double)(1024 + f), e - 25);",
     "v = ldexp((double)(1024 + f), e - 24);"),
    ("decode_subnormal_scale", "v = ldexp((double)f, -24);", "v = ldexp((double)f, -23);"),
    ("rounding_ties_away", "return (fmod(fl, 2.0) == 0.0) ? fl : fl + 1.0;", "return fl + 1.0;"),
    ("rounding_truncates", "if (frac > 0.5) return fl + 1.0;", "if (frac > 2.0) return fl + 1.0;"),
    ("overflow_threshold", "if (a >= 65520.0)", "if (a > 65504.0)"),
    ("thread_split_overlaps", "jobs[t].A = A_rows + (at - m_begin) * K;",
     "jobs[t].A = A_rows;"),
]


def _build_mutant(tmpdir, name, old, new):
    src = open(SRC).read()
    assert src.count(old) >= 1, "mutation anchor for %s not found in oracle.c" % name
    path_c = os.path.join(tmpdir, name + ".c")
    path_so = os.path.join(tmpdir, name + ".so")
    with open(path_c, "w") as f:
        f.write(src.replace(old, new))
    subprocess.run(["gcc", "-O1", "-std=c11", "-fPIC", "-shared", "-pthread", path_c, "-o",
                    path_so, "-lm"], check=True)
    return path_so


def test_pristine_oracle_passes_the_pins(tmp_path):
    so = _build_mutant(str(tmp_path), "pristine", "#include <math.h>", "#include <math.h>")
    env = dict(os.environ, ORACLE_LIB=so)
    r = subprocess.run([sys.executable, "-m", "pytest", "-q", "-x", "-p", "no:cacheprovider",
                        os.path.join(ROOT, "tests", "test_oracle_pins.py")],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stdout[-2000:]


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_pins_catch_planted_mistake(tmp_path, name, old, new):
    so = _build_mutant(str(tmp_path), name, old, new)
    env = dict(os.environ, ORACLE_LIB=so)
    r = subprocess.run([sys.executable, "-m", "pytest", "-q", "-x", "-p", "no:cacheprovider",
                        os.path.join(ROOT, "tests", "test_oracle_pins.py")],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode != 0, "mutant %s survived the pins:\n%s" % (name, r.stdout[-2000:])
