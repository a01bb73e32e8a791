"""The oracle's pins catch plausible mistakes.

Each case plants one mistake in a temporary copy of oracle/oracle.c (a transposed
operand, a wrong sign or index, a dropped term), builds it, and runs the pin suite
(tests/test_oracle.py) against it in a subprocess: the suite must fail.  The
committed oracle is never modified.
"""
import os
import shutil
import subprocess
import sys
import tempfile
from concurrent.futures import ThreadPoolExecutor

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "oracle.c")

MUTANTS = {
    "accept_operands_transposed": ("if (!(u[t] * b < a)) { n = t; break; }",
                                   "if (!(u[t] * a < b)) { n = t; break; }"),
    "residual_sign_flipped": ("r[x] = fmax(0.0, pt[x] - pd[x]);", "r[x] = fmax(0.0, pd[x] - pt[x]);"),
    "bonus_from_wrong_row": ("const double* pt = P + (size_t)n * V;",
                             "const double* pt = P + (size_t)(n == K ? 0 : n) * V;"),
    "temperature_multiplies": ("w[x] = isinf(l[x]) ? 0.0 : exp(l[x] / T - m);",
                               "w[x] = isinf(l[x]) ? 0.0 : exp(l[x] * T - lmax * T);"),
    "top_k_off_by_one": ("nkeep = top_k;", "nkeep = top_k + 1;"),
    "top_p_drops_crossing_token": ("if (cum / zk >= p) { cut = j; break; }",
                                   "if (cum / zk >= p) { cut = j > 0 ? j - 1 : 0; break; }"),
    "tie_break_reversed": ("return (p->x > q->x) - (p->x < q->x);", "return (p->x < q->x) - (p->x > q->x);"),
    "cdf_walks_backwards": ("for (int32_t x = 0; x < V; ++x) {\n    if (!(r[x] > 0.0)) continue;",
                            "for (int32_t x = V - 1; x >= 0; --x) {\n    if (!(r[x] > 0.0)) continue;"),
    "argmax_ties_to_last": ("if (best < 0 || l[x] > lmax) {", "if (best < 0 || l[x] >= lmax) {"),
    "normalise_over_all_tokens": ("if (kept[x]) zf += w[x];", "zf += w[x];"),
    "nan_not_detected": ("if (isnan(l[x]) || (isinf(l[x]) && l[x] > 0)) status = ORACLE_ERR_NONFINITE;",
                         "if (isinf(l[x]) && l[x] > 0) status = ORACLE_ERR_NONFINITE;"),
    "residual_uses_next_row": ("const double* pd = P + (size_t)(nt + n) * V;",
                               "const double* pd = P + (size_t)(nt + (n + 1 < K ? n + 1 : n)) * V;"),
    "histogram_drops_all_accepted": ("if (n >= 0 && n <= K)", "if (n >= 0 && n < K)"),
    "histogram_bins_off_by_one": ("hist[n] += 1;", "hist[n > 0 ? n - 1 : 0] += 1;"),
}


def _run_mutant(name, tmp):
    old, new = MUTANTS[name]
    src = open(SRC).read()
    assert src.count(old) == 1, "mutation site for %s not found exactly once" % name
    d = os.path.join(tmp, name)
    os.makedirs(d)
    shutil.copy(os.path.join(ROOT, "oracle", "oracle.h"), d)
    with open(os.path.join(d, "oracle.c"), "w") as f:
        f.write(src.replace(old, new))
    so = os.path.join(d, "libmutant.so")
    subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-o", so,
                           os.path.join(d, "oracle.c"), "-lm"])
    env = dict(os.environ, ORACLE_LIB=so)
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
                        os.path.join(ROOT, "tests", "test_oracle.py")],
                       env=env, cwd=ROOT, capture_output=True, text=True, timeout=900)
    return r.returncode


@pytest.fixture(scope="module")
def results():
    tmp = tempfile.mkdtemp(prefix="oracle_mutants_")
    try:
        with ThreadPoolExecutor(max_workers=min(8, os.cpu_count() or 1)) as ex:
            codes = dict(zip(MUTANTS, ex.map(lambda n: _run_mutant(n, tmp), MUTANTS)))
    finally:
        shutil.rmtree(tmp, ignore_errors=True)
    return codes


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_reject_mutant(results, name):
    assert results[name] != 0, "the pin suite passed with mutation %s planted" % name
