"""The oracle's pins catch plausible mistakes.

Each case plants one mistake in a temporary copy of oracle/oracle.c or oracle/oracle.h
(a transposed operand, a wrong sign or index, a dropped term, a misplaced or
mis-sized near-threshold band), builds it, and runs the pin suite
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
ORACLE_DIR = os.path.join(ROOT, "oracle")

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
    # the near-threshold flags, which decide every exclusion from bit-exact parity
    "draw_band_scaled_by_R": (
        "*near = fabs(u - prev / R) < ORACLE_NEAR_EPS || fabs(u - cum / R) < ORACLE_NEAR_EPS;",
        "*near = fabs(target - prev) < ORACLE_NEAR_EPS || fabs(target - cum) < ORACLE_NEAR_EPS;"),
    "draw_lower_edge_dropped": (
        "*near = fabs(u - prev / R) < ORACLE_NEAR_EPS || fabs(u - cum / R) < ORACLE_NEAR_EPS;",
        "*near = fabs(u - cum / R) < ORACLE_NEAR_EPS;"),
    "draw_upper_edge_dropped": (
        "*near = fabs(u - prev / R) < ORACLE_NEAR_EPS || fabs(u - cum / R) < ORACLE_NEAR_EPS;",
        "*near = fabs(u - prev / R) < ORACLE_NEAR_EPS;"),
    "accept_band_on_products": ("if (fabs(u[t] - ratio) < ORACLE_NEAR_EPS) fl |= ORACLE_NEAR_ACCEPT;",
                                "if (fabs(u[t] * b - a) < ORACLE_NEAR_EPS) fl |= ORACLE_NEAR_ACCEPT;"),
    "accept_flags_every_position": ("if (!(u[t] * b < a)) { n = t; break; }",
                                    "if (!(u[t] * b < a) && n == K) n = t;"),
    "topp_prev_edge_dropped": (
        "(fabs(cum / zk - p) < ORACLE_NEAR_EPS || (cut > 0 && fabs(prev / zk - p) < ORACLE_NEAR_EPS))",
        "(fabs(cum / zk - p) < ORACLE_NEAR_EPS)"),
    "topp_band_unnormalised": (
        "(fabs(cum / zk - p) < ORACLE_NEAR_EPS || (cut > 0 && fabs(prev / zk - p) < ORACLE_NEAR_EPS))",
        "(fabs(cum - p) < ORACLE_NEAR_EPS || (cut > 0 && fabs(prev - p) < ORACLE_NEAR_EPS))"),
    "near_band_ten_times_wider": ("#define ORACLE_NEAR_EPS 1e-6", "#define ORACLE_NEAR_EPS 1e-5", "oracle.h"),
    "near_band_ten_times_narrower": ("#define ORACLE_NEAR_EPS 1e-6", "#define ORACLE_NEAR_EPS 1e-7", "oracle.h"),
}


def _run_mutant(name, tmp):
    old, new, *where = MUTANTS[name]
    fname = where[0] if where else "oracle.c"
    d = os.path.join(tmp, name)
    os.makedirs(d)
    for f in ("oracle.c", "oracle.h"):
        shutil.copy(os.path.join(ORACLE_DIR, f), d)
    src = open(os.path.join(ORACLE_DIR, fname)).read()
    assert src.count(old) == 1, "mutation site for %s not found exactly once" % name
    with open(os.path.join(d, fname), "w") as f:
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
