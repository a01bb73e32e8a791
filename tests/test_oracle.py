"""Pins of the fp64 oracle against what the pages and the mathematics fix.

Every test here runs on the CPU.  None retypes the oracle's formulas: each
checks it against a printed value (tests/golden), a closed form, a theorem, an
invariant, a library routine, or brute-force enumeration (tests/brute.py).
"""
import math

import numpy as np
import pytest
from scipy import stats

import oracle
import workloads
from brute import chain_law, exact_law, expected_tokens
from conftest import read_golden


def logits_of(p):
    """fp32 logits whose softmax at T=1 is p (zero probability -> -inf)."""
    p = np.asarray(p, np.float64)
    with np.errstate(divide="ignore"):
        return np.log(p).astype(np.float32)


def probs_of(row, **kw):
    probs, _, _, _, s = oracle.row_probs(row, **kw)
    assert s == oracle.OK
    return probs


# --------------------------------------------------------------------------
# worked example ("Speculative Decoding", "Why the output doesn't change")


def test_worked_example_acceptance_and_residual():
    g = read_golden("worked_example.txt")
    tgt = probs_of(logits_of(g["target"]))
    drf = probs_of(logits_of(g["draft"]))
    np.testing.assert_allclose(tgt, g["target"], rtol=1e-6)
    np.testing.assert_allclose(drf, g["draft"], rtol=1e-6)
    assert abs(np.minimum(tgt, drf).sum() - g["acceptance"]) < 1e-6
    # the only positive residual is on word 0, so every rejection emits word 0
    r = np.maximum(0, tgt - drf)
    assert r[0] > 0 and np.all(r[1:] < 1e-7)


def _repeat_rows(rows, dtype=np.float32):
    """[R, V] rows laid out as one sequence, repeated B times through stride 0."""
    return np.ascontiguousarray(np.asarray(rows, dtype))


def test_worked_example_monte_carlo_follows_target_not_draft():
    g = read_golden("worked_example.txt")
    lt, ld = logits_of(g["target"]), logits_of(g["draft"])
    tgt_p, drf_p = probs_of(lt), probs_of(ld)
    B = 200_000
    rng = np.random.default_rng(11)
    target = _repeat_rows([lt, lt])       # K = 1: position 0 and the bonus row
    draft = _repeat_rows([ld])
    d = rng.choice(4, size=(B, 1), p=drf_p).astype(np.int32)
    u = rng.random((B, 2))
    res = oracle.verify(target, draft, d, u, tgt_strides=(0, 4), drf_strides=(0, 4), B=B)
    assert res["status"] == oracle.OK
    y0 = res["tokens"][:, 0]
    counts = np.bincount(y0, minlength=4)
    # acceptance rate 0.8 within 4 sigma
    acc = (res["num_accepted"] == 1).mean()
    assert abs(acc - 0.8) < 4 * math.sqrt(0.8 * 0.2 / B)
    # every rejection emits word 0 (the whole residual mass sits there)
    assert np.all(y0[res["num_accepted"] == 0] == 0)
    # emitted words follow the target (chi-square), and the draft is rejected
    assert stats.chisquare(counts, B * tgt_p).pvalue > 1e-3
    assert stats.chisquare(counts, B * drf_p).pvalue < 1e-12


# --------------------------------------------------------------------------
# closed form ("Speculative Decoding", "How much faster")


def test_closed_form_printed_numbers():
    g = read_golden("closed_form.txt")
    a, gam, c = g["alpha"], int(g["gamma"]), g["c"]
    tokens = (1 - a ** (gam + 1)) / (1 - a)
    assert abs(tokens - g["tokens_per_pass"]) < 0.005          # 3.3616 printed as 3.36
    assert abs(tokens / (gam * c + 1) - g["speedup"]) < 0.05    # 2.80 printed as 2.8
    assert abs(expected_tokens([a] * gam) - tokens) < 1e-12


@pytest.mark.parametrize("alpha,K", [(0.8, 4), (0.5, 3), (0.95, 2)])
def test_expected_tokens_per_round_closed_form(alpha, K):
    # rows built so that sum_x min(tgt, drf) = alpha exactly: draft on words 0..3,
    # target = alpha * draft + (1 - alpha) * uniform on words 4..7
    drf = np.array([0.4, 0.3, 0.2, 0.1, 0, 0, 0, 0])
    tgt = alpha * drf + (1 - alpha) * np.array([0, 0, 0, 0, .25, .25, .25, .25])
    lt, ld = logits_of(tgt), logits_of(drf)
    tp, dp = probs_of(lt), probs_of(ld)
    assert abs(np.minimum(tp, dp).sum() - alpha) < 1e-6
    B = 200_000
    rng = np.random.default_rng(5)
    target = _repeat_rows([lt] * (K + 1))
    draft = _repeat_rows([ld] * K)
    d = np.stack([rng.choice(8, size=B, p=dp) for _ in range(K)], 1).astype(np.int32)
    u = rng.random((B, K + 1))
    res = oracle.verify(target, draft, d, u, tgt_strides=(0, 8), drf_strides=(0, 8), B=B)
    n1 = res["num_accepted"] + 1
    want = (1 - alpha ** (K + 1)) / (1 - alpha)
    assert abs(n1.mean() - want) < 4 * n1.std() / math.sqrt(B)


@pytest.mark.parametrize("alpha,K", [(0.8, 4), (0.5, 3)])
def test_accept_histogram_follows_truncated_geometric_law(alpha, K):
    """Acceptance telemetry ("Speculative decoding: how to run large models faster",
    "Limitations and open issues").  With acceptance alpha at every position the
    accept tests are independent, so a round accepts j < K tokens with probability
    alpha^j (1 - alpha) and all K with alpha^K; the histogram's mean tokens per
    round is then the printed closed form."""
    drf = np.array([0.4, 0.3, 0.2, 0.1, 0, 0, 0, 0])
    tgt = alpha * drf + (1 - alpha) * np.array([0, 0, 0, 0, .25, .25, .25, .25])
    lt, ld = logits_of(tgt), logits_of(drf)
    dp = probs_of(ld)
    B = 100_000
    rng = np.random.default_rng(9)
    d = np.stack([rng.choice(8, size=B, p=dp) for _ in range(K)], 1).astype(np.int32)
    u = rng.random((B, K + 1))
    d[:50, 0] = 8                                   # 50 sequences with an out-of-range token
    res = oracle.verify(_repeat_rows([lt] * (K + 1)), _repeat_rows([ld] * K), d, u,
                        tgt_strides=(0, 8), drf_strides=(0, 8), B=B)
    hist = oracle.accept_histogram(res["num_accepted"], K)
    assert hist.shape == (K + 2,) and hist.sum() == B and hist[K + 1] == 50
    ok = B - 50
    law = np.array([alpha ** j * (1 - alpha) for j in range(K)] + [alpha ** K])
    assert stats.chisquare(hist[:K + 1], law * ok).pvalue > 1e-4
    mean_tokens = (np.arange(1, K + 2) * hist[:K + 1]).sum() / ok
    want = (1 - alpha ** (K + 1)) / (1 - alpha)
    assert abs(mean_tokens - want) < 4 * math.sqrt(K * K / ok)


def test_accept_histogram_bins_every_value():
    """Bins 0..K count exactly the sequences with that many accepted tokens; every
    other value (an error) lands in bin K+1 -- checked on all values in [-3, K+3]."""
    K = 5
    vals = np.arange(-3, K + 4, dtype=np.int32)
    counts = np.arange(1, vals.size + 1)
    n = np.repeat(vals, counts)
    np.random.default_rng(2).shuffle(n)
    hist = oracle.accept_histogram(n, K)
    for v, c in zip(vals, counts):
        if 0 <= v <= K:
            assert hist[v] == c
    assert hist[K + 1] == counts[(vals < 0) | (vals > K)].sum()
    assert hist.sum() == n.size


# --------------------------------------------------------------------------
# Theorem 1 and brute force


def _random_case(rng, V, K, T=1.0, top_k=0, top_p=1.0, peaked=1.0):
    tl = (rng.normal(0, 2 * peaked, (K + 1, V))).astype(np.float32)
    dl = (tl[:K] + rng.normal(0, 1.0, (K, V))).astype(np.float32)
    kw = dict(temperature=T, top_k=top_k, top_p=top_p)
    tp = [probs_of(r, **kw) for r in tl]
    dp = [probs_of(r, **kw) for r in dl]
    return tl, dl, tp, dp, kw


@pytest.mark.parametrize("seed,V,K,T,top_k,top_p", [
    (0, 4, 1, 1.0, 0, 1.0), (1, 5, 2, 0.7, 0, 1.0), (2, 6, 2, 1.3, 3, 1.0),
    (3, 8, 2, 1.0, 0, 0.8), (4, 7, 2, 0.9, 4, 0.9), (5, 3, 2, 1.0, 0, 1.0)])
def test_brute_force_equals_theorem1_chain_law(seed, V, K, T, top_k, top_p):
    rng = np.random.default_rng(seed)
    _, _, tp, dp, _ = _random_case(rng, V, K, T, top_k, top_p)
    ex, ch = exact_law(tp, dp), chain_law(tp, dp)
    keys = set(ex) | set(ch)
    assert max(abs(ex.get(k, 0) - ch.get(k, 0)) for k in keys) < 1e-12
    assert abs(sum(ex.values()) - 1) < 1e-12
    # every emitted position follows its target row (Theorem 1)
    for j in range(K + 1):
        reach = sum(v for k, v in ex.items() if len(k) > j)
        if reach > 1e-9:
            marg = np.zeros(V)
            for k, v in ex.items():
                if len(k) > j:
                    marg[k[j]] += v
            np.testing.assert_allclose(marg / reach, tp[j], atol=1e-12)


@pytest.mark.parametrize("seed,V,K,T,top_k,top_p", [
    (10, 5, 2, 1.0, 0, 1.0), (11, 6, 2, 0.8, 3, 1.0), (12, 8, 1, 1.0, 0, 0.85),
    (13, 4, 2, 1.2, 0, 1.0)])
def test_oracle_monte_carlo_matches_brute_force_law(seed, V, K, T, top_k, top_p):
    rng = np.random.default_rng(seed)
    tl, dl, tp, dp, kw = _random_case(rng, V, K, T, top_k, top_p)
    law = exact_law(tp, dp)
    B = 300_000
    d = np.stack([rng.choice(V, size=B, p=dp[t]) for t in range(K)], 1).astype(np.int32)
    u = rng.random((B, K + 1))
    res = oracle.verify(np.ascontiguousarray(tl), np.ascontiguousarray(dl), d, u,
                        tgt_strides=(0, V), drf_strides=(0, V), B=B, **kw)
    assert res["status"] == oracle.OK
    emp = {}
    for row, n in zip(res["tokens"], res["num_accepted"]):
        key = tuple(row[: n + 1])
        emp[key] = emp.get(key, 0) + 1
    assert set(emp) <= {k for k, v in law.items() if v > 0}
    keys = sorted(k for k, v in law.items() if v * B >= 5)
    obs = np.array([emp.get(k, 0) for k in keys], float)
    exp = np.array([law[k] for k in keys]) * B
    rest_o, rest_e = B - obs.sum(), B - exp.sum()
    if rest_e >= 5:
        obs, exp = np.append(obs, rest_o), np.append(exp, rest_e)
    exp *= obs.sum() / exp.sum()
    assert stats.chisquare(obs, exp).pvalue > 1e-4


def test_oracle_thresholds_match_brute_force_by_uniform_scan():
    """Scan one uniform over a fine lattice with everything else fixed: the measure of
    u giving each outcome is the brute-force probability (min(1, tgt/drf) for the test,
    r/R for the residual draw, tgt for the bonus)."""
    rng = np.random.default_rng(21)
    V, K = 6, 1
    tl, dl, tp, dp, kw = _random_case(rng, V, K)
    N = 100_000
    grid = (np.arange(N) + 0.5) / N
    target, draft = np.ascontiguousarray(tl), np.ascontiguousarray(dl)
    for dtok in range(V):
        d = np.full((N, 1), dtok, np.int32)
        u = np.stack([grid, np.full(N, 0.5)], 1)
        res = oracle.verify(target, draft, d, u, tgt_strides=(0, V), drf_strides=(0, V), B=N)
        acc = (res["num_accepted"] == 1).mean()
        assert abs(acc - min(1.0, tp[0][dtok] / dp[0][dtok])) <= 2.0 / N
    # residual draw: reject at 0 (u_0 close to 1 rejects any token with tgt < drf)
    dtok = int(np.argmax(dp[0] - tp[0]))
    d = np.full((N, 1), dtok, np.int32)
    u = np.stack([np.full(N, 1 - 1e-12), grid], 1)
    res = oracle.verify(target, draft, d, u, tgt_strides=(0, V), drf_strides=(0, V), B=N)
    assert np.all(res["num_accepted"] == 0)
    freq = np.bincount(res["tokens"][:, 0], minlength=V) / N
    r = np.maximum(0, tp[0] - dp[0])
    np.testing.assert_allclose(freq, r / r.sum(), atol=2.0 / N)
    # bonus draw: accept at 0 (u_0 = 0 accepts any token with tgt > 0)
    dtok = int(np.argmax(tp[0]))
    d = np.full((N, 1), dtok, np.int32)
    u = np.stack([np.zeros(N), grid], 1)
    res = oracle.verify(target, draft, d, u, tgt_strides=(0, V), drf_strides=(0, V), B=N)
    assert np.all(res["num_accepted"] == 1)
    freq = np.bincount(res["tokens"][:, 1], minlength=V) / N
    np.testing.assert_allclose(freq, tp[1], atol=2.0 / N)


# --------------------------------------------------------------------------
# special cases that reduce to textbook / library routines


def _softmax_numpy(row, T=1.0):
    # the temperature crosses the ABI as fp32, so the reference uses that value
    x = row.astype(np.float64) / float(np.float32(T))
    e = np.exp(x - x.max())
    return e / e.sum()


def test_unfiltered_row_is_numpy_softmax_and_logsumexp():
    rng = np.random.default_rng(3)
    for V, T in [(7, 1.0), (1000, 0.6), (33333, 1.7)]:
        row = (rng.normal(0, 3, V)).astype(np.float32)
        probs, amax, _, (m, zf), s = oracle.row_probs(row, temperature=T)
        np.testing.assert_allclose(probs, _softmax_numpy(row, T), rtol=1e-12, atol=1e-300)
        assert amax == int(np.argmax(row)) and m == float(row.max())
        T32 = float(np.float32(T))
        lse = math.log(math.fsum(math.exp((float(x) - m) / T32) for x in row))
        assert abs(math.log(zf) - lse) < 1e-12


def test_draft_equal_target_accepts_all_and_bonus_is_categorical():
    rng = np.random.default_rng(4)
    B, K, V = 500, 3, 50
    tl = rng.normal(0, 2, (B, K + 1, V)).astype(np.float32)
    dl = np.ascontiguousarray(tl[:, :K])
    d = np.zeros((B, K), np.int32)
    for b in range(B):
        for t in range(K):
            d[b, t] = rng.choice(V, p=_softmax_numpy(tl[b, t]))
    u = rng.random((B, K + 1))
    res = oracle.verify(tl, dl, d, u)
    assert np.all(res["num_accepted"] == K)
    np.testing.assert_array_equal(res["tokens"][:, :K], d)
    for b in range(B):
        cdf = np.cumsum(_softmax_numpy(tl[b, K]))
        want = int(np.searchsorted(cdf, u[b, K] * cdf[-1], side="right"))
        if not (res["flags"][b] & oracle.NEAR_DRAW):
            assert res["tokens"][b, K] == want


def test_greedy_is_argmax_longest_prefix():
    rng = np.random.default_rng(6)
    B, K, V = 400, 4, 64
    # bf16-rounded values give many exact ties; argmax ties go to the lowest index
    tl = workloads.to_bf16_bits(np.round(rng.normal(0, 2, (B, K + 1, V)) * 2) / 2)
    tf = workloads.bf16_bits_to_f32(tl)
    am = np.argmax(tf, axis=-1)
    d = np.where(rng.random((B, K)) < 0.7, am[:, :K], rng.integers(0, V, (B, K))).astype(np.int32)
    res = oracle.verify(tl, None, d, None, greedy=True)
    for b in range(B):
        n = 0
        while n < K and d[b, n] == am[b, n]:
            n += 1
        assert res["num_accepted"][b] == n
        assert list(res["tokens"][b, :n]) == list(d[b, :n])
        assert res["tokens"][b, n] == am[b, n]
        assert np.all(res["tokens"][b, n + 1:] == -1)


def _order(row):
    """Token order by (raw logit desc, index asc), via numpy's lexsort."""
    return np.lexsort((np.arange(len(row)), -row.astype(np.float64)))


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_filters_match_sort_definition_and_invariants(dtype):
    rng = np.random.default_rng(8)
    V = 3000
    for trial in range(12):
        raw = rng.normal(0, 3, V) - 1.1 * np.log(1 + rng.permutation(V))
        row = workloads.to_bf16_bits(raw) if dtype == "bf16" else raw.astype(np.float32)
        lf = workloads.bf16_bits_to_f32(row) if dtype == "bf16" else row
        T = [0.5, 0.8, 1.0, 1.6][trial % 4]
        top_k = [0, 1, 50, 2999][trial % 4]
        top_p = [1.0, 0.9, 0.5, 0.999][(trial // 4) % 4]
        probs, amax, near, (m, zf), s = oracle.row_probs(row, temperature=T, top_k=top_k,
                                                         top_p=top_p)
        assert s == oracle.OK
        kept = probs > 0
        order = _order(lf)
        nk = int(kept.sum())
        # the kept set is a prefix of the order
        assert kept[order[:nk]].all() and not kept[order[nk:]].any()
        if top_k:
            assert nk <= top_k
        # on the kept set, ratios follow the tempered logits (closed form)
        ks = order[:nk]
        np.testing.assert_allclose(probs[ks] / probs[ks[0]],
                                   np.exp((lf[ks].astype(np.float64) - lf[ks[0]]) / float(np.float32(T))),
                                   rtol=1e-9)
        assert abs(probs.sum() - 1) < 1e-12
        # the top-p crossing: mass before the last kept token < top_p <= mass with it
        if top_p < 1 and not near:
            w = np.exp((lf[order].astype(np.float64) - lf[order[0]]) / float(np.float32(T)))
            base = w[: (top_k or V)].sum()
            cum = np.cumsum(w[:nk]) / base
            assert cum[-1] >= top_p and (nk == 1 or cum[-2] < top_p)
        if top_k == 1:
            assert nk == 1 and probs[amax] == 1.0


def test_filter_degenerate_cases_reduce_to_unfiltered_or_argmax():
    rng = np.random.default_rng(9)
    row = rng.normal(0, 2, 500).astype(np.float32)
    base = probs_of(row, temperature=0.9)
    np.testing.assert_array_equal(probs_of(row, temperature=0.9, top_k=500), base)
    np.testing.assert_array_equal(probs_of(row, temperature=0.9, top_k=0, top_p=1.0), base)
    one = probs_of(row, temperature=0.9, top_p=1e-9)
    assert one[np.argmax(row)] == 1.0 and one.sum() == 1.0
    np.testing.assert_array_equal(probs_of(row, greedy=True), one)
    # all-equal logits: top-k keeps the k lowest indices
    flat = np.zeros(20, np.float32)
    pk = probs_of(flat, top_k=7)
    assert np.all(pk[:7] == pytest.approx(1 / 7)) and np.all(pk[7:] == 0)


# --------------------------------------------------------------------------
# errors and invariants


def test_errors_are_reported_per_sequence():
    rng = np.random.default_rng(12)
    B, K, V = 6, 2, 16
    tl = rng.normal(0, 1, (B, K + 1, V)).astype(np.float32)
    dl = rng.normal(0, 1, (B, K, V)).astype(np.float32)
    d = rng.integers(0, V, (B, K)).astype(np.int32)
    u = rng.random((B, K + 1))
    tl[1, 2, 3] = np.nan
    dl[2, 0, 5] = np.inf
    tl[3, 0, :] = -np.inf
    d[4, 1] = V
    tl[5, 1, :4] = -np.inf   # -inf entries are allowed (zero probability)
    res = oracle.verify(tl, dl, d, u)
    assert res["status"] in (oracle.ERR_NONFINITE, oracle.ERR_TOKEN_RANGE)
    for b in (1, 2, 3, 4):
        assert res["num_accepted"][b] == -1 and np.all(res["tokens"][b] == -1)
    for b in (0, 5):
        assert res["num_accepted"][b] >= 0
    # greedy reads no draft rows: a NaN there is not an error
    dl2 = np.full_like(dl, np.nan)
    res = oracle.verify(tl[:1], dl2[:1], d[:1], None, greedy=True)
    assert res["status"] == oracle.OK
    bad = oracle.verify(tl[:1], dl[:1], d[:1], u[:1], temperature=0.0)
    assert bad["status"] == oracle.ERR_INVALID_ARG
    bad = oracle.verify(tl[:1], dl[:1], d[:1], u[:1], top_p=1.5)
    assert bad["status"] == oracle.ERR_INVALID_ARG


@pytest.mark.parametrize("name", ["c1", "c2", "c3", "c4", "c5"])
def test_invariants_on_every_configuration(name):
    cfg = workloads.CONFIGS[name]
    B = min(cfg.B, 3)
    V = min(cfg.V, 20000)
    w = workloads.make(cfg, B=B, V=V)
    kw = dict(temperature=w["temperature"], top_k=w["top_k"], top_p=w["top_p"],
              greedy=w["greedy"])
    sd = oracle.sample_draft(w["draft"], w["u_draft"], **kw)
    assert sd["status"] == oracle.OK
    d = sd["tokens"]
    res = oracle.verify(w["target"], w["draft"], d, w["u_verify"], **kw)
    assert res["status"] == oracle.OK
    K = w["K"]
    for b in range(B):
        n = res["num_accepted"][b]
        assert 0 <= n <= K                                  # 1 <= emitted <= K+1
        assert list(res["tokens"][b, :n]) == list(d[b, :n])
        assert 0 <= res["tokens"][b, n] < V
        assert np.all(res["tokens"][b, n + 1:] == -1)


def test_sample_draft_is_categorical_by_library_routine():
    rng = np.random.default_rng(13)
    B, K, V = 50, 3, 777
    dl = rng.normal(0, 2, (B, K, V)).astype(np.float32)
    u = rng.random((B, K))
    res = oracle.sample_draft(dl, u, temperature=1.3)
    for b in range(B):
        for t in range(K):
            cdf = np.cumsum(_softmax_numpy(dl[b, t], 1.3))
            want = int(np.searchsorted(cdf, u[b, t] * cdf[-1], side="right"))
            if not res["flags"][b, t]:
                assert res["tokens"][b, t] == want
    g = oracle.sample_draft(dl, None, greedy=True)
    np.testing.assert_array_equal(g["tokens"], np.argmax(dl, axis=-1))


# --------------------------------------------------------------------------
# near-threshold flags: the only exclusions from bit-exact GPU parity.  A
# decision is flagged when its uniform (or, for top-p, the cumulative mass at
# the cut) lies within 1e-6 of the threshold it is compared with ("within
# hardware numerics": paperlayer.ai summary of "Accelerating Large Language
# Model Decoding with Speculative Sampling", abstract; the thresholds are those
# of "Speculative Decoding", roadtointelligence.com, "Draft, then verify",
# steps 3-4).  Each pin places the uniform or top_p at a known distance from a
# threshold computed independently with numpy in fp64: 0.5e-6 must flag, 2e-6
# and 5e-6 must not, and the decision itself must fall on the right side.

EPS = 1e-6
INSIDE, OUTSIDE = 0.5e-6, (2e-6, 5e-6)


def _np_probs(row, T=1.0):
    """Softmax of fp32 logits in fp64 (numpy), the reference for the thresholds."""
    return _softmax_numpy(np.asarray(row, np.float32), T)


def _flag_rows(seed=41, V=6):
    """One K=1 sequence: target rows 0 and 1, draft row 0 (fp32 logits)."""
    rng = np.random.default_rng(seed)
    tl = rng.normal(0, 1.2, (2, V)).astype(np.float32)
    dl = (tl[:1] + rng.normal(0, 1.2, (1, V))).astype(np.float32)
    return tl, dl


def _verify_one(tl, dl, d, u, **kw):
    res = oracle.verify(tl[None], dl[None], np.asarray([d], np.int32), np.asarray([u], np.float64), **kw)
    assert res["status"] == oracle.OK
    return int(res["num_accepted"][0]), res["tokens"][0], int(res["flags"][0])


def test_near_flag_accept_band():
    tl, dl = _flag_rows()
    tp, dp = _np_probs(tl[0]), _np_probs(dl[0])
    # a token the draft over-weights, with a small draft probability, so that a
    # band scaled by drf (|u drf - tgt| instead of |u - tgt/drf|) would be wider
    cand = [x for x in range(len(tp)) if tp[x] < dp[x] and dp[x] < 0.45]
    assert cand
    x = cand[0]
    ratio = tp[x] / dp[x]
    for off in (INSIDE, *OUTSIDE):
        for sign in (-1, 1):
            u0 = ratio + sign * off
            n, _, fl = _verify_one(tl, dl, [x], [u0, 0.37])
            assert n == (1 if sign < 0 else 0), (off, sign)          # accept iff u < ratio
            assert bool(fl & oracle.NEAR_ACCEPT) == (off < EPS), (off, sign, fl)


def test_near_flag_accept_only_for_tests_taken():
    rng = np.random.default_rng(43)
    V, K = 6, 2
    tl = rng.normal(0, 1.2, (K + 1, V)).astype(np.float32)
    dl = (tl[:K] + rng.normal(0, 1.2, (K, V))).astype(np.float32)
    tp = [_np_probs(r) for r in tl]
    dp = [_np_probs(r) for r in dl]
    x0 = int(np.argmax(dp[0] - tp[0]))     # tgt < drf at position 0: u near 1 rejects
    x1 = int(np.argmax(dp[1] - tp[1]))
    r1 = tp[1][x1] / dp[1][x1]
    assert tp[0][x0] / dp[0][x0] < 0.99 and r1 < 1
    # position 0 rejects, so the test at position 1 (u exactly at its ratio) is never taken
    res = oracle.verify(tl[None], dl[None], np.asarray([[x0, x1]], np.int32),
                        np.asarray([[1 - 1e-9, r1, 0.41]]))
    assert res["num_accepted"][0] == 0 and not (res["flags"][0] & oracle.NEAR_ACCEPT)
    # position 0 accepts (u = 0), so the test at position 1 is taken and flagged
    res = oracle.verify(tl[None], dl[None], np.asarray([[x0, x1]], np.int32),
                        np.asarray([[0.0, r1, 0.41]]))
    assert res["num_accepted"][0] >= 1 and (res["flags"][0] & oracle.NEAR_ACCEPT)


def _edges(w, x):
    """CDF edges cum(x-1)/R and cum(x)/R of token x under weights w (index order)."""
    c = np.cumsum(w)
    return (c[x - 1] if x > 0 else 0.0) / c[-1], c[x] / c[-1]


def test_near_flag_residual_draw_edges():
    tl, dl = _flag_rows(seed=47, V=8)
    tp, dp = _np_probs(tl[0]), _np_probs(dl[0])
    r = np.maximum(0.0, tp - dp)
    R = r.sum()
    assert 0.05 < R < 0.5      # a band scaled by R would be at least twice as wide
    d = int(np.argmax(dp - tp))
    pos = [x for x in range(len(r)) if r[x] > 0]
    x = pos[len(pos) // 2]
    assert x > pos[0]
    lo, hi = _edges(r, x)
    for off in (INSIDE, *OUTSIDE):
        for u1 in (lo + off, hi - off):
            n, tok, fl = _verify_one(tl, dl, [d], [1 - 1e-12, u1])
            assert n == 0 and tok[0] == x, (off, u1)
            assert bool(fl & oracle.NEAR_DRAW) == (off < EPS), (off, u1, fl)


def test_near_flag_bonus_draw_edges():
    tl, dl = _flag_rows(seed=53, V=8)
    tp1 = _np_probs(tl[1])
    d = int(np.argmax(_np_probs(tl[0])))
    x = 4
    lo, hi = _edges(tp1, x)
    for off in (INSIDE, *OUTSIDE):
        for u1 in (lo + off, hi - off):
            n, tok, fl = _verify_one(tl, dl, [d], [0.0, u1])
            assert n == 1 and tok[1] == x, (off, u1)
            assert bool(fl & oracle.NEAR_DRAW) == (off < EPS), (off, u1, fl)


def test_near_flag_sample_draft_edges():
    rng = np.random.default_rng(59)
    V = 10
    row = rng.normal(0, 1.5, (1, 1, V)).astype(np.float32)
    p = _np_probs(row[0, 0], 0.9)
    x = 6
    lo, hi = _edges(p, x)
    for off in (INSIDE, *OUTSIDE):
        for u in (lo + off, hi - off):
            res = oracle.sample_draft(row, np.asarray([[u]]), temperature=0.9)
            assert res["tokens"][0, 0] == x
            assert bool(res["flags"][0, 0] & oracle.NEAR_DRAW) == (off < EPS), (off, u)


def _crossing_masses(row, T=1.0, top_k=0):
    """Cumulative masses along (logit desc, index asc), relative to the top-k mass."""
    lf = np.asarray(row, np.float32)
    order = _order(lf)
    w = np.exp((lf[order].astype(np.float64) - lf[order[0]]) / float(np.float32(T)))
    if top_k:
        w = w[:top_k]
    return np.cumsum(w) / w.sum()


@pytest.mark.parametrize("top_k,j", [(0, 3), (0, 1), (6, 2)])
def test_near_flag_top_p_band(top_k, j):
    rng = np.random.default_rng(61 + j)
    V = 12
    row = rng.normal(0, 1.0, V).astype(np.float32)
    cm = _crossing_masses(row, top_k=top_k)
    c = cm[j]
    for off in (INSIDE, *OUTSIDE):
        for sign in (-1, 1):
            p32 = np.float32(c + sign * off)
            dist = abs(c - float(p32))
            probs, _, near, _, s = oracle.row_probs(row, top_k=top_k, top_p=float(p32))
            assert s == oracle.OK
            # kept: the prefix through j when top_p <= c, else through j + 1
            assert int((probs > 0).sum()) == (j + 1 if float(p32) <= c else j + 2), (off, sign)
            assert near == (dist < EPS), (off, sign, dist)
    # the same flag reaches verify's per-sequence bits (NEAR_TOPP) and sample_draft's
    tl = np.stack([row, row])
    p32 = float(np.float32(c + INSIDE))
    res = oracle.verify(tl[None], row[None, None], np.asarray([[0]], np.int32), np.asarray([[0.0, 0.5]]),
                        top_k=top_k, top_p=p32)
    assert res["flags"][0] & oracle.NEAR_TOPP
    sd = oracle.sample_draft(row[None, None], np.asarray([[0.5]]), top_k=top_k, top_p=p32)
    assert sd["flags"][0, 0] & oracle.NEAR_TOPP
    p32 = float(np.float32(c + OUTSIDE[1]))
    res = oracle.verify(tl[None], row[None, None], np.asarray([[0]], np.int32), np.asarray([[0.0, 0.5]]),
                        top_k=top_k, top_p=p32)
    assert not (res["flags"][0] & oracle.NEAR_TOPP)
