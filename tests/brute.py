"""Brute-force laws of one verification round, for tiny V and K.

Independent of the oracle: it takes the adjusted distributions as plain
probability vectors and integrates the procedure's randomness exactly.

`exact_law` enumerates every draft vector d in V^K (weight prod_t drf_t(d_t)),
and for each one integrates the uniforms analytically: the accept test at t
passes with probability min(1, tgt_t(d_t)/drf_t(d_t)); the first rejection at
n emits x with probability r_n(x)/R_n, r_n = max(0, tgt_n - drf_n); if all K
pass, the bonus token is x with probability tgt_K(x).  ("Speculative
Decoding", roadtointelligence.com, section "Draft, then verify", steps 1-4.)

`chain_law` is the closed form that Theorem 1 implies for the same round
("Accelerating Large Language Model Decoding with Speculative Sampling",
paperlayer.ai summary, section "Hyperparams", Theorem 1): an accepted draft
token at t has mass min(tgt_t, drf_t)(y), a rejection at n followed by y has
mass tgt_n(y) - min(tgt_n, drf_n)(y), so summed over both every emitted
position follows the target row.
"""
from __future__ import annotations

import itertools


def _residual(tgt, drf):
    r = [max(0.0, a - b) for a, b in zip(tgt, drf)]
    R = sum(r)
    if R <= 0.0:  # zero residual mass: fall back to the target row
        return list(tgt)
    return [x / R for x in r]


def exact_law(tgt_rows, drf_rows):
    """Law of the emitted tuple (y_0..y_n) for one round: dict tuple -> probability."""
    K = len(drf_rows)
    V = len(tgt_rows[0])
    law = {}
    for d in itertools.product(range(V), repeat=K):
        wd = 1.0
        for t in range(K):
            wd *= drf_rows[t][d[t]]
        if wd == 0.0:
            continue
        reach = wd
        for t in range(K):
            a, b = tgt_rows[t][d[t]], drf_rows[t][d[t]]
            acc = min(1.0, a / b)
            rej = reach * (1.0 - acc)
            if rej > 0.0:
                res = _residual(tgt_rows[t], drf_rows[t])
                for x in range(V):
                    if res[x] > 0.0:
                        key = tuple(d[:t]) + (x,)
                        law[key] = law.get(key, 0.0) + rej * res[x]
            reach *= acc
            if reach == 0.0:
                break
        if reach > 0.0:
            for x in range(V):
                if tgt_rows[K][x] > 0.0:
                    key = tuple(d) + (x,)
                    law[key] = law.get(key, 0.0) + reach * tgt_rows[K][x]
    return law


def chain_law(tgt_rows, drf_rows):
    """Closed-form law from Theorem 1 (same keys as exact_law)."""
    K = len(drf_rows)
    V = len(tgt_rows[0])
    mins = [[min(a, b) for a, b in zip(tgt_rows[t], drf_rows[t])] for t in range(K)]
    law = {}

    def rec(prefix, mass):
        t = len(prefix)
        if t == K:
            for x in range(V):
                if tgt_rows[K][x] > 0.0:
                    law[prefix + (x,)] = law.get(prefix + (x,), 0.0) + mass * tgt_rows[K][x]
            return
        for x in range(V):
            stop = tgt_rows[t][x] - mins[t][x]
            if stop > 0.0:
                law[prefix + (x,)] = law.get(prefix + (x,), 0.0) + mass * stop
            if mins[t][x] > 0.0:
                rec(prefix + (x,), mass * mins[t][x])

    rec((), 1.0)
    return law


def expected_tokens(alphas):
    """E[tokens per round] = sum_{j=0}^{K} prod_{t<j} alpha_t for per-position acceptance
    probabilities alpha_t; with all alpha_t = a this is (1 - a^(K+1)) / (1 - a)
    ("Speculative Decoding", section "How much faster")."""
    total, prod = 0.0, 1.0
    for j in range(len(alphas) + 1):
        total += prod
        if j < len(alphas):
            prod *= alphas[j]
    return total
