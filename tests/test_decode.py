"""The decode-round driver (the loop around verification) and the latency-vs-K model.

CPU tests pin the synthetic sources, the closed forms the model restates, and the
oracle's own decode loop; GPU tests compare the driver, round by round, with that
loop and check its tokens per round against the closed form.
"""
import math

import numpy as np
import pytest

import oracle
import workloads
from brute import expected_tokens
from conftest import read_golden


def oracle_rounds(src, first, K, rounds, seed, **prm):
    """The decode loop on the oracle: per round, K draft draws one token at a time,
    then one verification of the K+1 target rows; the next context ends with the
    emitted token.  Returns per round (tokens, num_accepted, flagged)."""
    B = len(first)
    last = np.asarray(first, np.int64)
    pos = np.zeros(B, np.int64)
    out = []
    for r in range(rounds):
        ud, uv = workloads.round_uniforms(seed, r, B, K)
        states = np.zeros((B, K + 1), np.int64)
        drafted = np.zeros((B, K), np.int32)
        flagged = np.zeros(B, bool)
        cur = last
        for j in range(K):
            st = workloads.state_of(cur, pos + j, src.S)
            states[:, j] = st
            d = oracle.sample_draft(np.ascontiguousarray(src.draft[st][:, None, :]), ud[:, j:j + 1], **prm)
            drafted[:, j] = d["tokens"][:, 0]
            flagged |= d["flags"][:, 0] != 0
            cur = d["tokens"][:, 0].astype(np.int64)
        states[:, K] = workloads.state_of(cur, pos + K, src.S)
        v = oracle.verify(np.ascontiguousarray(src.target[states]), np.ascontiguousarray(src.draft[states[:, :K]]),
                          drafted, uv, **prm)
        assert v["status"] == oracle.OK
        flagged |= v["flags"] != 0
        n = v["num_accepted"]
        last = v["tokens"][np.arange(B), n].astype(np.int64)
        pos = pos + n + 1
        out.append((v["tokens"], n, flagged))
    return out


# --------------------------------------------------------------------------
# CPU

def test_synthetic_source_has_exact_acceptance():
    """Every state's rows, read through the oracle's adjusted distributions, have
    sum_x min(target, draft) = alpha."""
    for alpha, dtype in ((0.8, "f32"), (0.55, "f32")):
        src = workloads.synthetic_source(V=128, S=13, alpha=alpha, seed=3, dtype=dtype)
        for s in range(src.S):
            p = oracle.row_probs(src.target[s])[0]
            q = oracle.row_probs(src.draft[s])[0]
            assert abs(np.minimum(p, q).sum() - alpha) < 1e-6


def test_closed_forms_reproduce_printed_numbers():
    """"Speculative Decoding" (roadtointelligence.com), "How much faster": 3.36 tokens
    per pass and a 2.8x speed-up at alpha 0.8, gamma 4, c 0.05; the chain law gives
    the same expectation at every alpha and K."""
    from speculative_sampling_verification_spec_gb300 import decode
    g = read_golden("closed_form.txt")
    a, gam, c = g["alpha"], int(g["gamma"]), g["c"]
    assert abs(decode.expected_tokens_per_round(a, gam) - g["tokens_per_pass"]) < 0.005
    assert abs(decode.speedup(a, gam, c) - g["speedup"]) < 0.05
    for alpha in (0.3, 0.6, 0.9, 0.99, 1.0):
        for K in (1, 2, 5, 8):
            assert abs(decode.expected_tokens_per_round(alpha, K) - expected_tokens([alpha] * K)) < 1e-12


def test_latency_model_reduces_to_the_page_and_verify_cost_only_lowers_it():
    from speculative_sampling_verification_spec_gb300 import decode
    for alpha, c in ((0.8, 0.05), (0.6, 0.2), (0.9, 0.128)):
        for K in range(1, 9):
            page = (1 - alpha ** (K + 1)) / ((1 - alpha) * (K * c + 1))
            assert abs(decode.speedup(alpha, K, c) - page) < 1e-12
            assert decode.speedup(alpha, K, c, 0.01) < decode.speedup(alpha, K, c)
        # the optimum over K is the brute-force argmax of the page's form
        want = max(range(1, 17), key=lambda k: (1 - alpha ** (k + 1)) / ((1 - alpha) * (k * c + 1)))
        assert decode.best_k(alpha, c, lambda k: 0.0) == want
        # a verification cost growing with K never moves the optimum to a larger K
        assert decode.best_k(alpha, c, lambda k: 0.002 * k) <= want


@pytest.mark.parametrize("alpha,K", [(0.8, 4), (0.6, 3)])
def test_oracle_decode_loop_follows_closed_form(alpha, K):
    src = workloads.synthetic_source(V=64, S=31, alpha=alpha, seed=4)
    B, rounds = 2000, 12
    first = np.random.default_rng(1).integers(0, 32, B)
    res = oracle_rounds(src, first, K, rounds, seed=8)
    n1 = np.concatenate([n for _, n, _ in res]) + 1
    want = (1 - alpha ** (K + 1)) / (1 - alpha)
    assert abs(n1.mean() - want) < 4 * n1.std() / math.sqrt(n1.size)


# --------------------------------------------------------------------------
# GPU

@pytest.mark.gpu
@pytest.mark.parametrize("kw", [dict(), dict(top_k=20), dict(temperature=0.8, top_p=0.9), dict(greedy=True),
                                dict(dtype="bf16", top_k=7, top_p=0.8)])
def test_decode_driver_matches_oracle_loop(kw):
    import torch
    from speculative_sampling_verification_spec_gb300 import decode
    kw = dict(kw)
    dtype = kw.pop("dtype", "f32")
    src = workloads.synthetic_source(V=300, S=53, seed=6, dtype=dtype)
    B, K, rounds, seed = 96, 4, 6, 21
    first = np.random.default_rng(2).integers(0, src.V, B)
    ref = oracle_rounds(src, first, K, rounds, seed, **kw)
    conv = (lambda a: torch.from_numpy(a.view(np.int16)).view(torch.bfloat16)) if dtype == "bf16" \
        else torch.from_numpy
    tt, dt = conv(src.target).cuda(), conv(src.draft).cuda()
    got = decode.decode_rounds(tt, dt, lambda last, pos: workloads.state_of(last, pos, src.S),
                               torch.from_numpy(first).cuda(), K, rounds,
                               lambda r: workloads.round_uniforms(seed, r, B, K), **kw)
    live = np.ones(B, bool)  # a sequence is compared until its first flagged round
    compared = 0
    for (gt, gn), (rt, rn, fl) in zip(got, ref):
        gt, gn = gt.cpu().numpy(), gn.cpu().numpy()
        ok = live & ~fl
        assert np.array_equal(gn[ok], rn[ok])
        assert np.array_equal(gt[ok], rt[ok])
        compared += int(ok.sum())
        live = ok
    assert compared >= 0.9 * B * rounds


@pytest.mark.gpu
def test_decode_driver_tokens_per_round_closed_form():
    import torch
    from speculative_sampling_verification_spec_gb300 import decode
    alpha, K, B, rounds = 0.8, 4, 8192, 8
    src = workloads.synthetic_source(V=512, S=101, alpha=alpha, seed=5)
    first = np.random.default_rng(3).integers(0, 256, B)
    got = decode.decode_rounds(torch.from_numpy(src.target).cuda(), torch.from_numpy(src.draft).cuda(),
                               lambda last, pos: workloads.state_of(last, pos, src.S),
                               torch.from_numpy(first).cuda(), K, rounds,
                               lambda r: workloads.round_uniforms(11, r, B, K))
    n1 = torch.cat([n for _, n in got]).cpu().numpy() + 1
    assert n1.min() >= 1
    want = decode.expected_tokens_per_round(alpha, K)
    assert abs(n1.mean() - want) < 4 * n1.std() / math.sqrt(n1.size)
