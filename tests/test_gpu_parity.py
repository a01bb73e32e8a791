"""Parity of the CUDA path (called through the C ABI) with the fp64 oracle.

Bar: out_tokens and out_num_accepted bit-exact, excluding only sequences the
oracle flags as having a uniform (or a top-p cumulative mass) within 1e-6 of a
decision threshold; per-row normalisers and draft-token probabilities within
1e-5 relative.  Flagged sequences are counted, and must stay rare.
"""
import math
import os
import zlib

import numpy as np
import pytest
import torch
from scipy import stats

import oracle
import workloads
from _gpu import check_invariants, compare_verify, params_of, to_dev
from _report import record

pytestmark = pytest.mark.gpu

DEV = "cuda:0"
NT = max(1, min(16, os.cpu_count() or 1))   # host threads for the oracle at full size


@pytest.fixture(scope="module")
def sv():
    import speculative_sampling_verification_spec_gb300 as m
    m.binding.lib()
    return m


def run_case(sv, w, check_stats=True, seqs=None, where="", max_flag_frac=0.1):
    """GPU verify on all of w's sequences; oracle on `seqs` (default all).  At most
    max_flag_frac of the compared sequences (and at least one) may be flagged."""
    prm = params_of(w)
    d = oracle.sample_draft_threaded(w["draft"], w["u_draft"], NT, **prm)
    assert d["status"] == oracle.OK
    tokens = d["tokens"]
    tgt, drf = to_dev(w["target"]), to_dev(w["draft"])
    ws = sv.workspace(sv.spec_verify_workspace_size(w["B"], w["K"], w["V"], sv.SPEC_BF16 if w["dtype"] == "bf16" else sv.SPEC_F32, w["greedy"]), torch.device(DEV))
    out_t, out_n = sv.spec_verify(tgt, drf, to_dev(tokens), to_dev(w["u_verify"]), ws=ws, **prm)
    torch.cuda.synchronize()
    gt, gn = out_t.cpu().numpy(), out_n.cpu().numpy()
    check_invariants(gt, gn, tokens, w["K"], w["V"])
    sel = np.arange(w["B"]) if seqs is None else np.asarray(seqs)
    ref = oracle.verify_threaded(w["target"][sel], w["draft"][sel], tokens[sel], w["u_verify"][sel], NT,
                                 with_stats=check_stats, **prm)
    assert ref["status"] == oracle.OK
    nflag = compare_verify(gt[sel], gn[sel], ref, where)
    assert nflag <= max(1, int(max_flag_frac * len(sel))), "%s: %d flagged sequences" % (where, nflag)
    if check_stats:
        dt = sv.SPEC_BF16 if w["dtype"] == "bf16" else sv.SPEC_F32
        rows = sv.spec_read_row_stats(w["B"], w["K"], w["V"], dt, True, ws, **prm)
        R = w["K"] + 1 if w["greedy"] else 2 * w["K"] + 1
        for bi, b in enumerate(sel):
            for r in range(R):
                g = rows[b * R + r]
                o = ref["row_stats"][bi, r]
                assert g["flags"] == 0
                assert g["m"] == o[0], (where, b, r)
                if not w["greedy"]:
                    assert abs(g["zf"] - o[1]) <= 1e-5 * o[1], (where, b, r, g["zf"], o[1])
                    if o[2] > 1e-300:
                        assert abs(g["p_tok"] - o[2]) <= 1e-5 * o[2], (where, b, r, g["p_tok"], o[2])
                    else:
                        assert g["p_tok"] < 1e-30
    return gt, gn, tokens


SMALL = [
    ("c1", {}),
    ("c2", {}),
    ("c3", dict(B=6, V=50001)),        # odd V: rows not 16-byte aligned (plain-load path)
    ("c3", dict(B=3)),                 # full V = 128256
    ("c4", dict(B=24)),                # full V = 50304, fp32 greedy
    ("c4", dict(B=16, V=20011)),
    ("c4_bf16", dict(B=24)),
    ("c5", dict(B=3)),                 # full V = 256000
    ("c5", dict(B=6, V=70003)),
]


@pytest.mark.parametrize("name,kw", SMALL, ids=["%s-%s" % (n, "-".join("%s%s" % kv for kv in k.items())) for n, k in SMALL])
def test_verify_matches_oracle(sv, name, kw):
    w = workloads.make(name, **kw)
    run_case(sv, w, where=name)


@pytest.mark.parametrize("name", ["c3", "c4", "c4_bf16", "c5"])
def test_full_size_every_sequence(sv, name):
    """The bench's launch configuration (full B, K, V): every sequence, and every
    row record, against the oracle."""
    w = workloads.make(name)
    run_case(sv, w, check_stats=True, where=name + "-full")


@pytest.mark.parametrize("name,kw", [("c1", {}), ("c2", {}), ("c3", dict(B=4, V=60007)),
                                     ("c5", dict(B=2)), ("c4", dict(B=8)),
                                     ("c5", {}), ("c3", {}), ("c4", {}), ("c4_bf16", {})],
                         ids=["c1", "c2", "c3-B4-V60007", "c5-B2", "c4-B8", "c5-full", "c3-full", "c4-full",
                              "c4_bf16-full"])
def test_sample_draft_matches_oracle(sv, name, kw):
    """Draft draws against the oracle's, row by row; the full-size cases are the
    bench's own spec_sample_draft launch (c5: B=32, K=8, V=256000)."""
    w = workloads.make(name, **kw)
    prm = params_of(w)
    ref = oracle.sample_draft_threaded(w["draft"], w["u_draft"], NT, **prm)
    assert ref["status"] == oracle.OK
    g = sv.spec_sample_draft(to_dev(w["draft"]), to_dev(w["u_draft"]), **prm).cpu().numpy()
    ok = ref["flags"] == 0
    bad = np.argwhere((g != ref["tokens"]) & ok)
    assert len(bad) == 0, "%d mismatching draft rows, e.g. %s" % (len(bad), bad[:5].tolist())
    record("sample_draft %s %s" % (name, kw or "full"), ok.size, int((~ok).sum()), "rows")
    assert (~ok).sum() <= max(1, ok.size // 10)


def _custom(B, K, V, rng, scale=2.0, dtype="f32"):
    tl = rng.normal(0, scale, (B, K + 1, V)).astype(np.float32)
    dl = (tl[:, :K] + rng.normal(0, 1.0, (B, K, V))).astype(np.float32)
    if dtype == "bf16":
        tl, dl = workloads.to_bf16_bits(tl), workloads.to_bf16_bits(dl)
    return dict(target=tl, draft=dl, u_draft=rng.random((B, K)), u_verify=rng.random((B, K + 1)),
                B=B, K=K, V=V, dtype=dtype, temperature=1.0, top_k=0, top_p=1.0, greedy=False)


@pytest.mark.parametrize("case", [
    dict(V=1, K=1, B=3),
    dict(V=7, K=1, B=40),
    dict(V=3000, K=2, B=6, top_k=1000),               # top-k beyond the on-chip sort: tie-cut path
    dict(V=3000, K=2, B=6, top_k=40, top_p=0.8),
    dict(V=20000, K=2, B=4, top_k=2000, top_p=0.95),  # top-p inside a tie-cut top-k set
    # huge nucleus (kept set of ~1500-1700 > the 512-entry stored list) over a near-flat row;
    # the tokens at the cut hold ~5e-4 of the mass each, so a cut falls within 1e-6 of top_p
    # in about 1 % of the rows (the oracle flags 1 of 64 and 1 of 32 sequences here)
    dict(V=2000, K=1, B=64, top_p=0.9, scale=0.3),
    dict(V=2000, K=2, B=32, top_p=0.85, scale=0.3),
    dict(V=5000, K=2, B=4, temperature=0.05),
    dict(V=5000, K=2, B=4, temperature=5.0, top_p=0.5),
    # top-p alone on 16-byte aligned rows: the streaming kernel's nucleus pool
    dict(V=4096, K=2, B=6, dtype="bf16", temperature=0.8, top_p=0.9),
    dict(V=12000, K=3, B=5, scale=3.0, top_p=0.7),
    dict(V=8192, K=2, B=4, dtype="bf16", scale=1.0, top_p=0.95),  # nuclei of hundreds of tokens
    # bf16 nuclei of ~1500 tokens: past the streaming kernel's pool, so the general path
    dict(V=2048, K=1, B=32, dtype="bf16", top_p=0.9, scale=0.3),
    dict(V=4099, K=3, B=5, dtype="bf16", top_k=13, temperature=0.7),
    dict(V=2048, K=4, B=8, greedy=True, dtype="bf16", scale=0.3),   # many exact ties
])
def test_edge_cases_match_oracle(sv, case):
    rng = np.random.default_rng(zlib.crc32(repr(sorted(case.items())).encode()))
    w = _custom(case["B"], case["K"], case["V"], rng, case.get("scale", 2.0), case.get("dtype", "f32"))
    for k in ("temperature", "top_k", "top_p", "greedy"):
        if k in case:
            w[k] = case[k]
    run_case(sv, w, where=str(case), max_flag_frac=case.get("max_flag_frac", 0.1))


def test_ties_all_equal_logits_cut_by_index(sv):
    B, K, V = 3, 2, 3000
    w = dict(target=np.zeros((B, K + 1, V), np.float32), draft=np.zeros((B, K, V), np.float32),
             u_draft=np.random.default_rng(1).random((B, K)),
             u_verify=np.random.default_rng(2).random((B, K + 1)),
             B=B, K=K, V=V, dtype="f32", temperature=1.0, top_k=7, top_p=1.0, greedy=False)
    gt, gn, _ = run_case(sv, w, where="flat-topk")
    assert np.all(gt[np.arange(B), gn] < 7)
    # every token holds 1/V of the mass; top_p = 0.3123 keeps ceil(0.3123 V) tokens, and the
    # crossing (937/3000 = 0.31233) stays clear of the 1e-6 band around top_p
    w["top_k"], w["top_p"] = 0, 0.3123
    gt, gn, _ = run_case(sv, w, where="flat-topp")
    assert np.all(gt[np.arange(B), gn] < 937)


def test_neg_inf_entries_and_layouts(sv):
    rng = np.random.default_rng(31)
    B, K, V = 5, 3, 1500
    w = _custom(B, K, V, rng)
    w["target"][:, :, ::3] = -np.inf
    w["draft"][:, :, 1::5] = -np.inf
    w["top_k"] = 30
    run_case(sv, w, where="-inf")
    # repeated rows through stride 0, and a padded row stride
    prm = params_of(w)
    one_t = to_dev(w["target"][:1])
    one_d = to_dev(w["draft"][:1])
    tgt = one_t.expand(B, K + 1, V)
    drf = one_d.expand(B, K, V)
    d = oracle.sample_draft(w["draft"][:1], w["u_draft"][:1], **prm)["tokens"].repeat(B, 0)
    out_t, out_n = sv.spec_verify(tgt, drf, to_dev(d), to_dev(w["u_verify"]), **prm)
    ref = oracle.verify(w["target"][:1], w["draft"][:1], d, w["u_verify"],
                        tgt_strides=(0, V), drf_strides=(0, V), B=B, **prm)
    compare_verify(out_t.cpu().numpy(), out_n.cpu().numpy(), ref, "stride0")
    pad_t = torch.zeros(B, K + 1, V + 13, device=DEV)[:, :, :V]
    pad_t.copy_(to_dev(w["target"]))
    pad_d = torch.zeros(B, K, V + 13, device=DEV)[:, :, :V]
    pad_d.copy_(to_dev(w["draft"]))
    d = oracle.sample_draft(w["draft"], w["u_draft"], **prm)["tokens"]
    out_t, out_n = sv.spec_verify(pad_t, pad_d, to_dev(d), to_dev(w["u_verify"]), **prm)
    ref = oracle.verify(w["target"], w["draft"], d, w["u_verify"], **prm)
    compare_verify(out_t.cpu().numpy(), out_n.cpu().numpy(), ref, "padded")


def test_errors_reported_per_sequence(sv):
    rng = np.random.default_rng(12)
    B, K, V = 6, 2, 300
    tl = rng.normal(0, 1, (B, K + 1, V)).astype(np.float32)
    dl = rng.normal(0, 1, (B, K, V)).astype(np.float32)
    d = rng.integers(0, V, (B, K)).astype(np.int32)
    u = rng.random((B, K + 1))
    tl[1, 2, 3] = np.nan
    dl[2, 0, 5] = np.inf
    tl[3, 0, :] = -np.inf
    d[4, 1] = V
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    out_t, out_n = sv.spec_verify(to_dev(tl), to_dev(dl), to_dev(d), to_dev(u), status=status)
    ref = oracle.verify(tl, dl, d, u)
    gn, gt = out_n.cpu().numpy(), out_t.cpu().numpy()
    np.testing.assert_array_equal(gn, ref["num_accepted"])
    for b in (1, 2, 3, 4):
        assert gn[b] == -1 and np.all(gt[b] == -1)
    assert int(status.item()) in (3, 4)
    compare_verify(gt[[0, 5]], gn[[0, 5]], {k: v[[0, 5]] if k != "status" else v for k, v in ref.items()})


def test_repeatable_bit_for_bit(sv):
    w = workloads.make("c3", B=8, V=30011)
    prm = params_of(w)
    d = to_dev(oracle.sample_draft(w["draft"], w["u_draft"], **prm)["tokens"])
    tgt, drf, u = to_dev(w["target"]), to_dev(w["draft"]), to_dev(w["u_verify"])
    outs = [tuple(x.cpu().numpy().copy() for x in sv.spec_verify(tgt, drf, d, u, **prm)) for _ in range(3)]
    for o in outs[1:]:
        assert np.array_equal(o[0], outs[0][0]) and np.array_equal(o[1], outs[0][1])


def test_workspace_shared_across_shapes(sv):
    """One zero-filled workspace serves calls of different shapes and modes: every
    call leaves the counter area (its first 64 KB) at zero, and the results of a
    call after the others still match the oracle."""
    ws = torch.zeros(48 << 20, dtype=torch.uint8, device=DEV)
    cases = [("c5", dict(B=3)), ("c3", dict(B=6, V=50001)), ("c2", {}), ("c4", dict(B=16)),
             ("c1", {}), ("c5", dict(B=2, V=70003))]
    for name, kw in cases:
        w = workloads.make(name, **kw)
        prm = params_of(w)
        drf = to_dev(w["draft"])
        tok = sv.spec_sample_draft(drf, None if w["greedy"] else to_dev(w["u_draft"]), ws=ws, **prm)
        torch.cuda.synchronize()
        assert int(ws[:65536].count_nonzero()) == 0, name
        ref_d = oracle.sample_draft(w["draft"], w["u_draft"], **prm)
        ok = ref_d["flags"] == 0
        assert np.array_equal(tok.cpu().numpy()[ok], ref_d["tokens"][ok]), name
        out_t, out_n = sv.spec_verify(to_dev(w["target"]), drf, to_dev(ref_d["tokens"]), to_dev(w["u_verify"]),
                                      ws=ws, **prm)
        torch.cuda.synchronize()
        assert int(ws[:65536].count_nonzero()) == 0, name
        ref = oracle.verify(w["target"], w["draft"], ref_d["tokens"], w["u_verify"], **prm)
        compare_verify(out_t.cpu().numpy(), out_n.cpu().numpy(), ref, "shared-ws-" + name)


def test_worked_example_distribution_on_gpu(sv):
    """"Speculative Decoding" (roadtointelligence.com), "Why the output doesn't change":
    acceptance 0.8 and emitted words in the target's proportions, not the draft's."""
    tgt_p = np.array([0.5, 0.25, 0.15, 0.10])
    drf_p = np.array([0.3, 0.4, 0.2, 0.1])
    lt, ld = np.log(tgt_p).astype(np.float32), np.log(drf_p).astype(np.float32)
    B = 200_000
    rng = np.random.default_rng(77)
    tp = oracle.row_probs(lt)[0]
    dp = oracle.row_probs(ld)[0]
    d = rng.choice(4, size=(B, 1), p=dp).astype(np.int32)
    u = rng.random((B, 2))
    tgt = torch.from_numpy(np.stack([lt, lt])).to(DEV).unsqueeze(0).expand(B, 2, 4)
    drf = torch.from_numpy(ld[None]).to(DEV).unsqueeze(0).expand(B, 1, 4)
    out_t, out_n = sv.spec_verify(tgt, drf, to_dev(d), to_dev(u))
    gt, gn = out_t.cpu().numpy(), out_n.cpu().numpy()
    acc = (gn == 1).mean()
    assert abs(acc - 0.8) < 4 * math.sqrt(0.16 / B)
    counts = np.bincount(gt[:, 0], minlength=4)
    assert stats.chisquare(counts, B * tp).pvalue > 1e-3
    assert stats.chisquare(counts, B * dp).pvalue < 1e-12
    ref = oracle.verify(np.stack([lt, lt])[None], ld[None, None], d, u, tgt_strides=(0, 4),
                        drf_strides=(0, 4), B=B)
    compare_verify(gt, gn, ref, "worked-example")


def test_accept_histogram_matches_oracle(sv):
    """Acceptance telemetry: the histogram the kernel adds to hist equals the
    oracle's histogram of the oracle's accepted counts, bin for bin; a second call
    accumulates; sequences that ended in an error land in bin K+1."""
    alpha, K, B = 0.8, 4, 40_000
    drf = np.array([0.4, 0.3, 0.2, 0.1, 0, 0, 0, 0])
    tgt = alpha * drf + (1 - alpha) * np.array([0, 0, 0, 0, .25, .25, .25, .25])
    with np.errstate(divide="ignore"):
        lt, ld = np.log(tgt).astype(np.float32), np.log(drf).astype(np.float32)
    rng = np.random.default_rng(31)
    d = np.stack([rng.choice(8, size=B, p=drf) for _ in range(K)], 1).astype(np.int32)
    u = rng.random((B, K + 1))
    d[:7, 1] = 8                                     # out-of-range draft tokens: errors
    target = np.ascontiguousarray(np.broadcast_to(lt, (B, K + 1, 8)))
    draft = np.ascontiguousarray(np.broadcast_to(ld, (B, K, 8)))
    out_t, out_n = sv.spec_verify(to_dev(target), to_dev(draft), to_dev(d), to_dev(u))
    ref = oracle.verify(target, draft, d, u)
    ok = ref["flags"] == 0
    gn = out_n.cpu().numpy()
    assert np.array_equal(gn[ok], ref["num_accepted"][ok])
    hist = sv.spec_accept_histogram(out_n, K)
    torch.cuda.synchronize()
    want = oracle.accept_histogram(gn, K)
    assert np.array_equal(hist.cpu().numpy(), want)
    assert want[K + 1] == 7
    assert np.array_equal(oracle.accept_histogram(ref["num_accepted"][ok], K), oracle.accept_histogram(gn[ok], K))
    sv.spec_accept_histogram(out_n, K, hist=hist)
    torch.cuda.synchronize()
    assert np.array_equal(hist.cpu().numpy(), 2 * want)
    # a full-size call's histogram (c5 shape) against the oracle's
    w = workloads.make("c5", B=4)
    prm = params_of(w)
    dd = oracle.sample_draft(w["draft"], w["u_draft"], **prm)["tokens"]
    o_t, o_n = sv.spec_verify(to_dev(w["target"]), to_dev(w["draft"]), to_dev(dd), to_dev(w["u_verify"]), **prm)
    h5 = sv.spec_accept_histogram(o_n, w["K"])
    torch.cuda.synchronize()
    r5 = oracle.verify(w["target"], w["draft"], dd, w["u_verify"], **prm)
    keep = r5["flags"] == 0
    assert np.array_equal(o_n.cpu().numpy()[keep], r5["num_accepted"][keep])
    assert np.array_equal(h5.cpu().numpy(), oracle.accept_histogram(o_n.cpu().numpy(), w["K"]))


@pytest.mark.parametrize("name,kw,prm", [
    ("c2", dict(K=1, B=64), {}),
    ("c3", dict(K=1, B=32), {}),
    ("c5", dict(K=1, B=16), {}),
    ("c5", dict(K=1, B=24, V=70003), {}),
    ("c1", dict(K=1, B=256), dict(top_k=5, top_p=0.9, temperature=1.3))])
def test_sample_verify_equals_draw_then_verify(sv, name, kw, prm):
    """The fused K = 1 step gives the oracle's draw from the draft row, then the
    oracle's verification of that token: draft token, emitted tokens and count."""
    w = workloads.make(name, **kw)
    p = dict(params_of(w), **prm)
    assert w["K"] == 1 and not p["greedy"]
    ud = w["u_draft"][:, 0].copy()
    dr = oracle.sample_draft(w["draft"], w["u_draft"], **p)
    ref = oracle.verify(w["target"], w["draft"], dr["tokens"], w["u_verify"], **p)
    assert ref["status"] == oracle.OK
    g_d, g_t, g_n = sv.spec_sample_verify(to_dev(w["target"]), to_dev(w["draft"]), to_dev(ud),
                                          to_dev(w["u_verify"]), **p)
    torch.cuda.synchronize()
    g_d, g_t, g_n = g_d.cpu().numpy(), g_t.cpu().numpy(), g_n.cpu().numpy()
    ok = (dr["flags"][:, 0] == 0) & (ref["flags"] == 0)
    assert ok.sum() >= 0.9 * w["B"]
    assert np.array_equal(g_d[ok], dr["tokens"][ok, 0])
    assert np.array_equal(g_n[ok], ref["num_accepted"][ok])
    assert np.array_equal(g_t[ok], ref["tokens"][ok])
    # and the same as the two separate calls on the GPU
    s_d = sv.spec_sample_draft(to_dev(w["draft"]), to_dev(w["u_draft"]), **p)
    s_t, s_n = sv.spec_verify(to_dev(w["target"]), to_dev(w["draft"]), s_d, to_dev(w["u_verify"]), **p)
    torch.cuda.synchronize()
    assert np.array_equal(s_d.cpu().numpy()[:, 0], g_d)
    assert np.array_equal(s_n.cpu().numpy(), g_n) and np.array_equal(s_t.cpu().numpy(), g_t)


@pytest.mark.parametrize("name,kw,prm", [
    ("c3", dict(B=24, V=30011), {}),
    ("c5", dict(B=12), {}),
    ("c4", dict(B=40, V=20011), {}),
    ("c1", dict(B=300), dict(top_k=6, top_p=0.85)),
    # 16-byte aligned rows: the streaming kernel's ragged rows (top-p, greedy)
    ("c3", dict(B=24, V=32768), {}),
    ("c4", dict(B=40, V=20000), {})])
def test_ragged_batch_equals_per_sequence_verify(sv, name, kw, prm):
    """Each sequence of a ragged call gives the oracle's verification with its own
    draft length K_b: the first K_b draft tokens, uniform columns 0..K_b."""
    w = workloads.make(name, **kw)
    p = dict(params_of(w), **prm)
    B, K = w["B"], w["K"]
    rng = np.random.default_rng(40 + K)
    lens = rng.integers(1, K + 1, B).astype(np.int32)
    lens[0] = K
    d = oracle.sample_draft(w["draft"], w["u_draft"], **p)["tokens"]
    g_t, g_n = sv.spec_verify_ragged(to_dev(w["target"]), to_dev(w["draft"]), to_dev(d),
                                     None if p["greedy"] else to_dev(w["u_verify"]), lens, **p)
    torch.cuda.synchronize()
    g_t, g_n = g_t.cpu().numpy(), g_n.cpu().numpy()
    compared = 0
    for kb in sorted(set(lens.tolist())):
        sel = np.nonzero(lens == kb)[0]
        ref = oracle.verify(np.ascontiguousarray(w["target"][sel, :kb + 1]), np.ascontiguousarray(w["draft"][sel, :kb]),
                            np.ascontiguousarray(d[sel, :kb]), np.ascontiguousarray(w["u_verify"][sel, :kb + 1]), **p)
        ok = ref["flags"] == 0
        assert np.array_equal(g_n[sel][ok], ref["num_accepted"][ok]), kb
        assert np.array_equal(g_t[sel][ok][:, :kb + 1], ref["tokens"][ok]), kb
        assert np.all(g_t[sel][:, kb + 1:] == -1)
        compared += int(ok.sum())
    assert compared >= 0.9 * B


@pytest.mark.parametrize("name,kw", [("c5", dict(B=6)), ("c4", dict(B=20, V=20011)), ("c3", dict(B=8, V=30011)),
                                     ("c2", {}), ("c3", dict(B=8, V=32768)), ("c4", dict(B=20, V=20000))])
def test_ragged_with_equal_lengths_is_spec_verify(sv, name, kw):
    """A ragged call whose lengths all equal K gives spec_verify's outputs bit for bit."""
    w = workloads.make(name, **kw)
    p = params_of(w)
    d = to_dev(oracle.sample_draft(w["draft"], w["u_draft"], **p)["tokens"])
    tgt, drf = to_dev(w["target"]), to_dev(w["draft"])
    u = None if p["greedy"] else to_dev(w["u_verify"])
    a_t, a_n = sv.spec_verify(tgt, drf, d, u, **p)
    b_t, b_n = sv.spec_verify_ragged(tgt, drf, d, u, np.full(w["B"], w["K"], np.int32), **p)
    torch.cuda.synchronize()
    assert np.array_equal(a_t.cpu().numpy(), b_t.cpu().numpy())
    assert np.array_equal(a_n.cpu().numpy(), b_n.cpu().numpy())
