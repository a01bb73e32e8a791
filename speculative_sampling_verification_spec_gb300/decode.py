"""Decode rounds around the verification step, and the latency-vs-K model.

The loop of the pages ("Speculative Decoding", roadtointelligence.com, section
"Draft, then verify", steps 1-4; Algorithm 2 in the paperlayer.ai summary of
"Accelerating Large Language Model Decoding with Speculative Sampling"): the
draft proposes K tokens one at a time, the target scores the K+1 positions in
one call, verification keeps n of them and emits one more, and the next round
starts after the n + 1 new tokens.

Here the "models" are tables of logit rows on the device and a state function
that maps a context (its last token and its position) to a row.  Drawing the
draft tokens (`spec_sample_draft`) and verifying (`spec_verify`) run in the
library's kernels; the driver only gathers the rows the tables assign to each
context, which stands in for the model calls.

`expected_tokens_per_round` and `speedup` restate the closed forms of the same
page, section "How much faster", and extend the round's cost by the measured
time of the verification step itself.
"""
from __future__ import annotations

import torch

from . import binding


def decode_rounds(target_table, draft_table, state_fn, first_tokens, K, rounds, uniforms, *,
                  temperature=1.0, top_k=0, top_p=1.0, greedy=False, record=True):
    """Run `rounds` decode rounds for B sequences on the device.

    target_table, draft_table  CUDA [S, V] logit rows (float32 or bfloat16)
    state_fn(last, position)   row index of a context (int64 CUDA tensors in and out)
    first_tokens               CUDA [B] integer: the last token of each prompt (position 0)
    uniforms(r)                host float64 arrays (u_draft [B, K], u_verify [B, K+1]) of round r
    Returns, when record, one (out_tokens [B, K+1], out_num_accepted [B]) pair per
    round (the library's outputs; n + 1 tokens are appended per sequence).
    """
    dev = target_table.device
    B = first_tokens.numel()
    V = target_table.shape[1]
    prm = dict(temperature=temperature, top_k=top_k, top_p=top_p, greedy=greedy)
    last = first_tokens.to(device=dev, dtype=torch.int64)
    pos = torch.zeros(B, dtype=torch.int64, device=dev)
    out = []
    for r in range(rounds):
        ud, uv = uniforms(r)
        ud_d = None if greedy else torch.from_numpy(ud).to(dev, non_blocking=True)
        uv_d = None if greedy else torch.from_numpy(uv).to(dev, non_blocking=True)
        states = torch.empty((B, K + 1), dtype=torch.int64, device=dev)
        drafted = torch.empty((B, K), dtype=torch.int32, device=dev)
        cur = last
        for j in range(K):  # the draft runs one token at a time
            st = state_fn(cur, pos + j)
            states[:, j] = st
            rows = draft_table.index_select(0, st).unsqueeze(1)  # [B, 1, V]
            tok = binding.spec_sample_draft(rows, None if greedy else ud_d[:, j:j + 1].contiguous(), **prm)
            drafted[:, j] = tok[:, 0]
            cur = tok[:, 0].to(torch.int64)
        states[:, K] = state_fn(cur, pos + K)
        # the target scores all K+1 positions of the round in one call
        target = target_table.index_select(0, states.reshape(-1)).view(B, K + 1, V)
        draft = None if greedy else draft_table.index_select(0, states[:, :K].reshape(-1)).view(B, K, V)
        out_t, out_n = binding.spec_verify(target, draft, drafted, uv_d, **prm)
        n = out_n.to(torch.int64)
        # the next context ends with the token emitted after the n accepted ones
        last = out_t.gather(1, n.clamp(min=0).unsqueeze(1)).squeeze(1).to(torch.int64)
        pos = pos + n + 1
        if record:
            out.append((out_t.clone(), out_n.clone()))
    return out


def expected_tokens_per_round(alpha, K):
    """E[tokens emitted per round] with acceptance alpha at every position:
    (1 - alpha^(K+1)) / (1 - alpha), and K + 1 at alpha = 1."""
    if alpha >= 1.0:
        return float(K + 1)
    return (1.0 - alpha ** (K + 1)) / (1.0 - alpha)


def speedup(alpha, K, c, verify_cost=0.0):
    """Tokens per unit time relative to one token per target call.  A round costs
    K draft calls (c each, in target-call units), one target call, and the
    verification step (verify_cost, in target-call units; 0 gives the page's form
    (1 - alpha^(K+1)) / ((1 - alpha)(K c + 1)))."""
    return expected_tokens_per_round(alpha, K) / (K * c + 1.0 + verify_cost)


def best_k(alpha, c, verify_cost_of_k, k_max=16):
    """The K in [1, k_max] with the largest speed-up, given the verification cost
    as a function of K (in target-call units)."""
    return max(range(1, k_max + 1), key=lambda k: speedup(alpha, k, c, verify_cost_of_k(k)))
