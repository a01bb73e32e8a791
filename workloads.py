"""Seeded synthetic inputs for speculative-sampling verification.

This module is the only code shared by the CUDA path's tests/bench and the
oracle's tests.  It holds none of the method's arithmetic: it draws logits,
uniforms and parameters, nothing else.  Draft tokens are NOT made here, because
drawing them is part of the method (`spec_sample_draft` on the GPU side,
`oracle.sample_draft` on the oracle side); the uniforms for that draw are.

The pages' workloads (Chinchilla 70B with a 4B draft on XSum and HumanEval;
"Accelerating Large Language Model Decoding with Speculative Sampling",
section "The result") need trained models and datasets that are not available.
These generators stand in for them with the shapes of the five configurations:

  c1  B=1   K=4 V=32     fp32  target ~ N(0, 2^2); draft = target + N(0, 1^2); T=1
  c2  B=1   K=4 V=32000  bf16  Zipf+Gaussian target; draft noise sigma=1.5; T=1
  c3  B=64  K=4 V=128256 bf16  sigma=1.0; T=0.8, top_p=0.9
  c4  B=256 K=3 V=50304  fp32  sigma=2.0; greedy          (c4_bf16: same values in bf16)
  c5  B=32  K=8 V=256000 bf16  sigma=0.5; T=1.0, top_k=50

Zipf+Gaussian target row: l_x = N(0, 3^2) - 1.1 * ln(rank_x), rank_x = 1 + pi(x) for one
seeded permutation pi of [0, V) per configuration; every (b, t) row draws its own noise;
draft row t = target row t + N(0, sigma^2).  bf16 values are the fp32 values rounded to
nearest-even.  Configuration i (0-based, c1 = 0) uses numpy.random.default_rng(i) with
the fixed draw order: permutation, target noise, draft noise, draft-token uniforms,
verify uniforms.
"""
from __future__ import annotations

import dataclasses

import numpy as np


@dataclasses.dataclass
class Config:
    name: str
    seed: int
    B: int
    K: int
    V: int
    dtype: str            # "f32" or "bf16"
    kind: str             # "gauss" (c1) or "zipf"
    sigma_draft: float
    temperature: float = 1.0
    top_k: int = 0
    top_p: float = 1.0
    greedy: bool = False

    def describe(self) -> str:
        mode = "greedy" if self.greedy else "T=%g%s%s" % (
            self.temperature, " top_k=%d" % self.top_k if self.top_k else "",
            " top_p=%g" % self.top_p if self.top_p < 1 else "")
        return "B=%d K=%d V=%d %s %s" % (self.B, self.K, self.V, self.dtype, mode)


CONFIGS = {
    "c1": Config("c1", 0, 1, 4, 32, "f32", "gauss", 1.0),
    "c2": Config("c2", 1, 1, 4, 32000, "bf16", "zipf", 1.5),
    "c3": Config("c3", 2, 64, 4, 128256, "bf16", "zipf", 1.0, temperature=0.8, top_p=0.9),
    "c4": Config("c4", 3, 256, 3, 50304, "f32", "zipf", 2.0, greedy=True),
    "c4_bf16": Config("c4_bf16", 3, 256, 3, 50304, "bf16", "zipf", 2.0, greedy=True),
    "c5": Config("c5", 4, 32, 8, 256000, "bf16", "zipf", 0.5, temperature=1.0, top_k=50),
}


def to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round fp32 values to bf16 (nearest-even) and return the raw uint16 bits."""
    b = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    rounded = (b + np.uint32(0x7FFF) + ((b >> np.uint32(16)) & np.uint32(1))) >> np.uint32(16)
    return rounded.astype(np.uint16)


def bf16_bits_to_f32(h: np.ndarray) -> np.ndarray:
    return (h.astype(np.uint32) << np.uint32(16)).view(np.float32)


def make(cfg: Config | str, B: int | None = None, V: int | None = None, K: int | None = None,
         seed: int | None = None) -> dict:
    """Draw one batch of inputs for a configuration (optionally resized / reseeded).

    Returns dict with target [B, K+1, V] and draft [B, K, V] (float32, or uint16 bf16
    bits), u_draft [B, K] and u_verify [B, K+1] (float64 in [0, 1)), and the
    sampling parameters of the configuration.
    """
    if isinstance(cfg, str):
        cfg = CONFIGS[cfg]
    B = cfg.B if B is None else B
    V = cfg.V if V is None else V
    K = cfg.K if K is None else K
    rng = np.random.default_rng(cfg.seed if seed is None else seed)
    perm = rng.permutation(V)
    if cfg.kind == "gauss":
        target = rng.standard_normal((B, K + 1, V), dtype=np.float32) * np.float32(2.0)
    else:
        bias = (np.float32(-1.1) * np.log((1 + perm).astype(np.float32))).astype(np.float32)
        target = rng.standard_normal((B, K + 1, V), dtype=np.float32)
        target *= np.float32(3.0)
        target += bias
    draft = rng.standard_normal((B, K, V), dtype=np.float32)
    draft *= np.float32(cfg.sigma_draft)
    draft += target[:, :K, :]
    u_draft = rng.random((B, K))
    u_verify = rng.random((B, K + 1))
    if cfg.dtype == "bf16":
        target, draft = to_bf16_bits(target), to_bf16_bits(draft)
    return dict(target=target, draft=draft, u_draft=u_draft, u_verify=u_verify,
                temperature=cfg.temperature, top_k=cfg.top_k, top_p=cfg.top_p,
                greedy=cfg.greedy, B=B, K=K, V=V, dtype=cfg.dtype, name=cfg.name)


# --------------------------------------------------------------------------
# Synthetic logit sources for the decode-round driver.
#
# The decode loop of the pages ("Speculative Decoding", roadtointelligence.com,
# section "Draft, then verify"; Algorithm 2 in the paperlayer.ai summary of
# "Accelerating Large Language Model Decoding with Speculative Sampling") calls
# a draft and a target model.  No weights are available, so each "model" here
# is a seeded table of S logit rows, and the row for a context is picked by a
# state computed from the context's last token and its position:
#     state = (last_token * STATE_A + position * STATE_B) mod S.
# Both the GPU driver and the oracle's loop index the same tables with the same
# integer formula, so they see bit-identical rows.

STATE_A, STATE_B = 7919, 104729


def state_of(last_token, position, S):
    """State index of a context (numpy or torch integer arrays; int64 math)."""
    return (last_token * STATE_A + position * STATE_B) % S


@dataclasses.dataclass
class SyntheticSource:
    V: int
    S: int
    target: np.ndarray      # [S, V] float32 logits (or uint16 bf16 bits)
    draft: np.ndarray       # [S, V]
    alpha: float | None     # the exact acceptance of every state, when built for one
    dtype: str


def synthetic_source(V=256, S=97, alpha=None, seed=0, dtype="f32", sigma_draft=1.0):
    """Target and draft tables of S rows.

    alpha=None: Zipf+Gaussian target rows as in make() and draft = target +
    N(0, sigma_draft^2).  alpha given: every state has sum_x min(p, q) = alpha
    exactly (in the probabilities the logits are the logs of): the draft q lives on
    tokens [0, V/2) with q = softmax(N(0, 1.5^2)) there; the target is
    p = alpha * q + (1 - alpha) * r with r uniform on [V/2, V), where q = 0.
    """
    rng = np.random.default_rng(seed)
    if alpha is None:
        perm = rng.permutation(V)
        bias = (np.float32(-1.1) * np.log((1 + perm).astype(np.float32))).astype(np.float32)
        target = rng.standard_normal((S, V), dtype=np.float32) * np.float32(3.0) + bias
        draft = target + rng.standard_normal((S, V), dtype=np.float32) * np.float32(sigma_draft)
    else:
        h = V // 2
        g = rng.standard_normal((S, h)) * 1.5
        q = np.exp(g - g.max(axis=1, keepdims=True))
        q /= q.sum(axis=1, keepdims=True)
        qf = np.zeros((S, V))
        qf[:, :h] = q
        r = np.zeros((S, V))
        r[:, h:] = 1.0 / (V - h)
        p = alpha * qf + (1 - alpha) * r
        with np.errstate(divide="ignore"):
            target, draft = np.log(p).astype(np.float32), np.log(qf).astype(np.float32)
    if dtype == "bf16":
        target, draft = to_bf16_bits(target), to_bf16_bits(draft)
    return SyntheticSource(V, S, np.ascontiguousarray(target), np.ascontiguousarray(draft), alpha, dtype)


def round_uniforms(seed, r, B, K):
    """Uniforms of decode round r: u_draft [B, K] (draft draws), u_verify [B, K+1]."""
    rng = np.random.default_rng([int(seed), int(r)])
    return rng.random((B, K)), rng.random((B, K + 1))
