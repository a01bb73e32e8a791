"""Shared helpers of the GPU tests: move seeded inputs to the device, run the CUDA
path through the binding (which calls the C ABI), and compare with the oracle."""
import numpy as np
import torch

import oracle
from _report import record

NEAR_ANY = oracle.NEAR_ACCEPT | oracle.NEAR_DRAW | oracle.NEAR_TOPP


def to_dev(arr, dev="cuda:0"):
    """numpy float32 -> float32 tensor; numpy uint16 (bf16 bits) -> bfloat16 tensor."""
    if arr.dtype == np.uint16:
        return torch.from_numpy(np.ascontiguousarray(arr).view(np.int16)).view(torch.bfloat16).to(dev)
    return torch.from_numpy(np.ascontiguousarray(arr)).to(dev)


def params_of(w):
    return dict(temperature=w["temperature"], top_k=w["top_k"], top_p=w["top_p"],
                greedy=w["greedy"])


def compare_verify(gpu_tokens, gpu_n, ref, where=""):
    """Bit-exact comparison, sequences flagged near a threshold excluded (and counted).
    Returns the number of flagged sequences."""
    gt, gn = np.asarray(gpu_tokens), np.asarray(gpu_n)
    flagged = (ref["flags"] & NEAR_ANY) != 0
    ok = ~flagged
    bad = np.nonzero((gn[ok] != ref["num_accepted"][ok]) |
                     np.any(gt[ok] != ref["tokens"][ok], axis=1))[0]
    if len(bad):
        idx = np.nonzero(ok)[0][bad[:5]]
        raise AssertionError("%s: %d mismatching sequences, e.g. %s: gpu n=%s tok=%s | oracle n=%s tok=%s" % (
            where, len(bad), idx.tolist(), gn[idx].tolist(), gt[idx].tolist(),
            ref["num_accepted"][idx].tolist(), ref["tokens"][idx].tolist()))
    record(where or "verify", len(gn), int(flagged.sum()))
    return int(flagged.sum())


def check_invariants(gpu_tokens, gpu_n, d, K, V):
    gt, gn = np.asarray(gpu_tokens), np.asarray(gpu_n)
    for b in range(len(gn)):
        n = gn[b]
        assert 0 <= n <= K
        assert np.array_equal(gt[b, :n], d[b, :n])
        assert 0 <= gt[b, n] < V
        assert np.all(gt[b, n + 1:] == -1)
