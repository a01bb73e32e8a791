"""fp64 CPU oracle for speculative-sampling verification (ctypes wrapper).

TEST INFRASTRUCTURE ONLY.  Only `tests/`, `__graft_entry__.smoke()` and the
`cpu_baseline` / `--impl reference` legs of `bench.py` may import this module.
The product package never imports it, and it never imports the product
package: the two share nothing but the seeded input generator in
`workloads.py`.

The arithmetic lives in `oracle.c` (plain C, fp64, single-threaded); this file
only builds it with gcc and marshals numpy arrays.  Every function follows the
definition stated in `oracle.h`, which cites the passages of the pages.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")

F32, BF16 = 0, 1
OK, ERR_INVALID_ARG, ERR_NONFINITE, ERR_TOKEN_RANGE = 0, 1, 3, 4
NEAR_ACCEPT, NEAR_DRAW, NEAR_TOPP = 1, 2, 4
NEAR_EPS = 1e-6


class Params(ctypes.Structure):
    _fields_ = [
        ("B", ctypes.c_int32), ("K", ctypes.c_int32), ("V", ctypes.c_int32),
        ("dtype", ctypes.c_int32),
        ("tgt_seq_stride", ctypes.c_int64), ("tgt_row_stride", ctypes.c_int64),
        ("drf_seq_stride", ctypes.c_int64), ("drf_row_stride", ctypes.c_int64),
        ("temperature", ctypes.c_float), ("top_k", ctypes.c_int32),
        ("top_p", ctypes.c_float), ("greedy", ctypes.c_int32),
    ]


_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile oracle.c into liboracle.so with gcc (portable flags only)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < max(
            os.path.getmtime(_SRC), os.path.getmtime(os.path.join(_HERE, "oracle.h"))):
        tmp = _LIB + ".tmp.%d" % os.getpid()
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-Wall",
                               "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def lib():
    global _lib
    with _lock:
        if _lib is None:
            # ORACLE_LIB lets the mutation tests load a deliberately broken copy
            path = os.environ.get("ORACLE_LIB") or build()
            L = ctypes.CDLL(path)
            P = ctypes.c_void_p
            L.oracle_row_probs.argtypes = [P, ctypes.c_int32, ctypes.c_int32, ctypes.c_float,
                                           ctypes.c_int32, ctypes.c_float, ctypes.c_int32,
                                           P, P, P, P]
            L.oracle_verify.argtypes = [P, P, P, P, ctypes.POINTER(Params), P, P, P, P]
            L.oracle_sample_draft.argtypes = [P, P, ctypes.POINTER(Params), P, P]
            for f in (L.oracle_row_probs, L.oracle_verify, L.oracle_sample_draft):
                f.restype = ctypes.c_int
            L.oracle_accept_histogram.argtypes = [P, ctypes.c_int64, ctypes.c_int32, P]
            L.oracle_accept_histogram.restype = None
            _lib = L
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data


def _dtype_code(arr):
    if arr.dtype == np.float32:
        return F32
    if arr.dtype == np.uint16:  # bf16 carried as raw bits
        return BF16
    raise TypeError("logits must be float32 or uint16 (bf16 bits), got %s" % arr.dtype)


def row_probs(row, temperature=1.0, top_k=0, top_p=1.0, greedy=False):
    """Adjusted distribution of one row -> (probs[V] fp64, argmax, near_topp, (max, Z_f), status)."""
    row = np.ascontiguousarray(row)
    V = row.shape[-1]
    probs = np.zeros(V, np.float64)
    amax = np.zeros(1, np.int32)
    near = np.zeros(1, np.int32)
    stats = np.zeros(2, np.float64)
    s = lib().oracle_row_probs(_ptr(row), _dtype_code(row), V, float(temperature), int(top_k),
                               float(top_p), int(bool(greedy)), _ptr(probs), _ptr(amax),
                               _ptr(near), _ptr(stats))
    return probs, int(amax[0]), bool(near[0]), (float(stats[0]), float(stats[1])), s


def _params(B, K, V, dtype, tgt_strides, drf_strides, temperature, top_k, top_p, greedy):
    return Params(B, K, V, dtype, tgt_strides[0], tgt_strides[1], drf_strides[0], drf_strides[1],
                  float(temperature), int(top_k), float(top_p), int(bool(greedy)))


def verify(target, draft, tokens, uniforms, temperature=1.0, top_k=0, top_p=1.0, greedy=False,
           with_stats=False, tgt_strides=None, drf_strides=None, B=None):
    """Oracle verification.  target [B, K+1, V], draft [B, K, V] (or None when greedy),
    tokens [B, K] int32, uniforms [B, K+1] fp64 (or None when greedy).  Strides (elements)
    default to the contiguous layout; pass (0, V) to repeat one sequence's rows B times.
    Returns dict(tokens, num_accepted, flags, status[, row_stats])."""
    tokens = np.ascontiguousarray(tokens, dtype=np.int32)
    if B is None:
        B = tokens.shape[0]
    K = tokens.shape[1]
    V = target.shape[-1]
    dt = _dtype_code(target)
    tgt_strides = tgt_strides or ((K + 1) * V, V)
    drf_strides = drf_strides or (K * V, V)
    if draft is not None:
        assert draft.dtype == target.dtype
    p = _params(B, K, V, dt, tgt_strides, drf_strides, temperature, top_k, top_p, greedy)
    out_t = np.full((B, K + 1), -7, np.int32)
    out_n = np.full(B, -7, np.int32)
    flags = np.zeros(B, np.int32)
    stats = np.zeros((B, 2 * K + 1, 3), np.float64) if with_stats else None
    u = None if uniforms is None else np.ascontiguousarray(uniforms, dtype=np.float64)
    s = lib().oracle_verify(_ptr(target), _ptr(draft), _ptr(tokens), _ptr(u), ctypes.byref(p),
                            _ptr(out_t), _ptr(out_n), _ptr(flags), _ptr(stats))
    res = dict(tokens=out_t, num_accepted=out_n, flags=flags, status=s)
    if with_stats:
        res["row_stats"] = stats
    return res


def sample_draft(draft, uniforms, temperature=1.0, top_k=0, top_p=1.0, greedy=False,
                 drf_strides=None, B=None, K=None):
    """Oracle draft-token drawing.  draft [B, K, V], uniforms [B, K] fp64 (None when greedy).
    Returns dict(tokens [B, K], flags [B, K], status)."""
    if B is None or K is None:
        B, K = draft.shape[0], draft.shape[1]
    V = draft.shape[-1]
    drf_strides = drf_strides or (K * V, V)
    p = _params(B, K, V, _dtype_code(draft), (0, 0), drf_strides, temperature, top_k, top_p, greedy)
    out_t = np.full((B, K), -7, np.int32)
    flags = np.zeros((B, K), np.int32)
    u = None if uniforms is None else np.ascontiguousarray(uniforms, dtype=np.float64)
    s = lib().oracle_sample_draft(_ptr(draft), _ptr(u), ctypes.byref(p), _ptr(out_t), _ptr(flags))
    return dict(tokens=out_t, flags=flags, status=s)


def accept_histogram(num_accepted, K):
    """int64 [K+2]: sequences per number of accepted draft tokens 0..K, then the
    sequences that ended in an error (oracle_accept_histogram in oracle.h)."""
    n = np.ascontiguousarray(num_accepted, dtype=np.int32)
    hist = np.zeros(int(K) + 2, dtype=np.int64)
    L = lib()
    L.oracle_accept_histogram(n.ctypes.data_as(ctypes.c_void_p), ctypes.c_int64(n.size), ctypes.c_int32(int(K)),
                              hist.ctypes.data_as(ctypes.c_void_p))
    return hist


def verify_threaded(target, draft, tokens, uniforms, threads, **kw):
    """Run `verify` over contiguous sequence slices on `threads` host threads (ctypes
    releases the GIL).  Same result as `verify` (row_stats included when asked for);
    used to time the oracle on many cores and to check full-size launches quickly."""
    B = tokens.shape[0]
    bounds = np.linspace(0, B, threads + 1).astype(int)
    parts = [None] * threads

    def work(i):
        a, b = bounds[i], bounds[i + 1]
        if b > a:
            parts[i] = verify(target[a:b], None if draft is None else draft[a:b], tokens[a:b],
                              None if uniforms is None else uniforms[a:b], **kw)

    ts = [threading.Thread(target=work, args=(i,)) for i in range(threads)]
    for t in ts:
        t.start()
    for t in ts:
        t.join()
    parts = [p for p in parts if p is not None]
    res = dict(tokens=np.concatenate([p["tokens"] for p in parts]),
               num_accepted=np.concatenate([p["num_accepted"] for p in parts]),
               flags=np.concatenate([p["flags"] for p in parts]),
               status=next((p["status"] for p in parts if p["status"]), 0))
    if kw.get("with_stats"):
        res["row_stats"] = np.concatenate([p["row_stats"] for p in parts])
    return res


def sample_draft_threaded(draft, uniforms, threads, **kw):
    """`sample_draft` over contiguous sequence slices on `threads` host threads; same
    result as `sample_draft` (the tests use it to check full-size launches quickly)."""
    B = draft.shape[0]
    bounds = np.linspace(0, B, threads + 1).astype(int)
    parts = [None] * threads

    def work(i):
        a, b = bounds[i], bounds[i + 1]
        if b > a:
            parts[i] = sample_draft(draft[a:b], None if uniforms is None else uniforms[a:b], **kw)

    ts = [threading.Thread(target=work, args=(i,)) for i in range(threads)]
    for t in ts:
        t.start()
    for t in ts:
        t.join()
    parts = [p for p in parts if p is not None]
    return dict(tokens=np.concatenate([p["tokens"] for p in parts]),
                flags=np.concatenate([p["flags"] for p in parts]),
                status=next((p["status"] for p in parts if p["status"]), 0))
