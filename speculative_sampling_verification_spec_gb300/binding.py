"""Python binding of libspecverify.so: argument marshalling only.

Each function here has the name of the C entry point it calls (see
include/spec_verify.h) and does nothing but turn torch CUDA tensors into
pointers, strides and a stream handle.  Every step of the computation runs in
the library's CUDA kernels; there is no CPU or PyTorch fallback, and a missing
library raises.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

from . import _build

SPEC_OK = 0
SPEC_F32, SPEC_BF16 = 0, 1
STATUS_NAMES = {0: "SPEC_OK", 1: "SPEC_ERR_INVALID_ARG", 2: "SPEC_ERR_CUDA", 3: "SPEC_ERR_NONFINITE",
                4: "SPEC_ERR_TOKEN_RANGE", 5: "SPEC_ERR_TIMEOUT", 6: "SPEC_ERR_UNSUPPORTED",
                7: "SPEC_ERR_SCRATCH_LIMIT"}
SPEC_NOALLOC_SCRATCH_BYTES = 8 << 20
EXPORTED = ("spec_verify", "spec_sample_draft", "spec_verify_workspace_size",
            "spec_sample_draft_workspace_size", "spec_read_row_stats", "spec_status_string",
            "spec_launch_count", "spec_verify_noalloc", "spec_accept_histogram", "spec_sample_verify",
            "spec_verify_ragged", "spec_verify_ragged_workspace_size")


class SpecParams(ctypes.Structure):
    _fields_ = [
        ("B", ctypes.c_int32), ("K", ctypes.c_int32), ("V", ctypes.c_int32),
        ("dtype", ctypes.c_int32),
        ("target_seq_stride", ctypes.c_int64), ("target_row_stride", ctypes.c_int64),
        ("draft_seq_stride", ctypes.c_int64), ("draft_row_stride", ctypes.c_int64),
        ("temperature", ctypes.c_float), ("top_k", ctypes.c_int32), ("top_p", ctypes.c_float),
        ("greedy", ctypes.c_int32),
        ("stream", ctypes.c_void_p), ("status", ctypes.c_void_p),
        ("workspace", ctypes.c_void_p), ("workspace_bytes", ctypes.c_size_t),
    ]


class SpecRowStat(ctypes.Structure):
    _fields_ = [
        ("zf", ctypes.c_double), ("p_tok", ctypes.c_double), ("m", ctypes.c_float),
        ("tau_val", ctypes.c_float), ("tau_idx", ctypes.c_int32), ("argmax", ctypes.c_int32),
        ("list_len", ctypes.c_int32), ("flags", ctypes.c_int32), ("token", ctypes.c_int32),
        ("pad_", ctypes.c_int32),
    ]


class SpecError(RuntimeError):
    def __init__(self, code, what):
        super().__init__("%s: %s (%s)" % (what, STATUS_NAMES.get(code, code), spec_status_string(code)))
        self.code = code


_lock = threading.Lock()
_lib = None


def lib() -> ctypes.CDLL:
    """The loaded library; raises if it has not been built (no fallback exists)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(_build.LIB):
                raise FileNotFoundError(
                    "libspecverify.so is missing: build it with "
                    "`python -c 'import __graft_entry__ as g; g.build()'`")
            L = ctypes.CDLL(_build.LIB)
            P = ctypes.c_void_p
            PP = ctypes.POINTER(SpecParams)
            L.spec_verify.argtypes = [P, P, P, P, PP, P, P]
            L.spec_verify.restype = ctypes.c_int
            L.spec_sample_draft.argtypes = [P, P, PP, P]
            L.spec_sample_draft.restype = ctypes.c_int
            L.spec_verify_workspace_size.argtypes = [PP]
            L.spec_verify_workspace_size.restype = ctypes.c_size_t
            L.spec_sample_draft_workspace_size.argtypes = [PP]
            L.spec_sample_draft_workspace_size.restype = ctypes.c_size_t
            L.spec_read_row_stats.argtypes = [PP, ctypes.c_int32, P, ctypes.c_int64]
            L.spec_read_row_stats.restype = ctypes.c_int
            L.spec_status_string.argtypes = [ctypes.c_int]
            L.spec_status_string.restype = ctypes.c_char_p
            L.spec_verify_noalloc.argtypes = [P, P, P, P, PP, P, P]
            L.spec_verify_noalloc.restype = ctypes.c_int
            L.spec_verify_ragged.argtypes = [P, P, P, P, P, PP, P, P]
            L.spec_verify_ragged.restype = ctypes.c_int
            L.spec_verify_ragged_workspace_size.argtypes = [PP]
            L.spec_verify_ragged_workspace_size.restype = ctypes.c_size_t
            L.spec_sample_verify.argtypes = [P, P, P, P, PP, P, P, P]
            L.spec_sample_verify.restype = ctypes.c_int
            L.spec_accept_histogram.argtypes = [P, ctypes.c_int32, ctypes.c_int32, P, P]
            L.spec_accept_histogram.restype = ctypes.c_int
            L.spec_launch_count.argtypes = []
            L.spec_launch_count.restype = ctypes.c_uint64
            _lib = L
    return _lib


def spec_status_string(code: int) -> str:
    return lib().spec_status_string(int(code)).decode()


def spec_launch_count() -> int:
    return int(lib().spec_launch_count())


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.float32:
        return SPEC_F32
    if t.dtype == torch.bfloat16:
        return SPEC_BF16
    raise TypeError("logits must be float32 or bfloat16, got %s" % t.dtype)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _check_cuda(*ts):
    for t in ts:
        if t is not None and not t.is_cuda:
            raise ValueError("spec_* calls take CUDA tensors (copy host data to the GPU first)")


_ws_cache = {}


def workspace(nbytes: int, device: torch.device) -> torch.Tensor:
    """A zero-filled device workspace of at least nbytes, cached per device (the
    kernels leave it reusable, so it is zeroed only when first allocated)."""
    key = (device.index if device.index is not None else torch.cuda.current_device())
    ws = _ws_cache.get(key)
    if ws is None or ws.numel() < nbytes:
        ws = torch.zeros(max(nbytes, 1 << 16), dtype=torch.uint8, device=device)
        _ws_cache[key] = ws
    return ws


def make_params(B, K, V, dtype, tgt_strides=(0, 0), drf_strides=(0, 0), temperature=1.0, top_k=0,
                top_p=1.0, greedy=False, stream=None, status=None, ws=None) -> SpecParams:
    return SpecParams(int(B), int(K), int(V), int(dtype), int(tgt_strides[0]), int(tgt_strides[1]),
                      int(drf_strides[0]), int(drf_strides[1]), float(temperature), int(top_k),
                      float(top_p), int(bool(greedy)), stream,
                      None if status is None else status.data_ptr(),
                      None if ws is None else ws.data_ptr(), 0 if ws is None else ws.numel())


def _stream_handle(stream):
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def spec_verify_workspace_size(B, K, V, dtype, greedy=False) -> int:
    p = make_params(B, K, V, dtype, greedy=greedy)
    return int(lib().spec_verify_workspace_size(ctypes.byref(p)))


def spec_sample_draft_workspace_size(B, K, V, dtype, greedy=False) -> int:
    p = make_params(B, K, V, dtype, greedy=greedy)
    return int(lib().spec_sample_draft_workspace_size(ctypes.byref(p)))


class _VerifyArgs:
    pass


def _verify_args(target, draft, draft_tokens, uniforms, B=None, out_tokens=None, out_num_accepted=None,
                 stream=None):
    """Checks and conversions shared by every verify entry point: CUDA tensors, one
    logit dtype (float32 or bfloat16) for both models, unit stride along V, int32
    tokens and float64 uniforms (both made contiguous), and the output tensors.
    Converted copies are recorded on `stream` so the allocator keeps them until the
    call's kernels have read them."""
    _check_cuda(target, draft, draft_tokens, uniforms)
    a = _VerifyArgs()
    a.K = draft_tokens.shape[1]
    a.B = draft_tokens.shape[0] if B is None else B
    a.V = target.shape[-1]
    a.dt = _dtype_code(target)
    if draft is not None and draft.dtype != target.dtype:
        raise TypeError("target and draft logits must share a dtype")
    if target.stride(-1) != 1 or (draft is not None and draft.stride(-1) != 1):
        raise ValueError("logit rows must be contiguous along the vocabulary")
    if uniforms is not None and uniforms.dtype != torch.float64:
        raise TypeError("uniforms must be float64")
    a.tstr = (target.stride(0), target.stride(1))
    a.dstr = (draft.stride(0), draft.stride(1)) if draft is not None else (0, 0)
    tok = draft_tokens if draft_tokens.dtype == torch.int32 else draft_tokens.to(torch.int32)
    a.tok = tok.contiguous()
    a.u = None if uniforms is None else uniforms.contiguous()
    if stream is not None:
        for t, orig in ((a.tok, draft_tokens), (a.u, uniforms)):
            if t is not None and t.data_ptr() != orig.data_ptr():
                t.record_stream(stream)
    dev = target.device
    a.out_tokens = torch.empty((a.B, a.K + 1), dtype=torch.int32, device=dev) if out_tokens is None else out_tokens
    a.out_n = torch.empty((a.B,), dtype=torch.int32, device=dev) if out_num_accepted is None else out_num_accepted
    for o, shape in ((a.out_tokens, (a.B, a.K + 1)), (a.out_n, (a.B,))):
        if o.dtype != torch.int32 or tuple(o.shape) != shape or not o.is_contiguous() or not o.is_cuda:
            raise ValueError("outputs must be contiguous int32 CUDA tensors of shape %s" % (shape,))
    return a


def spec_verify(target, draft, draft_tokens, uniforms, *, temperature=1.0, top_k=0, top_p=1.0,
                greedy=False, out_tokens=None, out_num_accepted=None, status=None, ws=None,
                stream=None, B=None):
    """target [B, K+1, V] and draft [B, K, V] CUDA logits (any element strides for the
    first two dims, unit stride along V), draft_tokens [B, K] int32, uniforms [B, K+1]
    float64.  Returns (out_tokens [B, K+1] int32, out_num_accepted [B] int32)."""
    a = _verify_args(target, draft, draft_tokens, uniforms, B, out_tokens, out_num_accepted, stream)
    p = make_params(a.B, a.K, a.V, a.dt, a.tstr, a.dstr, temperature, top_k, top_p, greedy,
                    _stream_handle(stream), status)
    if ws is None:
        ws = workspace(int(lib().spec_verify_workspace_size(ctypes.byref(p))), target.device)
    p.workspace, p.workspace_bytes = ws.data_ptr(), ws.numel()
    code = lib().spec_verify(_ptr(target), _ptr(draft), _ptr(a.tok), _ptr(a.u), ctypes.byref(p),
                             _ptr(a.out_tokens), _ptr(a.out_n))
    if code != SPEC_OK:
        raise SpecError(code, "spec_verify")
    return a.out_tokens, a.out_n


def spec_sample_draft(draft, uniforms, *, temperature=1.0, top_k=0, top_p=1.0, greedy=False,
                      out_tokens=None, status=None, ws=None, stream=None):
    """draft [B, K, V] CUDA logits, uniforms [B, K] float64 (None when greedy).
    Returns out_tokens [B, K] int32."""
    _check_cuda(draft, uniforms)
    B, K, V = draft.shape[0], draft.shape[1], draft.shape[-1]
    if draft.stride(-1) != 1:
        raise ValueError("logit rows must be contiguous along the vocabulary")
    dev = draft.device
    if out_tokens is None:
        out_tokens = torch.empty((B, K), dtype=torch.int32, device=dev)
    p = make_params(B, K, V, _dtype_code(draft), (0, 0), (draft.stride(0), draft.stride(1)),
                    temperature, top_k, top_p, greedy, _stream_handle(stream), status)
    if ws is None:
        ws = workspace(int(lib().spec_sample_draft_workspace_size(ctypes.byref(p))), dev)
    p.workspace, p.workspace_bytes = ws.data_ptr(), ws.numel()
    if uniforms is not None and uniforms.dtype != torch.float64:
        raise TypeError("uniforms must be float64")
    code = lib().spec_sample_draft(_ptr(draft), _ptr(None if uniforms is None else uniforms.contiguous()),
                                   ctypes.byref(p), _ptr(out_tokens))
    if code != SPEC_OK:
        raise SpecError(code, "spec_sample_draft")
    return out_tokens


def spec_read_row_stats(B, K, V, dtype, is_verify, ws, *, greedy=False, temperature=1.0, top_k=0,
                        top_p=1.0, stream=None):
    """Per-row records of the last call made with workspace `ws` (list of dicts)."""
    p = make_params(B, K, V, dtype, temperature=temperature, top_k=top_k, top_p=top_p,
                    greedy=greedy, stream=_stream_handle(stream), ws=ws)
    R = (K + 1 if greedy else 2 * K + 1) if is_verify else K
    n = B * R
    arr = (SpecRowStat * max(n, 1))()
    code = lib().spec_read_row_stats(ctypes.byref(p), int(bool(is_verify)), arr, n)
    if code != SPEC_OK:
        raise SpecError(code, "spec_read_row_stats")
    return [{f: getattr(arr[i], f) for f, _ in SpecRowStat._fields_ if f != "pad_"} for i in range(n)]


def spec_verify_noalloc(target, draft, draft_tokens, uniforms, *, temperature=1.0, top_k=0, top_p=1.0,
                        greedy=False, out_tokens=None, out_num_accepted=None, status=None, stream=None):
    """spec_verify with the library's fixed scratch array instead of a workspace, for
    callers that may not allocate device memory (see include/spec_verify.h).  Same
    arguments and results as spec_verify."""
    a = _verify_args(target, draft, draft_tokens, uniforms, None, out_tokens, out_num_accepted, stream)
    p = make_params(a.B, a.K, a.V, a.dt, a.tstr, a.dstr, temperature, top_k, top_p, greedy,
                    _stream_handle(stream), status)
    code = lib().spec_verify_noalloc(_ptr(target), _ptr(draft), _ptr(a.tok), _ptr(a.u), ctypes.byref(p),
                                     _ptr(a.out_tokens), _ptr(a.out_n))
    if code != SPEC_OK:
        raise SpecError(code, "spec_verify_noalloc")
    return a.out_tokens, a.out_n


def spec_accept_histogram(out_num_accepted, K, *, hist=None, stream=None):
    """Add the histogram of accepted-draft counts (out_num_accepted [B] int32 CUDA)
    to hist (int32 [K+2] CUDA; a zeroed one is made when None): bins 0..K count
    sequences by accepted tokens, bin K+1 the sequences that ended in an error.
    Returns hist."""
    _check_cuda(out_num_accepted)
    n = out_num_accepted if out_num_accepted.dtype == torch.int32 else out_num_accepted.to(torch.int32)
    n = n.contiguous()
    if hist is None:
        hist = torch.zeros((int(K) + 2,), dtype=torch.int32, device=n.device)
    _check_cuda(hist)
    if hist.dtype != torch.int32 or hist.numel() != int(K) + 2 or not hist.is_contiguous():
        raise ValueError("hist must be a contiguous int32 tensor of K + 2 entries")
    code = lib().spec_accept_histogram(_ptr(n), int(n.numel()), int(K), _ptr(hist), _stream_handle(stream))
    if code != SPEC_OK:
        raise SpecError(code, "spec_accept_histogram")
    return hist


def spec_sample_verify(target, draft, draft_uniforms, uniforms, *, temperature=1.0, top_k=0, top_p=1.0,
                       greedy=False, out_draft_tokens=None, out_tokens=None, out_num_accepted=None, status=None,
                       ws=None, stream=None):
    """K = 1 drafting step and verification in one call: target [B, 2, V] and draft
    [B, 1, V] CUDA logits, draft_uniforms [B] and uniforms [B, 2] float64.
    Returns (out_draft_tokens [B], out_tokens [B, 2], out_num_accepted [B]), int32.
    Sampling only (greedy has no draft draw to fuse)."""
    if greedy:
        raise ValueError("spec_sample_verify samples; use spec_sample_draft + spec_verify for greedy")
    _check_cuda(target, draft, draft_uniforms, uniforms)
    B, V = target.shape[0], target.shape[-1]
    if target.shape[1] != 2 or draft.shape[1] != 1:
        raise ValueError("spec_sample_verify takes K = 1: target [B, 2, V], draft [B, 1, V]")
    if draft.dtype != target.dtype:
        raise TypeError("target and draft logits must share a dtype")
    if target.stride(-1) != 1 or draft.stride(-1) != 1:
        raise ValueError("logit rows must be contiguous along the vocabulary")
    if draft_uniforms.dtype != torch.float64 or uniforms.dtype != torch.float64:
        raise TypeError("uniforms must be float64")
    dev = target.device
    if out_draft_tokens is None:
        out_draft_tokens = torch.empty((B,), dtype=torch.int32, device=dev)
    if out_tokens is None:
        out_tokens = torch.empty((B, 2), dtype=torch.int32, device=dev)
    if out_num_accepted is None:
        out_num_accepted = torch.empty((B,), dtype=torch.int32, device=dev)
    p = make_params(B, 1, V, _dtype_code(target), (target.stride(0), target.stride(1)),
                    (draft.stride(0), draft.stride(1)), temperature, top_k, top_p, False,
                    _stream_handle(stream), status)
    if ws is None:
        ws = workspace(int(lib().spec_verify_workspace_size(ctypes.byref(p))), dev)
    p.workspace, p.workspace_bytes = ws.data_ptr(), ws.numel()
    code = lib().spec_sample_verify(_ptr(target), _ptr(draft), _ptr(draft_uniforms.contiguous()),
                                    _ptr(uniforms.contiguous()), ctypes.byref(p), _ptr(out_draft_tokens),
                                    _ptr(out_tokens), _ptr(out_num_accepted))
    if code != SPEC_OK:
        raise SpecError(code, "spec_sample_verify")
    return out_draft_tokens, out_tokens, out_num_accepted


def spec_verify_ragged(target, draft, draft_tokens, uniforms, draft_lengths, *, temperature=1.0, top_k=0,
                       top_p=1.0, greedy=False, out_tokens=None, out_num_accepted=None, status=None, ws=None,
                       stream=None):
    """spec_verify with a draft length per sequence: target [B, K+1, V], draft
    [B, K, V] CUDA logits, draft_tokens [B, K], uniforms [B, K+1] (column K_b: the
    final draw), draft_lengths: host ints K_b in [1, K] (list, numpy or CPU tensor).
    Returns (out_tokens [B, K+1], out_num_accepted [B])."""
    import numpy as np
    a = _verify_args(target, draft, draft_tokens, uniforms, None, out_tokens, out_num_accepted, stream)
    lens = np.ascontiguousarray(np.asarray(draft_lengths.cpu() if torch.is_tensor(draft_lengths) else draft_lengths,
                                           dtype=np.int32))
    if lens.shape != (a.B,):
        raise ValueError("draft_lengths must hold one length per sequence")
    p = make_params(a.B, a.K, a.V, a.dt, a.tstr, a.dstr, temperature, top_k, top_p, greedy,
                    _stream_handle(stream), status)
    if ws is None:
        ws = workspace(int(lib().spec_verify_ragged_workspace_size(ctypes.byref(p))), target.device)
    p.workspace, p.workspace_bytes = ws.data_ptr(), ws.numel()
    code = lib().spec_verify_ragged(_ptr(target), _ptr(draft), _ptr(a.tok), _ptr(a.u),
                                    lens.ctypes.data_as(ctypes.c_void_p), ctypes.byref(p), _ptr(a.out_tokens),
                                    _ptr(a.out_n))
    if code != SPEC_OK:
        raise SpecError(code, "spec_verify_ragged")
    return a.out_tokens, a.out_n
