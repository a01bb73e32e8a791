"""spec_verify_noalloc: the variant for callers that may not allocate device memory.

Some callers cannot give the library a workspace: a plugin inside a serving
framework that has reserved the GPU's memory for its own pool and only hands
the plugin the tensors it works on, or a decode loop that must not allocate
between tokens.  spec_verify_noalloc serves them from a fixed scratch array
compiled into the library.  This test calls it through the C ABI (ctypes, no
binding logic) and checks that it returns exactly what spec_verify returns on
the same inputs, on two calls in a row (the array keeps the first call's
contents, which must not disturb the second).  The file is named to be
collected last.
"""
import ctypes

import numpy as np
import pytest
import torch

import workloads
from _gpu import params_of, to_dev

pytestmark = pytest.mark.gpu


def _c_call(L, b, tgt, drf, tok, u, prm, out_t, out_n):
    p = b.make_params(tok.shape[0], tok.shape[1], tgt.shape[-1], b._dtype_code(tgt),
                      (tgt.stride(0), tgt.stride(1)), (drf.stride(0), drf.stride(1)),
                      prm["temperature"], prm["top_k"], prm["top_p"], prm["greedy"],
                      ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    vp = lambda t: ctypes.c_void_p(t.data_ptr())  # noqa: E731
    return L.spec_verify_noalloc(vp(tgt), vp(drf), vp(tok), vp(u), ctypes.byref(p), vp(out_t), vp(out_n))


@pytest.mark.parametrize("name,kw", [("c5", dict(B=4)), ("c3", dict(B=6, V=50001)), ("c2", {}),
                                     ("c4", dict(B=16))])
def test_noalloc_matches_spec_verify_twice(name, kw):
    import speculative_sampling_verification_spec_gb300 as sv
    b = sv.binding
    L = b.lib()
    w = workloads.make(name, **kw)
    prm = params_of(w)
    tgt, drf = to_dev(w["target"]), to_dev(w["draft"])
    ud, uv = to_dev(w["u_draft"]), to_dev(w["u_verify"])
    tok = sv.spec_sample_draft(drf, None if w["greedy"] else ud, **prm)
    ref_t, ref_n = sv.spec_verify(tgt, drf, tok, uv, **prm)
    torch.cuda.synchronize()
    for _ in range(2):
        out_t = torch.full_like(ref_t, -9)
        out_n = torch.full_like(ref_n, -9)
        code = _c_call(L, b, tgt, drf, tok, uv, prm, out_t, out_n)
        assert code == 0, b.spec_status_string(code)
        torch.cuda.synchronize()
        assert torch.equal(out_t, ref_t) and torch.equal(out_n, ref_n)


def test_noalloc_across_changing_layouts():
    """Calls in a row that change B, K, V and the mode (greedy, top-k, unfiltered,
    top-p on unaligned rows) share the one array: each call must still return
    spec_verify's outputs, so no call may leave a stale counter behind."""
    import speculative_sampling_verification_spec_gb300 as sv
    b = sv.binding
    L = b.lib()
    order = [("c4", dict(B=16)), ("c5", dict(B=4)), ("c2", {}), ("c3", dict(B=6, V=50001)), ("c4", dict(B=16)),
             ("c5", dict(B=2, V=70003))]
    for name, kw in order:
        w = workloads.make(name, **kw)
        prm = params_of(w)
        tgt, drf = to_dev(w["target"]), to_dev(w["draft"])
        ud, uv = to_dev(w["u_draft"]), to_dev(w["u_verify"])
        tok = sv.spec_sample_draft(drf, None if w["greedy"] else ud, **prm)
        ref_t, ref_n = sv.spec_verify(tgt, drf, tok, uv, **prm)
        out_t = torch.full_like(ref_t, -9)
        out_n = torch.full_like(ref_n, -9)
        code = _c_call(L, b, tgt, drf, tok, uv, prm, out_t, out_n)
        assert code == 0, b.spec_status_string(code)
        torch.cuda.synchronize()
        assert torch.equal(out_t, ref_t) and torch.equal(out_n, ref_n), name


def test_noalloc_python_wrapper_checks_its_inputs():
    """The Python wrapper converts int64 draft tokens to int32 (the C entry point
    reads int32) and rejects logits that are not contiguous along V and uniforms
    that are not float64, as spec_verify's wrapper does."""
    import speculative_sampling_verification_spec_gb300 as sv
    w = workloads.make("c5", B=3, V=30000)
    prm = params_of(w)
    tgt, drf = to_dev(w["target"]), to_dev(w["draft"])
    uv = to_dev(w["u_verify"])
    tok = sv.spec_sample_draft(drf, to_dev(w["u_draft"]), **prm)
    ref_t, ref_n = sv.spec_verify(tgt, drf, tok, uv, **prm)
    got_t, got_n = sv.spec_verify_noalloc(tgt, drf, tok.to(torch.int64), uv, **prm)
    torch.cuda.synchronize()
    assert torch.equal(got_t, ref_t) and torch.equal(got_n, ref_n)
    strided = torch.zeros(3, 9, 2 * 30000, dtype=tgt.dtype, device=tgt.device)[:, :, ::2]
    strided.copy_(tgt)
    with pytest.raises(ValueError):
        sv.spec_verify_noalloc(strided, drf, tok, uv, **prm)
    with pytest.raises(TypeError):
        sv.spec_verify_noalloc(tgt, drf, tok, uv.float(), **prm)


def test_noalloc_rejects_requests_beyond_its_scratch():
    import speculative_sampling_verification_spec_gb300 as sv
    b = sv.binding
    L = b.lib()
    B, K, V = 4096, 8, 1000   # 4096 * 17 rows need far more than the fixed array
    assert sv.spec_verify_workspace_size(B, K, V, b.SPEC_F32) > b.SPEC_NOALLOC_SCRATCH_BYTES
    p = b.make_params(B, K, V, b.SPEC_F32, ((K + 1) * V, V), (K * V, V))
    fake = ctypes.c_void_p(0x1000)   # never dereferenced: the size check comes first
    assert L.spec_verify_noalloc(fake, fake, fake, fake, ctypes.byref(p), fake, fake) == 7
    assert "scratch" in b.spec_status_string(7)
