"""The C ABI library builds, loads and exports every entry point its header declares.

No GPU is needed: only host-side entry points are called (size queries, argument
validation that returns before any CUDA call, status strings).
"""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "spec_verify.h")


@pytest.fixture(scope="module")
def L():
    from speculative_sampling_verification_spec_gb300 import _build, binding
    _build.build()
    return binding.lib()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(spec_[a-z_]+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for must in ("spec_verify", "spec_sample_draft", "spec_verify_workspace_size",
                 "spec_status_string"):
        assert must in names


def test_library_exports_every_declared_symbol(L):
    for name in declared_functions():
        assert hasattr(L, name), name


def test_binding_names_match_header():
    from speculative_sampling_verification_spec_gb300 import binding
    assert set(binding.EXPORTED) == set(declared_functions())


def test_status_strings(L):
    from speculative_sampling_verification_spec_gb300 import binding
    for code in range(7):
        assert binding.spec_status_string(code)
    assert binding.spec_status_string(0) == "ok"


def test_workspace_size_is_host_only_and_grows_with_rows(L):
    from speculative_sampling_verification_spec_gb300 import binding as b
    s1 = b.spec_verify_workspace_size(64, 4, 128256, b.SPEC_BF16)
    s2 = b.spec_verify_workspace_size(128, 4, 128256, b.SPEC_BF16)
    g = b.spec_verify_workspace_size(64, 4, 128256, b.SPEC_BF16, greedy=True)
    assert 0 < s1 < s2 and 0 < g < s1
    assert b.spec_sample_draft_workspace_size(64, 4, 128256, b.SPEC_BF16) > 0
    # invalid parameters give 0
    assert b.spec_verify_workspace_size(-1, 4, 10, b.SPEC_BF16) == 0
    assert b.spec_verify_workspace_size(1, 0, 10, b.SPEC_BF16) == 0
    assert b.spec_verify_workspace_size(1, 1, 10, 7) == 0


def test_invalid_arguments_are_rejected_on_the_host(L):
    from speculative_sampling_verification_spec_gb300 import binding as b
    P = b.SpecParams
    good = dict(B=2, K=2, V=16, dtype=b.SPEC_F32, target_seq_stride=48, target_row_stride=16,
                draft_seq_stride=32, draft_row_stride=16, temperature=1.0, top_k=0, top_p=1.0,
                greedy=0, stream=None, status=None, workspace=None, workspace_bytes=0)

    def call(**over):
        kw = dict(good, **over)
        p = P(*[kw[f] for f, _ in P._fields_])
        fake = ctypes.c_void_p(0x1000)  # never dereferenced: validation fails first
        return L.spec_verify(fake, fake, fake, fake, ctypes.byref(p), fake, fake)

    assert call(temperature=0.0) == 1
    assert call(temperature=float("inf")) == 1
    assert call(top_p=0.0) == 1
    assert call(top_p=1.5) == 1
    assert call(top_k=-1) == 1
    assert call(B=-1) == 1
    assert call(K=0) == 1
    assert call(dtype=5) == 1
    assert call(target_row_stride=-1) == 1
    assert call(workspace=None) == 1              # missing workspace
    assert call(workspace=0x1001, workspace_bytes=1 << 30) == 1   # misaligned workspace
    assert call(B=0) == 0                         # nothing to do
    # greedy ignores temperature / top-p
    assert call(greedy=1, temperature=0.0, top_p=3.0) == 1       # still no workspace
    p = P(*[dict(good)[f] for f, _ in P._fields_])
    assert L.spec_verify(None, None, None, None, ctypes.byref(p), None, None) == 1


def test_accept_histogram_rejects_bad_arguments_on_the_host(L):
    fake = ctypes.c_void_p(0x1000)  # never dereferenced: validation fails first
    assert L.spec_accept_histogram(fake, -1, 4, fake, None) == 1
    assert L.spec_accept_histogram(fake, 3, 0, fake, None) == 1
    assert L.spec_accept_histogram(fake, 3, 8193, fake, None) == 1
    assert L.spec_accept_histogram(None, 3, 4, fake, None) == 1
    assert L.spec_accept_histogram(fake, 3, 4, None, None) == 1
    assert L.spec_accept_histogram(None, 0, 4, None, None) == 0   # nothing to count


def test_sample_verify_requires_k1_sampling_on_the_host(L):
    from speculative_sampling_verification_spec_gb300 import binding as b
    P = b.SpecParams
    good = dict(B=2, K=1, V=16, dtype=b.SPEC_F32, target_seq_stride=32, target_row_stride=16,
                draft_seq_stride=16, draft_row_stride=16, temperature=1.0, top_k=0, top_p=1.0,
                greedy=0, stream=None, status=None, workspace=None, workspace_bytes=0)

    def call(ptrs=None, **over):
        kw = dict(good, **over)
        p = P(*[kw[f] for f, _ in P._fields_])
        fake = ctypes.c_void_p(0x1000)  # never dereferenced: validation fails first
        args = ptrs if ptrs is not None else [fake] * 7
        return L.spec_sample_verify(args[0], args[1], args[2], args[3], ctypes.byref(p), args[4], args[5],
                                    args[6])

    assert call(K=2) == 1                    # K = 1 only
    assert call(greedy=1) == 1               # sampling only
    assert call(temperature=0.0) == 1
    assert call() == 1                       # no workspace
    fake = ctypes.c_void_p(0x1000)
    assert call(ptrs=[fake, fake, None, fake, fake, fake, fake]) == 1   # draft uniforms missing
    assert call(ptrs=[fake, fake, fake, fake, None, fake, fake]) == 1   # draft-token output missing
    assert call(B=0) == 0
    assert L.spec_sample_verify(None, None, None, None, None, None, None, None) == 1


def test_ragged_lengths_are_checked_on_the_host(L):
    from speculative_sampling_verification_spec_gb300 import binding as b
    P = b.SpecParams
    good = dict(B=3, K=4, V=16, dtype=b.SPEC_F32, target_seq_stride=80, target_row_stride=16,
                draft_seq_stride=64, draft_row_stride=16, temperature=1.0, top_k=0, top_p=1.0,
                greedy=0, stream=None, status=None, workspace=0x100000, workspace_bytes=1 << 40)
    p = P(*[good[f] for f, _ in P._fields_])
    fake = ctypes.c_void_p(0x1000)  # never dereferenced: validation fails first

    def call(lens):
        arr = (ctypes.c_int32 * 3)(*lens) if lens is not None else None
        return L.spec_verify_ragged(fake, fake, fake, fake, arr, ctypes.byref(p), fake, fake)

    assert call([1, 0, 4]) == 1      # a length below 1
    assert call([1, 5, 4]) == 1      # a length above K
    assert call(None) == 1           # no lengths
    # the ragged workspace holds the padded call's plus the rows' index
    pv = P(*[dict(good, workspace=None, workspace_bytes=0)[f] for f, _ in P._fields_])
    assert L.spec_verify_ragged_workspace_size(ctypes.byref(pv)) > L.spec_verify_workspace_size(ctypes.byref(pv))
