"""GB300-native speculative-sampling verification.

The computation lives in libspecverify.so (CUDA kernels for sm_103a behind the
C ABI in include/spec_verify.h).  This package holds the in-tree build, a thin
binding with the C entry points' names, and (decode.py) the decode-round driver
around the verification step with the latency-vs-K model.
"""
from .binding import (  # noqa: F401
    SPEC_BF16, SPEC_F32, SpecError, spec_accept_histogram, spec_launch_count, spec_read_row_stats,
    spec_sample_draft, spec_sample_draft_workspace_size, spec_sample_verify, spec_status_string, spec_verify,
    spec_verify_workspace_size, spec_verify_noalloc, spec_verify_ragged, workspace,
)
from . import decode  # noqa: F401
from ._build import build  # noqa: F401
