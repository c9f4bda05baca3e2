"""GB300-native verify/sample step of speculative decoding.

The computation lives in libspecverify.so (CUDA, sm_103a; C ABI in
include/specverify.h).  This package is its thin Python binding.
"""

from ._binding import (  # noqa: F401
    SV_DTYPE_BF16,
    SV_DTYPE_F16,
    SV_DTYPE_F32,
    SV_ERR_CUDA,
    SV_ERR_INVALID_ARG,
    SV_ERR_TIMEOUT,
    SV_ERR_UNSUPPORTED,
    SV_ERR_WORKSPACE,
    SV_NOALLOC_SCRATCH_BYTES,
    SV_OK,
    SV_SEQ_BAD_ROW,
    SV_SEQ_DRAFT_OUT_OF_RANGE,
    SV_SEQ_Q_NOT_POSITIVE,
    SV_SEQ_RESIDUAL_ZERO,
    SvError,
    alloc_qlogits_workspace,
    alloc_workspace,
    load_library,
    sv_last_kernels,
    sv_set_timing_events,
    sv_truncate_emitted,
    sv_status_string,
    sv_verify_greedy,
    sv_verify_greedy_noalloc,
    sv_verify_greedy_ragged,
    sv_qlogits_workspace_bytes,
    sv_verify_sample,
    sv_verify_sample_qlogits,
    sv_verify_sample_ragged,
    sv_workspace_bytes,
    truncate_emitted,
    verify_greedy,
    verify_sample,
    verify_sample_qlogits,
)
