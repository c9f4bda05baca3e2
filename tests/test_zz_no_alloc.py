"""sv_verify_greedy_noalloc: greedy verify for callers that cannot allocate
device memory (the library's own static scratch replaces the workspace).

Called through the C ABI, on two calls in a row, and compared bit-exactly
(the greedy tolerance) with the CPU oracle and with sv_verify_greedy (the
workspace entry point) on the same inputs.  This file is collected last so
that a stop-at-first-failure run has already run every other test; it also
passes alone in a fresh process.
"""

import numpy as np
import pytest
import torch

import workloads
import _parity as P

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def sv():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from speculative_decoding_verification_46_gb300 import build

    build.build_library()
    import speculative_decoding_verification_46_gb300 as pkg

    pkg.load_library()
    return pkg


def _noalloc(sv, logits, draft, stream):
    B, G1, V = logits.shape
    tok = torch.full((B, G1), -7, dtype=torch.int32, device=logits.device)
    n = torch.full((B,), -7, dtype=torch.int32, device=logits.device)
    st = torch.full((B,), -7, dtype=torch.int32, device=logits.device)
    dt = {torch.float32: sv.SV_DTYPE_F32, torch.bfloat16: sv.SV_DTYPE_BF16, torch.float16: sv.SV_DTYPE_F16}
    rc = sv.sv_verify_greedy_noalloc(B, G1 - 1, V, logits.data_ptr(), dt[logits.dtype], draft.data_ptr(),
                                     tok.data_ptr(), n.data_ptr(), st.data_ptr(), stream.cuda_stream)
    assert rc == sv.SV_OK, sv.sv_status_string(rc)
    return tok, n, st


@pytest.mark.parametrize("B,V,dtype", [(512, 128256, torch.bfloat16), (37, 1001, torch.float32),
                                       (9, 40003, torch.float16)])
def test_noalloc_matches_oracle_and_workspace_entry_point_on_two_calls(sv, B, V, dtype):
    w = workloads.WORKLOADS["greedy_b512_g4_v128256_bf16"].with_(V=V)
    inp = workloads.make_inputs(w, seed=B + V, device="cuda:0", B=B)
    logits = inp["logits"].to(dtype).contiguous()
    draft = inp["draft"]
    assert sv.sv_workspace_bytes(B, w.gamma, V, 0) <= sv.SV_NOALLOC_SCRATCH_BYTES
    stream = torch.cuda.current_stream()
    ref = P.oracle_greedy(dict(logits=logits, draft=draft))
    ws_out = sv.verify_greedy(logits, draft)
    for _ in range(2):
        got = _noalloc(sv, logits, draft, stream)
        torch.cuda.synchronize()
        P.compare_greedy(got, ref, V)
        assert np.array_equal(P.to_np(got[2]), ref["status"])
        for a, b in zip(got, ws_out):
            assert torch.equal(a, b)


def test_noalloc_rejects_problems_beyond_its_scratch(sv):
    """A problem whose workspace exceeds the scratch is refused before any
    pointer is used: every pointer here is NULL, so nothing can be read or
    written whatever the order of the checks."""
    B, G, V = 4096, 8, 152064
    assert sv.sv_workspace_bytes(B, G, V, 0) > sv.SV_NOALLOC_SCRATCH_BYTES
    rc = sv.sv_verify_greedy_noalloc(B, G, V, None, sv.SV_DTYPE_BF16, None, None, None, None, None)
    assert rc == sv.SV_ERR_WORKSPACE, sv.sv_status_string(rc)
