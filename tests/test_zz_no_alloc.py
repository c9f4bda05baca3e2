"""sv_verify_greedy_noalloc: greedy verify for callers that cannot allocate
device memory (the library's own static scratch replaces the workspace).

Called through the C ABI and compared with sv_verify_greedy (workspace
entry point) on the same inputs, on two calls in a row: the greedy tolerance
is bit-exact.  This file is collected last so that a stop-at-first-failure run
has already run every other test; it also passes alone in a fresh process.
"""

import numpy as np
import pytest
import torch

import workloads

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
def test_noalloc_matches_workspace_entry_point_on_two_calls(sv, B, V, dtype):
    w = workloads.WORKLOADS["greedy_b512_g4_v128256_bf16"].with_(V=V)
    inp = workloads.make_inputs(w, seed=B + V, device="cuda:0", B=B)
    logits = inp["logits"].to(dtype).contiguous()
    draft = inp["draft"]
    stream = torch.cuda.current_stream()
    ref = sv.verify_greedy(logits, draft)
    for _ in range(2):
        got = _noalloc(sv, logits, draft, stream)
        torch.cuda.synchronize()
        for a, b in zip(got, ref):
            assert torch.equal(a, b)


def test_noalloc_rejects_problems_beyond_its_scratch(sv):
    B, G, V = 4096, 8, 152064
    assert sv.sv_workspace_bytes(B, G, V, 0) > (8 << 20)
    rc = sv.sv_verify_greedy_noalloc(B, G, V, 1 << 20, sv.SV_DTYPE_BF16, 1 << 21, 1 << 22, 1 << 23, None, None)
    assert rc == sv.SV_ERR_WORKSPACE
