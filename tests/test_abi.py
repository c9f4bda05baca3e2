"""The C ABI library builds, loads and exports every declared symbol; host-side
argument validation returns the documented status codes.  No kernel is
launched here (these run without a GPU): every call below fails validation
before any CUDA call, or is the empty B = 0 call."""

import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def sv():
    from speculative_decoding_verification_46_gb300 import build

    build.build_library()
    import speculative_decoding_verification_46_gb300 as pkg

    pkg.load_library()
    return pkg


def _declared_functions():
    text = open(os.path.join(ROOT, "include", "specverify.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(sv_\w+)\s*\(", text)))


def test_exports_every_declared_symbol(sv):
    lib = ctypes.CDLL(sv.load_library()._name)
    names = _declared_functions()
    assert set(names) == {"sv_workspace_bytes", "sv_verify_sample", "sv_verify_greedy", "sv_status_string",
                          "sv_set_timing_events", "sv_verify_greedy_noalloc", "sv_last_kernels",
                          "sv_verify_sample_ragged", "sv_verify_greedy_ragged", "sv_truncate_emitted",
                          "sv_qlogits_workspace_bytes", "sv_verify_sample_qlogits", "sv_shard_workspace_bytes",
                          "sv_shard_row_stats", "sv_shard_scan", "sv_shard_draw_sums", "sv_shard_draw_pick",
                          "sv_shard_topk_candidates", "sv_shard_topk_finish", "sv_pointer_device_readable"}
    for n in names:
        assert hasattr(lib, n), n


def test_status_strings(sv):
    for code in range(6):
        assert sv.sv_status_string(code).startswith("SV_")
    assert "unknown" in sv.sv_status_string(99)


def test_workspace_bytes(sv):
    a = sv.sv_workspace_bytes(64, 4, 128256, 0)
    b = sv.sv_workspace_bytes(128, 4, 128256, 0)
    assert 0 < a < b and a % 256 == 0
    assert sv.sv_workspace_bytes(256, 8, 152064, 50) > sv.sv_workspace_bytes(256, 8, 152064, 0)
    for bad in [(-1, 4, 10, 0), (4, -1, 10, 0), (4, 65, 10, 0), (4, 4, 0, 0), (4, 4, (1 << 24) + 1, 0),
                (4, 4, 10, -1), (4, 4, 10, 1025)]:
        assert sv.sv_workspace_bytes(*bad) == 0, bad


# fake, never dereferenced device addresses (validation fails before any use)
A = 1 << 20


def _sample(sv, **kw):
    args = dict(B=4, gamma=3, V=100, logits=A, logits_dtype=sv.SV_DTYPE_BF16, q=A + 4096, draft_tokens=A + 8192,
                uniforms=A + 12288, temperature=1.0, top_k=0, top_p=1.0, out_tokens=A + 16384,
                out_num_accepted=A + 20480, out_accept_prob=None, out_status=None, workspace=A + 65536,
                workspace_bytes=1 << 30, stream=None)
    args.update(kw)
    return sv.sv_verify_sample(*args.values())


def _greedy(sv, **kw):
    args = dict(B=4, gamma=3, V=100, logits=A, logits_dtype=sv.SV_DTYPE_BF16, draft_tokens=A + 8192,
                out_tokens=A + 16384, out_num_accepted=A + 20480, out_status=None, workspace=A + 65536,
                workspace_bytes=1 << 30, stream=None)
    args.update(kw)
    return sv.sv_verify_greedy(*args.values())


@pytest.mark.parametrize("kw", [dict(B=-1), dict(gamma=-1), dict(gamma=65), dict(V=0), dict(V=(1 << 24) + 1),
                                dict(logits_dtype=7), dict(temperature=0.0), dict(temperature=-1.0),
                                dict(temperature=float("inf")), dict(temperature=float("nan")), dict(top_k=-1),
                                dict(top_k=1025), dict(top_p=0.0), dict(top_p=1.5), dict(top_p=float("nan")),
                                dict(logits=None), dict(draft_tokens=None), dict(uniforms=None),
                                dict(out_tokens=None), dict(out_num_accepted=None), dict(logits=A + 2),
                                dict(q=A + 4100)])
def test_sample_rejects_invalid_arguments(sv, kw):
    assert _sample(sv, **kw) == sv.SV_ERR_INVALID_ARG


def test_sample_workspace_and_unsupported(sv):
    assert _sample(sv, workspace=None) == sv.SV_ERR_WORKSPACE
    assert _sample(sv, workspace_bytes=16) == sv.SV_ERR_WORKSPACE
    assert _sample(sv, workspace=A + 3) == sv.SV_ERR_WORKSPACE
    # top-p without top-k over a vocabulary larger than the largest list: the
    # per-row threshold path, which validates its workspace before any launch
    assert _sample(sv, V=5000, top_k=0, top_p=0.9, workspace_bytes=16) == sv.SV_ERR_WORKSPACE
    # gamma = 0 needs neither q nor drafts; B = 0 is an empty call
    assert _sample(sv, B=0) == sv.SV_OK
    assert _sample(sv, gamma=0, q=None, draft_tokens=None, workspace_bytes=16) == sv.SV_ERR_WORKSPACE
    # q = NULL with gamma > 0 is valid (deterministic drafts): it reaches the workspace check
    assert _sample(sv, q=None, workspace_bytes=16) == sv.SV_ERR_WORKSPACE


@pytest.mark.parametrize("kw", [dict(B=-1), dict(gamma=-1), dict(V=0), dict(logits_dtype=3), dict(logits=None),
                                dict(draft_tokens=None), dict(out_tokens=None), dict(out_num_accepted=None),
                                dict(logits=A + 8)])
def test_greedy_rejects_invalid_arguments(sv, kw):
    assert _greedy(sv, **kw) == sv.SV_ERR_INVALID_ARG


def test_greedy_workspace(sv):
    assert _greedy(sv, workspace_bytes=8) == sv.SV_ERR_WORKSPACE
    assert _greedy(sv, B=0) == sv.SV_OK


def test_torch_wrappers_refuse_cpu_tensors(sv):
    import torch

    L = torch.zeros(2, 3, 10, dtype=torch.bfloat16)
    d = torch.zeros(2, 2, dtype=torch.int32)
    with pytest.raises(ValueError):
        sv.verify_greedy(L, d)
    with pytest.raises(ValueError):
        sv.verify_sample(L, torch.zeros(2, 2, 10), d, torch.zeros(2, 3), 1.0)


def test_timing_hook_validation(sv):
    lib = sv.load_library()
    assert lib.sv_set_timing_events(None, 0) == sv.SV_OK
    assert lib.sv_set_timing_events(None, 3) == sv.SV_ERR_INVALID_ARG
    assert lib.sv_set_timing_events(None, 2) == sv.SV_ERR_INVALID_ARG


def test_last_kernels_empty_without_launch(sv):
    lib = sv.load_library()
    assert sv.sv_last_kernels() == []
    # an argument error and the empty batch launch nothing
    assert lib.sv_verify_greedy(1, 2, 0, None, 0, None, None, None, None, None, 0, None) == sv.SV_ERR_INVALID_ARG
    assert sv.sv_last_kernels() == []
    assert lib.sv_verify_greedy(0, 2, 10, None, 0, None, None, None, None, None, 0, None) == sv.SV_OK
    assert sv.sv_last_kernels() == []


def test_ragged_and_truncate_validation(sv):
    lib = sv.load_library()
    # ragged calls need gamma_b (the empty batch needs nothing)
    assert sv.sv_verify_sample_ragged(4, 3, 100, A, sv.SV_DTYPE_BF16, A + 4096, A + 8192, A + 12288, None, 1.0, 0,
                                      1.0, A + 16384, A + 20480, None, None, A + 65536, 1 << 30,
                                      None) == sv.SV_ERR_INVALID_ARG
    assert sv.sv_verify_greedy_ragged(4, 3, 100, A, sv.SV_DTYPE_BF16, A + 8192, None, A + 16384, A + 20480, None,
                                      A + 65536, 1 << 30, None) == sv.SV_ERR_INVALID_ARG
    assert sv.sv_verify_greedy_ragged(0, 3, 100, None, sv.SV_DTYPE_BF16, None, None, None, None, None, None, 0,
                                      None) == sv.SV_OK
    # a ragged call with gamma_b given goes on to the usual checks
    assert sv.sv_verify_sample_ragged(4, 3, 100, A, sv.SV_DTYPE_BF16, A + 4096, A + 8192, A + 12288, A + 32768, 1.0,
                                      0, 1.0, A + 16384, A + 20480, None, None, A + 65536, 16,
                                      None) == sv.SV_ERR_WORKSPACE
    T = lib.sv_truncate_emitted
    assert T(-1, 3, A, A, None, 0, None, A, None) == sv.SV_ERR_INVALID_ARG
    assert T(4, 65, A, A, None, 0, None, A, None) == sv.SV_ERR_INVALID_ARG
    assert T(4, 3, A, A, None, 65, None, A, None) == sv.SV_ERR_INVALID_ARG
    assert T(4, 3, A, A, None, 2, None, A, None) == sv.SV_ERR_INVALID_ARG      # n_stop > 0 needs the ids
    assert T(4, 3, None, A, None, 0, None, A, None) == sv.SV_ERR_INVALID_ARG
    assert T(0, 3, None, None, None, 0, None, None, None) == sv.SV_OK


def test_qlogits_validation(sv):
    """Draft logits: the workspace adds float32 q after the usual layout;
    argument errors launch nothing (every call below fails validation)."""
    B, G, V = 4, 3, 100
    base = sv.sv_workspace_bytes(B, G, V, 0)
    ws = sv.sv_qlogits_workspace_bytes(B, G, V)
    assert ws >= base + 4 * B * G * V and ws % 256 == 0
    assert sv.sv_qlogits_workspace_bytes(-1, G, V) == 0 and sv.sv_qlogits_workspace_bytes(B, 65, V) == 0

    def call(**kw):
        a = dict(B=B, gamma=G, V=V, logits=A, ldt=sv.SV_DTYPE_BF16, ql=A + 8192, qdt=sv.SV_DTYPE_BF16,
                 d=A + 16384, u=A + 20480, T=1.0, k=0, p=1.0, tok=A + 24576, n=A + 28672, ws=A + 65536,
                 wsb=ws)
        a.update(kw)
        return sv.sv_verify_sample_qlogits(a["B"], a["gamma"], a["V"], a["logits"], a["ldt"], a["ql"], a["qdt"],
                                           a["d"], a["u"], a["T"], a["k"], a["p"], a["tok"], a["n"], None, None,
                                           a["ws"], a["wsb"], None)
    assert call(k=2000) == sv.SV_ERR_INVALID_ARG             # top_k above SV_MAX_TOP_K
    assert call(V=2000, p=0.9) == sv.SV_ERR_UNSUPPORTED       # q from draft logits: top-p alone over > SV_MAX_TOP_K
    assert call(k=10, wsb=sv.sv_qlogits_workspace_bytes(B, G, V, 10) - 256) == sv.SV_ERR_WORKSPACE
    assert call(qdt=7) == sv.SV_ERR_INVALID_ARG
    assert call(T=0.0) == sv.SV_ERR_INVALID_ARG
    assert call(ql=None) == sv.SV_ERR_INVALID_ARG
    assert call(ql=A + 8194) == sv.SV_ERR_INVALID_ARG         # not 16-byte aligned
    assert call(wsb=ws - 256) == sv.SV_ERR_WORKSPACE
    assert call(B=0, logits=None, ql=None) == sv.SV_OK
    assert sv.sv_last_kernels() == []


def test_noalloc_scratch_size_matches_header(sv):
    """The binding's SV_NOALLOC_SCRATCH_BYTES is the header's value."""
    text = open(os.path.join(ROOT, "include", "specverify.h")).read()
    m = re.search(r"#define\s+SV_NOALLOC_SCRATCH_BYTES\s+\((\d+)u\s*<<\s*(\d+)\)", text)
    assert m, "SV_NOALLOC_SCRATCH_BYTES not found in the header"
    assert sv.SV_NOALLOC_SCRATCH_BYTES == int(m.group(1)) << int(m.group(2))


def test_shard_entry_points_validate_before_launch(sv):
    """Invalid shard arguments are refused on the host (no device needed):
    shard counts and ranks, ranges outside the vocabulary, dtypes, missing
    pointers, workspaces too small."""
    bf = sv.SV_DTYPE_BF16
    ok = sv.SV_ERR_INVALID_ARG
    # row stats: v0 + V beyond Vg, negative v0, V = 0, bad dtype, bad temperature, NULL output
    assert sv.sv_shard_row_stats(4, 4, 100, 950, 1000, A, bf, A, A, 1.0, 0, A, None) == ok
    assert sv.sv_shard_row_stats(4, 4, 100, -1, 1000, A, bf, A, A, 1.0, 0, A, None) == ok
    assert sv.sv_shard_row_stats(4, 4, 0, 0, 1000, A, bf, A, A, 1.0, 0, A, None) == ok
    assert sv.sv_shard_row_stats(4, 4, 100, 0, 1000, A, 7, A, A, 1.0, 0, A, None) == ok
    assert sv.sv_shard_row_stats(4, 4, 100, 0, 1000, A, bf, A, A, 0.0, 0, A, None) == ok
    assert sv.sv_shard_row_stats(4, 4, 100, 0, 1000, A, bf, A, A, 1.0, 0, None, None) == ok
    assert sv.sv_shard_row_stats(4, 4, 100, 0, 1000, A + 4, bf, A, A, 1.0, 0, A, None) == ok   # misaligned
    assert sv.sv_shard_row_stats(0, 4, 100, 0, 1000, None, bf, None, None, 1.0, 0, None, None) == sv.SV_OK
    # scan: shard counts
    for S in (0, sv.SV_MAX_SHARDS + 1):
        assert sv.sv_shard_scan(S, 4, 4, 100, 1000, A, A, A, 1.0, 0, A, A, A, A, A, 1 << 20, None) == ok
    ws_need = sv.sv_shard_workspace_bytes(4, 4, 100)
    assert ws_need > 0
    assert sv.sv_shard_scan(2, 4, 4, 100, 1000, A, A, A, 1.0, 0, A, A, A, A, A, ws_need - 1, None) == \
        sv.SV_ERR_WORKSPACE
    assert sv.sv_shard_scan(2, 4, 4, 100, 1000, A, A, None, 1.0, 0, A, A, A, A, A, ws_need, None) == ok
    # pick: rank outside [0, nshard)
    for rank in (-1, 2):
        assert sv.sv_shard_draw_pick(2, rank, 4, 4, 100, 0, 1000, A, bf, A, A, A, 1.0, A, A, A, A, ws_need,
                                     None) == ok
    # draw sums: NULL totals, workspace too small
    assert sv.sv_shard_draw_sums(4, 4, 100, 0, 1000, A, bf, A, A, 1.0, None, A, ws_need, None) == ok
    assert sv.sv_shard_draw_sums(4, 4, 100, 0, 1000, A, bf, A, A, 1.0, A, A, ws_need - 1, None) == \
        sv.SV_ERR_WORKSPACE


def test_shard_topk_entry_points_validate_before_launch(sv):
    bf = sv.SV_DTYPE_BF16
    ws = sv.sv_workspace_bytes(4, 4, 1024, 50)
    # top_k outside 1..1024, a range not of whole 16-byte vectors, too many candidates to merge
    assert sv.sv_shard_topk_candidates(4, 4, 1024, 0, 4096, A, bf, A, A, 1.0, 0, A, A, ws, None) == \
        sv.SV_ERR_INVALID_ARG
    assert sv.sv_shard_topk_candidates(4, 4, 1020, 0, 4096, A, bf, A, A, 1.0, 50, A, A, ws, None) == \
        sv.SV_ERR_UNSUPPORTED
    assert sv.sv_shard_topk_candidates(4, 4, 1024, 0, 4096, A, bf, A, A, 1.0, 50, A, A, ws - 1, None) == \
        sv.SV_ERR_WORKSPACE
    assert sv.sv_shard_topk_finish(4, 4, 4, 4096, A, A, A, 1.0, 1024, 0.9, A, A, A, A, None) == \
        sv.SV_ERR_UNSUPPORTED
    assert sv.sv_shard_topk_finish(2, 4, 4, 4096, A, A, A, 1.0, 50, 0.0, A, A, A, A, None) == sv.SV_ERR_INVALID_ARG
    assert sv.sv_shard_topk_finish(2, 4, 4, 4096, A, A, None, 1.0, 50, 0.9, A, A, A, A, None) == \
        sv.SV_ERR_INVALID_ARG


def test_pointer_device_readable_on_host_memory(sv):
    """No device pointer on a machine without a usable GPU (or NULL / a
    pageable host address anywhere): 0, and no CUDA error is left behind."""
    import numpy as np

    buf = np.zeros(64, np.uint8)
    assert not sv.sv_pointer_device_readable(None)
    assert not sv.sv_pointer_device_readable(buf.ctypes.data)
