"""q supplied as the draft model's logits (sv_verify_sample_qlogits) on the GPU
against the oracle's verify_sample_qlogits (q_i = softmax(q_logits_i / T) in
float64), on both of its paths: fused into the streaming and final-draw
kernels (one dtype, 16-byte rows), or q formed by its own kernel first.
Acceptance probabilities within 1e-5 relative; tokens equal except at
boundary draws, where the oracle also flags a final draw within 1e-6
(absolute, probability units) of a CDF step, the reach of a float32 q."""

import numpy as np
import pytest
import torch

import _parity as P
from oracle import svref

pytestmark = pytest.mark.gpu

DEV = "cuda:0"
DTYPES = {"f32": torch.float32, "bf16": torch.bfloat16, "f16": torch.float16}


@pytest.fixture(scope="module")
def sv():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from speculative_decoding_verification_46_gb300 import build

    build.build_library()
    import speculative_decoding_verification_46_gb300 as pkg

    pkg.load_library()
    return pkg


@pytest.fixture(params=["auto", "grid", "cluster", "slices"])
def path(request, monkeypatch):
    if request.param != "auto":
        monkeypatch.setenv("SPECVERIFY_PATH", request.param)
    else:
        monkeypatch.delenv("SPECVERIFY_PATH", raising=False)
    return request.param


def _ql_case(seed, B, G, V, ldt, qdt, spread=1.5, noise=0.8):
    """Target logits, draft logits = target logits plus noise, drafts drawn
    from softmax(draft logits) with the Gumbel trick."""
    g = torch.Generator().manual_seed(seed)
    L = (torch.randn(B, G + 1, V, generator=g) * spread).to(ldt)
    Q = (L[:, :G].float() + noise * torch.randn(B, G, V, generator=g)).to(qdt)
    gum = -torch.log(-torch.log(torch.rand(B, G, V, generator=g).clamp_min(1e-12)))
    draft = (Q.float() + gum).argmax(-1).to(torch.int32)
    u = torch.rand(B, G + 1, generator=g)
    return dict(logits=L.contiguous(), q_logits=Q.contiguous(), draft=draft.contiguous(), uniforms=u)


def _gpu(inp):
    return {k: (v.to(DEV) if v is not None else None) for k, v in inp.items()}


def _oracle(inp, T, rows=None):
    L, Q, d, u = (P.to_np(inp[k]) for k in ("logits", "q_logits", "draft", "uniforms"))
    if rows is not None:
        L, Q, d, u = L[rows], Q[rows], d[rows], u[rows]
    return svref.verify_sample_qlogits(L, Q, d, u, T)


@pytest.mark.parametrize("ldt,qdt", [("bf16", "bf16"), ("f32", "f32"), ("f16", "bf16"), ("bf16", "f32")])
@pytest.mark.parametrize("V,G,B,T", [(257, 3, 16, 1.0), (1000, 4, 12, 0.7), (32000, 5, 3, 0.7),
                                     (128256, 4, 4, 1.0), (4096, 0, 5, 1.0), (4096, 1, 30, 1.3),
                                     (4096, 64, 6, 0.9)])
def test_qlogits_small(sv, path, ldt, qdt, V, G, B, T):
    inp = _ql_case(3000 + V + G, B, G, V, DTYPES[ldt], DTYPES[qdt])
    g = _gpu(inp)
    out = sv.verify_sample_qlogits(g["logits"], g["q_logits"], g["draft"], g["uniforms"], T)
    P.compare_sample(out, _oracle(inp, T), V)


@pytest.mark.parametrize("k,tp", [(0, 1.0), (50, 1.0), (50, 0.9)])
def test_qlogits_bad_draft_rows(sv, path, k, tp):
    """Draft rows with NaN, +inf or only -inf give q = 0 (the q(d) <= 0 bit
    where tested), untruncated and truncated."""
    B, G, V = 6, 3, 1000
    inp = _ql_case(77, B, G, V, torch.bfloat16, torch.bfloat16)
    Q = inp["q_logits"]
    Q[0, 0, 5] = float("nan")
    Q[1, 0, :] = -float("inf")
    Q[2, 0, 9] = float("inf")
    Q[3, 1, :] = -float("inf")            # tested only if position 0 is accepted
    g = _gpu(inp)
    out = sv.verify_sample_qlogits(g["logits"], g["q_logits"], g["draft"], g["uniforms"], 1.0, k, tp)
    L, Qn, d, u = (P.to_np(inp[x]) for x in ("logits", "q_logits", "draft", "uniforms"))
    ref = svref.verify_sample_qlogits(L, Qn, d, u, 1.0, k, tp)
    assert np.all(ref["status"][:3] & svref.SEQ_Q_NOT_POSITIVE)
    P.compare_sample(out, ref, V)


def test_qlogits_full_size(sv):
    """B = 64, gamma = 4, V = 128256 bfloat16 (the untruncated workload's
    shapes), in the launch configuration the bench uses; every sequence
    against the oracle."""
    B, G, V, T = 64, 4, 128256, 0.7
    inp = _ql_case(4242, B, G, V, torch.bfloat16, torch.bfloat16, spread=2.0)
    g = _gpu(inp)
    out = sv.verify_sample_qlogits(g["logits"], g["q_logits"], g["draft"], g["uniforms"], T)
    # one dtype on both sides and 16-byte rows: the fused path (q never written out)
    assert sv.sv_last_kernels() == ["stream_dense_kernel", "final_draw_kernel"]
    arrays = [P.to_np(inp[k]) for k in ("logits", "q_logits", "draft", "uniforms")]
    st = P.compare_sample(out, P.oracle_pool("qlogits", arrays, (T, 0, 1.0)), V)
    assert st["sequences"] == B


def test_qlogits_mixed_dtypes_materialise_q(sv):
    """Draft logits in another dtype than the target's: q is formed by its own
    kernel first (then the usual path)."""
    inp = _ql_case(8, 16, 4, 32000, torch.bfloat16, torch.float32)
    g = _gpu(inp)
    out = sv.verify_sample_qlogits(g["logits"], g["q_logits"], g["draft"], g["uniforms"], 0.9)
    assert sv.sv_last_kernels()[0] == "q_softmax_kernel"
    P.compare_sample(out, _oracle(inp, 0.9), 32000)


@pytest.mark.parametrize("tk_path", ["auto", "slices"])
@pytest.mark.parametrize("ldt", ["bf16", "f32", "bf16/f32"])
@pytest.mark.parametrize("V,G,B,k,tp,T", [(1000, 4, 12, 50, 1.0, 0.8), (1000, 4, 12, 50, 0.9, 0.8),
                                          (40000, 3, 6, 50, 0.9, 1.0), (700, 2, 10, 0, 0.9, 1.2),
                                          (5000, 4, 8, 1, 1.0, 1.0), (33, 3, 20, 40, 0.95, 0.7)])
def test_qlogits_truncated(sv, monkeypatch, tk_path, ldt, V, G, B, k, tp, T):
    """top-k / top-p applied to q_i as to p_i (the draft row's own kept set)."""
    if tk_path == "slices":
        monkeypatch.setenv("SPECVERIFY_PATH", "slices")
    else:
        monkeypatch.delenv("SPECVERIFY_PATH", raising=False)
    l_dt, q_dt = (ldt.split("/") * 2)[:2]   # "bf16/f32": target bf16, draft logits f32 (q materialised)
    inp = _ql_case(6000 + V + k, B, G, V, DTYPES[l_dt], DTYPES[q_dt], spread=1.0, noise=0.5)
    g = _gpu(inp)
    out = sv.verify_sample_qlogits(g["logits"], g["q_logits"], g["draft"], g["uniforms"], T, k, tp)
    L, Q, d, u = (P.to_np(inp[x]) for x in ("logits", "q_logits", "draft", "uniforms"))
    P.compare_sample(out, svref.verify_sample_qlogits(L, Q, d, u, T, k, tp), V)


def test_qlogits_truncation_limits(sv):
    inp = _gpu(_ql_case(5, 2, 2, 2000, torch.bfloat16, torch.bfloat16))
    with pytest.raises(sv.SvError) as e:   # top-p over 2000 tokens with no top-k
        sv.verify_sample_qlogits(inp["logits"], inp["q_logits"], inp["draft"], inp["uniforms"], 1.0, 0, 0.9)
    assert e.value.status == sv.SV_ERR_UNSUPPORTED


@pytest.mark.parametrize("kind", ["fused", "materialised", "truncated", "truncated_materialised"])
def test_qlogits_leaves_workspace_zero_filled(sv, kind):
    """Every path leaves the whole workspace (layout, q scratch, kept lists)
    zero-filled, as the contract says."""
    B, G, V, T = 8, 4, 32000, 0.9
    qdt = torch.float32 if kind in ("materialised", "truncated_materialised") else torch.bfloat16
    k, tp = (50, 0.9) if kind.startswith("truncated") else (0, 1.0)
    inp = _ql_case(31, B, G, V, torch.bfloat16, qdt)
    g = _gpu(inp)
    ws = sv.alloc_qlogits_workspace(B, G, V, k, device=DEV)
    for _ in range(2):
        out = sv.verify_sample_qlogits(g["logits"], g["q_logits"], g["draft"], g["uniforms"], T, k, tp, workspace=ws)
        torch.cuda.synchronize()
        assert int(torch.count_nonzero(ws)) == 0
        L, Q, d, u = (P.to_np(inp[x]) for x in ("logits", "q_logits", "draft", "uniforms"))
        P.compare_sample(out, svref.verify_sample_qlogits(L, Q, d, u, T, k, tp), V)
    names = sv.sv_last_kernels()
    if kind == "truncated":       # one dtype: the draft rows go through the streaming top-k kernel
        assert names == ["stream_topk_kernel"], names
    elif kind == "truncated_materialised":
        assert names[0] == "q_truncate_kernel" and names[-1] == "q_clear_kernel", names
    elif kind == "materialised":
        assert names[0] == "q_softmax_kernel", names
    else:
        assert names == ["stream_dense_kernel", "final_draw_kernel"], names


def test_qlogits_workspace_shared_with_plain_calls(sv):
    """The q scratch sits after the usual layout: a plain call on the same
    workspace afterwards finds its part zero-filled and is exact."""
    B, G, V, T = 8, 4, 4096, 0.9
    inp = _ql_case(99, B, G, V, torch.bfloat16, torch.bfloat16)
    g = _gpu(inp)
    ws = sv.alloc_qlogits_workspace(B, G, V, device=DEV)
    for _ in range(2):
        out = sv.verify_sample_qlogits(g["logits"], g["q_logits"], g["draft"], g["uniforms"], T, workspace=ws)
        P.compare_sample(out, _oracle(inp, T), V)
        q = torch.softmax(g["q_logits"].double() / float(np.float32(T)), -1).float().contiguous()
        out2 = sv.verify_sample(g["logits"], q, g["draft"], g["uniforms"], T, workspace=ws)
        P.compare_sample(out2, P.oracle_sample(dict(inp, q=q.cpu()), T), V)
