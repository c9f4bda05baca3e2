"""Deterministic drafts (q passed as NULL: each q_i one-hot at its drafted
token) on the GPU against the oracle given the same None.  Same tolerance
and boundary rules as the other parity tests (tests/_parity.py)."""

import numpy as np
import pytest
import torch

import workloads
import _parity as P

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


def _det_case(seed, B, G, V, dtype, spread=1.5, noise=0.7, oob=False):
    """Target logits; drafts = argmax of the target logits plus noise (the
    guess of a cheap deterministic drafter: often right, sometimes not)."""
    g = torch.Generator().manual_seed(seed)
    L = (torch.randn(B, G + 1, V, generator=g) * spread).to(dtype)
    guess = L[:, :G].float() + noise * torch.randn(B, G, V, generator=g)
    draft = guess.argmax(-1).to(torch.int32)
    if oob and B > 1 and G > 0:
        draft[1, 0] = V
    u = torch.rand(B, G + 1, generator=g)
    return dict(logits=L.contiguous(), q=None, draft=draft.contiguous(), uniforms=u)


def _gpu(inp):
    return {k: (v.to(DEV) if v is not None else None) for k, v in inp.items()}


@pytest.mark.parametrize("dt", ["f32", "bf16", "f16"])
@pytest.mark.parametrize("V,G,B,T", [(7, 3, 40, 1.0), (1000, 4, 12, 0.7), (40003, 4, 6, 1.0), (32000, 5, 3, 0.7),
                                     (128256, 4, 4, 1.0), (4096, 1, 30, 1.3)])
def test_deterministic_small(sv, path, dt, V, G, B, T):
    inp = _det_case(1000 + V + G, B, G, V, DTYPES[dt], oob=(V == 1000))
    g = _gpu(inp)
    out = sv.verify_sample(g["logits"], None, g["draft"], g["uniforms"], T)
    P.compare_sample(out, P.oracle_sample(inp, T), V)


@pytest.mark.parametrize("tk_path", ["auto", "slices"])
@pytest.mark.parametrize("V,G,B,k,tp", [(5000, 4, 12, 50, 0.9), (40000, 8, 6, 50, 0.9), (33, 3, 40, 40, 0.95)])
def test_deterministic_topk(sv, monkeypatch, tk_path, V, G, B, k, tp):
    if tk_path == "slices":
        monkeypatch.setenv("SPECVERIFY_PATH", "slices")
    else:
        monkeypatch.delenv("SPECVERIFY_PATH", raising=False)
    inp = _det_case(2000 + V + k, B, G, V, torch.bfloat16, spread=1.0)
    g = _gpu(inp)
    out = sv.verify_sample(g["logits"], None, g["draft"], g["uniforms"], 0.8, k, tp)
    P.compare_sample(out, P.oracle_sample(inp, 0.8, k, tp), V)


def test_deterministic_single_sequence_rounds(sv):
    """B = 1, gamma = 5, V = 32000 bf16 (the single-sequence shape), fresh
    inputs every round, drafts from the noisy-argmax drafter."""
    ws = sv.alloc_workspace(1, 5, 32000, 0, DEV)
    totals = dict(hard=0, boundary_mismatch=0, draws=0)
    accepted = 0
    for rnd in range(60):
        inp = _det_case(50_000 + rnd, 1, 5, 32000, torch.bfloat16, spread=2.0)
        g = _gpu(inp)
        out = sv.verify_sample(g["logits"], None, g["draft"], g["uniforms"], 0.7, workspace=ws)
        st = P.compare_sample(out, P.oracle_sample(inp, 0.7), 32000)
        for k2 in totals:
            totals[k2] += st[k2]
        accepted += int(out[1].item())
    assert totals["hard"] == 0
    assert accepted > 0


def test_deterministic_full_size_b64(sv):
    w = workloads.WORKLOADS["sample_b64_g4_v128256_bf16_s0.7"]
    inp = workloads.make_inputs(w, device=DEV)
    guess = inp["logits"][:, : w.gamma].float() + 0.7 * torch.randn(w.B, w.gamma, w.V, device=DEV,
                                                                      generator=torch.Generator(DEV).manual_seed(3))
    inp = dict(inp, q=None, draft=guess.argmax(-1).to(torch.int32).contiguous())
    out = sv.verify_sample(inp["logits"], None, inp["draft"], inp["uniforms"], w.temperature)
    st = P.compare_sample(out, P.oracle_sample_pool(inp, w.temperature), w.V)
    assert st["sequences"] == w.B
