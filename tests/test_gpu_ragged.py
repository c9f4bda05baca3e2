"""Ragged rounds (per-sequence gamma_b) and the stop-token / max_new_tokens
truncation on the GPU, against the oracle (oracle/svref.py
verify_sample_ragged, verify_greedy_ragged, truncate_emitted)."""

import numpy as np
import pytest
import torch

import workloads
from oracle import svref
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


def _case(seed, B, G, V, dtype, T=1.0, top_k=0, top_p=1.0, deterministic=False):
    """Random inputs plus gamma_b in [0, G]; rows, q rows and drafts beyond
    gamma_b hold junk (NaN rows, out-of-range drafts) that must be ignored."""
    g = torch.Generator().manual_seed(seed)
    L = torch.randn(B, G + 1, V, generator=g) * 1.5
    w = workloads.Workload("case", B, G, V, "f32", "sample", T, top_k=top_k, top_p=top_p, draft_sigma=1.0)
    q = workloads._draft_proposal(w, L[:, :G].float(), g)
    draft = torch.multinomial(q.view(B * G, V), 1, generator=g).view(B, G).to(torch.int32)
    if deterministic:
        q = None
    gb = torch.randint(0, G + 1, (B,), generator=g, dtype=torch.int32)
    gb[0] = G
    if B > 1:
        gb[1] = 0
    for b in range(B):
        L[b, gb[b] + 1:, ::7] = float("nan")
        draft[b, gb[b]:] = V + 3
    u = torch.rand(B, G + 1, generator=g)
    inp = dict(logits=L.to(dtype).contiguous(), q=None if q is None else q.contiguous(), draft=draft.contiguous(),
               uniforms=u)
    return inp, gb


def _gpu(inp):
    return {k: (v.to(DEV) if v is not None else None) for k, v in inp.items()}


def _oracle(inp, gb, T, top_k=0, top_p=1.0):
    L = P.to_np(inp["logits"])
    q = P.to_np(inp["q"])
    return svref.verify_sample_ragged(L, q, P.to_np(inp["draft"]), P.to_np(inp["uniforms"]), T, gb.numpy(),
                                      top_k, top_p)


@pytest.mark.parametrize("dt", ["f32", "bf16"])
@pytest.mark.parametrize("V,G,B,T", [(7, 3, 40, 1.0), (1000, 4, 12, 0.7), (40003, 5, 6, 1.0), (32000, 5, 4, 0.7),
                                     (128256, 4, 4, 1.0), (4096, 64, 20, 0.9)])
@pytest.mark.parametrize("det", [False, True])
def test_ragged_sample(sv, path, dt, V, G, B, T, det):
    inp, gb = _case(700 + V + G, B, G, V, DTYPES[dt], T, deterministic=det)
    g = _gpu(inp)
    out = sv.verify_sample(g["logits"], g["q"], g["draft"], g["uniforms"], T, gamma_b=gb.to(DEV))
    ref = _oracle(inp, gb, T)
    P.compare_sample(out, ref, V)
    a = out[2].cpu().numpy()
    for b in range(B):
        assert np.all(a[b, int(gb[b]):] == 0.0)


@pytest.mark.parametrize("tk_path", ["auto", "slices"])
@pytest.mark.parametrize("V,G,B,k,tp", [(5000, 4, 12, 50, 0.9), (40000, 8, 6, 50, 0.9), (4096, 64, 12, 30, 0.9)])
def test_ragged_topk(sv, monkeypatch, tk_path, V, G, B, k, tp):
    if tk_path == "slices":
        monkeypatch.setenv("SPECVERIFY_PATH", "slices")
    else:
        monkeypatch.delenv("SPECVERIFY_PATH", raising=False)
    inp, gb = _case(900 + V + k, B, G, V, torch.bfloat16, 0.8, k, tp)
    g = _gpu(inp)
    out = sv.verify_sample(g["logits"], g["q"], g["draft"], g["uniforms"], 0.8, k, tp, gamma_b=gb.to(DEV))
    P.compare_sample(out, _oracle(inp, gb, 0.8, k, tp), V)


@pytest.mark.parametrize("V,G,B", [(7, 4, 33), (40003, 4, 9), (128256, 4, 6), (32000, 5, 3), (4096, 64, 16)])
def test_ragged_greedy(sv, path, V, G, B):
    inp, gb = _case(1100 + V, B, G, V, torch.bfloat16)
    L = inp["logits"].float()
    best = L[:, :G].nan_to_num(nan=-1e9).argmax(-1).to(torch.int32)
    keep = torch.rand(B, G, generator=torch.Generator().manual_seed(V)) < 0.7
    d = torch.where(keep, best, inp["draft"])
    for b in range(B):
        d[b, gb[b]:] = V + 3
    g = _gpu(dict(inp, draft=d.contiguous()))
    out = sv.verify_greedy(g["logits"], g["draft"], gamma_b=gb.to(DEV))
    ref = svref.verify_greedy_ragged(P.to_np(inp["logits"]), d.numpy(), gb.numpy())
    P.compare_greedy(out, ref, V)


def test_ragged_full_size_b64(sv):
    w = workloads.WORKLOADS["sample_b64_g4_v128256_bf16_s0.7"]
    inp = workloads.make_inputs(w, device=DEV)
    gb = torch.randint(0, w.gamma + 1, (w.B,), generator=torch.Generator().manual_seed(9), dtype=torch.int32)
    out = sv.verify_sample(inp["logits"], inp["q"], inp["draft"], inp["uniforms"], w.temperature, gamma_b=gb.to(DEV))
    arrays = [P.to_np(inp[k]) for k in ("logits", "q", "draft", "uniforms")] + [gb.numpy()]
    st = P.compare_sample(out, P.oracle_pool("ragged", arrays, (w.temperature, 0, 1.0)), w.V)
    assert st["sequences"] == w.B


@pytest.mark.parametrize("n_stop,with_budget", [(0, True), (1, False), (3, True), (64, True)])
def test_truncate_emitted(sv, n_stop, with_budget):
    rng = np.random.default_rng(n_stop + 7)
    B, G = 513, 8
    tok = rng.integers(0, 100, size=(B, G + 1)).astype(np.int32)
    n = rng.integers(0, G + 1, size=B).astype(np.int32)
    for b in range(B):
        tok[b, n[b] + 1:] = -1
    stops = rng.choice(100, size=n_stop, replace=False).astype(np.int32)
    budget = rng.integers(-1, G + 3, size=B).astype(np.int32) if with_budget else None
    t = torch.from_numpy(tok).to(DEV)
    emitted = sv.truncate_emitted(t, torch.from_numpy(n).to(DEV),
                                  torch.from_numpy(stops).to(DEV) if n_stop else None,
                                  torch.from_numpy(budget).to(DEV) if with_budget else None)
    rt, re = svref.truncate_emitted(tok, n, stops, budget)
    np.testing.assert_array_equal(t.cpu().numpy(), rt)
    np.testing.assert_array_equal(emitted.cpu().numpy(), re)
