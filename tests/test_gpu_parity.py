"""Parity of the CUDA path (through the C ABI) with the CPU oracle.

Small cases span several vocabulary slices and residual chunks plus a ragged
tail (V not a multiple of the vector width or the slice), all three logits
dtypes, gamma in {0, 1, 4, 8}, forced ties and degenerate rows.  The full-size
workloads run in the same launch configuration the bench times; where the
oracle would be slow it checks a seeded sample of sequences.
"""

import numpy as np
import pytest
import torch

import workloads
from oracle import svref
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


DEV = "cuda:0"
DTYPES = {"f32": torch.float32, "bf16": torch.bfloat16, "f16": torch.float16}


def _gpu(inp):
    return {k: (v.to(DEV) if v is not None else None) for k, v in inp.items()}


def _random_case(seed, B, G, V, dtype, T=1.0, ties=False, spread=2.0, top_k=0, top_p=1.0):
    """Random rows (optionally with many exact ties), q = a truncated or full
    softmax of noisy logits, d ~ q, uniforms U[0,1)."""
    g = torch.Generator().manual_seed(seed)
    L = torch.randn(B, G + 1, V, generator=g) * spread
    if ties:
        L = torch.round(L * 2) / 2
    L = L.to(dtype)
    w = workloads.Workload("case", B, G, V, "f32", "sample", T, top_k=top_k, top_p=top_p, draft_sigma=1.0)
    q = workloads._draft_proposal(w, L[:, :G].float(), g) if G > 0 else torch.zeros(B, 0, V)
    if G > 0:
        draft = torch.multinomial(q.view(B * G, V), 1, generator=g).view(B, G).to(torch.int32)
    else:
        draft = torch.zeros(B, 0, dtype=torch.int32)
    u = torch.rand(B, G + 1, generator=g)
    return dict(logits=L.contiguous(), q=q.contiguous(), draft=draft, uniforms=u)


# ------------------------------------------------------------------ greedy

@pytest.fixture(params=["auto", "grid", "cluster", "slices"])
def path(request, monkeypatch):
    """Which kernel path the library takes: its own choice (small problems go
    to the one-cluster-per-sequence kernel, larger ones to the streaming
    kernels), or forced: grid = streaming kernels (when V is a multiple of the
    vector width), cluster, slices = the per-slice grid kernels."""
    if request.param != "auto":
        monkeypatch.setenv("SPECVERIFY_PATH", request.param)
    else:
        monkeypatch.delenv("SPECVERIFY_PATH", raising=False)
    return request.param


@pytest.mark.parametrize("dt", ["f32", "bf16", "f16"])
@pytest.mark.parametrize("V,G,B", [(1, 2, 5), (7, 4, 33), (1000, 1, 17), (40003, 4, 9), (128256, 4, 6),
                                   (4096, 8, 3), (32000, 5, 2)])
def test_greedy_small(sv, path, dt, V, G, B):
    inp = _random_case(10 + V + G, B, G, V, DTYPES[dt], ties=True)
    # drafts: the row argmax most of the time, so that long accepted prefixes occur
    best = inp["logits"][:, :G].float().argmax(-1).to(torch.int32)
    coin = torch.rand(B, G, generator=torch.Generator().manual_seed(V)) < 0.8
    inp["draft"] = torch.where(coin, best, inp["draft"])
    g = _gpu(inp)
    out = sv.verify_greedy(g["logits"], g["draft"])
    P.compare_greedy(out, P.oracle_greedy(inp), V)


def test_greedy_degenerate_rows(sv, path):
    B, G, V = 6, 3, 300
    L = torch.randn(B, G + 1, V)
    L[0, 1, 17] = float("nan")
    L[1, :, :] = -float("inf")              # all -inf: argmax is index 0
    L[2, 2, :] = 0.0
    L[2, 2, 5] = -0.0                      # -0.0 == +0.0: lowest index wins
    L[3, 0, 3] = float("inf")
    d = torch.randint(0, V, (B, G), dtype=torch.int32)
    d[4, 1] = V + 5                          # out of range
    d[5, 0] = -1
    for dt in DTYPES.values():
        inp = dict(logits=L.to(dt), draft=d)
        g = _gpu(inp)
        out = sv.verify_greedy(g["logits"], g["draft"])
        P.compare_greedy(out, P.oracle_greedy(inp), V)


def test_greedy_full_size(sv):
    w = workloads.WORKLOADS["greedy_b512_g4_v128256_bf16"]
    inp = workloads.make_inputs(w, device=DEV)
    out = sv.verify_greedy(inp["logits"], inp["draft"])
    st = P.compare_greedy(out, P.oracle_greedy(inp), w.V)
    assert st["sequences"] == w.B


# ------------------------------------------------------------------ sampling, no truncation

@pytest.mark.parametrize("dt", ["f32", "bf16", "f16"])
@pytest.mark.parametrize("V,G,B,T", [(2, 4, 300, 1.0), (3, 1, 200, 0.7), (7, 8, 100, 1.3), (1024, 4, 40, 1.0),
                                     (32000, 5, 8, 0.7), (40003, 0, 8, 1.0), (40003, 8, 6, 0.9),
                                     (4096, 0, 5, 1.0), (8192, 8, 4, 0.8), (32000, 1, 3, 1.1)])
def test_sample_small(sv, path, dt, V, G, B, T):
    inp = _random_case(100 + V + G, B, G, V, DTYPES[dt], T=T, spread=1.5)
    g = _gpu(inp)
    out = sv.verify_sample(g["logits"], g["q"], g["draft"], g["uniforms"], T)
    P.compare_sample(out, P.oracle_sample(inp, T), V)


def test_sample_config_b4_g4_v1024_f32_rounds(sv):
    """The small workload as stated: 10k rounds, each with fresh seeds, one
    launch of B=4 per round (the launch configuration the bench times); the
    rounds' inputs are staged on the device together and every round's call
    reads its own slice."""
    w = workloads.WORKLOADS["sample_b4_g4_v1024_f32"]
    rounds = 10_000
    ins = [workloads.make_inputs(w, seed=10_000 + rnd) for rnd in range(rounds)]
    cat = {k: torch.cat([x[k] for x in ins]) for k in ("logits", "q", "draft", "uniforms")}
    g = _gpu(cat)
    ws = sv.alloc_workspace(w.B, w.gamma, w.V, 0, DEV)
    B, G = w.B, w.gamma
    out = (torch.empty(rounds * B, G + 1, dtype=torch.int32, device=DEV),
           torch.empty(rounds * B, dtype=torch.int32, device=DEV),
           torch.empty(rounds * B, G, dtype=torch.float32, device=DEV),
           torch.empty(rounds * B, dtype=torch.int32, device=DEV))
    for rnd in range(rounds):
        s = slice(rnd * B, (rnd + 1) * B)
        sv.verify_sample(g["logits"][s], g["q"][s], g["draft"][s], g["uniforms"][s], w.temperature, workspace=ws,
                         outputs=tuple(o[s] for o in out))
        assert sv.sv_last_kernels() == ["cluster_kernel"]
    torch.cuda.synchronize()
    st = P.compare_sample(out, P.oracle_sample(cat, w.temperature), w.V)
    assert st["sequences"] == rounds * B
    assert st["hard"] == 0
    assert st["boundary_mismatch"] <= P.BOUNDARY_FRACTION * st["draws"]


@pytest.mark.parametrize("force", [None, "grid", "slices"])
def test_sample_config_b1_g5_v32000_bf16_rounds(sv, force, monkeypatch):
    if force:
        monkeypatch.setenv("SPECVERIFY_PATH", force)
    w = workloads.WORKLOADS["sample_b1_g5_v32000_bf16"]
    ws = sv.alloc_workspace(w.B, w.gamma, w.V, 0, DEV)
    acc = []
    for rnd in range(200):
        inp = workloads.make_inputs(w, seed=20_000 + rnd)
        g = _gpu(inp)
        out = sv.verify_sample(g["logits"], g["q"], g["draft"], g["uniforms"], w.temperature, workspace=ws)
        P.compare_sample(out, P.oracle_sample(inp, w.temperature), w.V)
        acc.append(P.to_np(out[1]))


@pytest.mark.parametrize("name", ["sample_b64_g4_v128256_bf16_s0.3", "sample_b64_g4_v128256_bf16_s0.7",
                                  "sample_b64_g4_v128256_bf16_s1.5"])
def test_sample_full_size_b64(sv, name):
    w = workloads.WORKLOADS[name]
    inp = workloads.make_inputs(w, device=DEV)
    out = sv.verify_sample(inp["logits"], inp["q"], inp["draft"], inp["uniforms"], w.temperature)
    st = P.compare_sample(out, P.oracle_sample(inp, w.temperature), w.V)
    assert st["sequences"] == w.B


# ------------------------------------------------------------------ top-k / top-p

@pytest.fixture(params=["auto", "slices"])
def topk_path(request, monkeypatch):
    """Top-k kernel: the streaming per-row one (library's choice when V is a
    multiple of the vector width) or the per-slice one (forced)."""
    if request.param == "slices":
        monkeypatch.setenv("SPECVERIFY_PATH", "slices")
    else:
        monkeypatch.delenv("SPECVERIFY_PATH", raising=False)
    return request.param


@pytest.mark.parametrize("dt", ["f32", "bf16", "f16"])
@pytest.mark.parametrize("V,G,B,k,tp", [(7, 2, 50, 3, 1.0), (100, 4, 30, 1, 1.0), (5000, 4, 12, 50, 0.9),
                                        (40003, 8, 4, 50, 0.9), (40003, 3, 4, 200, 0.5), (600, 2, 20, 0, 0.8),
                                        (33, 3, 40, 40, 0.95), (40000, 8, 6, 50, 0.9), (16384, 4, 8, 600, 0.7),
                                        (1024, 2, 16, 1000, 0.99), (152064, 4, 4, 1024, 0.95)])
def test_topk_small(sv, topk_path, dt, V, G, B, k, tp):
    inp = _random_case(300 + V + k, B, G, V, DTYPES[dt], T=0.8, ties=True, spread=1.0, top_k=k, top_p=tp)
    g = _gpu(inp)
    out = sv.verify_sample(g["logits"], g["q"], g["draft"], g["uniforms"], 0.8, k, tp)
    P.compare_sample(out, P.oracle_sample(inp, 0.8, k, tp), V)


def _topp_kernel(V, esize, forced_row=False):
    """The threshold kernel the library runs for top-p alone: a row of whole
    16-byte vectors that fits 8 slices of 64 KB sits in a cluster's shared
    memory; any other row streams through one CTA."""
    fits = V % (16 // esize) == 0 and -(-V * esize // 65536) <= 8
    return "topp_cluster_kernel" if fits and not forced_row else "topp_row_kernel"


@pytest.mark.parametrize("path", ["auto", "topprow"])
@pytest.mark.parametrize("dt", ["bf16", "f16", "f32"])
@pytest.mark.parametrize("V,G,B,tp,T", [(40003, 4, 6, 0.9, 1.0), (128256, 4, 4, 0.5, 1.0), (152064, 8, 2, 0.99, 0.8),
                                        (5000, 3, 10, 0.95, 0.7), (1030, 2, 12, 0.6, 1.3), (32768, 2, 5, 0.9, 1.0),
                                        (65544, 3, 4, 0.8, 1.0), (262144, 2, 2, 0.9, 0.5), (262152, 2, 2, 0.9, 0.5)])
def test_topp_only_any_vocab(sv, monkeypatch, path, dt, V, G, B, tp, T):
    """top-p with no top-k beyond SV_MAX_TOP_K tokens (the threshold path):
    Zipf-like rows with heavy tails (large kept sets) and exact ties; the
    cluster-resident kernel (1 to 8 slices, the last one short) and the
    per-row kernel on the same inputs.  The largest rows (2^18 tokens, the
    cluster kernel's limit and one vector past it) run at T = 0.5: with a
    few draws per case, a flatter row would put one of them within 1e-6 of
    a CDF step more often than the 1e-4 boundary-mismatch bound allows."""
    if path == "topprow":
        monkeypatch.setenv("SPECVERIFY_PATH", "topprow")
    else:
        monkeypatch.delenv("SPECVERIFY_PATH", raising=False)
    w = workloads.Workload("topp", B, G, V, dt, "sample", T, top_k=0, top_p=tp, draft_sigma=0.7, seed=V + G)
    inp = workloads.make_inputs(w, seed=V + int(tp * 100))
    g = _gpu(inp)
    out = sv.verify_sample(g["logits"], g["q"], g["draft"], g["uniforms"], T, 0, tp)
    esize = {"bf16": 2, "f16": 2, "f32": 4}[dt]
    assert sv.sv_last_kernels() == [_topp_kernel(V, esize, path == "topprow"), "final_draw_kernel"]
    P.compare_sample(out, P.oracle_sample(inp, T, 0, tp), V)


@pytest.mark.parametrize("V,G,B,tp", [(7, 2, 40, 0.8), (600, 2, 20, 0.9), (1024, 4, 10, 0.5)])
def test_topp_only_threshold_path_forced_small_vocab(sv, monkeypatch, V, G, B, tp):
    """The threshold path forced where the list path would run, with many
    exact ties (rounded logits) and deterministic drafts too."""
    monkeypatch.setenv("SPECVERIFY_PATH", "topp")
    inp = _random_case(700 + V, B, G, V, torch.bfloat16, T=0.9, ties=True, spread=1.0, top_k=0, top_p=tp)
    g = _gpu(inp)
    out = sv.verify_sample(g["logits"], g["q"], g["draft"], g["uniforms"], 0.9, 0, tp)
    assert sv.sv_last_kernels() == [_topp_kernel(V, 2), "final_draw_kernel"]
    P.compare_sample(out, P.oracle_sample(inp, 0.9, 0, tp), V)
    out = sv.verify_sample(g["logits"], None, g["draft"], g["uniforms"], 0.9, 0, tp)
    P.compare_sample(out, P.oracle_sample(dict(inp, q=None), 0.9, 0, tp), V)


def test_topp_only_degenerate_rows(sv):
    B, G, V = 6, 3, 3000
    inp = _random_case(17, B, G, V, torch.float32, top_k=0, top_p=0.9)
    inp["logits"][0, 2, 100] = float("nan")
    inp["logits"][1, 0, :] = -float("inf")
    inp["logits"][2, 1, 5] = float("inf")
    inp["draft"][3, 1] = V
    inp["logits"][4, :, 1000:] = -float("inf")
    for dt in DTYPES.values():
        case = dict(inp, logits=inp["logits"].to(dt))
        g = _gpu(case)
        out = sv.verify_sample(g["logits"], g["q"], g["draft"], g["uniforms"], 1.0, 0, 0.9)
        P.compare_sample(out, P.oracle_sample(case, 1.0, 0, 0.9), V)


def test_topk_heavy_ties_take_the_exact_fallback(sv):
    """All-equal rows: every element ties at the threshold, the candidate
    buffers overflow and the exact (value, index) bisection must pick the
    k lowest indices."""
    B, G, V = 3, 2, 20000
    inp = _random_case(5, B, G, V, torch.bfloat16, top_k=50, top_p=1.0)
    inp["logits"][:, 1, :] = 1.0
    g = _gpu(inp)
    out = sv.verify_sample(g["logits"], g["q"], g["draft"], g["uniforms"], 1.0, 50, 1.0)
    P.compare_sample(out, P.oracle_sample(inp, 1.0, 50, 1.0), V)


def test_topk_full_size(sv):
    """The headline workload (B=256, gamma=8, V=152064, top-k 50 then top-p
    0.9), every sequence against the oracle."""
    w = workloads.WORKLOADS["topk50_topp0.9_b256_g8_v152064_bf16"]
    inp = workloads.make_inputs(w, device=DEV)
    out = sv.verify_sample(inp["logits"], inp["q"], inp["draft"], inp["uniforms"], w.temperature, w.top_k, w.top_p)
    ref = P.oracle_sample_pool(inp, w.temperature, w.top_k, w.top_p)
    st = P.compare_sample(out, ref, w.V)
    assert st["sequences"] == w.B


# ------------------------------------------------------------------ degenerate data, edges, reuse

def test_sample_degenerate_rows_and_flags(sv, path):
    B, G, V = 8, 3, 257
    inp = _random_case(7, B, G, V, torch.float32)
    inp["logits"][0, 2, 100] = float("nan")
    inp["logits"][1, 0, :] = -float("inf")
    inp["logits"][2, 1, 5] = float("inf")
    inp["draft"][3, 1] = V
    inp["q"][4, 0, inp["draft"][4, 0]] = 0.0
    inp["logits"][5, :, 200:] = -float("inf")      # masked tail: allowed, weight 0
    for dt in DTYPES.values():
        case = dict(inp, logits=inp["logits"].to(dt))
        g = _gpu(case)
        for k, tp in [(0, 1.0), (10, 0.9)]:
            out = sv.verify_sample(g["logits"], g["q"], g["draft"], g["uniforms"], 1.0, k, tp)
            P.compare_sample(out, P.oracle_sample(case, 1.0, k, tp), V)


def test_empty_batch_and_gamma_zero(sv):
    L = torch.zeros(0, 3, 10, device=DEV)
    out = sv.verify_sample(L, torch.zeros(0, 2, 10, device=DEV), torch.zeros(0, 2, dtype=torch.int32, device=DEV),
                           torch.zeros(0, 3, device=DEV), 1.0)
    assert out[0].numel() == 0
    inp = _random_case(3, 50, 0, 33, torch.bfloat16)
    g = _gpu(inp)
    out = sv.verify_sample(g["logits"], None, None, g["uniforms"], 1.0)
    P.compare_sample(out, P.oracle_sample(inp, 1.0), 33)


def test_workspace_reuse_and_determinism(sv):
    """One workspace across calls of different kinds and shapes: the tickets
    are left reset, and repeated calls give identical outputs."""
    ws = sv.alloc_workspace(64, 8, 40003, 50, DEV)
    cases = [_random_case(s, B, G, V, torch.bfloat16, top_k=k, top_p=tp)
             for s, (B, G, V, k, tp) in enumerate([(64, 8, 40003, 50, 0.9), (5, 2, 777, 0, 1.0),
                                                    (64, 4, 40003, 0, 1.0), (3, 8, 1000, 50, 1.0)])]
    first = []
    for rep in range(3):
        for ci, (c, kt) in enumerate(zip(cases, [(50, 0.9), (0, 1.0), (0, 1.0), (50, 1.0)])):
            g = _gpu(c)
            out = sv.verify_sample(g["logits"], g["q"], g["draft"], g["uniforms"], 1.0, kt[0], kt[1], workspace=ws)
            o = [P.to_np(x) for x in out]
            if rep == 0:
                first.append(o)
                P.compare_sample(out, P.oracle_sample(c, 1.0, *kt), c["logits"].shape[2])
            else:
                for x, y in zip(o, first[ci]):
                    assert np.array_equal(x, y)
        gd = _gpu(cases[1])
        sv.verify_greedy(gd["logits"], gd["draft"], workspace=ws)


def test_outputs_stay_inside_their_buffers(sv):
    """Guard bands around every output: nothing is written outside them."""
    B, G, V = 16, 4, 20001
    inp = _random_case(11, B, G, V, torch.bfloat16)
    g = _gpu(inp)
    pad = 64
    sentinel = -123456
    bt = torch.full((B * (G + 1) + 2 * pad,), sentinel, dtype=torch.int32, device=DEV)
    bn = torch.full((B + 2 * pad,), sentinel, dtype=torch.int32, device=DEV)
    ba = torch.full((B * G + 2 * pad,), -7.0, dtype=torch.float32, device=DEV)
    bs = torch.full((B + 2 * pad,), sentinel, dtype=torch.int32, device=DEV)
    outs = (bt[pad:-pad].view(B, G + 1), bn[pad:-pad], ba[pad:-pad].view(B, G), bs[pad:-pad])
    for k, tp in [(0, 1.0), (20, 0.9)]:
        sv.verify_sample(g["logits"], g["q"], g["draft"], g["uniforms"], 1.0, k, tp, outputs=outs)
        sv.verify_greedy(g["logits"], g["draft"], outputs=(outs[0], outs[1], outs[3]))
        torch.cuda.synchronize()
        for buf, s in ((bt, sentinel), (bn, sentinel), (ba, -7.0), (bs, sentinel)):
            assert torch.all(buf[:pad] == s) and torch.all(buf[-pad:] == s)


# ------------------------------------------------------------------ statistics through the kernel

@pytest.mark.parametrize("V", [2, 4, 8])
def test_gpu_chi_square_preserves_target(sv, V):
    import scipy.special
    import scipy.stats

    rng = np.random.default_rng(V)
    B, G = 200_000, 2
    row = rng.normal(0, 1.2, size=(G + 1, V)).astype(np.float32)
    qrow = rng.dirichlet(np.ones(V) * 0.5, size=G).astype(np.float32)
    qn = qrow.astype(np.float64) / qrow.astype(np.float64).sum(-1, keepdims=True)
    draft = np.stack([rng.choice(V, size=B, p=qn[i]) for i in range(G)], 1).astype(np.int32)
    L = torch.from_numpy(row).expand(B, G + 1, V).contiguous().to(DEV)
    q = torch.from_numpy(qrow).expand(B, G, V).contiguous().to(DEV)
    u = torch.from_numpy(rng.random((B, G + 1)).astype(np.float32)).to(DEV)
    tok, n, _, _ = sv.verify_sample(L, q, torch.from_numpy(draft).to(DEV), u, 1.0)
    tok, n = P.to_np(tok), P.to_np(n)
    P0 = scipy.special.softmax(row[0].astype(np.float64))
    P1 = scipy.special.softmax(row[1].astype(np.float64))
    assert scipy.stats.chisquare(np.bincount(tok[:, 0], minlength=V), B * P0).pvalue > 1e-3
    sel = n >= 1
    assert scipy.stats.chisquare(np.bincount(tok[sel, 1], minlength=V), sel.sum() * P1).pvalue > 1e-3


@pytest.mark.parametrize("alpha,gamma", [(0.7, 4), (0.7, 8)])
def test_gpu_expected_tokens_closed_form(sv, alpha, gamma):
    B = 400_000
    L = torch.log(torch.tensor([alpha, 1 - alpha])).expand(B, gamma + 1, 2).contiguous().to(DEV)
    q = torch.tensor([1.0, 0.0]).expand(B, gamma, 2).contiguous().to(DEV)
    d = torch.zeros(B, gamma, dtype=torch.int32, device=DEV)
    u = torch.rand(B, gamma + 1, generator=torch.Generator(device=DEV).manual_seed(gamma), device=DEV)
    _, n, a, _ = sv.verify_sample(L, q, d, u, 1.0)
    emitted = P.to_np(n).astype(np.float64) + 1
    e = svref.expected_tokens_per_round(alpha, gamma)
    assert abs(emitted.mean() - e) < 4 * emitted.std(ddof=1) / np.sqrt(B)
    np.testing.assert_allclose(P.to_np(a), alpha, rtol=1e-6)


# ------------------------------------------------------------------ gamma = 64 (the largest: 65 rows)

@pytest.mark.parametrize("mode", ["sample", "topk", "topp", "greedy"])
@pytest.mark.parametrize("V,B,forced", [(4096, 20, None), (4096, 20, "slices"), (1000, 2, "cluster")])
def test_gamma_64_bonus_row(sv, monkeypatch, mode, V, B, forced):
    """gamma = 64: row 64 is the bonus row.  Half the sequences have q = p
    (every draft accepted, the bonus drawn from row 64), half a noisy q."""
    if forced:
        monkeypatch.setenv("SPECVERIFY_PATH", forced)
    else:
        monkeypatch.delenv("SPECVERIFY_PATH", raising=False)
    G, T = 64, 0.9
    top_k, top_p = {"sample": (0, 1.0), "topk": (40, 0.9), "topp": (0, 0.8), "greedy": (0, 1.0)}[mode]
    if mode == "topp" and forced == "cluster":
        pytest.skip("top-p alone has its own rows path")
    g = torch.Generator().manual_seed(64 + V + B)
    L = (torch.randn(B, G + 1, V, generator=g) * 2.0).to(torch.bfloat16)
    w = workloads.Workload("case", B, G, V, "f32", "sample", T, top_k=top_k, top_p=top_p, draft_sigma=1.0)
    q = workloads._draft_proposal(w, L[:, :G].float(), g)
    same = workloads.Workload("case", B, G, V, "f32", "sample", T, top_k=top_k, top_p=top_p, draft_sigma=0.0)
    q_exact = workloads._proposal_of(same, L[:, :G].float() / T)
    half = B // 2
    q[:half] = q_exact[:half]
    draft = torch.multinomial(q.reshape(B * G, V), 1, generator=g).view(B, G).to(torch.int32)
    if mode == "greedy":
        am = L[:, :G].float().argmax(-1).to(torch.int32)
        draft[:half] = am[:half]
    u = torch.rand(B, G + 1, generator=g)
    inp = dict(logits=L.contiguous(), q=q.contiguous(), draft=draft, uniforms=u)
    d = _gpu(inp)
    if mode == "greedy":
        got = sv.verify_greedy(d["logits"], d["draft"])
        torch.cuda.synchronize()
        ref = P.oracle_greedy(inp)
        P.compare_greedy(got, ref, V)
        assert (ref["n_accepted"][:half] == G).all()
        return
    got = sv.verify_sample(d["logits"], d["q"], d["draft"], d["uniforms"], T, top_k, top_p)
    torch.cuda.synchronize()
    ref = P.oracle_sample(inp, T, top_k, top_p)
    P.compare_sample(got, ref, V)
    # the bonus row is drawn from (q = p up to the draft's own tie order at the cut)
    assert (ref["n_accepted"][:half] == G).sum() >= (half - 1 if mode == "sample" else min(2, half))


# ------------------------------------------------------------------ the largest vocabulary

@pytest.mark.parametrize("mode", ["sample", "greedy"])
def test_max_vocabulary(sv, monkeypatch, mode):
    """V = SV_MAX_VOCAB (2^24): 8192 final-draw items per row, the largest
    search stash, the streaming kernel's shortest grid."""
    monkeypatch.delenv("SPECVERIFY_PATH", raising=False)
    V, G, B = 1 << 24, 2, 2
    inp = _random_case(24, B, G, V, torch.bfloat16, T=1.0, spread=3.0)
    d = _gpu(inp)
    if mode == "greedy":
        got = sv.verify_greedy(d["logits"], d["draft"])
        torch.cuda.synchronize()
        P.compare_greedy(got, P.oracle_greedy(inp), V)
    else:
        got = sv.verify_sample(d["logits"], d["q"], d["draft"], d["uniforms"], 1.0)
        torch.cuda.synchronize()
        P.compare_sample(got, P.oracle_sample(inp, 1.0), V)


def test_large_batch(sv, monkeypatch):
    """B = 4096 sequences (V = 1024, gamma = 4): the grids and workspace of a
    large batch; every sequence against the oracle (process pool)."""
    monkeypatch.delenv("SPECVERIFY_PATH", raising=False)
    V, G, B = 1024, 4, 4096
    inp = _random_case(4096, B, G, V, torch.float32, T=0.9)
    d = _gpu(inp)
    got = sv.verify_sample(d["logits"], d["q"], d["draft"], d["uniforms"], 0.9)
    torch.cuda.synchronize()
    ref = P.oracle_sample_pool(inp, 0.9)
    stats = P.compare_sample(got, ref, V)
    assert stats["sequences"] == B
    got_g = sv.verify_greedy(d["logits"], d["draft"])
    torch.cuda.synchronize()
    P.compare_greedy(got_g, P.oracle_greedy(inp), V)
