"""Vocabulary-sharded verify on one GPU: the shards are column slices of one
problem (``sharded.simulate``), each run through the library's shard entry
points, their records exchanged by stacking.  The result must be the CPU
oracle's for the whole rows, under the same tolerance as the unsharded path:
greedy bit-exact, sampling a_i within 1e-5 relative and tokens equal except
boundary draws.  Shard counts 1..8, splits that leave ragged and unaligned
ranges, all three logits dtypes, dense and one-hot q, degenerate rows, and the
full-size B=64 V=128256 and B=512 greedy workloads.
"""

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


@pytest.fixture(scope="module")
def sharded(sv):
    from speculative_decoding_verification_46_gb300 import sharded as m

    return m


def _case(seed, B, G, V, dtype, T=1.0, ties=False, one_hot=False):
    g = torch.Generator().manual_seed(seed)
    L = torch.randn(B, G + 1, V, generator=g) * 2.0
    if ties:
        L = torch.round(L * 2) / 2
    L = L.to(dtype)
    w = workloads.Workload("case", B, G, V, "f32", "sample", T, draft_sigma=1.0)
    q = workloads._draft_proposal(w, L[:, :G].float(), g) if G > 0 else torch.zeros(B, 0, V)
    draft = (torch.multinomial(q.view(B * G, V), 1, generator=g).view(B, G).to(torch.int32) if G > 0
             else torch.zeros(B, 0, dtype=torch.int32))
    u = torch.rand(B, G + 1, generator=g)
    return dict(logits=L.contiguous(), q=None if one_hot else q.contiguous(), draft=draft, uniforms=u)


def _dev(inp):
    return {k: (v.to(DEV) if v is not None else None) for k, v in inp.items()}


@pytest.mark.parametrize("S", [1, 2, 3, 4, 8])
@pytest.mark.parametrize("dt", ["f32", "bf16", "f16"])
@pytest.mark.parametrize("V,G,B", [(8, 3, 7), (1001, 4, 9), (40003, 4, 5), (32000, 8, 3), (128256, 4, 4),
                                   (2048, 64, 3)])
def test_sharded_sample_matches_oracle(sharded, S, dt, V, G, B):
    if S > V:
        pytest.skip("more shards than tokens")
    inp = _case(1000 + S * 7 + V + G, B, G, V, DTYPES[dt], T=0.8, ties=(V == 1001))
    d = _dev(inp)
    got = sharded.simulate(d["logits"], d["q"], d["draft"], d["uniforms"], S, greedy=False, temperature=0.8)
    torch.cuda.synchronize()
    ref = P.oracle_sample(inp, 0.8)
    P.compare_sample(got, ref, V)


@pytest.mark.parametrize("S", [1, 2, 5, 8])
@pytest.mark.parametrize("dt", ["f32", "bf16"])
@pytest.mark.parametrize("V,G,B", [(9, 2, 6), (1000, 4, 17), (40003, 8, 5), (128256, 4, 6), (2048, 64, 4)])
def test_sharded_greedy_matches_oracle(sharded, S, dt, V, G, B):
    inp = _case(2000 + S + V + G, B, G, V, DTYPES[dt], ties=True)
    L = inp["logits"].float()
    g = torch.Generator().manual_seed(S + V)
    am = L[:, :G].argmax(-1).to(torch.int32)
    keep = torch.rand(B, G, generator=g) < 0.8
    inp["draft"] = torch.where(keep, am, torch.randint(0, V, (B, G), generator=g, dtype=torch.int32))
    d = _dev(inp)
    got = sharded.simulate(d["logits"], None, d["draft"], None, S, greedy=True)
    torch.cuda.synchronize()
    P.compare_greedy(got[:2] + (got[3],), P.oracle_greedy(inp), V)


@pytest.mark.parametrize("S", [2, 4])
def test_sharded_one_hot_drafts(sharded, S):
    """q = NULL (deterministic drafts): a_i = p_i(d_i), residual = p_n without d_n."""
    inp = _case(77 + S, 12, 4, 5003, torch.bfloat16, T=1.0, one_hot=True)
    d = _dev(inp)
    got = sharded.simulate(d["logits"], None, d["draft"], d["uniforms"], S, greedy=False, temperature=1.0)
    torch.cuda.synchronize()
    P.compare_sample(got, P.oracle_sample(inp, 1.0), 5003)


@pytest.mark.parametrize("S", [2, 3])
def test_sharded_degenerate_rows_and_bad_drafts(sharded, S):
    """NaN rows, rows of only -inf, a row whose mass sits in one shard, and
    draft ids outside [0, V): status bits as the oracle's, outputs in range."""
    B, G, V = 6, 4, 3001
    inp = _case(5 + S, B, G, V, torch.float32, T=1.0)
    L = inp["logits"]
    L[1, 2, 17] = float("nan")
    L[2, 0, :] = float("-inf")
    L[3, 1, :] = float("-inf")
    L[3, 1, V - 1] = 5.0        # all of row 1's mass in the last shard
    inp["draft"][4, 1] = V + 3
    inp["draft"][5, 0] = -2
    d = _dev(inp)
    got = sharded.simulate(d["logits"], d["q"], d["draft"], d["uniforms"], S, greedy=False, temperature=1.0)
    torch.cuda.synchronize()
    P.compare_sample(got, P.oracle_sample(inp, 1.0), V)
    got_g = sharded.simulate(d["logits"], None, d["draft"], None, S, greedy=True)
    torch.cuda.synchronize()
    P.compare_greedy(got_g[:2] + (got_g[3],), P.oracle_greedy(inp), V)


@pytest.mark.parametrize("S", [2, 4])
def test_sharded_full_size_b64(sharded, S):
    """B=64, gamma=4, V=128256 bf16 (sigma 0.7): every sequence against the
    oracle, which runs on a process pool."""
    w = workloads.WORKLOADS["sample_b64_g4_v128256_bf16_s0.7"]
    inp = workloads.make_inputs(w, device=DEV)
    got = sharded.simulate(inp["logits"], inp["q"], inp["draft"], inp["uniforms"], S, greedy=False,
                           temperature=w.temperature)
    torch.cuda.synchronize()
    ref = P.oracle_sample_pool(inp, w.temperature)
    stats = P.compare_sample(got, ref, w.V)
    assert stats["sequences"] == w.B


def test_sharded_greedy_full_size_b512(sharded):
    w = workloads.WORKLOADS["greedy_b512_g4_v128256_bf16"]
    inp = workloads.make_inputs(w, device=DEV)
    got = sharded.simulate(inp["logits"], None, inp["draft"], None, 4, greedy=True)
    torch.cuda.synchronize()
    P.compare_greedy(got[:2] + (got[3],), P.oracle_greedy(inp), w.V)


def test_sharded_steps_launch_the_library_kernels(sv, sharded):
    """Each step runs the library's own kernel (no fallback), and a second call
    on the same workspaces gives the same result (the workspace is left zeroed)."""
    inp = _dev(_case(3, 4, 4, 4099, torch.bfloat16))
    shards = []
    for r, (v0, Vr) in enumerate(sharded.split_vocab(4099, 2)):
        shards.append(sharded.Shard(logits=inp["logits"][:, :, v0:v0 + Vr].contiguous(),
                                    q=inp["q"][:, :, v0:v0 + Vr].contiguous(), draft=inp["draft"],
                                    uniforms=inp["uniforms"], v0=v0, Vg=4099, rank=r))
    steps = sharded.CudaSteps()
    seen = []

    class Spy:
        def __getattr__(self, name):
            fn = getattr(steps, name)

            def call(*a, **k):
                out = fn(*a, **k)
                seen.append(sv.sv_last_kernels())
                return out
            return call

    r1 = sharded.run_shards(shards, sharded.LocalExchange(), 2, greedy=False, temperature=1.0, steps=Spy())
    first = [t.clone() for t in r1[0] if t is not None]
    r2 = sharded.run_shards(shards, sharded.LocalExchange(), 2, greedy=False, temperature=1.0)
    torch.cuda.synchronize()
    for a, b in zip(first, [t for t in r2[0] if t is not None]):
        assert torch.equal(a, b)
    assert ["shard_stats_kernel"] in seen and ["shard_scan_kernel"] in seen
    assert ["final_draw_kernel"] in seen and ["shard_pick_kernel"] in seen
    for ws in (sh.workspace for sh in shards):
        assert int(ws.count_nonzero()) == 0


# ------------------------------------------------------------ truncation (top-k, then top-p)

def _case_trunc(seed, B, G, V, dtype, T, top_k, top_p, one_hot=False):
    g = torch.Generator().manual_seed(seed)
    L = (torch.randn(B, G + 1, V, generator=g) * 2.0).to(dtype)
    w = workloads.Workload("case", B, G, V, "f32", "sample", T, top_k=top_k, top_p=top_p, draft_sigma=1.0)
    q = workloads._draft_proposal(w, L[:, :G].float(), g)
    draft = torch.multinomial(q.view(B * G, V), 1, generator=g).view(B, G).to(torch.int32)
    u = torch.rand(B, G + 1, generator=g)
    return dict(logits=L.contiguous(), q=None if one_hot else q.contiguous(), draft=draft, uniforms=u)


@pytest.mark.parametrize("S", [1, 2, 3, 4, 8])
@pytest.mark.parametrize("dt", ["bf16", "f32", "f16"])
@pytest.mark.parametrize("V,G,B,k,p", [(1000, 4, 9, 50, 0.9), (40000, 4, 5, 50, 1.0), (152064, 8, 3, 50, 0.9),
                                       (4096, 3, 6, 200, 0.8), (20000, 2, 4, 1, 1.0), (2048, 64, 3, 30, 0.9)])
def test_sharded_topk_topp_matches_oracle(sharded, S, dt, V, G, B, k, p):
    align = 4 if dt == "f32" else 8
    if S * k > 2048:
        pytest.skip("more candidates than one merge holds")
    inp = _case_trunc(3000 + S + V + k, B, G, V, DTYPES[dt], 0.8, k, p)
    d = _dev(inp)
    got = sharded.simulate(d["logits"], d["q"], d["draft"], d["uniforms"], S, greedy=False, temperature=0.8,
                           top_k=k, top_p=p, align=align)
    torch.cuda.synchronize()
    P.compare_sample(got, P.oracle_sample(inp, 0.8, k, p), V)


@pytest.mark.parametrize("S", [2, 4])
def test_sharded_topk_one_hot_drafts(sharded, S):
    inp = _case_trunc(91 + S, 8, 4, 32000, torch.bfloat16, 1.0, 50, 0.9, one_hot=True)
    d = _dev(inp)
    got = sharded.simulate(d["logits"], None, d["draft"], d["uniforms"], S, greedy=False, temperature=1.0,
                           top_k=50, top_p=0.9, align=8)
    torch.cuda.synchronize()
    P.compare_sample(got, P.oracle_sample(inp, 1.0, 50, 0.9), 32000)


@pytest.mark.parametrize("S", [2, 4])
def test_sharded_topk_full_size_b256(sharded, S):
    """The top-k 50 then top-p 0.9 workload (B=256, gamma=8, V=152064): every
    sequence against the oracle (process pool)."""
    w = workloads.WORKLOADS["topk50_topp0.9_b256_g8_v152064_bf16"]
    inp = workloads.make_inputs(w, device=DEV)
    got = sharded.simulate(inp["logits"], inp["q"], inp["draft"], inp["uniforms"], S, greedy=False,
                           temperature=w.temperature, top_k=w.top_k, top_p=w.top_p, align=8)
    torch.cuda.synchronize()
    stats = P.compare_sample(got, P.oracle_sample_pool(inp, w.temperature, w.top_k, w.top_p), w.V)
    assert stats["sequences"] == w.B


def test_sharded_topk_launches_and_leaves_workspace_zeroed(sv, sharded):
    inp = _dev(_case_trunc(5, 4, 4, 8192, torch.bfloat16, 1.0, 50, 0.9))
    shards = []
    for r, (v0, Vr) in enumerate(sharded.split_vocab(8192, 2, 8)):
        shards.append(sharded.Shard(logits=inp["logits"][:, :, v0:v0 + Vr].contiguous(),
                                    q=inp["q"][:, :, v0:v0 + Vr].contiguous(), draft=inp["draft"],
                                    uniforms=inp["uniforms"], v0=v0, Vg=8192, rank=r))
    steps = sharded.CudaSteps()
    seen = []

    class Spy:
        def __getattr__(self, name):
            fn = getattr(steps, name)

            def call(*a, **k):
                out = fn(*a, **k)
                seen.append(sv.sv_last_kernels())
                return out
            return call

    r1 = sharded.run_shards(shards, sharded.LocalExchange(), 2, greedy=False, temperature=1.0, top_k=50, top_p=0.9,
                            steps=Spy())
    first = [t.clone() for t in r1[0] if t is not None]
    r2 = sharded.run_shards(shards, sharded.LocalExchange(), 2, greedy=False, temperature=1.0, top_k=50, top_p=0.9)
    torch.cuda.synchronize()
    for a, b in zip(first, [t for t in r2[0] if t is not None]):
        assert torch.equal(a, b)
    assert ["stream_topk_kernel"] in seen and ["shard_topk_finish_kernel"] in seen
    for sh in shards:
        assert int(sh.workspace.count_nonzero()) == 0


@pytest.mark.parametrize("greedy", [False, True])
def test_sharded_max_shards(sharded, greedy):
    """SV_MAX_SHARDS (32) shards of V = 128256."""
    inp = _case(32, 6, 4, 128256, torch.bfloat16, T=1.0)
    d = _dev(inp)
    got = sharded.simulate(d["logits"], None if greedy else d["q"], d["draft"], None if greedy else d["uniforms"], 32,
                           greedy=greedy, temperature=1.0)
    torch.cuda.synchronize()
    if greedy:
        P.compare_greedy(got[:2] + (got[3],), P.oracle_greedy(inp), 128256)
    else:
        P.compare_sample(got, P.oracle_sample(inp, 1.0), 128256)
