"""q left in pinned host memory (read in place by the kernels across the
host link): every path gives the same outputs, bit for bit, as with q in
device memory, and matches the oracle; pageable host memory is refused."""

import pytest
import torch

import workloads
import _parity as P

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


@pytest.fixture(scope="module")
def sv():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from speculative_decoding_verification_46_gb300 import build

    build.build_library()
    import speculative_decoding_verification_46_gb300 as pkg

    pkg.load_library()
    return pkg


def _dev(inp):
    return {k: (v.to(DEV) if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}


# (workload recipe, B, forced path): untruncated streaming, the small-batch
# cluster kernel and the per-row kernels, top-k then top-p, top-p alone in
# the cluster-resident and the per-row threshold kernels, a ragged round
CASES = [
    ("sample_b64_g4_v128256_bf16_s0.7", 12, "auto"),
    ("sample_b1_g5_v32000_bf16", 2, "auto"),
    ("sample_b1_g5_v32000_bf16", 2, "grid"),
    ("sample_b4_g4_v1024_f32", 4, "auto"),
    ("topk50_topp0.9_b256_g8_v152064_bf16", 6, "auto"),
    ("topp0.9_b64_g4_v128256_bf16", 6, "auto"),
    ("topp0.9_b64_g4_v128256_bf16", 6, "topprow"),
    ("sample_ragged_b64_g8_v128256_bf16", 8, "auto"),
]


@pytest.mark.parametrize("name,B,path", CASES)
def test_host_q_matches_device_q(sv, monkeypatch, name, B, path):
    if path == "auto":
        monkeypatch.delenv("SPECVERIFY_PATH", raising=False)
    else:
        monkeypatch.setenv("SPECVERIFY_PATH", path)
    w = workloads.WORKLOADS[name]
    inp = workloads.make_inputs(w, seed=w.seed + 11, B=B)
    g = _dev(inp)
    q_host = inp["q"].contiguous().pin_memory()
    assert sv.sv_pointer_device_readable(q_host.data_ptr())
    gb = g.get("gamma_b")
    ref = sv.verify_sample(g["logits"], g["q"], g["draft"], g["uniforms"], w.temperature, w.top_k, w.top_p,
                           gamma_b=gb)
    kern = sv.sv_last_kernels()
    got = sv.verify_sample(g["logits"], q_host, g["draft"], g["uniforms"], w.temperature, w.top_k, w.top_p,
                           gamma_b=gb)
    torch.cuda.synchronize()
    assert sv.sv_last_kernels() == kern
    for a, b in zip(ref, got):
        assert torch.equal(a, b)
    if not w.ragged:
        P.compare_sample(got, P.oracle_sample(inp, w.temperature, w.top_k, w.top_p), w.V)


def test_pageable_host_q_is_refused(sv):
    w = workloads.WORKLOADS["sample_b4_g4_v1024_f32"]
    inp = workloads.make_inputs(w, seed=3)
    g = _dev(inp)
    q_pageable = inp["q"].contiguous()
    assert not q_pageable.is_pinned()
    assert not sv.sv_pointer_device_readable(q_pageable.data_ptr())
    with pytest.raises(ValueError):
        sv.verify_sample(g["logits"], q_pageable, g["draft"], g["uniforms"], w.temperature)
    assert sv.sv_pointer_device_readable(g["q"].data_ptr())
    assert not sv.sv_pointer_device_readable(0)
