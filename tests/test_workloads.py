"""The seeded input generators produce inputs of the stated shapes and
distributions (checked on the CPU at reduced batch)."""

import pytest
import torch

import workloads


@pytest.mark.parametrize("name", sorted(workloads.WORKLOADS))
def test_shapes_and_support(name):
    w = workloads.WORKLOADS[name]
    inp = workloads.make_inputs(w, B=2)
    G, V = w.gamma, w.V
    assert inp["logits"].shape == (2, G + 1, V) and inp["logits"].dtype == w.torch_dtype
    assert inp["draft"].shape == (2, G) and inp["draft"].dtype == torch.int32
    assert inp["uniforms"].shape == (2, G + 1) and inp["uniforms"].dtype == torch.float32
    assert torch.all((inp["uniforms"] >= 0) & (inp["uniforms"] < 1))
    assert torch.all((inp["draft"] >= 0) & (inp["draft"] < V))
    if w.qlogits:
        # the draft's logits in the workload's dtype; q is formed by the library
        assert inp["q"] is None
        ql = inp["q_logits"]
        assert ql.shape == (2, G, V) and ql.dtype == w.torch_dtype and torch.isfinite(ql.float()).all()
    elif w.mode == "greedy" or w.deterministic:
        assert inp["q"] is None
    else:
        q = inp["q"]
        assert q.shape == (2, G, V) and q.dtype == torch.float32
        torch.testing.assert_close(q.double().sum(-1), torch.ones(2, G, dtype=torch.float64), atol=1e-5, rtol=0)
        qd = q.gather(-1, inp["draft"].long().unsqueeze(-1))
        assert torch.all(qd > 0)            # every draft was drawn from q
        if w.top_k > 0:
            assert torch.all((q > 0).sum(-1) <= w.top_k)


def test_seeded_and_reproducible():
    w = workloads.WORKLOADS["sample_b4_g4_v1024_f32"]
    a = workloads.make_inputs(w, seed=3)
    b = workloads.make_inputs(w, seed=3)
    c = workloads.make_inputs(w, seed=4)
    for k in ("logits", "q", "draft", "uniforms"):
        assert torch.equal(a[k], b[k])
    assert not torch.equal(a["logits"], c["logits"])
