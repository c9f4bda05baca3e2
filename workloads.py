"""Seeded synthetic inputs for the speculative-decoding verify/sample step.

This module is the only code that both the CUDA path's tests/bench and the CPU
oracle see.  It holds none of the verify step's arithmetic: it only draws the
step's INPUTS - target logits, the draft's actual proposal q (the draft model's
own sampling transform, upstream of the step), the drafted tokens and the
uniforms - from torch's seeded generators.  Nothing here decides acceptance,
forms a residual or samples an output token.

The pages measure on models and datasets that are not available here (T5-XXL
with T5-small/base/large drafts on WMT En-De and CNN/DM); these synthetic rows
stand in for them with the shapes and value distributions below:

* ``gauss``: target logits ~ N(0, sigma^2) iid; draft logits = scale * target
  + N(0, draft_sigma^2); q = softmax(draft / T).
* ``zipf``: target logit of token v = -1.1 * ln(rank(v)) + N(0, 0.5^2), with
  rank a seeded random permutation of 1..V per row (a heavy-tailed LM-like
  row), rounded to the logits dtype; draft logits = target + N(0, draft_sigma^2);
  q = softmax(draft / T), optionally truncated by top-k then top-p and
  renormalised (the draft's actual proposal), stored dense in float32.
* draft tokens d_i ~ q_i (torch.multinomial); uniforms ~ U[0, 1) float32.
* greedy rows: d_i = the row's argmax with probability 0.7, else a uniform
  random token.
"""

from __future__ import annotations

import dataclasses

import torch

_DTYPES = {"f32": torch.float32, "bf16": torch.bfloat16, "f16": torch.float16}


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    B: int
    gamma: int
    V: int
    dtype: str                 # logits dtype: "f32" | "bf16" | "f16"
    mode: str                  # "sample" | "greedy"
    temperature: float = 1.0
    top_k: int = 0
    top_p: float = 1.0
    target: str = "zipf"       # "zipf" | "gauss"
    target_sigma: float = 0.5  # noise std of the target logits
    draft_scale: float = 1.0
    draft_sigma: float = 0.7
    seed: int = 0
    deterministic: bool = False   # q = None: the drafter's guess argmax(target + noise)
    ragged: bool = False          # per-sequence gamma_b in [1, gamma], stop tokens and token budgets
    n_stop: int = 0               # stop-token ids of a ragged round
    qlogits: bool = False         # the draft's proposal supplied as its logits (w's dtype), q formed on the GPU

    @property
    def rows(self) -> int:
        return self.B * (self.gamma + 1)

    @property
    def torch_dtype(self):
        return _DTYPES[self.dtype]

    def with_(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


# The five workloads of the verify step (sizes and distributions as stated for
# the step's headline measurements), plus the two other draft-noise levels of
# the B=64 sweep, the deterministic-draft (q one-hot, passed as None) case, a
# ragged round (per-sequence gamma_b, stop tokens, token budgets), q given as
# the draft's logits, and top-p alone over the whole vocabulary.
WORKLOADS = {
    w.name: w
    for w in [
        Workload("sample_b4_g4_v1024_f32", 4, 4, 1024, "f32", "sample", 1.0,
                 target="gauss", target_sigma=2.0, draft_scale=0.9, draft_sigma=1.0, seed=47),
        Workload("sample_b1_g5_v32000_bf16", 1, 5, 32000, "bf16", "sample", 0.7,
                 draft_sigma=0.7, seed=48),
        Workload("sample_b64_g4_v128256_bf16_s0.7", 64, 4, 128256, "bf16", "sample", 1.0,
                 draft_sigma=0.7, seed=49),
        Workload("sample_b64_g4_v128256_bf16_s0.3", 64, 4, 128256, "bf16", "sample", 1.0,
                 draft_sigma=0.3, seed=49),
        Workload("sample_b64_g4_v128256_bf16_s1.5", 64, 4, 128256, "bf16", "sample", 1.0,
                 draft_sigma=1.5, seed=49),
        Workload("greedy_b512_g4_v128256_bf16", 512, 4, 128256, "bf16", "greedy", seed=50),
        Workload("sample_det_b64_g4_v128256_bf16", 64, 4, 128256, "bf16", "sample", 1.0,
                 draft_sigma=0.7, seed=52, deterministic=True),
        Workload("sample_ragged_b64_g8_v128256_bf16", 64, 8, 128256, "bf16", "sample", 1.0,
                 draft_sigma=0.7, seed=53, ragged=True, n_stop=4),
        Workload("topk50_topp0.9_b256_g8_v152064_bf16", 256, 8, 152064, "bf16", "sample", 0.8,
                 top_k=50, top_p=0.9, draft_sigma=0.7, seed=51),
        Workload("sample_qlogits_b64_g4_v128256_bf16", 64, 4, 128256, "bf16", "sample", 1.0,
                 draft_sigma=0.7, seed=54, qlogits=True),
        Workload("topk50_topp0.9_qlogits_b256_g8_v152064_bf16", 256, 8, 152064, "bf16", "sample", 0.8,
                 top_k=50, top_p=0.9, draft_sigma=0.7, seed=55, qlogits=True),
        Workload("topp0.9_b64_g4_v128256_bf16", 64, 4, 128256, "bf16", "sample", 1.0,
                 top_p=0.9, draft_sigma=0.7, seed=56),
    ]
}

# the largest single-GPU workload: the one the bench line reports by default
HEADLINE = "topk50_topp0.9_b256_g8_v152064_bf16"


def _target_logits(w: Workload, B: int, g: torch.Generator, device) -> torch.Tensor:
    G1, V = w.gamma + 1, w.V
    if w.target == "gauss":
        L = torch.randn(B, G1, V, generator=g, device=device) * w.target_sigma
    else:
        keys = torch.rand(B * G1, V, generator=g, device=device)
        rank = keys.argsort(dim=1).to(torch.float32) + 1.0   # random permutation of 1..V
        del keys
        L = (-1.1 * torch.log(rank)).view(B, G1, V)
        del rank
        L += w.target_sigma * torch.randn(B, G1, V, generator=g, device=device)
    return L.to(w.torch_dtype)


def _draft_proposal(w: Workload, Lf: torch.Tensor, g: torch.Generator) -> torch.Tensor:
    """The draft's actual proposal q_i over the vocabulary (float32, dense)."""
    B, G, V = Lf.shape
    dl = w.draft_scale * Lf + w.draft_sigma * torch.randn(B, G, V, generator=g, device=Lf.device)
    z = dl / w.temperature
    del dl
    return _proposal_of(w, z)


def _proposal_of(w: Workload, z: torch.Tensor) -> torch.Tensor:
    """softmax(z) after w's top-k / top-p (z = draft logits / T), float32 dense."""
    B, G, V = z.shape
    if w.top_k <= 0 and w.top_p >= 1.0:
        return torch.softmax(z, dim=-1)
    k = V if w.top_k <= 0 else min(w.top_k, V)
    dev = z.device
    vals, idx = torch.topk(z, k, dim=-1, sorted=True)
    del z
    pk = torch.softmax(vals.double(), dim=-1)
    if w.top_p < 1.0:
        cum = pk.cumsum(-1)
        # keep the shortest prefix whose mass reaches top_p (crossing token kept)
        drop = (cum - pk) >= w.top_p
        pk = pk.masked_fill(drop, 0.0)
        pk = pk / pk.sum(-1, keepdim=True)
    q = torch.zeros(B, G, V, dtype=torch.float32, device=dev)
    q.scatter_(-1, idx, pk.float())
    return q


def make_inputs(w: Workload, seed: int | None = None, device="cpu", B: int | None = None) -> dict:
    """Draw one batch of inputs for workload ``w``.

    Returns dict(logits [B, gamma+1, V] (w's dtype), q [B, gamma, V] float32 or
    None in greedy mode, draft [B, gamma] int32, uniforms [B, gamma+1] float32).
    """
    B = w.B if B is None else B
    seed = w.seed if seed is None else seed
    device = torch.device(device)
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    G = w.gamma
    logits = _target_logits(w, B, g, device)
    Lf = logits[:, :G].float()
    q = None
    if w.mode == "greedy":
        # planted drafts: the row's argmax with probability 0.7, else uniform
        best = Lf.argmax(dim=-1)
        coin = torch.rand(B, G, generator=g, device=device) < 0.7
        rnd = torch.randint(0, w.V, (B, G), generator=g, device=device)
        draft = torch.where(coin, best, rnd)
    elif w.qlogits:
        # the draft model's logits (target logits plus noise, w's dtype); its
        # proposal softmax(q_logits / T) is formed by the library
        ql = (w.draft_scale * Lf + w.draft_sigma * torch.randn(B, G, w.V, generator=g, device=device)).to(w.torch_dtype)
        if G > 0:
            qp = _proposal_of(w, ql.float() / w.temperature)   # the draft samples from its actual proposal
            draft = torch.multinomial(qp.view(B * G, w.V), 1, generator=g).view(B, G)
            del qp
        else:
            draft = torch.zeros(B, 0, dtype=torch.int64, device=device)
    elif w.deterministic:
        # a deterministic drafter (n-gram / prompt lookup stand-in): its guess
        # is the argmax of the target logits plus noise; q is one-hot (None)
        guess = w.draft_scale * Lf + w.draft_sigma * torch.randn(B, G, w.V, generator=g, device=device)
        draft = guess.argmax(dim=-1)
        del guess
    else:
        q = _draft_proposal(w, Lf, g)
        if G > 0:
            draft = torch.multinomial(q.view(B * G, w.V), 1, generator=g).view(B, G)
        else:
            draft = torch.zeros(B, 0, dtype=torch.int64, device=device)
    del Lf
    uniforms = torch.rand(B, G + 1, generator=g, device=device, dtype=torch.float32)
    out = dict(logits=logits.contiguous(), q=None if q is None else q.contiguous(),
               draft=draft.to(torch.int32).contiguous(), uniforms=uniforms.contiguous())
    if w.qlogits:
        out["q_logits"] = ql.contiguous()
    if w.ragged:
        # gamma_b uniform in [1, gamma]; the stop ids are frequent target tokens
        # (the argmax of sequence 0's rows) so that some rounds stop early;
        # budgets uniform in [1, gamma + 2]
        out["gamma_b"] = torch.randint(1, G + 1, (B,), generator=g, device=device, dtype=torch.int32)
        stops = logits[0, : w.n_stop].float().argmax(-1).to(torch.int32)
        out["stop_tokens"] = stops.contiguous()
        out["max_new"] = torch.randint(1, G + 3, (B,), generator=g, device=device, dtype=torch.int32)
    return out
