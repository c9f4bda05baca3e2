"""Vocabulary-sharded verify: the rows' logits (and q) split by token range.

When a tensor-parallel output layer leaves each process the logits of one
token range, the verify round ("11.1 核心原理", section 11.1.2 and listing
10-1) still needs sums over the whole vocabulary: every row's softmax
normaliser and the inverse CDF of the final draw.  Each shard reduces its own
range with the library's kernels (``sv_shard_*`` in include/specverify.h) and
the shards exchange a few records per row:

  1. row statistics of the local range         -> all-gather
  2. merged scan (a_i, n, outputs), greedy done
  3. row-n sums of the local range             -> all-gather
  4. the shard holding the draw picks its token -> all-reduce MAX of the tokens

With top-k (then top-p) the rows' candidate lists replace all of this: each
shard's top-k per row with q there -> all-gather -> every shard finishes the
round on the merged lists (one exchange).

The driver below runs these steps for a list of shards held by this process:
one shard per process with ``TorchDistributedExchange`` (NCCL or gloo), or
all shards of a problem in one process with ``LocalExchange`` (their records
are exchanged by stacking).  Every step of the computation runs on the GPU;
the exchange only moves records.
"""

from __future__ import annotations

from dataclasses import dataclass, field
from typing import List, Optional, Sequence

import torch

from . import _binding as sv


@dataclass
class Shard:
    """One shard's inputs: tokens [v0, v0 + V) of a vocabulary of Vg.

    logits [B, gamma+1, V] and q [B, gamma, V] (float32, or None: one-hot
    drafts) are this shard's columns, contiguous CUDA tensors; draft [B, gamma]
    int32 and uniforms [B, gamma+1] float32 hold global token ids / values and
    are the same on every shard."""

    logits: torch.Tensor
    q: Optional[torch.Tensor]
    draft: torch.Tensor
    uniforms: Optional[torch.Tensor]
    v0: int
    Vg: int
    rank: int
    workspace: Optional[torch.Tensor] = None
    out: dict = field(default_factory=dict)

    @property
    def V(self) -> int:
        return self.logits.shape[2]


class LocalExchange:
    """All shards in this process: a gather stacks the shards' tensors."""

    def all_gather(self, tensors: Sequence[torch.Tensor]) -> List[torch.Tensor]:
        stacked = torch.stack(list(tensors))
        return [stacked for _ in tensors]

    def all_reduce_max(self, tensors: Sequence[torch.Tensor]) -> None:
        m = torch.stack(list(tensors)).amax(dim=0)
        for t in tensors:
            t.copy_(m)


class TorchDistributedExchange:
    """One shard per process over torch.distributed (ranks in token order)."""

    def __init__(self, group=None):
        import torch.distributed as dist

        self.dist = dist
        self.group = group
        self.world = dist.get_world_size(group)

    def all_gather(self, tensors: Sequence[torch.Tensor]) -> List[torch.Tensor]:
        (t,) = tensors
        out = [torch.empty_like(t) for _ in range(self.world)]
        self.dist.all_gather(out, t.contiguous(), group=self.group)
        return [torch.stack(out)]

    def all_reduce_max(self, tensors: Sequence[torch.Tensor]) -> None:
        (t,) = tensors
        self.dist.all_reduce(t, op=self.dist.ReduceOp.MAX, group=self.group)


def _check(st: int, what: str) -> None:
    if st != sv.SV_OK:
        raise sv.SvError(st, what)


class CudaSteps:
    """The four shard-local steps on the GPU (the library's kernels)."""

    def row_stats(self, sh: Shard, greedy: bool, temperature: float) -> torch.Tensor:
        B, G1, V = sh.logits.shape
        G = G1 - 1
        stats = torch.empty(B, G1, sv.SV_SHARD_STAT_WORDS, dtype=torch.int32, device=sh.logits.device)
        _check(sv.sv_shard_row_stats(B, G, V, sh.v0, sh.Vg, sh.logits.data_ptr(), sv._TORCH_DTYPE[sh.logits.dtype],
                                     None if (greedy or sh.q is None or G == 0) else sh.q.data_ptr(),
                                     sh.draft.data_ptr() if G > 0 else None, temperature, int(greedy),
                                     stats.data_ptr(), sv._stream_handle(sh.logits.device, None)),
               "sv_shard_row_stats")
        return stats

    def scan(self, sh: Shard, stats_all: torch.Tensor, greedy: bool, temperature: float, nshard: int) -> None:
        B, G1, V = sh.logits.shape
        G = G1 - 1
        dev = sh.logits.device
        o = sh.out
        o["tokens"] = torch.empty(B, G1, dtype=torch.int32, device=dev)
        o["n"] = torch.empty(B, dtype=torch.int32, device=dev)
        o["a"] = None if (greedy or G == 0) else torch.empty(B, G, dtype=torch.float32, device=dev)
        o["status"] = torch.empty(B, dtype=torch.int32, device=dev)
        if sh.workspace is None and not greedy:
            sh.workspace = alloc_shard_workspace(B, G, V, dev)
        ws = sh.workspace
        _check(sv.sv_shard_scan(nshard, B, G, V, sh.Vg, stats_all.data_ptr(), sh.draft.data_ptr() if G > 0 else None,
                                None if greedy else sh.uniforms.data_ptr(), temperature, int(greedy),
                                o["tokens"].data_ptr(), o["n"].data_ptr(), sv._addr(o["a"]), o["status"].data_ptr(),
                                None if ws is None else ws.data_ptr(), 0 if ws is None else ws.numel(),
                                sv._stream_handle(dev, None)),
               "sv_shard_scan")

    def draw_sums(self, sh: Shard, temperature: float) -> torch.Tensor:
        B, G1, V = sh.logits.shape
        G = G1 - 1
        dev = sh.logits.device
        tot = torch.empty(B, sv.SV_SHARD_TOTAL_WORDS, dtype=torch.float32, device=dev)
        ws = sh.workspace
        _check(sv.sv_shard_draw_sums(B, G, V, sh.v0, sh.Vg, sh.logits.data_ptr(), sv._TORCH_DTYPE[sh.logits.dtype],
                                     None if (sh.q is None or G == 0) else sh.q.data_ptr(),
                                     sh.draft.data_ptr() if G > 0 else None, temperature, tot.data_ptr(),
                                     ws.data_ptr(), ws.numel(), sv._stream_handle(dev, None)),
               "sv_shard_draw_sums")
        return tot

    def topk_candidates(self, sh: Shard, temperature: float, top_k: int) -> torch.Tensor:
        B, G1, V = sh.logits.shape
        G = G1 - 1
        dev = sh.logits.device
        cand = torch.empty(B, G1, top_k + 1, sv.SV_SHARD_CAND_BYTES // 4, dtype=torch.int32, device=dev)
        if sh.workspace is None:
            sh.workspace = sv.alloc_workspace(B, G, V, top_k, dev)
        ws = sh.workspace
        _check(sv.sv_shard_topk_candidates(B, G, V, sh.v0, sh.Vg, sh.logits.data_ptr(),
                                           sv._TORCH_DTYPE[sh.logits.dtype],
                                           None if (sh.q is None or G == 0) else sh.q.data_ptr(),
                                           sh.draft.data_ptr() if G > 0 else None, temperature, top_k,
                                           cand.data_ptr(), ws.data_ptr(), ws.numel(), sv._stream_handle(dev, None)),
               "sv_shard_topk_candidates")
        return cand

    def topk_finish(self, sh: Shard, cand_all: torch.Tensor, temperature: float, top_k: int, top_p: float,
                    nshard: int) -> None:
        B, G1, V = sh.logits.shape
        G = G1 - 1
        dev = sh.logits.device
        o = sh.out
        o["tokens"] = torch.empty(B, G1, dtype=torch.int32, device=dev)
        o["n"] = torch.empty(B, dtype=torch.int32, device=dev)
        o["a"] = None if G == 0 else torch.empty(B, G, dtype=torch.float32, device=dev)
        o["status"] = torch.empty(B, dtype=torch.int32, device=dev)
        _check(sv.sv_shard_topk_finish(nshard, B, G, sh.Vg, cand_all.data_ptr(),
                                       sh.draft.data_ptr() if G > 0 else None, sh.uniforms.data_ptr(), temperature,
                                       top_k, top_p, o["tokens"].data_ptr(), o["n"].data_ptr(), sv._addr(o["a"]),
                                       o["status"].data_ptr(), sv._stream_handle(dev, None)),
               "sv_shard_topk_finish")

    def draw_pick(self, sh: Shard, totals_all: torch.Tensor, temperature: float, nshard: int) -> None:
        B, G1, V = sh.logits.shape
        G = G1 - 1
        dev = sh.logits.device
        o = sh.out
        ws = sh.workspace
        _check(sv.sv_shard_draw_pick(nshard, sh.rank, B, G, V, sh.v0, sh.Vg, sh.logits.data_ptr(),
                                     sv._TORCH_DTYPE[sh.logits.dtype],
                                     None if (sh.q is None or G == 0) else sh.q.data_ptr(),
                                     sh.draft.data_ptr() if G > 0 else None, sh.uniforms.data_ptr(), temperature,
                                     totals_all.data_ptr(), o["tokens"].data_ptr(), o["status"].data_ptr(),
                                     ws.data_ptr(), ws.numel(), sv._stream_handle(dev, None)),
               "sv_shard_draw_pick")


def alloc_shard_workspace(B: int, gamma: int, V: int, device=None) -> torch.Tensor:
    """A zero-filled workspace for one shard of V tokens."""
    n = sv.sv_shard_workspace_bytes(B, gamma, V)
    if n == 0 and B > 0:
        raise sv.SvError(sv.SV_ERR_INVALID_ARG, "sv_shard_workspace_bytes")
    return torch.zeros(max(n, 256), dtype=torch.uint8, device=device)


def run_shards(shards: Sequence[Shard], exchange, nshard: int, *, greedy: bool, temperature: float = 1.0,
               top_k: int = 0, top_p: float = 1.0, steps=None):
    """The sharded verify of one call for the shards this process holds.

    top_k (1..1024, then top_p) truncates p as the unsharded path does; top-p
    without top-k is not offered sharded.  Returns, per shard, (out_tokens
    [B, gamma+1], n [B], accept_prob [B, gamma] or None, status [B]); every
    shard's result is the whole problem's."""
    steps = CudaSteps() if steps is None else steps
    Vg = shards[0].Vg if shards else 0
    truncate = not greedy and ((0 < top_k < Vg) or top_p < 1.0)
    if truncate:
        if not 0 < top_k < Vg:
            raise sv.SvError(sv.SV_ERR_UNSUPPORTED, "sharded verify: top-p without top-k")
        cands = [steps.topk_candidates(sh, temperature, top_k) for sh in shards]
        cands_all = exchange.all_gather(cands)
        for sh, ca in zip(shards, cands_all):
            steps.topk_finish(sh, ca, temperature, top_k, top_p, nshard)
        return [(sh.out["tokens"], sh.out["n"], sh.out["a"], sh.out["status"]) for sh in shards]
    stats = [steps.row_stats(sh, greedy, temperature) for sh in shards]
    stats_all = exchange.all_gather(stats)
    for sh, st in zip(shards, stats_all):
        steps.scan(sh, st, greedy, temperature, nshard)
    if not greedy:
        tots = [steps.draw_sums(sh, temperature) for sh in shards]
        tots_all = exchange.all_gather(tots)
        for sh, tt in zip(shards, tots_all):
            steps.draw_pick(sh, tt, temperature, nshard)
        exchange.all_reduce_max([sh.out["tokens"] for sh in shards])
    return [(sh.out["tokens"], sh.out["n"], sh.out["a"], sh.out["status"]) for sh in shards]


def split_vocab(V: int, nshard: int, align: int = 1) -> List[tuple]:
    """Contiguous token ranges [(v0, V_r)] of a vocabulary split nshard ways,
    every boundary a multiple of `align` (the truncated path wants ranges of
    whole 16-byte vectors: 8 for 16-bit logits, 4 for float32)."""
    bounds = [min(V, (V * r // nshard) // align * align) for r in range(nshard)] + [V]
    return [(bounds[r], bounds[r + 1] - bounds[r]) for r in range(nshard)]


def simulate(logits, q, draft, uniforms, nshard: int, *, greedy: bool, temperature: float = 1.0, top_k: int = 0,
             top_p: float = 1.0, align: int = 1, steps=None):
    """All nshard shards of one problem in this process (whole-row tensors in,
    the shards' column slices copied out): the sharded path's result, which
    equals verify_sample / verify_greedy on the whole rows."""
    B, G1, Vg = logits.shape
    shards = []
    for r, (v0, Vr) in enumerate(split_vocab(Vg, nshard, align)):
        shards.append(Shard(logits=logits[:, :, v0:v0 + Vr].contiguous(),
                            q=None if (q is None or greedy) else q[:, :, v0:v0 + Vr].contiguous(),
                            draft=draft, uniforms=uniforms, v0=v0, Vg=Vg, rank=r))
    res = run_shards(shards, LocalExchange(), nshard, greedy=greedy, temperature=temperature, top_k=top_k,
                     top_p=top_p, steps=steps)
    return res[0]
