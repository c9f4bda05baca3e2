"""The vocabulary-sharded driver's exchange on CPU: two gloo processes, one
shard each, run ``sharded.run_shards`` with ``TorchDistributedExchange``.

The GPU kernels cannot run here, so the four shard-local steps are stand-ins
written in float64 numpy below (the same protocol: per-row records, merge in
shard order, per-shard row-n totals, the owner shard's local inverse CDF).
What is under test is the driver and the exchange: every rank must end with
the whole problem's result, equal to the CPU oracle's (tests/_parity.py
tolerance), and the same on both ranks.  The GPU steps themselves are checked
against the oracle in tests/test_gpu_sharded.py.
"""

import os
import socket
import sys

import numpy as np
import pytest
import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
for p in (ROOT, os.path.join(ROOT, "tests")):
    if p not in sys.path:
        sys.path.insert(0, p)

from oracle import svref  # noqa: E402
import _parity as P  # noqa: E402
from speculative_decoding_verification_46_gb300 import sharded  # noqa: E402

SEQ_OOB, SEQ_QBAD, SEQ_BADROW, SEQ_RESID0 = 1, 2, 4, 8


class CpuSteps:
    """float64 stand-ins of the shard steps (records are float64 tensors)."""

    def row_stats(self, sh, greedy, T):
        L = sh.logits.double().numpy()
        B, G1, V = L.shape
        G = G1 - 1
        d = sh.draft.numpy()
        q = None if (sh.q is None or greedy) else sh.q.double().numpy()
        rec = np.zeros((B, G1, 8))
        for b in range(B):
            for i in range(G1):
                x = L[b, i] / (1.0 if greedy else T)
                nan = bool(np.isnan(x).any())
                xf = np.where(np.isnan(x), -np.inf, x)
                m = xf.max()
                s = np.exp(xf - m).sum() if np.isfinite(m) else 0.0
                arg = sh.v0 + int(np.argmax(L[b, i] == np.nanmax(np.where(np.isnan(L[b, i]), -np.inf, L[b, i]))))
                has, ld, qd = 0, 0.0, 0.0
                if i < G:
                    dl = int(d[b, i]) - sh.v0
                    if d[b, i] >= 0 and 0 <= dl < V:
                        has, ld = 1, L[b, i, dl]
                        qd = 1.0 if q is None else q[b, i, dl]
                rec[b, i] = (m, s, arg, ld, qd, has, nan, 0)
        return torch.from_numpy(rec)

    def scan(self, sh, stats_all, greedy, T, nshard):
        R = stats_all.numpy()                     # [S, B, G1, 8]
        S, B, G1, _ = R.shape
        G = G1 - 1
        d = sh.draft.numpy()
        u = None if greedy else sh.uniforms.double().numpy()
        tok = np.full((B, G1), -1, np.int32)
        n_out = np.zeros(B, np.int32)
        a_out = np.zeros((B, G), np.float32)
        st_out = np.zeros(B, np.int32)
        state = []
        for b in range(B):
            M = np.full(G1, -np.inf)
            s = np.zeros(G1)
            arg = np.zeros(G1, np.int64)
            nan = np.zeros(G1, bool)
            ld = np.zeros(G1)
            qd = np.zeros(G1)
            has = np.zeros(G1, bool)
            for i in range(G1):
                best = -np.inf
                for r in range(S):
                    m, sr, ar, l_, q_, h, nn, _ = R[r, b, i]
                    nan[i] |= bool(nn)
                    M[i] = max(M[i], m)
                    if m > best or (best == -np.inf and r == 0):
                        best, arg[i] = m, int(ar)
                    if h:
                        has[i], ld[i], qd[i] = True, l_, q_
                if np.isfinite(M[i]):
                    s[i] = sum(R[r, b, i, 1] * np.exp(R[r, b, i, 0] - M[i]) for r in range(S) if R[r, b, i, 0] > -np.inf)
            bits = 0
            for i in range(G1):
                if nan[i] or (not greedy and (not np.isfinite(M[i]) or not s[i] > 0)):
                    bits |= SEQ_BADROW
            rej = np.zeros(G, bool)
            for i in range(G):
                di = int(d[b, i])
                if di < 0 or di >= sh.Vg or not has[i]:
                    bits |= SEQ_OOB
                    rej[i] = True
                elif greedy:
                    rej[i] = di != (0 if nan[i] else int(arg[i]))
                else:
                    pd = np.exp(ld[i] / T - M[i]) / s[i] if (np.isfinite(M[i]) and s[i] > 0) else 0.0
                    if qd[i] > 0:
                        a = min(1.0, pd / qd[i])
                    else:
                        a = 1.0 if pd > 0 else 0.0
                        bits |= SEQ_QBAD
                    a_out[b, i] = a
                    rej[i] = not (u[b, i] < a)
            n = int(np.argmax(rej)) if rej.any() else G
            tok[b, :n] = d[b, :n]
            if greedy:
                tok[b, n] = 0 if nan[n] else int(arg[n])
            n_out[b] = n
            st_out[b] = bits
            state.append((n, M[n], s[n], bits))
        sh.out.update(tokens=torch.from_numpy(tok), n=torch.from_numpy(n_out),
                      a=None if greedy or G == 0 else torch.from_numpy(a_out), status=torch.from_numpy(st_out))
        sh.out["state"] = state

    def draw_sums(self, sh, T):
        L = sh.logits.double().numpy()
        B, G1, V = L.shape
        G = G1 - 1
        q = None if sh.q is None else sh.q.double().numpy()
        d = sh.draft.numpy()
        tot = np.zeros((B, 8))
        for b in range(B):
            n, M, s1, bits = sh.out["state"][b]
            w = np.exp(L[b, n] / T - M) if np.isfinite(M) else np.zeros(V)
            if n < G:
                if q is None:
                    qn = np.zeros(V)
                    dl = int(d[b, n]) - sh.v0
                    if 0 <= dl < V:
                        qn[dl] = np.inf
                else:
                    qn = q[b, n]
                sup = w > s1 * qn
                A = (w[sup] - s1 * qn[sup]).sum()
                Q = qn[sup].sum()
            else:
                A, Q = w.sum(), 0.0
            tot[b, :3] = (w.sum(), A, Q)
        return torch.from_numpy(tot)

    # ---- truncated protocol: candidate lists (value, global index, q, valid)
    def topk_candidates(self, sh, T, k):
        L = sh.logits.double().numpy()
        B, G1, V = L.shape
        G = G1 - 1
        d = sh.draft.numpy()
        q = None if sh.q is None else sh.q.double().numpy()
        rec = np.zeros((B, G1, k + 1, 4))
        for b in range(B):
            for i in range(G1):
                x = L[b, i]
                nan = bool(np.isnan(x).any())
                ok = np.nonzero(~np.isnan(x) & (x > -np.inf))[0]
                order = ok[np.lexsort((ok, -x[ok]))][:k]       # value descending, index ascending
                has, qd = 0, 0.0
                if i < G:
                    dl = int(d[b, i]) - sh.v0
                    if d[b, i] >= 0 and 0 <= dl < V:
                        has, qd = 1, (1.0 if q is None else q[b, i, dl])
                rec[b, i, 0] = (len(order), qd, has, nan)
                for e, v in enumerate(order):
                    qv = 0.0
                    if i < G:
                        qv = (1.0 if v + sh.v0 == d[b, i] else 0.0) if q is None else q[b, i, v]
                    rec[b, i, 1 + e] = (x[v], sh.v0 + v, qv, 1)
        return torch.from_numpy(rec)

    def topk_finish(self, sh, cand_all, T, k, top_p, nshard):
        C = cand_all.numpy()                       # [S, B, G1, k+1, 4]
        S, B, G1 = C.shape[:3]
        G = G1 - 1
        d = sh.draft.numpy()
        u = sh.uniforms.double().numpy()
        tok = np.full((B, G1), -1, np.int32)
        n_out = np.zeros(B, np.int32)
        a_out = np.zeros((B, G), np.float32)
        st_out = np.zeros(B, np.int32)

        def row(b, i):
            ent = [C[r, b, i, 1 + e] for r in range(S) for e in range(k) if C[r, b, i, 1 + e, 3]]
            nan = any(C[r, b, i, 0, 3] for r in range(S))
            ent.sort(key=lambda t: (-t[0], t[1]))
            ent = ent[:k]
            if nan or not ent or not np.isfinite(ent[0][0]):
                return [], nan or True, 0.0, 0
            w = np.exp(np.array([t[0] for t in ent]) / T - ent[0][0] / T)
            W = w.sum()
            J = len(ent)
            if top_p < 1.0:
                cum = np.cumsum(w)
                J = int(np.argmax(cum >= top_p * W)) + 1
            pk = w[:J] / w[:J].sum()
            hd = [C[r, b, i, 0] for r in range(S) if C[r, b, i, 0, 2]]
            qd, has = (hd[0][1], 1) if hd else (0.0, 0)
            return [(int(t[1]), pk[j], t[2]) for j, t in enumerate(ent[:J])], False, qd, has

        for b in range(B):
            bits = 0
            a = np.zeros(G)
            for i in range(G):
                kept, bad, qd, has = row(b, i)
                if bad:
                    bits |= SEQ_BADROW
                di = int(d[b, i])
                if di < 0 or di >= sh.Vg or not has:
                    bits |= SEQ_OOB
                    continue
                pd = next((pv for v, pv, _ in kept if v == di), 0.0)
                if qd > 0:
                    a[i] = min(1.0, pd / qd)
                else:
                    a[i] = 1.0 if pd > 0 else 0.0
                    bits |= SEQ_QBAD
            rej = [i for i in range(G) if not (u[b, i] < a[i])]
            n = rej[0] if rej else G
            if row(b, G)[1]:
                bits |= SEQ_BADROW
            kept = sorted(row(b, n)[0])
            r = np.array([max(pv - qv, 0.0) if n < G else pv for _, pv, qv in kept]) if kept else np.zeros(0)
            if n < G and not r.sum() > 0:
                bits |= SEQ_RESID0
                r = np.array([pv for _, pv, _ in kept])
            t = u[b, G] * r.sum()
            c = np.cumsum(r)
            hit = np.nonzero(c > t)[0]
            pos = np.nonzero(r > 0)[0]
            token = kept[hit[0]][0] if len(hit) else (kept[pos[-1]][0] if len(pos) else 0)
            tok[b, :n] = d[b, :n]
            tok[b, n] = token
            n_out[b] = n
            a_out[b] = a
            st_out[b] = bits
        sh.out.update(tokens=torch.from_numpy(tok), n=torch.from_numpy(n_out),
                      a=None if G == 0 else torch.from_numpy(a_out), status=torch.from_numpy(st_out))

    def draw_pick(self, sh, totals_all, T, nshard):
        Tt = totals_all.numpy()                   # [S, B, 8]
        L = sh.logits.double().numpy()
        B, G1, V = L.shape
        G = G1 - 1
        q = None if sh.q is None else sh.q.double().numpy()
        d = sh.draft.numpy()
        u = sh.uniforms.double().numpy()
        tok = sh.out["tokens"].numpy()
        st = sh.out["status"].numpy()
        for b in range(B):
            n, M, s1, bits = sh.out["state"][b]
            resid = n < G
            s = Tt[:, b, 0].sum()
            ds = s - s1
            use_q = resid
            Rr = np.maximum(Tt[:, b, 1] - ds * Tt[:, b, 2], 0.0) if use_q else Tt[:, b, 0].copy()
            r0 = 0
            if resid and not Rr.sum() > 0:
                r0, use_q, Rr = 1, False, Tt[:, b, 0].copy()
            Rt = Rr.sum()
            t = u[b, G] * Rt
            start = np.concatenate([[0.0], np.cumsum(Rr)[:-1]])
            cand = [r for r in range(Rr.shape[0]) if Rr[r] > 0 and start[r] <= t]
            owner = cand[-1] if (cand and Rt > 0 and not bits & SEQ_BADROW) else -1
            val = -1
            if owner == sh.rank:
                w = np.exp(L[b, n] / T - M)
                if use_q:
                    if q is None:
                        qn = np.zeros(V)
                        dl = int(d[b, n]) - sh.v0
                        if 0 <= dl < V:
                            qn[dl] = np.inf
                    else:
                        qn = q[b, n]
                    w = np.maximum(w - s * qn, 0.0)
                c = np.cumsum(w)
                hit = np.nonzero(c > t - start[owner])[0]
                pos = np.nonzero(w > 0)[0]
                val = sh.v0 + int(hit[0] if len(hit) else pos[-1])
            elif owner < 0 and sh.rank == 0:
                val = 0
            tok[b, n] = val
            st[b] = bits | (SEQ_RESID0 if r0 else 0)


def _case(B=5, G=4, V=1001, seed=11):
    g = torch.Generator().manual_seed(seed)
    L = torch.randn(B, G + 1, V, generator=g) * 2.0
    q = torch.softmax(L[:, :G] + torch.randn(B, G, V, generator=g), -1)
    draft = torch.multinomial(q.reshape(B * G, V), 1, generator=g).view(B, G).to(torch.int32)
    am = L[:, :G].argmax(-1).to(torch.int32)
    draft_g = torch.where(torch.rand(B, G, generator=g) < 0.7, am, draft)
    u = torch.rand(B, G + 1, generator=g)
    return dict(logits=L, q=q.float(), draft=draft, draft_g=draft_g, uniforms=u)


def _case_trunc(B=5, G=4, V=1000, seed=23, k=20, p=0.8):
    g = torch.Generator().manual_seed(seed)
    L = torch.randn(B, G + 1, V, generator=g) * 2.0
    z = (L[:, :G] + torch.randn(B, G, V, generator=g)) / 0.9
    vals, idx = torch.topk(z, k, dim=-1)
    pk = torch.softmax(vals.double(), -1)
    cum = pk.cumsum(-1)
    pk = pk.masked_fill((cum - pk) >= p, 0.0)
    pk = pk / pk.sum(-1, keepdim=True)
    q = torch.zeros(B, G, V, dtype=torch.float64).scatter_(-1, idx, pk).float()
    draft = torch.multinomial(q.reshape(B * G, V), 1, generator=g).view(B, G).to(torch.int32)
    u = torch.rand(B, G + 1, generator=g)
    return dict(logits=L, q=q, draft=draft, draft_g=draft, uniforms=u)


def _shard_of(inp, rank, nshard, greedy):
    V = inp["logits"].shape[2]
    v0, Vr = sharded.split_vocab(V, nshard)[rank]
    return sharded.Shard(logits=inp["logits"][:, :, v0:v0 + Vr].contiguous(),
                         q=None if greedy else inp["q"][:, :, v0:v0 + Vr].contiguous(),
                         draft=inp["draft_g"] if greedy else inp["draft"], uniforms=inp["uniforms"], v0=v0, Vg=V,
                         rank=rank)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, ws, port, queue):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(ws))
    import torch.distributed as dist

    dist.init_process_group("gloo", rank=rank, world_size=ws)
    try:
        inp = _case()
        out = {}
        for greedy in (False, True):
            sh = _shard_of(inp, rank, ws, greedy)
            (res,) = sharded.run_shards([sh], sharded.TorchDistributedExchange(), ws, greedy=greedy,
                                        temperature=0.9, steps=CpuSteps())
            out[greedy] = [None if t is None else t.numpy().copy() for t in res]
        tin = _case_trunc()
        sh = _shard_of(tin, rank, ws, False)
        (res,) = sharded.run_shards([sh], sharded.TorchDistributedExchange(), ws, greedy=False, temperature=0.9,
                                    top_k=20, top_p=0.8, steps=CpuSteps())
        out["trunc"] = [None if t is None else t.numpy().copy() for t in res]
        queue.put((rank, out))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def _compare(res, inp, greedy):
    tok, n, a, st = (None if x is None else torch.from_numpy(x) for x in res)
    if greedy:
        ref = svref.verify_greedy(inp["logits"].numpy(), inp["draft_g"].numpy())
        P.compare_greedy((tok, n, st), ref, inp["logits"].shape[2])
    else:
        ref = svref.verify_sample(inp["logits"].numpy(), inp["q"].numpy(), inp["draft"].numpy(),
                                  inp["uniforms"].numpy(), 0.9, 0, 1.0)
        P.compare_sample((tok, n, a, st), ref, inp["logits"].shape[2])


def test_two_gloo_ranks_reach_the_whole_problem_result():
    ctx = mp.get_context("spawn")
    queue = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, queue)) for r in range(2)]
    for p in procs:
        p.start()
    got = dict(queue.get(timeout=300) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    inp = _case()
    for greedy in (False, True):
        for r in (0, 1):
            _compare(got[r][greedy], inp, greedy)
        for x, y in zip(got[0][greedy], got[1][greedy]):
            assert (x is None and y is None) or np.array_equal(x, y)
    tin = _case_trunc()
    ref = svref.verify_sample(tin["logits"].numpy(), tin["q"].numpy(), tin["draft"].numpy(), tin["uniforms"].numpy(),
                              0.9, 20, 0.8)
    for r in (0, 1):
        tok, n, a, st = (None if x is None else torch.from_numpy(x) for x in got[r]["trunc"])
        P.compare_sample((tok, n, a, st), ref, 1000)
    for x, y in zip(got[0]["trunc"], got[1]["trunc"]):
        assert (x is None and y is None) or np.array_equal(x, y)


@pytest.mark.parametrize("nshard", [1, 3, 7])
def test_local_exchange_with_cpu_steps(nshard):
    """The same driver with all shards in one process (LocalExchange),
    untruncated, greedy, and top-k then top-p."""
    inp = _case(B=6, V=503, seed=nshard)
    for greedy in (False, True):
        shards = [_shard_of(inp, r, nshard, greedy) for r in range(nshard)]
        res = sharded.run_shards(shards, sharded.LocalExchange(), nshard, greedy=greedy, temperature=0.9,
                                 steps=CpuSteps())
        for r in range(nshard):
            _compare([None if t is None else t.numpy() for t in res[r]], inp, greedy)
    tin = _case_trunc(seed=40 + nshard)
    shards = [_shard_of(tin, r, nshard, False) for r in range(nshard)]
    res = sharded.run_shards(shards, sharded.LocalExchange(), nshard, greedy=False, temperature=0.9, top_k=20,
                             top_p=0.8, steps=CpuSteps())
    ref = svref.verify_sample(tin["logits"].numpy(), tin["q"].numpy(), tin["draft"].numpy(), tin["uniforms"].numpy(),
                              0.9, 20, 0.8)
    for r in range(nshard):
        tok, n, a, st = (None if t is None else t for t in res[r])
        P.compare_sample((tok, n, a, st), ref, 1000)
