"""Comparison of the CUDA path with the CPU oracle under the stated tolerance.

* greedy: bit-exact tokens, counts and status bits;
* sampling: acceptance probabilities within 1e-5 relative (plus 1e-30 absolute,
  for float32 underflow of probabilities below ~1e-38); tokens and counts
  equal, except for sequences where the oracle flags a boundary draw (a uniform
  within 1e-6 of an acceptance threshold or CDF step, or a top-p sum within
  1e-6 of top_p); such boundary mismatches must stay below 1e-4 of all draws.
* sequences whose rows hold NaN / +inf / only -inf: the status bit must be
  set and the outputs in range; their values are undefined.
"""

import numpy as np

from oracle import svref

RTOL = 1e-5
ATOL = 1e-30
BOUNDARY_FRACTION = 1e-4
RESID_TINY = 1e-6


def to_np(t):
    if t is None:
        return None
    t = t.detach().cpu()
    if t.dtype in (__import__("torch").bfloat16, __import__("torch").float16):
        t = t.float()
    return t.numpy()


def oracle_sample(inp, T, top_k=0, top_p=1.0, rows=None):
    L, q, d, u = (to_np(inp[k]) for k in ("logits", "q", "draft", "uniforms"))
    if rows is not None:
        L, d, u = L[rows], d[rows], u[rows]
        q = q[rows] if q is not None else None
    return svref.verify_sample(L, q, d, u, T, top_k, top_p)


def _oracle_chunk(job):
    kind, arrays, scal = job
    if kind == "sample":
        return svref.verify_sample(*arrays, *scal)
    if kind == "qlogits":
        return svref.verify_sample_qlogits(*arrays, *scal)
    L, q, d, u, gb = arrays          # ragged
    T, top_k, top_p = scal
    return svref.verify_sample_ragged(L, q, d, u, T, gb, top_k, top_p)


def oracle_pool(kind, arrays, scal, workers=8, chunk=8):
    """An oracle entry point ("sample": verify_sample(L, q, d, u, T, k, p);
    "qlogits": verify_sample_qlogits(L, Q, d, u, T, k, p); "ragged":
    verify_sample_ragged(L, q, d, u, T, gamma_b, k, p)) over the whole batch,
    sequences split across a pool of `spawn` processes (the oracle works per
    sequence; spawn, not fork, because the parent holds a CUDA context).
    `arrays` are per-sequence numpy arrays (None allowed), `scal` the
    trailing scalars.  Returns the oracle's result dict for the batch."""
    import multiprocessing as mp

    B = arrays[0].shape[0]
    jobs = [(kind, [None if a is None else a[s:s + chunk] for a in arrays], scal) for s in range(0, B, chunk)]
    with mp.get_context("spawn").Pool(max(1, min(workers, len(jobs), mp.cpu_count()))) as pool:
        parts = pool.map_async(_oracle_chunk, jobs).get(timeout=900)
    return {k: np.concatenate([r[k] for r in parts]) for k in parts[0]}


def oracle_sample_pool(inp, T, top_k=0, top_p=1.0):
    """oracle_sample over the whole batch on a process pool."""
    L, q, d, u = (to_np(inp[k]) for k in ("logits", "q", "draft", "uniforms"))
    return oracle_pool("sample", [L, q, d, u], (T, top_k, top_p))


def oracle_greedy(inp, rows=None):
    L, d = to_np(inp["logits"]), to_np(inp["draft"])
    if rows is not None:
        L, d = L[rows], d[rows]
    return svref.verify_greedy(L, d)


def compare_sample(gpu, ref, V, rows=None):
    tok, n, a, st = (to_np(x) for x in gpu)
    if rows is not None:
        tok, n, st = tok[rows], n[rows], st[rows]
        a = a[rows] if a is not None else None
    G = tok.shape[1] - 1
    bad = (ref["status"] & svref.SEQ_BAD_ROW) != 0
    good = ~bad
    assert np.all((tok >= -1) & (tok < V)), "token out of range"
    assert np.all((n >= 0) & (n <= G))
    assert np.all((st[bad] & svref.SEQ_BAD_ROW) != 0), "bad row not flagged"
    stats = dict(sequences=int(good.sum()), hard=0, boundary_mismatch=0, draws=0, boundary_flagged=0,
                 max_rel_err_a=0.0)
    if G > 0 and a is not None:
        ar = ref["accept_prob"]
        excess = np.abs(a.astype(np.float64) - ar) - (RTOL * np.abs(ar) + ATOL)
        stats["max_rel_err_a"] = float(np.max((np.abs(a - ar) / np.maximum(np.abs(ar), 1e-300))[good], initial=0))
        assert np.all(excess[good] <= 0), f"accept_prob off by more than {RTOL} relative"
    mism = (tok != ref["out_tokens"]).any(1) | (n != ref["n_accepted"])
    hard = mism & ~ref["boundary"] & good
    stats["hard"] = int(hard.sum())
    stats["boundary_mismatch"] = int((mism & ref["boundary"] & good).sum())
    stats["boundary_flagged"] = int((ref["boundary"] & good).sum())
    stats["draws"] = int((np.minimum(ref["n_accepted"] + 1, G) + 1)[good].sum())
    # Every status bit is compared exactly.  The one exception is
    # SEQ_RESIDUAL_ZERO on a rejection whose exact residual mass R is below
    # RESID_TINY: the step forms the residual in float32 (probabilities
    # rounded at ~6e-8 relative), so a float64 R of that size may round to
    # zero (bit set, draw from p_n) or stay positive; both are the pages'
    # rule applied to the values the step holds.
    keep = np.full(st.shape, -1, dtype=np.int64)
    if "residual_mass" in ref:
        keep[ref["residual_mass"] < RESID_TINY] &= ~np.int64(svref.SEQ_RESIDUAL_ZERO)
    assert np.array_equal((st & keep)[good], (ref["status"] & keep)[good]), "status bits differ"
    if stats["hard"]:
        lines = []
        for bidx in np.nonzero(hard)[0][:5]:
            lines.append(f"seq {bidx}: gpu n={n[bidx]} tok={tok[bidx].tolist()} | ref n={ref['n_accepted'][bidx]} "
                         f"tok={ref['out_tokens'][bidx].tolist()} a_ref={np.round(ref['accept_prob'][bidx], 7).tolist()}"
                         + (f" a_gpu={np.round(a[bidx], 7).tolist()}" if a is not None and G > 0 else ""))
        raise AssertionError(f"{stats['hard']} non-boundary mismatches:\n" + "\n".join(lines))
    assert stats["boundary_mismatch"] <= BOUNDARY_FRACTION * max(stats["draws"], 1), stats
    return stats


def compare_greedy(gpu, ref, V, rows=None):
    tok, n, st = (to_np(x) for x in gpu)
    if rows is not None:
        tok, n, st = tok[rows], n[rows], st[rows]
    bad = (ref["status"] & svref.SEQ_BAD_ROW) != 0
    good = ~bad
    assert np.all((tok >= -1) & (tok < V))
    assert np.all((st[bad] & svref.SEQ_BAD_ROW) != 0)
    assert np.array_equal(tok[good], ref["out_tokens"][good])
    assert np.array_equal(n[good], ref["n_accepted"][good])
    assert np.array_equal(st[good], ref["status"][good])
    return dict(sequences=int(good.sum()))
