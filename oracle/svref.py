"""Plain float64 CPU oracle for the batched verify/sample step of speculative decoding.

TEST INFRASTRUCTURE ONLY.  Only the tests, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import this
module.  The product path (the CUDA library and its Python binding) never
imports, links or calls it, and this module imports nothing from the product.

Every function below is written out from the pages, slowly and in float64:

* "11.1 核心原理: Draft + Verify 与 Rejection Sampling" (textbook chapter 11.1),
  cited as [Ch11.1]:
    - §11.1.1: row i of the one target forward predicts draft token d_{i+1};
      row gamma gives the bonus distribution;
    - §11.1.2: greedy rule (accept while d_i == argmax p_i, emit the target
      argmax at the first mismatch); sampling rule a_i = min(1, p_i(d_i)/q_i(d_i));
      residual r_i = max(p_i - q_i, 0) / sum; temperature / top-k / top-p are
      applied to p_i and q_i before the test; q is the draft's ACTUAL proposal;
    - code listing 10-1 (the verify round: scan in order, break at the first
      rejection and sample the residual, else sample the bonus from p_gamma;
      emitted = draft[:accepted] + [next_token]);
    - §11.1.3: the proof min(p,q) + max(p-q,0) = p and the worked example.
* "Fast Inference from Transformers via Speculative Decoding" (reading notes),
  cited as [SD-notes]: the speculative-sampling paragraph (accept with
  probability min(1, p(x)/q(x)), on rejection resample from
  norm(max(0, p(x) - q(x)))), the "at least one, at most gamma+1 tokens" remark
  and the E[N] equation.

Readings taken where the pages are silent (each one is listed with its reason
in the repository's design notes):

* uniforms: gamma + 1 per sequence; U[b, i] is the accept test of position i,
  U[b, gamma] is the single final draw (residual or bonus);
* accept iff u < a (strict, as in listing 10-1);
* categorical sampling is the inverse CDF in token-index order: the smallest v
  with C(v) = sum_{w <= v} r(w) > u * R, R = C(V-1); if rounding leaves no such
  v, the largest v with r(v) > 0;
* truncation order: temperature, then top-k ranked by (logit desc, index asc),
  renormalise, then top-p = the shortest prefix of that ranking whose
  renormalised mass reaches top_p (the crossing token is kept), renormalise;
* q is used exactly as given (it already is the draft's actual, truncated
  proposal); the step does not re-truncate it;
* q_i(d_i) <= 0: a_i = 1 if p_i(d_i) > 0 else 0, with a status bit;
  d_i outside [0, V): a_i = 0 (rejected), with a status bit;
  residual mass 0 after a rejection: sample from p_n, with a status bit;
  a row holding NaN or +inf, or only -inf: status bit, outputs undefined
  (but in range);
* greedy argmax ties go to the lowest index;
* q supplied as the draft's logits: q_i is the draft row transformed exactly
  as p_i (temperature, then top-k / top-p); a row with no distribution gives
  q_i = 0; a final draw within QLOGITS_CDF_BAND of a CDF step is a boundary
  draw (the step forms q in float32).

Parity pins (tests/test_oracle_*.py): the worked example of [Ch11.1] §11.1.3,
the exact output law of the §11.1.3 proof by brute-force enumeration on tiny
inputs, chi-square tests of distribution preservation, the E[N] closed form of
[SD-notes] and its worked numbers in the lmnt.cn blog §2.3 by Monte Carlo,
gamma = 0 against a library inverse CDF of scipy's softmax, greedy against
numpy.argmax, brute-force properties of top-k / top-p, the closed forms of a
one-hot q and of ragged rounds, and for q from draft logits: constant rows
(uniforms), shift invariance, scipy's softmax fed to the plain step, and q = p
accepting every draft.
"""

from __future__ import annotations

import numpy as np

# Per-sequence status bits.  The same values are stated in include/specverify.h;
# they are written here independently (no shared source).
SEQ_DRAFT_OUT_OF_RANGE = 1
SEQ_Q_NOT_POSITIVE = 2
SEQ_BAD_ROW = 4
SEQ_RESIDUAL_ZERO = 8

# A draw whose uniform lies this close to an acceptance threshold or to a CDF
# step (or a top-p cumulative sum this close to top_p) is a "boundary draw":
# a float32 implementation may legitimately decide it the other way.
BOUNDARY_EPS = 1e-6


def _f32(x) -> float:
    """The exact float64 value of x rounded to float32 (how the step receives
    temperature, top_p and the uniforms)."""
    return float(np.float32(x))


def row_is_bad(row) -> bool:
    """A row with a NaN or +inf logit, or with no finite logit at all, defines
    no distribution."""
    L = np.asarray(row, dtype=np.float64)
    return bool(np.isnan(L).any() or np.isposinf(L).any() or np.isneginf(L).all())


def truncation_keep_set(row, temperature, top_k=0, top_p=1.0):
    """Indices kept by top-k then top-p ([Ch11.1] §11.1.2: temperature,
    top-k / top-p are applied before verification).

    Returns (kept_indices in ranking order, top_p_boundary flag).  With no
    truncation every index is kept, in index order.
    """
    L = np.asarray(row, dtype=np.float64)
    V = L.shape[0]
    T = _f32(temperature)
    tp = _f32(top_p)
    k = V if top_k <= 0 else min(int(top_k), V)
    if k == V and tp >= 1.0:
        return np.arange(V), False
    # rank by (logit descending, index ascending); dividing by T > 0 keeps the order
    order = np.lexsort((np.arange(V), -L))
    kept = order[:k]
    boundary = False
    if tp < 1.0:
        z = L[kept] / T
        w = np.exp(z - z.max())
        pk = w / w.sum()                      # renormalised top-k distribution
        cum = np.cumsum(pk)
        reach = np.nonzero(cum >= tp)[0]
        J = int(reach[0]) + 1 if reach.size else k
        boundary = bool(np.any(np.abs(cum - tp) < BOUNDARY_EPS))
        kept = kept[:J]
    return kept, boundary


def target_distribution(row, temperature, top_k=0, top_p=1.0):
    """p = softmax(logits / T) over the kept set, zero elsewhere.

    [Ch11.1] §11.1.2 ("p_i is the target's actual sampling distribution, after
    temperature, top-k / top-p"); softmax of logits / temperature as in the
    lmnt.cn blog §3.3.  Returns (p float64 [V], bad_row, top_p_boundary).
    """
    L = np.asarray(row, dtype=np.float64)
    V = L.shape[0]
    if row_is_bad(L):
        return np.zeros(V), True, False
    kept, boundary = truncation_keep_set(L, temperature, top_k, top_p)
    z = L[kept] / _f32(temperature)
    w = np.exp(z - z.max())
    p = np.zeros(V)
    p[kept] = w / w.sum()
    return p, False, boundary


def accept_probability(p_d: float, q_d: float):
    """a = min(1, p(d) / q(d))  ([SD-notes] speculative sampling; [Ch11.1]
    §11.1.2).  Returns (a, q_not_positive flag)."""
    if not (q_d > 0.0):
        return (1.0 if p_d > 0.0 else 0.0), True
    return min(1.0, p_d / q_d), False


def residual(p, q):
    """Unnormalised residual r(v) = max(p(v) - q(v), 0)  ([Ch11.1] §11.1.2;
    [SD-notes] norm(max(0, p - q)))."""
    return np.maximum(np.asarray(p, np.float64) - np.asarray(q, np.float64), 0.0)


def inverse_cdf(weights, u):
    """Categorical draw from unnormalised weights with one uniform u in [0,1):
    the smallest v with C(v) > u * R, C the running sum in index order and
    R = C(V-1).  Returns (v, boundary flag)."""
    r = np.asarray(weights, dtype=np.float64)
    C = np.cumsum(r)
    R = C[-1]
    t = _f32(u) * R
    hit = np.nonzero(C > t)[0]
    if hit.size:
        v = int(hit[0])
    else:
        nz = np.nonzero(r > 0.0)[0]
        v = int(nz[-1]) if nz.size else 0
    lower, upper = C[v] - r[v], C[v]
    boundary = bool(abs(t - lower) < BOUNDARY_EPS * R or abs(upper - t) < BOUNDARY_EPS * R)
    return v, boundary


def deterministic_proposal(draft, V):
    """q of a deterministic draft (n-gram / prompt lookup, [SD-notes] notes an
    arbitrary drafting model M_q; [Ch11.1] §11.1.2 asks for the draft's actual
    q): all mass on the drafted token, q_i = one-hot(d_i).  An out-of-range
    draft gets no mass anywhere."""
    draft = np.asarray(draft, dtype=np.int64)
    B, G = draft.shape
    q = np.zeros((B, G, V))
    for b in range(B):
        for i in range(G):
            if 0 <= draft[b, i] < V:
                q[b, i, draft[b, i]] = 1.0
    return q


def verify_sample(logits, q, draft, uniforms, temperature, top_k=0, top_p=1.0):
    """The sampling verify step for a batch, following listing 10-1 of [Ch11.1].

    logits   [B, gamma+1, V]  target logits (any float dtype holding the exact
                              values), row i predicts d_{i+1} (§11.1.1)
    q        [B, gamma, V]    the draft's actual proposal probabilities, or None
                              for a deterministic draft (q_i = one-hot at d_i)
    draft    [B, gamma]       drafted token ids
    uniforms [B, gamma+1]     U[b, i] accept test i, U[b, gamma] final draw

    Returns a dict of numpy arrays: out_tokens [B, gamma+1] (-1 padded),
    n_accepted [B], accept_prob [B, gamma], status [B], boundary [B] (True
    where any evaluated draw lay within BOUNDARY_EPS of a decision boundary)
    and residual_mass [B] (R = sum max(p_n - q_n, 0) after a rejection, 1 for
    the bonus draw; reported so that a comparison can tell a rejection whose
    residual is zero only through rounding).
    """
    logits = np.asarray(logits)
    B, G1, V = logits.shape
    gamma = G1 - 1
    draft = np.asarray(draft, dtype=np.int64).reshape(B, gamma)
    if gamma == 0:
        q = np.zeros((B, 0, V))
    elif q is None:
        q = deterministic_proposal(draft, V)
    else:
        q = np.asarray(q)
    uniforms = np.asarray(uniforms, dtype=np.float32).reshape(B, G1)

    out = np.full((B, G1), -1, dtype=np.int64)
    n_acc = np.zeros(B, dtype=np.int64)
    acc_prob = np.zeros((B, gamma), dtype=np.float64)
    status = np.zeros(B, dtype=np.int64)
    boundary = np.zeros(B, dtype=bool)
    rmass = np.ones(B, dtype=np.float64)

    for b in range(B):
        P = []
        for i in range(G1):
            p, bad, tb = target_distribution(logits[b, i], temperature, top_k, top_p)
            P.append(p)
            if bad:
                status[b] |= SEQ_BAD_ROW
            boundary[b] |= tb
        # acceptance probabilities of every drafted position
        for i in range(gamma):
            d = int(draft[b, i])
            if d < 0 or d >= V:
                status[b] |= SEQ_DRAFT_OUT_OF_RANGE
                acc_prob[b, i] = 0.0
                continue
            a, qbad = accept_probability(P[i][d], float(q[b, i, d]))
            acc_prob[b, i] = a
            if qbad:
                status[b] |= SEQ_Q_NOT_POSITIVE
        # sequential scan, stopping at the first rejection
        n = gamma
        for i in range(gamma):
            u = _f32(uniforms[b, i])
            if abs(u - acc_prob[b, i]) < BOUNDARY_EPS:
                boundary[b] = True
            if not (u < acc_prob[b, i]):
                n = i
                break
        # one final draw: residual after a rejection, else the bonus from p_gamma
        if n < gamma:
            r = residual(P[n], q[b, n])
            rmass[b] = r.sum()
            if not (r.sum() > 0.0):
                status[b] |= SEQ_RESIDUAL_ZERO
                r = P[n]
        else:
            r = P[gamma]
        if r.sum() > 0.0:
            tok, tb = inverse_cdf(r, uniforms[b, gamma])
        else:
            tok, tb = 0, False
        boundary[b] |= tb
        out[b, :n] = draft[b, :n]
        out[b, n] = tok
        n_acc[b] = n
    return dict(out_tokens=out, n_accepted=n_acc, accept_prob=acc_prob,
                status=status, boundary=boundary, residual_mass=rmass)


def first_argmax(row) -> int:
    """Lowest index holding the largest logit (exact comparison of values;
    -0.0 and +0.0 compare equal)."""
    L = np.asarray(row, dtype=np.float64)
    if np.isnan(L).any():
        return 0
    return int(np.nonzero(L == L.max())[0][0])


def verify_greedy(logits, draft):
    """Greedy verify ([Ch11.1] §11.1.2): accept while d_i == argmax p_i; at the
    first mismatch emit the target argmax and stop; if all gamma drafts match,
    emit argmax p_gamma.  Temperature, top-k and top-p do not move the argmax.

    Returns dict(out_tokens [B, gamma+1] (-1 padded), n_accepted [B], status [B]).
    """
    logits = np.asarray(logits)
    B, G1, V = logits.shape
    gamma = G1 - 1
    draft = np.asarray(draft, dtype=np.int64).reshape(B, gamma)
    out = np.full((B, G1), -1, dtype=np.int64)
    n_acc = np.zeros(B, dtype=np.int64)
    status = np.zeros(B, dtype=np.int64)
    for b in range(B):
        g = []
        for i in range(G1):
            if np.isnan(np.asarray(logits[b, i], np.float64)).any():
                status[b] |= SEQ_BAD_ROW
            g.append(first_argmax(logits[b, i]))
        for i in range(gamma):
            if not (0 <= draft[b, i] < V):
                status[b] |= SEQ_DRAFT_OUT_OF_RANGE
        n = gamma
        for i in range(gamma):
            if draft[b, i] != g[i]:
                n = i
                break
        out[b, :n] = draft[b, :n]
        out[b, n] = g[n]
        n_acc[b] = n
    return dict(out_tokens=out, n_accepted=n_acc, status=status)


def expected_tokens_per_round(alpha: float, gamma: int) -> float:
    """E[N] = (1 - alpha^(gamma+1)) / (1 - alpha)  ([SD-notes] E[N] equation;
    the lmnt.cn blog §2.3 works it out as 2.77 at alpha=0.7, gamma=4 and 3.20
    at gamma=8)."""
    if alpha == 1.0:
        return float(gamma + 1)
    return (1.0 - alpha ** (gamma + 1)) / (1.0 - alpha)


# ----------------------------------------------------------------- ragged rounds

def verify_sample_ragged(logits, q, draft, uniforms, temperature, gamma_b, top_k=0, top_p=1.0):
    """A ragged batch ([SD-notes] and the lmnt.cn blog §3.2 let gamma change
    from round to round, per sequence): sequence b drafted only gamma_b[b] <=
    gamma tokens.  Reading: b is then exactly the single-sequence step with
    gamma = gamma_b[b] on its first gamma_b[b] + 1 logit rows, gamma_b[b] q
    rows and drafts, and uniforms U[b, 0..gamma_b[b]] (U[b, gamma_b[b]] for
    the final draw).  Rows and drafts beyond gamma_b[b] are not read.  Outputs
    are padded to gamma + 1 with -1 (accept_prob with 0)."""
    logits = np.asarray(logits)
    B, G1, V = logits.shape
    gamma = G1 - 1
    draft = np.asarray(draft, dtype=np.int64).reshape(B, gamma)
    uniforms = np.asarray(uniforms, dtype=np.float32).reshape(B, G1)
    gamma_b = np.asarray(gamma_b, dtype=np.int64).reshape(B)
    out = np.full((B, G1), -1, dtype=np.int64)
    n_acc = np.zeros(B, dtype=np.int64)
    acc_prob = np.zeros((B, gamma), dtype=np.float64)
    status = np.zeros(B, dtype=np.int64)
    boundary = np.zeros(B, dtype=bool)
    rmass = np.ones(B, dtype=np.float64)
    for b in range(B):
        g = int(gamma_b[b])
        if not (0 <= g <= gamma):
            raise ValueError("gamma_b must lie in [0, gamma]")
        qb = None if q is None else np.asarray(q)[b:b + 1, :g]
        r = verify_sample(logits[b:b + 1, :g + 1], qb, draft[b:b + 1, :g], uniforms[b:b + 1, :g + 1],
                          temperature, top_k, top_p)
        out[b, :g + 1] = r["out_tokens"][0]
        n_acc[b] = r["n_accepted"][0]
        acc_prob[b, :g] = r["accept_prob"][0]
        status[b] = r["status"][0]
        boundary[b] = r["boundary"][0]
        rmass[b] = r["residual_mass"][0]
    return dict(out_tokens=out, n_accepted=n_acc, accept_prob=acc_prob, status=status, boundary=boundary,
                residual_mass=rmass)


def verify_greedy_ragged(logits, draft, gamma_b):
    """Greedy verify of a ragged batch, with the same reading as
    verify_sample_ragged."""
    logits = np.asarray(logits)
    B, G1, V = logits.shape
    gamma = G1 - 1
    draft = np.asarray(draft, dtype=np.int64).reshape(B, gamma)
    gamma_b = np.asarray(gamma_b, dtype=np.int64).reshape(B)
    out = np.full((B, G1), -1, dtype=np.int64)
    n_acc = np.zeros(B, dtype=np.int64)
    status = np.zeros(B, dtype=np.int64)
    for b in range(B):
        g = int(gamma_b[b])
        if not (0 <= g <= gamma):
            raise ValueError("gamma_b must lie in [0, gamma]")
        r = verify_greedy(logits[b:b + 1, :g + 1], draft[b:b + 1, :g])
        out[b, :g + 1] = r["out_tokens"][0]
        n_acc[b] = r["n_accepted"][0]
        status[b] = r["status"][0]
    return dict(out_tokens=out, n_accepted=n_acc, status=status)


def truncate_emitted(out_tokens, n_accepted, stop_tokens=(), max_new=None):
    """End a round early ([Ch11.1] listing 10-1's comment: EOS / stop tokens
    and max_new_tokens may end the round, and no bonus is forced): the round
    emitted out_tokens[b, :n_b + 1]; keep them up to and including the first
    stop token, and at most max_new[b] of them.  Returns (tokens [B, gamma+1]
    with -1 after the cut, num_emitted [B])."""
    tok = np.array(out_tokens, dtype=np.int64, copy=True)
    n = np.asarray(n_accepted, dtype=np.int64)
    B, G1 = tok.shape
    stops = set(int(s) for s in stop_tokens)
    emitted = np.zeros(B, dtype=np.int64)
    for b in range(B):
        k = int(n[b]) + 1
        for j in range(k):
            if int(tok[b, j]) in stops:
                k = j + 1
                break
        if max_new is not None:
            k = min(k, max(int(max_new[b]), 0))
        tok[b, k:] = -1
        emitted[b] = k
    return tok, emitted


# An absolute band on the final draw's CDF steps for q formed from the
# draft's logits: the step materialises q in float32 (relative error of each
# q(v) a few 1e-7, so sum_v |dq(v)| < 1e-6), and the residual max(p - q, 0)
# moves by no more than q does.
QLOGITS_CDF_BAND = 1e-6


def draft_proposal_from_logits(q_logits, temperature, top_k=0, top_p=1.0):
    """q_i from the draft model's logits, transformed exactly as the target's
    ([Ch11.1] §11.1.2: temperature and top-k / top-p are applied to p_i and
    q_i alike, and q must be the draft's actual proposal).

    q_logits [B, gamma, V].  Returns (q float64 [B, gamma, V], top_p_boundary
    [B, gamma]).  A draft row that defines no distribution (NaN, +inf, only
    -inf) gives q_i = 0 everywhere, so its q_i(d_i) <= 0.
    """
    Q = np.asarray(q_logits, dtype=np.float64)
    B, G, V = Q.shape
    q = np.zeros((B, G, V))
    tb = np.zeros((B, G), dtype=bool)
    for b in range(B):
        for i in range(G):
            qi, _bad, bd = target_distribution(Q[b, i], temperature, top_k, top_p)
            q[b, i] = qi
            tb[b, i] = bd
    return q, tb


def verify_sample_qlogits(logits, q_logits, draft, uniforms, temperature, top_k=0, top_p=1.0):
    """The sampling verify step with the draft's proposal supplied as its
    logits: q_i = the truncated softmax of q_logits_i / T (the same transform
    as p_i), then the step of verify_sample.  The boundary flag also marks a
    final draw whose u * R lies within QLOGITS_CDF_BAND (absolute, in
    probability units) of the drawn token's CDF step."""
    q, qtb = draft_proposal_from_logits(q_logits, temperature, top_k, top_p)
    r = verify_sample(logits, q, draft, uniforms, temperature, top_k, top_p)
    L = np.asarray(logits)
    B, G1, V = L.shape
    gamma = G1 - 1
    U = np.asarray(uniforms, dtype=np.float32).reshape(B, G1)
    # reported separately: the sequences flagged only by the bands this
    # function adds (not by the 1e-6 bands of verify_sample)
    plain = r["boundary"].copy()
    for b in range(B):
        r["boundary"][b] |= bool(qtb[b].any())
        if r["status"][b] & SEQ_BAD_ROW:
            continue
        n = int(r["n_accepted"][b])
        p_n, _, _ = target_distribution(L[b, n], temperature, top_k, top_p)
        w = residual(p_n, q[b, n]) if n < gamma else p_n
        if not (w.sum() > 0.0):
            w = p_n
        C = np.cumsum(w)
        t = _f32(U[b, gamma]) * C[-1]
        v = int(r["out_tokens"][b, n])
        lower, upper = C[v] - w[v], C[v]
        if abs(t - lower) < QLOGITS_CDF_BAND or abs(upper - t) < QLOGITS_CDF_BAND:
            r["boundary"][b] = True
    r["qlogits_band_only"] = r["boundary"] & ~plain
    return r
