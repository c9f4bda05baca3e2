"""Pins of the CPU oracle to things other than itself.

Each test checks the oracle against something the pages or the mathematics fix:
the worked example printed in "11.1 核心原理: Draft + Verify 与 Rejection
Sampling" §11.1.3, the exact output law that the same section proves
(brute-force enumeration on tiny inputs, integrating the uniforms exactly by
bisection on the oracle's own decisions), special cases that reduce to library
routines (scipy's softmax, numpy's searchsorted and argmax), and brute-force
properties of top-k / top-p.  The planted-mistake tests show that the pins
catch the biased "resample from p" variant and a dropped clamp.
"""

import itertools
import json
import math
import os

import numpy as np
import pytest
import scipy.special

from oracle import svref

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _load(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


# ---------------------------------------------------------------- worked example

def _worked_example_law(ex):
    """Run the full oracle step on the worked example (V = 2, gamma = 1) and
    integrate the first emitted token's law exactly: d is weighted by q and the
    two uniforms run over midpoint grids whose fractions are exact for a = 0.75."""
    p, q = np.array(ex["p"]), np.array(ex["q"], dtype=np.float32)
    N = 40
    grid = (np.arange(N) + 0.5) / N
    logits, qs, drafts, us, weights = [], [], [], [], []
    for d in range(2):
        for u0 in grid:
            for u1 in grid:
                logits.append([np.log(p), np.log(p)])
                qs.append([q])
                drafts.append([d])
                us.append([u0, u1])
                weights.append(float(q[d]) / (N * N))
    res = svref.verify_sample(np.array(logits), np.array(qs), np.array(drafts),
                              np.array(us, dtype=np.float32), 1.0)
    law = np.zeros(2)
    for w, tok in zip(weights, res["out_tokens"][:, 0]):
        law[tok] += w
    return law


def test_worked_example_pieces():
    ex = _load("worked_example_ch11_1_3.json")
    p_ref, q = np.array(ex["p"]), np.array(ex["q"])
    p, bad, _ = svref.target_distribution(np.log(p_ref), 1.0)
    assert not bad
    np.testing.assert_allclose(p, p_ref, rtol=0, atol=1e-15)
    a = [svref.accept_probability(p[d], q[d])[0] for d in range(2)]
    np.testing.assert_allclose(a, ex["accept_prob"], atol=1e-15)
    np.testing.assert_allclose(q * np.array(a), ex["accepted_mass"], atol=1e-15)
    r = svref.residual(p, q)
    assert r.sum() == pytest.approx(ex["rejection_prob"], abs=1e-15)
    np.testing.assert_allclose(r / r.sum(), ex["residual"], atol=1e-15)
    final = q * np.array(a) + r
    np.testing.assert_allclose(final, ex["final"], atol=1e-15)


def test_worked_example_end_to_end():
    ex = _load("worked_example_ch11_1_3.json")
    np.testing.assert_allclose(_worked_example_law(ex), ex["final"], atol=1e-12)


def test_worked_example_catches_biased_resample(monkeypatch):
    """Planted mistake: resample from p after a rejection (the variant the page
    shows is biased).  The same pin must then read the page's biased numbers."""
    ex = _load("worked_example_ch11_1_3.json")
    monkeypatch.setattr(svref, "residual", lambda p, q: np.asarray(p, np.float64))
    law = _worked_example_law(ex)
    np.testing.assert_allclose(law, ex["biased_final_if_resampled_from_p"], atol=1e-12)
    assert abs(law[0] - ex["final"][0]) > 0.1


def test_distribution_identity_min_plus_max():
    """§11.1.3: q(v) min(1, p(v)/q(v)) + max(p(v) - q(v), 0) = p(v) for every v,
    and the rejection mass equals 1 - sum min(p, q)."""
    rng = np.random.default_rng(1)
    for _ in range(2000):
        V = int(rng.integers(1, 9))
        p = rng.dirichlet(np.ones(V) * rng.uniform(0.2, 3))
        q = rng.dirichlet(np.ones(V) * rng.uniform(0.2, 3))
        a = np.array([svref.accept_probability(p[v], q[v])[0] for v in range(V)])
        r = svref.residual(p, q)
        np.testing.assert_allclose(q * a + r, p, rtol=0, atol=1e-15)
        assert r.sum() == pytest.approx(1.0 - np.minimum(p, q).sum(), abs=1e-14)


# ------------------------------------------------------------- exact output law

def _threshold(pred, lo=0.0, hi=1.0, iters=48):
    """sup{x in [lo, hi): pred(x)} for a predicate that is true below a single
    threshold (float32 uniforms, so 48 halvings are exact to the float grid)."""
    if not pred(lo):
        return lo
    if pred(np.nextafter(np.float32(hi), np.float32(0))):
        return hi
    for _ in range(iters):
        mid = 0.5 * (lo + hi)
        if pred(mid):
            lo = mid
        else:
            hi = mid
    return 0.5 * (lo + hi)


def _oracle_law(L, q, T):
    """Exact law of the emitted sequence of the oracle step, by enumerating
    every draft d ~ q and integrating the uniforms through the oracle's own
    decisions (acceptance is monotone in u_i, the token is monotone in u_gamma)."""
    G1, V = L.shape
    G = G1 - 1
    law = {}
    one_minus = float(np.nextafter(np.float32(1), np.float32(0)))

    def run(d, us):
        res = svref.verify_sample(L[None], q[None], np.array([d]),
                                  np.array([us], dtype=np.float32), T)
        return int(res["n_accepted"][0]), [int(t) for t in res["out_tokens"][0]]

    def accept_uniforms(n, x):
        # positions before n accept (u = 0 < a), position n tests x
        return [0.0] * n + [x] + [0.0] * (G - n)

    def final_uniforms(n, x):
        # positions before n accept, position n (if a draft) rejects, the final draw is x
        stop = [one_minus] if n < G else []
        return [0.0] * n + stop + [0.0] * (G - n - len(stop)) + [x]

    for d in itertools.product(range(V), repeat=G):
        wd = float(np.prod([q[i, d[i]] for i in range(G)])) if G else 1.0
        if wd == 0.0:
            continue
        reach = 1.0                       # P(positions 0..n-1 all accepted | d)
        for n in range(G1):
            if reach == 0.0:
                break
            a_n = _threshold(lambda x: run(d, accept_uniforms(n, x))[0] > n) if n < G else 0.0
            p_stop = 1.0 - a_n            # P(the round ends at n | reached n)
            if p_stop > 0.0:
                below = 0.0               # P(token <= v-1) over the final uniform
                for v in range(V):
                    upto = _threshold(lambda x: run(d, final_uniforms(n, x))[1][n] <= v)
                    if upto - below > 0.0:
                        key = tuple(d[:n]) + (v,)
                        law[key] = law.get(key, 0.0) + wd * reach * p_stop * (upto - below)
                    below = upto
            reach *= a_n
    return law


def _theorem_law(L, q, T):
    """The law that §11.1.3 proves: accepted prefix tokens carry min(p_i, q_i),
    a rejection at n emits from max(p_n - q_n, 0), full acceptance emits from
    p_gamma.  p_i here is scipy's softmax of logits / T."""
    G1, V = L.shape
    G = G1 - 1
    P = [scipy.special.softmax(L[i] / np.float64(np.float32(T))) for i in range(G1)]
    Q = q.astype(np.float64)
    law = {}
    for n in range(G1):
        for prefix in itertools.product(range(V), repeat=n):
            w = 1.0
            for i, v in enumerate(prefix):
                w *= min(P[i][v], Q[i, v])
            for t in range(V):
                last = max(P[n][t] - Q[n, t], 0.0) if n < G else P[G][t]
                if w * last > 0:
                    law[prefix + (t,)] = w * last
    return law


@pytest.mark.parametrize("V,G,T,seed", [(2, 1, 1.0, 0), (3, 1, 0.7, 1), (2, 2, 1.3, 2), (3, 2, 1.0, 3)])
def test_exact_output_law_bruteforce(V, G, T, seed):
    rng = np.random.default_rng(seed)
    L = rng.normal(0, 1.5, size=(G + 1, V))
    q = rng.dirichlet(np.ones(V), size=G).astype(np.float32)
    law = _oracle_law(L, q, T)
    ref = _theorem_law(L, q, T)
    keys = set(law) | set(ref)
    for k in keys:
        assert law.get(k, 0.0) == pytest.approx(ref.get(k, 0.0), abs=2e-6), k
    assert sum(law.values()) == pytest.approx(1.0, abs=1e-6)
    # losslessness: the first emitted token is distributed as p_0
    first = np.zeros(V)
    for k, m in law.items():
        first[k[0]] += m
    np.testing.assert_allclose(first, scipy.special.softmax(L[0] / np.float64(np.float32(T))), atol=2e-6)


def test_exact_law_catches_dropped_clamp(monkeypatch):
    """Planted mistake: residual without the max(., 0) clamp."""
    rng = np.random.default_rng(7)
    L = rng.normal(0, 1.5, size=(2, 3))
    q = rng.dirichlet(np.ones(3), size=1).astype(np.float32)
    ref = _theorem_law(L, q, 1.0)
    monkeypatch.setattr(svref, "residual", lambda p, qq: np.asarray(p, np.float64) - np.asarray(qq, np.float64))
    law = _oracle_law(L, q, 1.0)
    err = max(abs(law.get(k, 0.0) - ref.get(k, 0.0)) for k in set(law) | set(ref))
    assert err > 1e-3


def test_exact_law_catches_misaligned_bonus_row(monkeypatch):
    """Planted mistake: the bonus drawn from row gamma-1 instead of row gamma."""
    rng = np.random.default_rng(11)
    L = rng.normal(0, 1.5, size=(2, 3))
    q = rng.dirichlet(np.ones(3), size=1).astype(np.float32)
    ref = _theorem_law(L, q, 1.0)
    orig = svref.target_distribution

    def shifted(row, *a, **k):
        return orig(L[0] if np.array_equal(np.asarray(row, np.float64), L[1]) else row, *a, **k)

    monkeypatch.setattr(svref, "target_distribution", shifted)
    law = _oracle_law(L, q, 1.0)
    err = max(abs(law.get(k, 0.0) - ref.get(k, 0.0)) for k in set(law) | set(ref))
    assert err > 1e-3


# ------------------------------------------------------------ special cases

def test_gamma0_is_library_inverse_cdf_of_softmax():
    """gamma = 0: the step samples the bonus token from softmax(logits / T)
    with one uniform; compare with scipy's softmax and numpy's searchsorted."""
    rng = np.random.default_rng(3)
    for _ in range(300):
        V = int(rng.integers(1, 300))
        T = float(np.float32(rng.uniform(0.3, 2.0)))
        L = rng.normal(0, 3, size=V).astype(np.float32)
        u = np.float32(rng.random())
        p, bad, _ = svref.target_distribution(L, T)
        ref = scipy.special.softmax(L.astype(np.float64) / T)
        np.testing.assert_allclose(p, ref, rtol=1e-12, atol=1e-300)
        res = svref.verify_sample(L[None, None, :], None, np.zeros((1, 0), int),
                                  np.array([[u]], np.float32), T)
        C = np.cumsum(ref)
        tok_ref = int(np.searchsorted(C, float(u) * C[-1], side="right"))
        if not res["boundary"][0]:
            assert res["out_tokens"][0, 0] == min(tok_ref, V - 1)
        assert res["n_accepted"][0] == 0


def _argmax_rows(rng, n, V, ties):
    L = rng.normal(0, 1, size=(n, V)).astype(np.float32)
    if ties:
        L = np.round(L * 2) / 2          # many exact ties
    return L


def test_greedy_matches_numpy_argmax_with_ties():
    rng = np.random.default_rng(4)
    for V in (1, 2, 5, 64, 1000):
        L = _argmax_rows(rng, 200, V, ties=True)
        for row in L:
            assert svref.first_argmax(row) == int(np.argmax(row))
    # -0.0 and +0.0 are the same value: the lower index wins
    assert svref.first_argmax(np.array([-1.0, -0.0, 0.0], np.float32)) == 1


def test_greedy_reproduces_target_greedy_path():
    """lmnt.cn blog §4.3 (check greedy equality with plain decoding first):
    every emitted token is the target argmax of its row, the accepted prefix is
    exactly the drafts that equal those argmaxes."""
    rng = np.random.default_rng(5)
    B, G, V = 300, 4, 37
    L = _argmax_rows(rng, B * (G + 1), V, ties=True).reshape(B, G + 1, V)
    g = L.argmax(-1)
    draft = np.where(rng.random((B, G)) < 0.6, g[:, :G], rng.integers(0, V, (B, G)))
    res = svref.verify_greedy(L, draft)
    for b in range(B):
        n = res["n_accepted"][b]
        assert np.all(draft[b, :n] == g[b, :n])
        assert n == G or draft[b, n] != g[b, n]
        assert np.all(res["out_tokens"][b, : n + 1] == g[b, : n + 1])
        assert np.all(res["out_tokens"][b, n + 1:] == -1)


def test_topk1_sampling_equals_greedy():
    rng = np.random.default_rng(6)
    B, G, V = 200, 3, 50
    L = _argmax_rows(rng, B * (G + 1), V, ties=True).reshape(B, G + 1, V)
    q = rng.dirichlet(np.ones(V), size=(B, G)).astype(np.float32)
    g = L.argmax(-1)
    draft = np.where(rng.random((B, G)) < 0.5, g[:, :G], rng.integers(0, V, (B, G)))
    us = rng.random((B, G + 1)).astype(np.float32)
    s = svref.verify_sample(L, q, draft, us, 0.9, top_k=1)
    gr = svref.verify_greedy(L, draft)
    np.testing.assert_array_equal(s["out_tokens"], gr["out_tokens"])
    np.testing.assert_array_equal(s["n_accepted"], gr["n_accepted"])


def test_q_equal_p_accepts_everything():
    rng = np.random.default_rng(8)
    B, G, V = 100, 5, 40
    T = 0.8
    L = rng.normal(0, 2, size=(B, G + 1, V))
    q = scipy.special.softmax(L[:, :G] / np.float64(np.float32(T)), axis=-1)
    draft = np.array([[rng.choice(V, p=q[b, i]) for i in range(G)] for b in range(B)])
    us = (rng.random((B, G + 1)) * 0.999).astype(np.float32)
    res = svref.verify_sample(L, q, draft, us, T)
    assert np.all(res["n_accepted"] == G)
    np.testing.assert_allclose(res["accept_prob"], 1.0, atol=1e-12)


def test_disjoint_supports_reject_first_and_sample_p():
    """p lives on tokens {0, 1}, q on {2, 3}: every draft is rejected at once and
    the residual is p itself, so the first token follows p_0."""
    rng = np.random.default_rng(9)
    B, G, V = 400, 2, 4
    L = np.full((B, G + 1, V), -np.inf)
    L[:, :, :2] = rng.normal(0, 1, size=(B, G + 1, 2))
    q = np.zeros((B, G, V), np.float32)
    q[:, :, 2:] = rng.dirichlet(np.ones(2), size=(B, G))
    draft = rng.integers(2, 4, size=(B, G))
    us = rng.random((B, G + 1)).astype(np.float32)
    res = svref.verify_sample(L, q, draft, us, 1.0)
    assert np.all(res["n_accepted"] == 0)
    assert np.all(res["accept_prob"] == 0.0)
    for b in range(B):
        p0 = scipy.special.softmax(L[b, 0, :2])
        tok = int(np.searchsorted(np.cumsum(p0), float(us[b, G]) * np.cumsum(p0)[-1], side="right"))
        if not res["boundary"][b]:
            assert res["out_tokens"][b, 0] == tok


# ------------------------------------------------------------ truncation

def test_topk_keep_set_bruteforce():
    """Exactly min(k, V) tokens are kept; each kept logit >= each dropped one;
    among tokens tied with the k-th kept value, the kept ones have the lower
    indices (ties broken by index)."""
    rng = np.random.default_rng(10)
    for _ in range(500):
        V = int(rng.integers(1, 30))
        k = int(rng.integers(1, V + 3))
        L = np.round(rng.normal(0, 1, size=V) * 2) / 2
        kept, _ = svref.truncation_keep_set(L, 1.0, top_k=k)
        assert len(kept) == min(k, V) and len(set(kept.tolist())) == len(kept)
        dropped = np.setdiff1d(np.arange(V), kept)
        if dropped.size:
            kmin = L[kept].min()
            assert np.all(L[dropped] <= kmin)
            tied_kept = kept[L[kept] == kmin]
            tied_drop = dropped[L[dropped] == kmin]
            if tied_drop.size:
                assert tied_kept.max() < tied_drop.min()


def test_topp_shortest_prefix_bruteforce():
    """top-p keeps the shortest prefix of the (logit desc, index asc) ranking
    whose renormalised top-k mass reaches top_p, checked against every prefix."""
    rng = np.random.default_rng(12)
    for _ in range(500):
        V = int(rng.integers(1, 12))
        k = int(rng.integers(0, V + 1))
        tp = float(np.float32(rng.uniform(0.05, 0.999)))
        T = float(np.float32(rng.uniform(0.5, 1.5)))
        L = np.round(rng.normal(0, 1, size=V) * 4) / 4
        kept, boundary = svref.truncation_keep_set(L, T, top_k=k, top_p=tp)
        if boundary:
            continue
        kk = V if k == 0 else min(k, V)
        ranked = sorted(range(V), key=lambda v: (-L[v], v))[:kk]
        w = np.exp(L[ranked] / T - np.max(L[ranked] / T))
        pk = w / w.sum()
        masses = [pk[:j].sum() for j in range(1, kk + 1)]
        J = next((j + 1 for j, m in enumerate(masses) if m >= tp), kk)
        assert list(kept) == ranked[:J]


def test_tiny_top_p_is_greedy():
    rng = np.random.default_rng(13)
    B, G, V = 100, 3, 20
    L = np.round(rng.normal(0, 1, size=(B, G + 1, V)) * 2) / 2
    q = rng.dirichlet(np.ones(V), size=(B, G)).astype(np.float32)
    g = L.argmax(-1)
    draft = np.where(rng.random((B, G)) < 0.5, g[:, :G], rng.integers(0, V, (B, G)))
    us = rng.random((B, G + 1)).astype(np.float32)
    s = svref.verify_sample(L, q, draft, us, 1.0, top_k=0, top_p=1e-7)
    gr = svref.verify_greedy(L, draft)
    np.testing.assert_array_equal(s["out_tokens"], gr["out_tokens"])


def test_no_truncation_when_k_covers_vocab():
    rng = np.random.default_rng(14)
    L = rng.normal(0, 2, size=33)
    p_full, _, _ = svref.target_distribution(L, 0.7)
    p_k, _, _ = svref.target_distribution(L, 0.7, top_k=33)
    np.testing.assert_allclose(p_full, p_k, atol=1e-16)
    np.testing.assert_allclose(p_full, scipy.special.softmax(L / np.float64(np.float32(0.7))), rtol=1e-12)


# ------------------------------------------------------------ status bits / edges

def test_status_flags_and_ranges():
    V, G = 5, 3
    L = np.zeros((4, G + 1, V))
    L[1, 2, 3] = np.nan
    L[2, 0, :] = -np.inf
    q = np.full((4, G, V), 0.2, np.float32)
    q[3, 0, :] = 0.0
    draft = np.array([[0, 7, 1], [0, 1, 2], [1, 1, 1], [2, 2, 2]])
    us = np.full((4, G + 1), 0.5, np.float32)
    res = svref.verify_sample(L, q, draft, us, 1.0)
    assert res["status"][0] & svref.SEQ_DRAFT_OUT_OF_RANGE
    assert res["accept_prob"][0, 1] == 0.0
    assert res["status"][1] & svref.SEQ_BAD_ROW
    assert res["status"][2] & svref.SEQ_BAD_ROW
    assert res["status"][3] & svref.SEQ_Q_NOT_POSITIVE
    assert res["accept_prob"][3, 0] == 1.0
    assert np.all((res["out_tokens"] >= -1) & (res["out_tokens"] < V))
    gr = svref.verify_greedy(L, draft)
    assert gr["status"][0] & svref.SEQ_DRAFT_OUT_OF_RANGE
    assert gr["status"][1] & svref.SEQ_BAD_ROW
    assert np.all((gr["out_tokens"] >= -1) & (gr["out_tokens"] < V))


def test_emitted_counts_between_one_and_gamma_plus_one():
    """[SD-notes]: a round emits at least one and at most gamma + 1 tokens."""
    rng = np.random.default_rng(15)
    B, G, V = 200, 4, 16
    L = rng.normal(0, 1, size=(B, G + 1, V))
    q = rng.dirichlet(np.ones(V), size=(B, G)).astype(np.float32)
    draft = np.array([[rng.choice(V, p=q[b, i] / q[b, i].sum()) for i in range(G)] for b in range(B)])
    us = rng.random((B, G + 1)).astype(np.float32)
    res = svref.verify_sample(L, q, draft, us, 1.0)
    emitted = (res["out_tokens"] >= 0).sum(1)
    assert np.all(emitted == res["n_accepted"] + 1)
    assert np.all((emitted >= 1) & (emitted <= G + 1))
    for b in range(B):
        n = res["n_accepted"][b]
        assert np.all(res["out_tokens"][b, :n] == draft[b, :n])


def test_expected_tokens_closed_form_matches_blog_numbers():
    gold = _load("expected_tokens_per_round_blog_2_3.json")
    for c in gold["cases"]:
        e = svref.expected_tokens_per_round(c["alpha"], c["gamma"])
        assert round(e, gold["decimals"]) == pytest.approx(c["expected_tokens"], abs=1e-12)
        # and the geometric series it sums: 1 + alpha + ... + alpha^gamma
        assert e == pytest.approx(sum(c["alpha"] ** j for j in range(c["gamma"] + 1)), rel=1e-14)
    assert not math.isclose(svref.expected_tokens_per_round(0.7, 4), 1 + 0.7 * 4)


# ------------------------------------------------- deterministic drafts (q = None)

def _oracle_law_deterministic(L, d, T):
    """Exact law of the emitted sequence for one fixed deterministic draft d
    (q passed as None), by integrating the uniforms through the oracle."""
    G1, V = L.shape
    G = G1 - 1
    law = {}
    one_minus = float(np.nextafter(np.float32(1), np.float32(0)))

    def run(us):
        res = svref.verify_sample(L[None], None, np.array([d]), np.array([us], dtype=np.float32), T)
        return int(res["n_accepted"][0]), [int(t) for t in res["out_tokens"][0]]

    reach = 1.0
    for n in range(G1):
        a_n = _threshold(lambda x: run([0.0] * n + [x] + [0.0] * (G - n))[0] > n) if n < G else 0.0
        p_stop = 1.0 - a_n
        if p_stop > 0.0:
            stop = [one_minus] if n < G else []
            below = 0.0
            for v in range(V):
                us = lambda x: [0.0] * n + stop + [0.0] * (G - n - len(stop)) + [x]
                upto = _threshold(lambda x: run(us(x))[1][n] <= v)
                if upto - below > 0.0:
                    key = tuple(d[:n]) + (v,)
                    law[key] = law.get(key, 0.0) + reach * p_stop * (upto - below)
                below = upto
        reach *= a_n
    return law


@pytest.mark.parametrize("V,G,T,seed", [(3, 1, 1.0, 5), (4, 2, 0.8, 6), (3, 3, 1.2, 7)])
def test_deterministic_draft_law_closed_form(V, G, T, seed):
    """q = one-hot(d_i): a_i = p_i(d_i) (min(1, p/1)), and a rejection at n
    draws from p_n with d_n removed, renormalised (max(p - onehot, 0))."""
    rng = np.random.default_rng(seed)
    L = rng.normal(0, 1.5, size=(G + 1, V))
    d = [int(x) for x in rng.integers(0, V, size=G)]
    P = [scipy.special.softmax(L[i] / np.float64(np.float32(T))) for i in range(G + 1)]
    ref = {}
    reach = 1.0
    for n in range(G + 1):
        if n < G:
            stop = 1.0 - P[n][d[n]]
            for v in range(V):
                if v != d[n] and P[n][v] > 0:
                    ref[tuple(d[:n]) + (v,)] = reach * stop * P[n][v] / (1.0 - P[n][d[n]])
            reach *= P[n][d[n]]
        else:
            for v in range(V):
                ref[tuple(d) + (v,)] = reach * P[G][v]
    law = _oracle_law_deterministic(L, d, T)
    for k in set(law) | set(ref):
        assert law.get(k, 0.0) == pytest.approx(ref.get(k, 0.0), abs=2e-6), k


def test_deterministic_draft_accept_prob_is_target_prob():
    rng = np.random.default_rng(11)
    B, G, V, T = 5, 3, 50, 0.9
    L = rng.normal(0, 2, size=(B, G + 1, V))
    d = rng.integers(0, V, size=(B, G))
    u = rng.random((B, G + 1)).astype(np.float32)
    r = svref.verify_sample(L, None, d, u, T)
    for b in range(B):
        for i in range(G):
            p = scipy.special.softmax(L[b, i] / np.float64(np.float32(T)))
            assert r["accept_prob"][b, i] == pytest.approx(p[d[b, i]], rel=1e-12)
    # a rejected position never re-emits its own draft
    for b in range(B):
        n = r["n_accepted"][b]
        if n < G:
            assert r["out_tokens"][b, n] != d[b, n]


# ------------------------------------------------------------- ragged rounds

def test_ragged_with_full_gamma_is_the_plain_step():
    rng = np.random.default_rng(21)
    B, G, V = 6, 4, 30
    L = rng.normal(0, 2, size=(B, G + 1, V))
    q = rng.dirichlet(np.ones(V), size=(B, G))
    d = np.array([[rng.choice(V, p=q[b, i]) for i in range(G)] for b in range(B)])
    u = rng.random((B, G + 1)).astype(np.float32)
    a = svref.verify_sample(L, q, d, u, 0.9)
    r = svref.verify_sample_ragged(L, q, d, u, 0.9, [G] * B)
    for k in ("out_tokens", "n_accepted", "status"):
        np.testing.assert_array_equal(a[k], r[k])
    np.testing.assert_allclose(a["accept_prob"], r["accept_prob"], rtol=0, atol=0)


@pytest.mark.parametrize("V,g,T,seed", [(3, 1, 1.0, 31), (2, 0, 0.8, 32), (3, 2, 1.1, 33)])
def test_ragged_sequence_law_is_the_theorem_law_for_its_gamma(V, g, T, seed):
    """One sequence of a batch padded to gamma = 3 that drafted only g tokens:
    its emitted law is the theorem's law for gamma = g on its first g + 1 rows
    (rows and uniforms beyond are filled with junk that must not matter)."""
    G = 3
    rng = np.random.default_rng(seed)
    L = rng.normal(0, 1.5, size=(G + 1, V))
    L[g + 1:] = rng.normal(0, 50, size=(G - g, V))          # junk rows beyond gamma_b
    q = rng.dirichlet(np.ones(V), size=G).astype(np.float32)
    law = {}
    one_minus = float(np.nextafter(np.float32(1), np.float32(0)))

    def run(d, us):
        res = svref.verify_sample_ragged(L[None], q[None], np.array([list(d) + [0] * (G - g)]),
                                         np.array([us + [0.5] * (G - g)], dtype=np.float32), T, [g])
        return int(res["n_accepted"][0]), [int(t) for t in res["out_tokens"][0]]

    for d in itertools.product(range(V), repeat=g):
        wd = float(np.prod([q[i, d[i]] for i in range(g)])) if g else 1.0
        reach = 1.0
        for n in range(g + 1):
            a_n = _threshold(lambda x: run(d, [0.0] * n + [x] + [0.0] * (g - n))[0] > n) if n < g else 0.0
            p_stop = 1.0 - a_n
            if p_stop > 0.0:
                stop = [one_minus] if n < g else []
                below = 0.0
                for v in range(V):
                    us = lambda x: [0.0] * n + stop + [0.0] * (g - n - len(stop)) + [x]
                    upto = _threshold(lambda x: run(d, us(x))[1][n] <= v)
                    if upto - below > 0.0:
                        key = tuple(d[:n]) + (v,)
                        law[key] = law.get(key, 0.0) + wd * reach * p_stop * (upto - below)
                    below = upto
            reach *= a_n
    ref = _theorem_law(L[:g + 1], q[:g], T)
    for k in set(law) | set(ref):
        assert law.get(k, 0.0) == pytest.approx(ref.get(k, 0.0), abs=2e-6), k


def test_ragged_ignores_rows_and_drafts_beyond_gamma_b():
    rng = np.random.default_rng(41)
    B, G, V = 4, 4, 20
    L = rng.normal(0, 1, size=(B, G + 1, V))
    q = rng.dirichlet(np.ones(V), size=(B, G))
    d = rng.integers(0, V, size=(B, G))
    u = rng.random((B, G + 1)).astype(np.float32)
    gb = np.array([2, 0, 4, 1])
    L2, d2 = L.copy(), d.copy()
    for b in range(B):
        L2[b, gb[b] + 1:] = np.nan          # would flag a bad row if read
        d2[b, gb[b]:] = V + 5              # would flag an out-of-range draft if read
    a = svref.verify_sample_ragged(L, q, d, u, 1.0, gb)
    r = svref.verify_sample_ragged(L2, q, d2, u, 1.0, gb)
    for k in ("out_tokens", "n_accepted", "status"):
        np.testing.assert_array_equal(a[k], r[k])
    assert np.all(r["status"] == 0)
    assert np.all(r["n_accepted"] <= gb)
    assert np.all(r["out_tokens"][np.arange(G + 1)[None, :] > gb[:, None]] == -1)
    g = svref.verify_greedy_ragged(L2, d2, gb)
    for b in range(B):
        gg = int(gb[b])
        best = [int(np.argmax(L[b, i])) for i in range(gg + 1)]
        n = next((i for i in range(gg) if d[b, i] != best[i]), gg)
        assert g["n_accepted"][b] == n
        assert list(g["out_tokens"][b, :n + 1]) == [int(x) for x in d[b, :n]] + [best[n]]
        assert g["status"][b] == 0


def test_truncate_emitted_is_the_longest_valid_prefix():
    """Brute force: the kept length is the largest k such that every kept
    token was emitted (k <= n + 1), no stop token precedes the k-th, and k <=
    max_new."""
    rng = np.random.default_rng(51)
    B, G = 200, 6
    tok = rng.integers(0, 8, size=(B, G + 1))
    n = rng.integers(0, G + 1, size=B)
    for b in range(B):
        tok[b, n[b] + 1:] = -1
    stops = [3, 6]
    max_new = rng.integers(0, G + 3, size=B)
    t, e = svref.truncate_emitted(tok, n, stops, max_new)
    for b in range(B):
        best = 0
        for k in range(0, G + 2):
            ok = k <= n[b] + 1 and k <= max_new[b] and all(tok[b, j] not in stops for j in range(max(k - 1, 0)))
            if ok:
                best = k
        assert e[b] == best, b
        assert list(t[b, :best]) == list(tok[b, :best]) and np.all(t[b, best:] == -1)
    # no stops and a large budget: nothing changes
    t2, e2 = svref.truncate_emitted(tok, n, (), None)
    np.testing.assert_array_equal(t2, tok)
    np.testing.assert_array_equal(e2, n + 1)


# ---------------------------------------------------------------- q as draft logits

def test_qlogits_constant_rows_give_closed_form_uniforms():
    """softmax of a constant row is uniform; top-k of a constant row keeps the k
    lowest indices (ties rank by index); top-p of a uniform keeps the shortest
    prefix reaching top_p, ceil(top_p * V) tokens."""
    B, G, V = 2, 3, 40
    Q = np.full((B, G, V), 1.75)
    q, tb = svref.draft_proposal_from_logits(Q, 0.7)
    assert np.allclose(q, 1.0 / V, rtol=0, atol=1e-15) and not tb.any()
    q, _ = svref.draft_proposal_from_logits(Q, 0.7, top_k=7)
    assert np.allclose(q[..., :7], 1.0 / 7, rtol=0, atol=1e-15) and np.all(q[..., 7:] == 0.0)
    q, _ = svref.draft_proposal_from_logits(Q, 1.3, top_p=0.5)
    J = math.ceil(np.float32(0.5) * V)
    assert np.allclose(q[..., :J], 1.0 / J, rtol=0, atol=1e-15) and np.all(q[..., J:] == 0.0)


def test_qlogits_shift_invariance():
    rng = np.random.default_rng(11)
    Q = rng.normal(size=(3, 2, 64)) * 3.0
    shift = rng.normal(size=(3, 2, 1)) * 50.0
    a, _ = svref.draft_proposal_from_logits(Q, 0.9, top_k=20, top_p=0.8)
    b, _ = svref.draft_proposal_from_logits(Q + shift, 0.9, top_k=20, top_p=0.8)
    assert np.allclose(a, b, rtol=1e-12, atol=1e-15)


@pytest.mark.parametrize("seed", range(4))
def test_qlogits_step_is_the_step_with_library_softmax_q(seed):
    """Untruncated: q_i = scipy.special.softmax(q_logits_i / T) fed to the plain
    step gives the same tokens and acceptance probabilities."""
    rng = np.random.default_rng(100 + seed)
    B, G, V, T = 6, 4, 30, 0.8
    L = rng.normal(size=(B, G + 1, V)) * 2.0
    Q = L[:, :G] + rng.normal(size=(B, G, V))
    d = rng.integers(0, V, size=(B, G))
    u = rng.random(size=(B, G + 1)).astype(np.float32)
    q_lib = scipy.special.softmax(Q / float(np.float32(T)), axis=-1)
    ref = svref.verify_sample(L, q_lib, d, u, T)
    got = svref.verify_sample_qlogits(L, Q, d, u, T)
    assert np.array_equal(got["out_tokens"], ref["out_tokens"])
    assert np.array_equal(got["n_accepted"], ref["n_accepted"])
    assert np.allclose(got["accept_prob"], ref["accept_prob"], rtol=1e-12, atol=0)


def test_qlogits_equal_to_target_logits_accept_every_draft():
    """q = p: every a_i = 1, so every draft is accepted and the bonus is the
    inverse CDF (numpy searchsorted) of scipy's softmax of row gamma."""
    rng = np.random.default_rng(7)
    B, G, V, T = 8, 3, 25, 1.1
    L = rng.normal(size=(B, G + 1, V)) * 1.5
    d = rng.integers(0, V, size=(B, G))
    u = rng.random(size=(B, G + 1)).astype(np.float32)
    r = svref.verify_sample_qlogits(L, L[:, :G].copy(), d, u, T)
    assert np.all(r["n_accepted"] == G)
    assert np.allclose(r["accept_prob"], 1.0, rtol=0, atol=1e-12)
    for b in range(B):
        pg = scipy.special.softmax(L[b, G] / float(np.float32(T)))
        tok = int(np.searchsorted(np.cumsum(pg), float(np.float32(u[b, G])) * pg.sum(), side="right"))
        assert r["out_tokens"][b, G] == min(tok, V - 1)
        assert np.array_equal(r["out_tokens"][b, :G], d[b])


def test_qlogits_bad_draft_row_is_a_zero_q():
    rng = np.random.default_rng(3)
    B, G, V = 2, 2, 16
    L = rng.normal(size=(B, G + 1, V))
    Q = rng.normal(size=(B, G, V))
    Q[0, 0, 5] = np.nan
    Q[1, 0, :] = -np.inf
    d = np.array([[1, 2], [3, 4]])
    u = np.full((B, G + 1), 0.5, dtype=np.float32)
    r = svref.verify_sample_qlogits(L, Q, d, u, 1.0)
    assert np.all(r["accept_prob"][:, 0] == 1.0)          # q_0(d_0) = 0 with p_0(d_0) > 0
    assert np.all(r["status"] & svref.SEQ_Q_NOT_POSITIVE)


def test_inverse_cdf_fallback_when_no_step_exceeds_the_target():
    """The branch where no running sum exceeds t = u R: all-zero weights draw
    index 0 (no mass anywhere); a target at the total (u = 1, outside the
    uniforms' range, the case rounding can reach) takes the last entry of
    positive mass, the same token as u just below 1, and skips trailing
    zero-weight entries."""
    assert svref.inverse_cdf([0.0, 0.0, 0.0], 0.5) == (0, False)
    w = [0.2, 0.5, 0.3, 0.0, 0.0]
    v_end, _ = svref.inverse_cdf(w, 1.0)
    v_below, _ = svref.inverse_cdf(w, float(np.float32(1.0) - np.float32(2.0 ** -24)))
    assert v_end == 2 and v_below == 2
    # the ordinary branch next to it: the smallest v whose running sum exceeds u R
    assert svref.inverse_cdf(w, 0.25)[0] == 1 and svref.inverse_cdf(w, 0.1)[0] == 0
