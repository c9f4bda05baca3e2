"""Statistical pins of the CPU oracle.

* Distribution preservation ("11.1 核心原理" §11.1.3; "Fast Inference from
  Transformers via Speculative Decoding" notes): with d_i ~ q_i drawn by the
  harness, the first emitted token follows p_0 and, after an accepted first
  draft, the second emitted token follows p_1 (chi-square, p-value > 1e-3).
  The planted biased variant (resample from p after a rejection) must fail.
* Accepted-count law: E[N] = (1 - alpha^(gamma+1)) / (1 - alpha) (the notes'
  E[N] equation; 2.77 / 3.20 in the lmnt.cn blog §2.3) by Monte Carlo, with
  p = (alpha, 1 - alpha) and q = (1, 0) so that every position accepts with
  probability alpha; and its per-row form 1 + sum_k prod_{i<k} beta_i,
  beta_i = sum_v min(p_i(v), q_i(v)), for independent synthetic rows.
"""

import numpy as np
import pytest
import scipy.special
import scipy.stats

from oracle import svref


def _first_two_token_pvalues(seed, V, G=2, B=20000, T=1.0, same_rows=True):
    rng = np.random.default_rng(seed)
    row = rng.normal(0, 1.2, size=(G + 1, V))
    qrow = rng.dirichlet(np.ones(V) * 0.5, size=G).astype(np.float32)
    L = np.broadcast_to(row, (B, G + 1, V)).copy()
    q = np.broadcast_to(qrow, (B, G, V)).copy()
    qn = qrow.astype(np.float64) / qrow.astype(np.float64).sum(-1, keepdims=True)
    draft = np.stack([rng.choice(V, size=B, p=qn[i]) for i in range(G)], 1)
    us = rng.random((B, G + 1)).astype(np.float32)
    res = svref.verify_sample(L, q, draft, us, T)
    P = [scipy.special.softmax(row[i] / T) for i in range(G + 1)]
    first = np.bincount(res["out_tokens"][:, 0], minlength=V)
    p1 = scipy.stats.chisquare(first, B * P[0]).pvalue
    sel = res["n_accepted"] >= 1
    second = np.bincount(res["out_tokens"][sel, 1], minlength=V)
    p2 = scipy.stats.chisquare(second, sel.sum() * P[1]).pvalue
    return p1, p2


@pytest.mark.parametrize("V,seed", [(2, 100), (4, 101), (8, 102)])
def test_chi_square_emitted_tokens_follow_target(V, seed):
    p1, p2 = _first_two_token_pvalues(seed, V)
    assert p1 > 1e-3 and p2 > 1e-3, (p1, p2)


def test_chi_square_catches_biased_resample(monkeypatch):
    monkeypatch.setattr(svref, "residual", lambda p, q: np.asarray(p, np.float64))
    p1, _ = _first_two_token_pvalues(100, 4)
    assert p1 < 1e-6


@pytest.mark.parametrize("alpha,gamma", [(0.7, 4), (0.7, 8), (0.3, 4)])
def test_expected_tokens_monte_carlo(alpha, gamma):
    rng = np.random.default_rng(int(alpha * 100) + gamma)
    B = 20000
    L = np.broadcast_to(np.log([alpha, 1 - alpha]), (B, gamma + 1, 2)).copy()
    q = np.zeros((B, gamma, 2), np.float32)
    q[:, :, 0] = 1.0
    draft = np.zeros((B, gamma), int)
    us = rng.random((B, gamma + 1)).astype(np.float32)
    res = svref.verify_sample(L, q, draft, us, 1.0)
    np.testing.assert_allclose(res["accept_prob"], alpha, rtol=1e-12)
    emitted = res["n_accepted"] + 1
    e = svref.expected_tokens_per_round(alpha, gamma)
    se = emitted.std(ddof=1) / np.sqrt(B)
    assert abs(emitted.mean() - e) < 4 * se, (emitted.mean(), e, se)


def test_expected_tokens_per_row_overlap_law():
    rng = np.random.default_rng(200)
    B, G, V, T = 20000, 4, 6, 1.0
    row = rng.normal(0, 1.0, size=(G + 1, V))
    qrow = rng.dirichlet(np.ones(V), size=G).astype(np.float32)
    L = np.broadcast_to(row, (B, G + 1, V)).copy()
    q = np.broadcast_to(qrow, (B, G, V)).copy()
    qn = qrow.astype(np.float64) / qrow.astype(np.float64).sum(-1, keepdims=True)
    draft = np.stack([rng.choice(V, size=B, p=qn[i]) for i in range(G)], 1)
    us = rng.random((B, G + 1)).astype(np.float32)
    res = svref.verify_sample(L, q, draft, us, T)
    beta = [np.minimum(scipy.special.softmax(row[i] / T), qrow[i].astype(np.float64)).sum() for i in range(G)]
    e = 1.0 + sum(np.prod(beta[:k]) for k in range(1, G + 1))
    emitted = res["n_accepted"] + 1
    se = emitted.std(ddof=1) / np.sqrt(B)
    assert abs(emitted.mean() - e) < 4 * se, (emitted.mean(), e, se)
