"""Statistical laws of speculative sampling, checked on the CPU oracle.

* Accepted-length law: with fixed rows, draft tokens drawn from q_i and fresh
  uniforms, ``P(n >= i) = prod_{j<i} alpha_j`` with
  ``alpha_j = sum_v min(phat_j(v), qhat_j(v))`` (spec-verify card, "Measured"
  and "Correctness": the accepted-length histogram tracks the analytic law of
  rejection sampling; PocketLLM dspark.md, length gate: E[tokens(n)] = 1 +
  sum_{i<n} prod_{j<=i} p_j).  Chi-square over n in {0..K}, p > 0.01.
* Expected tokens per round with a constant acceptance: ``1 + a + a^2`` = 2.44
  at a = 0.8, gamma = 2 (llmstudio.ru, section 30).
"""

import numpy as np
import pytest
from scipy import stats

import oracle as o
from conftest import load_golden

F32 = np.float32


def law_probs(p, q):
    ph = p.astype(np.float64) / p.astype(np.float64).sum(axis=1, keepdims=True)
    qh = q.astype(np.float64) / q.astype(np.float64).sum(axis=1, keepdims=True)
    alpha = np.minimum(ph[: len(q)], qh).sum(axis=1)
    K = len(q)
    surv = np.concatenate([[1.0], np.cumprod(alpha)])  # P(n >= i), i = 0..K
    pn = surv[:-1] - surv[1:]
    return np.concatenate([pn, [surv[-1]]]), alpha


def simulate_rounds(p, q, rounds, seed):
    """Batch ``rounds`` copies of one sequence with fresh draft tokens t_i ~ q_i
    and fresh 24-bit uniforms; return the oracle's n_accepted."""
    rng = np.random.default_rng(seed)
    K, V = q.shape
    qh = q.astype(np.float64) / q.astype(np.float64).sum(axis=1, keepdims=True)
    cdf = np.cumsum(qh, axis=1)
    tok = np.empty((rounds, K), np.int32)
    for i in range(K):
        tok[:, i] = np.minimum(np.searchsorted(cdf[i], rng.random(rounds) * cdf[i, -1],
                                               side="right"), V - 1)
    u = (rng.integers(0, 1 << 24, (rounds, K + 1)) * 2.0 ** -24).astype(F32)
    P = np.tile(p, (rounds, 1))
    Q = np.tile(q, (rounds, 1))
    res = o.accept(P, Q, tok.reshape(-1), u.reshape(-1), rounds, K)
    assert (res.status & ~np.uint32(o.NEAR_BOUNDARY | o.DRAW_CERTIFIED)).max() == 0
    return res.n_accepted


def chi2_pvalue(counts, probs):
    exp = probs * counts.sum()
    keep = exp > 0
    return stats.chisquare(counts[keep], exp[keep] * counts[keep].sum() / exp[keep].sum()).pvalue


@pytest.mark.slow
def test_accepted_length_law_chi_square():
    rng = np.random.default_rng(20240601)
    K, V = 4, 16
    tl = rng.normal(0, 1.5, (K + 1, V))
    p = np.exp(tl).astype(F32)
    q = np.exp(tl[:K] + rng.normal(0, 1.0, (K, V))).astype(F32)
    rounds = 100_000
    n = simulate_rounds(p, q, rounds, seed=1)
    probs, alpha = law_probs(p, q)
    counts = np.bincount(n, minlength=K + 1)
    pv = chi2_pvalue(counts, probs)
    assert pv > 0.01, (counts, probs * rounds, alpha, pv)


def test_accepted_length_law_detects_a_different_law():
    # the same statistic rejects the law of a different draft (power check)
    rng = np.random.default_rng(99)
    K, V = 3, 12
    tl = rng.normal(0, 1.5, (K + 1, V))
    p = np.exp(tl).astype(F32)
    q = np.exp(tl[:K] + rng.normal(0, 1.0, (K, V))).astype(F32)
    q_other = np.exp(tl[:K] + rng.normal(0, 2.0, (K, V))).astype(F32)
    n = simulate_rounds(p, q, 20_000, seed=2)
    probs_other, _ = law_probs(p, q_other)
    assert chi2_pvalue(np.bincount(n, minlength=K + 1), probs_other) < 1e-6


@pytest.mark.slow
def test_expected_tokens_closed_form():
    g = load_golden("llmstudio_s30_expected_tokens.txt")
    a, gam = g["alpha"], int(g["gamma"])
    # rows with sum(min(p, q)) = a exactly: q = a * p + (1 - a) * w, w disjoint from p
    V = 16
    rng = np.random.default_rng(4)
    p = np.zeros((gam + 1, V))
    q = np.zeros((gam, V))
    for i in range(gam + 1):
        p[i, :8] = rng.dirichlet(np.ones(8))
    for i in range(gam):
        q[i] = a * p[i]
        q[i, 8:] = (1 - a) * rng.dirichlet(np.ones(8))
    p, q = p.astype(F32), q.astype(F32)
    probs, alpha = law_probs(p, q)
    assert np.allclose(alpha, a, atol=1e-6)
    closed = (1 - a ** (gam + 1)) / (1 - a)
    assert abs(closed - g["expected_tokens"]) < 1e-12
    rounds = 100_000
    n = simulate_rounds(p, q, rounds, seed=3)
    mean_tokens = (n + 1).mean()  # accepted prefix plus the correction / bonus token
    se = (n + 1).std() / np.sqrt(rounds)
    assert abs(mean_tokens - g["expected_tokens"]) < 5 * se, (mean_tokens, se)
