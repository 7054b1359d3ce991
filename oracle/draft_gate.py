"""Plain reference of the draft-length gate (test infrastructure only).

The gate picks, per sequence, how many of the already drafted tokens to
submit to verification, from the drafter's per-position confidence scores and
a calibration table of P(draft token matches | confidence bucket)
(PocketLLM docs/dspark.md, the draft-length gate section):

* expected tokens of a round that submits n drafts,
  ``E(n) = 1 + sum_{i<n} prod_{j<=i} p_j``, with p_j the calibrated match
  probability of position j's confidence bucket;
* its cost, ``cost(0) = plain_ms`` (no verify: a plain decode step) and
  ``cost(n) = draft_ms + verify_base_ms + verify_slope_ms * n`` for n > 0
  (the page's fit ``verify(n) ~= 300 ms + 109 ms * n``, draft 196 ms, plain
  303 ms);
* ``n* = argmax_n E(n) / cost(n)``, taken only when it beats the full draft
  by the margin factor (1.15 by default); never fewer than ``min_draft``
  drafts; and a round whose committed-token logit margin (top1 - top2) is
  below ``margin_threshold`` (when that is > 0) skips drafting (n = 0).
* The table is estimated online from verified rounds: a round that submitted
  K_b drafts of which n were accepted records hits for positions 0..n-1 and
  one miss at position n when n < K_b; later positions are censored (never
  recorded).  Counts decay by ``decay`` per round before the new ones are
  added.

Readings where the page is silent:

* Buckets are half-open intervals of the confidence, ``[e_{i-1}, e_i)``, with
  ``e_{-1} = -inf`` and ``e_{NB-1} = +inf``; a NaN confidence falls in bucket 0.
* A bucket with no observations (total == 0) has p = 1: a cold gate keeps the
  full draft (it would otherwise skip drafting and never learn).
* Ties of E(n)/cost(n) go to the smaller n; truncation is taken when its
  ratio is at least ``margin`` times the full draft's.
* ``min_draft`` floors the post-draft choice (capped at K_b); the pre-draft
  margin skip overrides it.

Arithmetic.  The page fixes no precision, so the decision here is the rule
itself in exact rational arithmetic: p = hits / total, the costs and the
margin are the exact values of the (double) parameters, and E, cost and their
ratio are Fractions.  An implementation that evaluates the ratios in floating
point can pick another n only where two compared quantities lie within its
rounding error of each other; ``gate_decision`` reports such near-ties, for
the fp32 evaluation order of ``ratio_error_bound``.  The calibration counts
are decayed and added in fp64, one rounding per operation (decay, then add):
that is the update rule written out in the counts' own type.
"""

from dataclasses import dataclass
from fractions import Fraction

import numpy as np

F32_UNIT = 2.0 ** -24  # unit roundoff of fp32


@dataclass
class GateParams:
    """Defaults are the page's (PocketLLM dspark.md, the gate's environment
    variables and cost fit)."""
    margin: float = 1.15
    min_draft: int = 0
    decay: float = 0.9
    draft_ms: float = 196.0
    verify_base_ms: float = 300.0
    verify_slope_ms: float = 109.0
    plain_ms: float = 303.0
    margin_threshold: float = 0.0


def bucket_of(conf, edges):
    """Index of the half-open bucket holding ``conf`` (NaN -> 0)."""
    c = float(conf)
    if c != c:
        return 0
    b = 0
    for e in edges:
        if c >= float(e):
            b += 1
    return b


def match_prob(hits, total):
    """Calibrated P(match) of one bucket, exactly; 1 when it has no observations."""
    h, t = Fraction(float(hits)), Fraction(float(total))
    return h / t if t > 0 else Fraction(1)


def round_cost(n, prm):
    """cost(n) in ms, exactly (a Fraction of the double parameters)."""
    if n == 0:
        return Fraction(float(prm.plain_ms))
    return (Fraction(float(prm.draft_ms)) + Fraction(float(prm.verify_base_ms))
            + Fraction(float(prm.verify_slope_ms)) * n)


def expected_tokens(p, n):
    """E(n) = 1 + sum_{i<n} prod_{j<=i} p_j (running product, running sum);
    exact when p holds Fractions."""
    e, prod = Fraction(1), Fraction(1)
    for i in range(n):
        prod = prod * (p[i] if isinstance(p[i], Fraction) else Fraction(float(p[i])))
        e = e + prod
    return e


def gate_ratios(p, k_b, prm):
    """E(n) / cost(n) for n = 0..k_b, exactly.  A zero cost gives +inf."""
    out = []
    for n in range(k_b + 1):
        c = round_cost(n, prm)
        out.append(expected_tokens(p, n) / c if c > 0 else float("inf"))
    return out


def ratio_error_bound(n):
    """Relative error bound of E(n)/cost(n) evaluated in fp32 with one rounding
    per operation: p rounded once (u), n products (2n u over the product of
    rounded factors), n additions of positive terms into E (n u), cost from
    fp32-rounded parameters (two inputs and two operations: 4 u), the
    quotient (u); (3n + 6) u covers the first-order sum with room for the
    second-order terms."""
    return (3 * n + 6) * F32_UNIT


def _near(a, b, rel):
    if a == float("inf") or b == float("inf"):
        return a == b
    return abs(a - b) <= Fraction(rel) * max(a, b)


def gate_decision(conf_row, k_b, logit_margin, edges, hits, total, prm):
    """(n, near): the number of drafts (0..k_b) one sequence submits, and
    whether a comparison that decided it was within an fp32 evaluation's error
    bound (a near-tie, where such an evaluation may pick another n)."""
    if prm.margin_threshold > 0.0 and logit_margin is not None and \
            np.float32(logit_margin) < np.float32(prm.margin_threshold):
        return 0, False
    p = [match_prob(hits[bucket_of(c, edges)], total[bucket_of(c, edges)]) for c in conf_row[:k_b]]
    r = gate_ratios(p, k_b, prm)
    n_lo = min(int(prm.min_draft), k_b)
    best_n = n_lo
    for n in range(n_lo + 1, k_b + 1):
        if r[n] > r[best_n]:
            best_n = n
    near = any(_near(r[n], r[best_n], ratio_error_bound(n) + ratio_error_bound(best_n))
               for n in range(n_lo, k_b + 1) if n != best_n)
    if best_n == k_b:
        return k_b, near
    m = Fraction(float(prm.margin))
    full = r[k_b] * m if r[k_b] != float("inf") else (float("inf") if m > 0 else float("nan"))
    near = near or (full == full and _near(r[best_n], full,
                                           ratio_error_bound(best_n) + ratio_error_bound(k_b) + 2 * F32_UNIT))
    if full == full and r[best_n] >= full:
        return best_n, near
    return k_b, near


def gate_length(conf_row, k_b, logit_margin, edges, hits, total, prm):
    """Number of drafts (0..k_b) one sequence submits."""
    return gate_decision(conf_row, k_b, logit_margin, edges, hits, total, prm)[0]


def gate_batch(conf, k_per_seq, logit_margin, edges, hits, total, prm, with_near=False):
    """Per-sequence lengths and their exclusive prefix sum ``cu_k[B+1]``
    (and, with ``with_near``, the per-sequence near-tie flags).

    ``conf`` is ``[B, K]`` (row b holds sequence b's K drafted positions);
    ``k_per_seq[b]`` <= K drafts were made for b (all K when None)."""
    conf = np.asarray(conf)
    B, K = conf.shape
    n = np.zeros(B, dtype=np.int32)
    near = np.zeros(B, dtype=bool)
    for b in range(B):
        kb = K if k_per_seq is None else int(k_per_seq[b])
        lm = None if logit_margin is None else logit_margin[b]
        n[b], near[b] = gate_decision(conf[b], kb, lm, edges, hits, total, prm)
    cu = np.zeros(B + 1, dtype=np.int32)
    cu[1:] = np.cumsum(n)
    return (n, cu, near) if with_near else (n, cu)


def update_table(conf, n_submitted, n_accepted, edges, hits, total, decay):
    """One round of calibration: decay, then add the recorded observations.

    Returns new (hits, total) as float64 arrays."""
    conf = np.asarray(conf)
    nb = len(hits)
    new_h = [0] * nb
    new_t = [0] * nb
    for b in range(conf.shape[0]):
        ks, na = int(n_submitted[b]), int(n_accepted[b])
        for i in range(na):
            k = bucket_of(conf[b, i], edges)
            new_h[k] += 1
            new_t[k] += 1
        if na < ks:
            new_t[bucket_of(conf[b, na], edges)] += 1
    d = float(decay)
    h2 = np.array([d * float(hits[k]) + float(new_h[k]) for k in range(nb)], dtype=np.float64)
    t2 = np.array([d * float(total[k]) + float(new_t[k]) for k in range(nb)], dtype=np.float64)
    return h2, t2


__all__ = ["GateParams", "bucket_of", "match_prob", "round_cost", "expected_tokens", "gate_ratios",
           "ratio_error_bound", "gate_decision", "gate_length", "gate_batch", "update_table"]
