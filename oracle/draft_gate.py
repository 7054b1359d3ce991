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

Readings where the page is silent (stated in the design doc as well):

* Buckets are half-open intervals of the confidence, ``[e_{i-1}, e_i)``, with
  ``e_{-1} = -inf`` and ``e_{NB-1} = +inf``; a NaN confidence falls in bucket 0.
* A bucket with no observations (total == 0) has p = 1: a cold gate keeps the
  full draft (it would otherwise skip drafting and never learn).
* Ties of E(n)/cost(n) go to the smaller n; truncation is taken when its
  ratio is at least ``margin`` times the full draft's.
* ``min_draft`` floors the post-draft choice (capped at K_b); the pre-draft
  margin skip overrides it.

The decision (E, cost, their ratio, the margin test) is taken in fp32, the
kernel's precision, since it only decides an integer; p = hits / total is an
fp64 quotient rounded to fp32, and the calibration counts stay fp64.  Each
operation rounds once, in the order written here (the GPU kernels follow the
same order, so results compare bit for bit).
"""

from dataclasses import dataclass

import numpy as np


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
    """Calibrated P(match) of one bucket; 1 when it has no observations."""
    h, t = float(hits), float(total)
    return h / t if t > 0.0 else 1.0


def round_cost(n, prm):
    if n == 0:
        return float(prm.plain_ms)
    return float(prm.draft_ms) + float(prm.verify_base_ms) + float(prm.verify_slope_ms) * float(n)


def expected_tokens(p, n):
    """E(n) = 1 + sum_{i<n} prod_{j<=i} p_j (running product, running sum)."""
    e, prod = 1.0, 1.0
    for i in range(n):
        prod = prod * float(p[i])
        e = e + prod
    return e


def ratios_f32(p, k_b, prm):
    """E(n) / cost(n) for n = 0..k_b as the gate decides them: in fp32 (the
    kernel's precision), one rounding per operation, E by running product
    and sum, cost as (draft_ms + verify_base_ms) + verify_slope_ms * n."""
    f = np.float32
    fixed = f(f(prm.draft_ms) + f(prm.verify_base_ms))
    e, prod = f(1.0), f(1.0)
    out = []
    for n in range(0, k_b + 1):
        if n > 0:
            prod = f(prod * f(p[n - 1]))
            e = f(e + prod)
        cost = f(prm.plain_ms) if n == 0 else f(fixed + f(f(prm.verify_slope_ms) * f(n)))
        out.append(f(e / cost))
    return out


def gate_length(conf_row, k_b, logit_margin, edges, hits, total, prm):
    """Number of drafts (0..k_b) one sequence submits."""
    if prm.margin_threshold > 0.0 and logit_margin is not None and \
            np.float32(logit_margin) < np.float32(prm.margin_threshold):
        return 0
    p = [np.float32(match_prob(hits[bucket_of(c, edges)], total[bucket_of(c, edges)])) for c in conf_row[:k_b]]
    r = ratios_f32(p, k_b, prm)
    n_lo = min(int(prm.min_draft), k_b)
    best_n = n_lo
    for n in range(n_lo + 1, k_b + 1):
        if r[n] > r[best_n]:
            best_n = n
    if best_n < k_b and r[best_n] >= np.float32(np.float32(prm.margin) * r[k_b]):
        return best_n
    return k_b


def gate_batch(conf, k_per_seq, logit_margin, edges, hits, total, prm):
    """Per-sequence lengths and their exclusive prefix sum ``cu_k[B+1]``.

    ``conf`` is ``[B, K]`` (row b holds sequence b's K drafted positions);
    ``k_per_seq[b]`` <= K drafts were made for b (all K when None)."""
    conf = np.asarray(conf)
    B, K = conf.shape
    n = np.zeros(B, dtype=np.int32)
    for b in range(B):
        kb = K if k_per_seq is None else int(k_per_seq[b])
        lm = None if logit_margin is None else logit_margin[b]
        n[b] = gate_length(conf[b], kb, lm, edges, hits, total, prm)
    cu = np.zeros(B + 1, dtype=np.int32)
    cu[1:] = np.cumsum(n)
    return n, cu


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


__all__ = ["GateParams", "bucket_of", "match_prob", "round_cost", "expected_tokens", "ratios_f32",
           "gate_length", "gate_batch", "update_table"]
