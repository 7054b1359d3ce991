"""Top-k and top-p sampler filters on logit rows (test infrastructure).

TEST INFRASTRUCTURE ONLY: the rules of the package docstring apply (tests,
``smoke()`` and the bench's CPU legs import it; the product never does).

llmstudio.ru, "Как работает speculative decoding и MTP при инференсе LLM",
section 38: a sampling pipeline turns the raw logits into the effective
distribution in the order penalties, temperature, top-k, top-p, other
filters, normalisation; the draft's q goes through the same pipeline, and the
accept / resample rule compares those effective distributions.  So the filters
below are applied alike to every target row and every draft row of a sampled
sequence, after the temperature and before the verification.  Section 39
(stateful samplers: penalties, grammars, bans) is not modelled here.

Readings this file fixes (the page names the filters, not their tie rules):

* Top-k keeps every token whose logit is >= the k-th largest logit (equal
  logits at the boundary are all kept).  k <= 0, or k at least the number of
  non-NaN logits, keeps everything.
* Top-p acts on what top-k kept, renormalised: with weights
  ``w_v = exp((l_v - m) / T)`` (m the row maximum) and ``Z`` their total over
  the top-k set, token v is kept iff the weight of the top-k tokens with a
  strictly larger logit is ``< p * Z``.  The kept set is thus the smallest
  prefix of the ranking (largest logits first) whose mass reaches ``p``, with
  equal logits kept or dropped together.  ``p >= 1`` keeps everything;
  ``p`` NaN or ``<= 0`` is an invalid parameter.
* Both filters keep ``{v : l_v >= floor}`` for a per-row floor (``-inf`` keeps
  everything).  The floor is the row's own logit value, so it is exact in the
  row's dtype.  NaN logits take no part in the ranking; a row whose maximum is
  not finite gets floor ``-inf`` (the verification reports such rows).
* The top-p boundary is decided in fp64 here.  When ``p * Z`` lies within
  ``FILTER_REL_TOL * Z`` of the mass above the lowest kept logit, or of the
  mass above the next logit down, the row is flagged ``near``: an
  implementation whose weights are accurate to that tolerance may keep either
  set there.
"""

from __future__ import annotations

import math
from typing import Optional, Tuple

import numpy as np

FILTER_REL_TOL = 1e-5


def _ranked(x: np.ndarray):
    """Distinct non-NaN values in decreasing order and their multiplicities."""
    v = x[~np.isnan(x)]
    vals, counts = np.unique(v, return_counts=True)  # increasing
    return vals[::-1], counts[::-1]


def _weights(vals: np.ndarray, counts: np.ndarray, T: float) -> np.ndarray:
    """Total weight of each group of equal logits: count * exp((l - m) / T)."""
    return counts * np.exp((vals - vals[0]) / T)


def top_k_floor(x: np.ndarray, k: Optional[int]) -> float:
    """The k-th largest non-NaN value of ``x`` (``-inf`` when top-k keeps all)."""
    vals, counts = _ranked(np.asarray(x, np.float64))
    n = int(counts.sum())
    if k is None or k <= 0 or k >= n:
        return -math.inf
    seen = 0
    for v, c in zip(vals, counts):
        seen += int(c)
        if seen >= k:
            return float(v)
    raise AssertionError("unreachable")


def filter_floor(logits64: np.ndarray, T: float, top_k: Optional[int],
                 top_p: Optional[float]) -> Tuple[float, bool, bool]:
    """``(floor, near, bad)`` of one row of logits at temperature ``T > 0``.

    ``bad`` marks an invalid top-p (floor NaN); ``near`` marks a top-p
    boundary within ``FILTER_REL_TOL`` (see the module docstring).
    """
    if top_p is not None and not (top_p > 0.0):
        return math.nan, False, True
    x = np.asarray(logits64, np.float64)
    vals, counts = _ranked(x)
    if vals.size == 0 or not math.isfinite(vals[0]):
        return -math.inf, False, False
    floor = top_k_floor(x, top_k)                      # top-k first
    if top_p is None or top_p >= 1.0:
        return floor, False, False
    keep = vals >= floor                               # then top-p on what top-k kept
    vals, counts = vals[keep], counts[keep]
    w = _weights(vals, counts, float(T))
    Z = math.fsum(w)
    above = np.concatenate(([0.0], np.cumsum(w)[:-1]))  # mass of strictly larger logits
    pz = float(top_p) * Z
    J = int(np.flatnonzero(above < pz)[-1])            # the lowest kept group
    tol = FILTER_REL_TOL * Z
    near = abs(above[J] - pz) <= tol or (J + 1 < vals.size and abs(above[J + 1] - pz) <= tol)
    return float(vals[J]), bool(near), False


def floor_is_valid(logits64: np.ndarray, T: float, top_k: Optional[int],
                   top_p: Optional[float], floor: float) -> bool:
    """Whether ``floor`` is a correct floor for the row within the tolerance:
    the top-k part exactly, the top-p boundary up to ``FILTER_REL_TOL * Z``."""
    ref, near, bad = filter_floor(logits64, T, top_k, top_p)
    if bad:
        return math.isnan(floor)
    if floor == ref:
        return True
    if not near:
        return False
    x = np.asarray(logits64, np.float64)
    vals, counts = _ranked(x)
    fk = top_k_floor(x, top_k)
    keep = vals >= fk
    vals, counts = vals[keep], counts[keep]
    if floor not in set(vals.tolist()):
        return False
    w = _weights(vals, counts, float(T))
    Z = math.fsum(w)
    above = np.concatenate(([0.0], np.cumsum(w)[:-1]))
    j = int(np.flatnonzero(vals == floor)[0])
    pz, tol = float(top_p) * Z, FILTER_REL_TOL * Z
    kept_ok = above[j] < pz + tol                       # the floor's group may be kept
    next_ok = j + 1 >= vals.size or above[j + 1] >= pz - tol  # the next group may be dropped
    return bool(kept_ok and next_ok)


def apply_floor(logits64: np.ndarray, floor: float) -> np.ndarray:
    """Logits below the floor become -inf (NaN stays NaN)."""
    x = np.asarray(logits64, np.float64).copy()
    x[x < floor] = -math.inf
    return x


def _seq_rows(B: int, K: int, cu_k: Optional[np.ndarray]):
    for b in range(B):
        if cu_k is None:
            yield b, K, b * (K + 1), b * K
        else:
            lo, hi = int(cu_k[b]), int(cu_k[b + 1])
            yield b, hi - lo, lo + b, lo


def floors_batch(target: np.ndarray, draft: Optional[np.ndarray], decode, temperature: np.ndarray,
                 top_k: Optional[np.ndarray], top_p: Optional[np.ndarray], B: int, K: int,
                 cu_k: Optional[np.ndarray] = None):
    """Floors of every target row (``[sum(K_b + 1)]``) and draft row
    (``[sum K_b]``), with their ``near`` flags.  Greedy sequences (T = 0) and
    invalid temperatures get ``-inf``.  ``decode(row)`` gives the fp64 logits
    of one stored row."""
    nt = target.shape[0]
    nd = 0 if draft is None else draft.shape[0]
    ft, fd = np.full(nt, -np.inf), np.full(nd, -np.inf)
    nrt, nrd = np.zeros(nt, bool), np.zeros(nd, bool)
    for b, kb, t0, d0 in _seq_rows(B, K, cu_k):
        T = float(np.float32(temperature[b]))
        if not (T > 0.0) or T == math.inf:
            continue
        k = None if top_k is None else int(top_k[b])
        p = None if top_p is None else float(np.float32(top_p[b]))
        for i in range(kb + 1):
            ft[t0 + i], nrt[t0 + i], _ = filter_floor(decode(target[t0 + i]), T, k, p)
            if i < kb:
                fd[d0 + i], nrd[d0 + i], _ = filter_floor(decode(draft[d0 + i]), T, k, p)
    return ft, fd, nrt, nrd
