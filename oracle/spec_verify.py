"""Plain single-threaded reference of the verification step (test infrastructure).

Readings of the pages that this file fixes (each restated where it is used):

* Row pairing.  Target row ``i`` of a sequence is the distribution after the
  committed token and drafts ``t_0..t_{i-1}``; it scores ``t_i``; row ``K_b``
  is the bonus row (spec-verify card, "Usage": ``target_probs [K+1, V]``,
  "Method": "all K matched emit argmax(target_K)").
* Greedy.  Accept ``t_i`` while it equals ``argmax(target_i)``; at the first
  miss emit that argmax; if all match emit ``argmax(target_K)`` (card,
  "Method"; llmstudio.ru section 13).  Ties go to the lowest index; NaN never
  wins (it ranks below -inf); an all-NaN row yields index 0.
* Sampling.  Accept ``t_i`` with probability ``min(1, p_i(t_i)/q_i(t_i))``
  using the explicit uniform ``u_i``; on the first rejection resample from
  ``norm(max(0, p_i - q_i))``; if all are accepted draw the bonus from
  ``p_K`` (card, "Method"; llmstudio.ru sections 15-17, 47, 48).
  Rows need not be normalised and "masses are summed exactly" (card,
  "Correctness"): every probability is divided by the exact real sum of its
  f32 row.  The decision is the exact real predicate
  ``u_i * q_i(t_i) * Zp_i < p_i(t_i) * Zq_i``, which for ``u`` in [0, 1) is
  ``u < min(1, phat/qhat)``.
* Uniforms.  A sequence owns ``K_b + 1`` uniforms: ``u_0..u_{K_b-1}`` drive
  the accept tests and ``u_{K_b}`` is the single draw used by whichever of
  resample or bonus happens ("randomness enters only through explicit
  uniform draws", card "Method").
* Inverse CDF.  ``next = min{v : C_v > u * R}`` with ``C`` the running sum of
  the (normalised) weights and ``R`` their total; strict ``>`` so zero-mass
  tokens are never emitted.  The draw is computed in fp64 and flagged
  ``NEAR_BOUNDARY`` when ``u * R`` lies within ``1e-5 * R`` of a CDF step.
* Logits.  ``T_b = 0`` means greedy on the raw logits; ``T_b > 0`` means both
  target and draft rows become ``softmax(logits / T_b)`` (computed in fp64,
  max-subtracted, then rounded to f32) and the sampling rule runs on those
  rows (llmstudio.ru section 38: p and q are the distributions after the
  sampling transforms, warped identically).  An implementation that forms
  the weights ``2^((l - m) log2(e) / T)`` in fp32 with a hardware exp2 of
  relative error ``e`` can take another accept decision only where the
  oracle's test is within ``softmax_decision_tol`` of its threshold; such
  decisions set the oracle-only ``NEAR_DECISION`` bit.
* Empty residual.  After a rejection the exact residual mass is positive
  (q(t) > p(t) there) but may be tiny; one whose mass lies within the fp32
  error band of zero (``EMPTY_PROB_TOL`` for probability rows, the row pair's
  softmax band for warped rows, the same bound on sum |d(phat - qhat)|) may
  come out empty in fp32 arithmetic, so the oracle flags it ``NEAR_EMPTY``
  (and ``NEAR_BOUNDARY``: which id it names is decided by rounding).

Error conventions (a sequence stops at the first row where one applies):
``BAD_LAYOUT`` ragged offsets out of range (n = 0, next = -1);
``BAD_TOKEN`` a draft id outside [0, V) (greedy: counts as a miss and emits
the row argmax; sampling: next = -1); ``BAD_VALUE`` NaN / +-Inf / negative
probability, NaN / +Inf logit, uniform outside [0, 1) or bad temperature
(sampling: next = -1; greedy: NaN only flags, the argmax ignores it);
``ZERO_MASS`` a needed row whose mass is zero (next = -1), or a zero residual
after a rejection, in which case the draw falls back to ``p_j``.
"""

from __future__ import annotations

import dataclasses
from fractions import Fraction
from typing import Callable, Optional, Tuple

import numpy as np

BAD_TOKEN = 1
BAD_VALUE = 2
ZERO_MASS = 4
NEAR_BOUNDARY = 8
BAD_LAYOUT = 64
NEAR_FILTER = 256  # oracle only: a top-p boundary within the filter tolerance
NEAR_DECISION = 512  # oracle only: an accept test within the softmax tolerance of its threshold
DRAW_CERTIFIED = 2048  # oracle only: a bonus draw whose id holds within TIGHT_BONUS_REL (below)
NEAR_EMPTY = 4096  # oracle only: a residual mass within the fp32 error band of zero (below)

BOUNDARY_REL_TOL = 1e-5
# A bonus draw from f32 probability rows, normalised by any mass Z' (the
# common factor Z/Z' cancels in the normalised CDF), weighted with one f32
# rounding per element (relative u = 2^-24) and floored to 64-bit fixed point
# with a total near 2^(62 - bitlen V): every normalised CDF value moves by at
# most 2u + 2^(2 bitlen V - 61), below 2^-21 for V <= 2^18.  A uniform
# farther than that from every step therefore names the same id.
TIGHT_BONUS_REL = 2.0 ** -21
TIGHT_BONUS_MAX_V = 1 << 18
# After a rejection the residual mass R = sum_v max(0, phat_v - qhat_v) is
# positive in exact arithmetic, but it can be as small as (1 - u) qhat(t).
# Normalising f32 probability rows in fp32 (a rounded reciprocal of the mass,
# a rounded product, a rounded difference) moves each term by at most
# 4u (phat_v + qhat_v) + u |phat_v - qhat_v|, so R by at most 9u < 2^-20.  A
# residual with R at or below that band may come out empty (ZERO_MASS and a
# draw from phat) or not, and its draw is decided by rounding: NEAR_EMPTY and
# NEAR_BOUNDARY.  Warped rows use the softmax band of the row pair instead.
EMPTY_PROB_TOL = 2.0 ** -20

_TWO_M149 = Fraction(1, 1 << 149)


@dataclasses.dataclass
class Result:
    n_accepted: np.ndarray  # int32 [B]
    next_token: np.ndarray  # int32 [B]
    status: np.ndarray  # uint32 [B]


# ------------------------------------------------------------------ inputs

def decode_rows(arr: np.ndarray, dtype: str) -> np.ndarray:
    """Exact conversion of stored rows to float64 ('f32', 'f16', 'bf16'
    given as uint16 bit patterns, or 'f64' as they are)."""
    if dtype == "f64":
        return np.asarray(arr, np.float64)
    if dtype == "bf16":
        bits = np.asarray(arr, np.uint16).astype(np.uint32) << 16
        return bits.view(np.float32).astype(np.float64)
    if dtype == "f16":
        return np.asarray(arr, np.float16).astype(np.float64)
    if dtype == "f32":
        return np.asarray(arr, np.float32).astype(np.float64)
    raise ValueError(dtype)


# ------------------------------------------------------------------ masses

def exact_mass_int(row: np.ndarray) -> int:
    """Exact sum of a row of non-negative finite f32 values, as the integer
    ``S`` with ``sum = S * 2**-149`` (card, "Correctness": masses are summed
    exactly).

    Every finite f32 ``x >= 0`` is ``M * 2**(s - 149)`` with an integer
    significand ``M < 2**24`` and ``s`` in [0, 253]; the sum is accumulated per
    exponent in int64 (no rounding) and the buckets are combined with Python
    integers.
    """
    bits = np.ascontiguousarray(row, dtype=np.float32).view(np.uint32)
    expo = (bits >> 23) & 0xFF
    frac = bits & 0x7FFFFF
    sig = np.where(expo > 0, frac | 0x800000, frac).astype(np.int64)
    shift = np.where(expo > 0, expo - 1, 0).astype(np.int64)
    buckets = np.zeros(254, np.int64)
    np.add.at(buckets, shift, sig)
    total = 0
    for s in np.flatnonzero(buckets):
        total += int(buckets[s]) << int(s)
    return total


def exact_mass(row: np.ndarray) -> Fraction:
    return exact_mass_int(row) * _TWO_M149


def _row_is_bad_prob(row: np.ndarray) -> bool:
    r = np.asarray(row, np.float32)
    return bool(np.isnan(r).any() or np.isinf(r).any() or (r < 0).any())


def _uniform_ok(u) -> bool:
    u = float(np.float32(u))
    return 0.0 <= u < 1.0


# ------------------------------------------------------------------ greedy

def argmax_lowest(row64: np.ndarray) -> Tuple[int, bool]:
    """Index of the largest value, lowest index on ties, NaN never wins.

    Returns ``(index, saw_nan)``; an all-NaN row gives index 0.
    """
    x = np.asarray(row64, np.float64)
    nan = np.isnan(x)
    if nan.all():
        return 0, bool(nan.any())
    key = np.where(nan, -np.inf, x)
    best = key.max()
    cand = np.flatnonzero((key == best) & ~nan)
    return int(cand[0]), bool(nan.any())


def _greedy_sequence(rows: Callable[[int], np.ndarray], tokens: np.ndarray,
                     k: int, V: int) -> Tuple[int, int, int]:
    status = 0
    for i in range(k + 1):
        a, saw_nan = argmax_lowest(rows(i))
        if saw_nan:
            status |= BAD_VALUE
        if i == k:
            return k, a, status
        t = int(tokens[i])
        if not 0 <= t < V:
            return i, a, status | BAD_TOKEN
        if t != a:
            return i, a, status
    raise AssertionError("unreachable")


# ------------------------------------------------------------------ sampling

def accept_decision(u: float, p_t: float, q_t: float, zp_int: int, zq_int: int) -> bool:
    """Exact real predicate ``u * q(t) * Zp < p(t) * Zq``.

    ``u``, ``p_t``, ``q_t`` are f32 values (converted exactly); the masses are
    the exact integers of :func:`exact_mass_int` (their common 2**-149 factor
    cancels).  Equals ``u < min(1, phat(t) / qhat(t))`` for ``u`` in [0, 1)
    (card, "Method"; llmstudio.ru sections 15-16).
    """
    lhs = Fraction(float(np.float32(u))) * Fraction(float(np.float32(q_t))) * zp_int
    rhs = Fraction(float(np.float32(p_t))) * zq_int
    return lhs < rhs


def inverse_cdf_draw(weights64: np.ndarray, u: float, tol: float = BOUNDARY_REL_TOL) -> Tuple[int, bool]:
    """``min{v : C_v > u * R}`` over fp64 running sums ``C`` of ``weights64``,
    ``R = C[-1]``; also whether ``u * R`` is within ``tol * R`` (default
    ``1e-5 * R``) of a CDF step (a boundary case)."""
    c = np.cumsum(np.asarray(weights64, np.float64))
    total = float(c[-1])
    tau = float(np.float32(u)) * total
    idx = int(np.searchsorted(c, tau, side="right"))
    idx = min(idx, len(c) - 1)
    lo = float(c[idx - 1]) if idx > 0 else 0.0
    hi = float(c[idx])
    near = min(abs(tau - lo), abs(hi - tau)) <= tol * total
    return idx, bool(near)


EX2_REL = 2.0 ** -21  # relative error bound taken for a hardware exp2 (checked by a GPU test)
F32_U = 2.0 ** -24


def softmax_weight_tol(row_max: float, temperature: float) -> float:
    """Relative error bound of one fp32 weight ``2^((l - m) k)``, k = log2(e)/T,
    against the exact one, for a row of maximum ``m``: the exp2 (e), the
    argument formed as ``l k - m k`` with ``m k`` rounded once and k rounded
    once (at most ``(|m k| + 2 * 126) u`` in the exponent, weights below
    2^-126 being flushed), and the rounding of the weight (u)."""
    mk = abs(float(row_max)) * 1.4426950408889634 / float(temperature)
    return EX2_REL + 0.6931471805599453 * (mk + 2 * 126.0) * F32_U + F32_U


def softmax_decision_tol(tol_p: float, tol_q: float) -> float:
    """Relative band of an accept test ``u qhat(t) < phat(t)`` from weights
    within ``tol_p`` / ``tol_q`` of exact: phat(t) = w_t / Z moves by at most
    2 tol_p (weight and mass), qhat(t) by 2 tol_q, plus the oracle's own f32
    rounding of both probabilities (2 u)."""
    return 2.0 * tol_p + 2.0 * tol_q + 2.0 * F32_U


def _near_decision(u: float, p_t: float, q_t: float, zp_int: int, zq_int: int, tol: float) -> bool:
    """Whether ``u q(t) Zp`` and ``p(t) Zq`` are within ``tol`` (relative) of each other."""
    lhs = Fraction(float(np.float32(u))) * Fraction(float(np.float32(q_t))) * zp_int
    rhs = Fraction(float(np.float32(p_t))) * zq_int
    return abs(lhs - rhs) <= Fraction(tol) * max(lhs, rhs)


def _frac_to_f64(num: int) -> float:
    """Correctly rounded float64 of ``num * 2**-149``."""
    return float(num * _TWO_M149)


RowGetter = Callable[[int], Tuple[Optional[np.ndarray], int]]


def _accept_sequence(get_p: RowGetter, get_q: RowGetter, tokens: np.ndarray,
                     u: np.ndarray, k: int, V: int,
                     decision_tol: Optional[Callable[[int], float]] = None,
                     certify_bonus: bool = False) -> Tuple[int, int, int]:
    """One sequence of speculative sampling.  ``get_p(i)`` / ``get_q(i)``
    return ``(f32 row, error_bits)``; a row is fetched only when the
    left-to-right walk reaches it (llmstudio.ru section 48).  With
    ``decision_tol`` (row -> relative band, for warped rows), a decision
    within the band of its threshold sets ``NEAR_DECISION``, and the same
    band bounds the residual mass that sets ``NEAR_EMPTY`` (sum_v of
    |d phat_v| <= 2 tol_p + u and of |d qhat_v| <= 2 tol_q + u).  With
    ``certify_bonus`` (probability rows given as they are), a bonus draw
    farther than ``TIGHT_BONUS_REL`` from every step sets ``DRAW_CERTIFIED``."""
    flags = 0
    for i in range(k + 1):
        if i < k:
            t = int(tokens[i])
            if not 0 <= t < V:
                return i, -1, BAD_TOKEN | flags
        p, perr = get_p(i)
        if perr:
            return i, -1, perr | flags
        if i < k:
            q, qerr = get_q(i)
            if qerr:
                return i, -1, qerr | flags
        if not _uniform_ok(u[i]):
            return i, -1, BAD_VALUE | flags
        zp = exact_mass_int(p)
        if zp == 0:
            return i, -1, ZERO_MASS | flags
        if i == k:
            # all K_b accepted: bonus draw from p_K (card, "Method").
            w = p.astype(np.float64) / _frac_to_f64(zp)
            idx, near = inverse_cdf_draw(w, u[i])
            if certify_bonus and V <= TIGHT_BONUS_MAX_V and not inverse_cdf_draw(w, u[i], TIGHT_BONUS_REL)[1]:
                flags |= DRAW_CERTIFIED
            return k, idx, flags | (NEAR_BOUNDARY if near else 0)
        zq = exact_mass_int(q)
        if zq == 0:
            return i, -1, ZERO_MASS | flags
        if decision_tol is not None and _near_decision(u[i], p[t], q[t], zp, zq, decision_tol(i)):
            flags = NEAR_DECISION
        if accept_decision(u[i], p[t], q[t], zp, zq):
            continue
        # first rejection: resample from norm(max(0, phat - qhat)) with u_K.
        if not _uniform_ok(u[k]):
            return i, -1, BAD_VALUE | flags
        phat = p.astype(np.float64) / _frac_to_f64(zp)
        qhat = q.astype(np.float64) / _frac_to_f64(zq)
        resid = np.maximum(0.0, phat - qhat)
        status = 0
        band = decision_tol(i) if decision_tol is not None else EMPTY_PROB_TOL
        if not resid.sum() > band:
            flags |= NEAR_EMPTY | NEAR_BOUNDARY
        if not resid.sum() > 0.0:
            resid, status = phat, ZERO_MASS
        idx, near = inverse_cdf_draw(resid, u[k])
        return i, idx, status | flags | (NEAR_BOUNDARY if near else 0)
    raise AssertionError("unreachable")


# ------------------------------------------------------------------ layout

def _layouts(B: int, K: int, cu_k: Optional[np.ndarray], sum_k: int):
    """Per sequence ``(k_b, target_row0, draft_row0)`` or ``None`` when the
    ragged offsets are out of range.  Tokens start at ``draft_row0`` and
    uniforms at ``target_row0``."""
    out = []
    for b in range(B):
        if cu_k is None:
            out.append((K, b * (K + 1), b * K))
            continue
        lo, hi = int(cu_k[b]), int(cu_k[b + 1])
        if lo < 0 or hi < lo or hi > sum_k or hi - lo > K:
            out.append(None)
        else:
            out.append((hi - lo, lo + b, lo))
    return out


def _new_result(B: int) -> Result:
    return Result(np.zeros(B, np.int32), np.full(B, -1, np.int32), np.zeros(B, np.uint32))


def _sum_k(B, K, cu_k, tokens):
    return len(tokens) if cu_k is not None else B * K


# ------------------------------------------------------------------ public

def verify_greedy(target: np.ndarray, dtype: str, tokens: np.ndarray, B: int, K: int,
                  cu_k: Optional[np.ndarray] = None) -> Result:
    """Greedy verification of B sequences (card, "Method", first bullet)."""
    V = target.shape[1]
    res = _new_result(B)
    for b, lay in enumerate(_layouts(B, K, cu_k, _sum_k(B, K, cu_k, tokens))):
        if lay is None:
            res.status[b] = BAD_LAYOUT
            continue
        k, t0, d0 = lay
        n, nxt, st = _greedy_sequence(lambda i: decode_rows(target[t0 + i], dtype),
                                      tokens[d0:d0 + k], k, V)
        res.n_accepted[b], res.next_token[b], res.status[b] = n, nxt, st
    return res


def accept(p: np.ndarray, q: np.ndarray, tokens: np.ndarray, u: np.ndarray, B: int,
           K: int, cu_k: Optional[np.ndarray] = None) -> Result:
    """Speculative sampling of B sequences from f32 probability rows."""
    V = p.shape[1]
    res = _new_result(B)

    def getter(rows, start):
        def get(i):
            r = np.asarray(rows[start + i], np.float32)
            return r, (BAD_VALUE if _row_is_bad_prob(r) else 0)
        return get

    for b, lay in enumerate(_layouts(B, K, cu_k, _sum_k(B, K, cu_k, tokens))):
        if lay is None:
            res.status[b] = BAD_LAYOUT
            continue
        k, t0, d0 = lay
        n, nxt, st = _accept_sequence(getter(p, t0), getter(q, d0), tokens[d0:d0 + k],
                                      u[t0:t0 + k + 1], k, V, certify_bonus=True)
        res.n_accepted[b], res.next_token[b], res.status[b] = n, nxt, st
    return res


def softmax_fp64(logits64: np.ndarray, temperature: float) -> Tuple[Optional[np.ndarray], int]:
    """``softmax(l / T)`` of one row in fp64, max-subtracted.

    Returns ``(probabilities, error_bits)``: NaN or +Inf logits are
    ``BAD_VALUE``; a row whose logits are all -Inf is ``ZERO_MASS``.
    """
    x = np.asarray(logits64, np.float64)
    if np.isnan(x).any() or np.isposinf(x).any():
        return None, BAD_VALUE
    m = x.max()
    if m == -np.inf:
        return None, ZERO_MASS
    e = np.exp((x - m) / float(temperature))
    return e / e.sum(), 0


def warped_rows_f32(logits: np.ndarray, dtype: str, temperature: float) -> np.ndarray:
    """f32 rounding of the fp64 softmax of every row (NaN rows for errors)."""
    out = np.full(logits.shape, np.nan, np.float32)
    for r in range(logits.shape[0]):
        pr, err = softmax_fp64(decode_rows(logits[r], dtype), temperature)
        if not err:
            out[r] = pr.astype(np.float32)
    return out


def accept_from_logits(target: np.ndarray, draft: np.ndarray, dtype: str,
                       temperature: np.ndarray, tokens: np.ndarray, u: np.ndarray,
                       B: int, K: int, cu_k: Optional[np.ndarray] = None,
                       top_k: Optional[np.ndarray] = None,
                       top_p: Optional[np.ndarray] = None) -> Result:
    """Mixed greedy / sampled verification from logits with per-sequence T.

    ``T_b = 0`` runs greedy on the raw logits; ``T_b > 0`` warps target and
    draft rows identically to ``softmax(l / T_b)`` (fp64, rounded to f32) and
    runs speculative sampling on them (llmstudio.ru sections 13, 37, 38).
    With ``top_k`` / ``top_p`` (per sequence), every sampled row is first cut
    to the tokens the filters keep (``sampler_filter``; section 38: the
    filters come after the temperature and apply to p and q alike).  An
    invalid top-p is ``BAD_VALUE`` at row 0; a row whose top-p boundary is
    within the filter tolerance sets the oracle-only ``NEAR_FILTER`` bit.
    """
    from . import sampler_filter as sf
    V = target.shape[1]
    res = _new_result(B)
    near_rows = [False]
    row_tol = {}

    def getter(rows, start, T, k=None, p=None, tag="p"):
        def get(i):
            x = decode_rows(rows[start + i], dtype)
            finite = x[np.isfinite(x)]
            row_tol[(tag, i)] = softmax_weight_tol(finite.max() if finite.size else 0.0, T)
            if k is not None or p is not None:
                floor, near, bad = sf.filter_floor(x, T, k, p)
                if bad:
                    return None, BAD_VALUE
                near_rows[0] = near_rows[0] or near
                x = sf.apply_floor(x, floor)
            pr, err = softmax_fp64(x, T)
            if err == ZERO_MASS:
                # all -Inf: a row of zero weights, reported by the mass check
                return np.zeros(V, np.float32), 0
            return (None, err) if err else (pr.astype(np.float32), 0)
        return get

    for b, lay in enumerate(_layouts(B, K, cu_k, _sum_k(B, K, cu_k, tokens))):
        if lay is None:
            res.status[b] = BAD_LAYOUT
            continue
        k, t0, d0 = lay
        T = float(np.float32(temperature[b]))
        if not (T >= 0.0) or T == np.inf:
            res.status[b] = BAD_VALUE
            continue
        if T == 0.0:
            n, nxt, st = _greedy_sequence(lambda i: decode_rows(target[t0 + i], dtype),
                                          tokens[d0:d0 + k], k, V)
        else:
            fk = None if top_k is None else int(top_k[b])
            fp = None if top_p is None else float(np.float32(top_p[b]))
            near_rows[0] = False
            row_tol.clear()
            n, nxt, st = _accept_sequence(getter(target, t0, T, fk, fp, "p"), getter(draft, d0, T, fk, fp, "q"),
                                          tokens[d0:d0 + k], u[t0:t0 + k + 1], k, V,
                                          lambda i: softmax_decision_tol(row_tol[("p", i)], row_tol[("q", i)]))
            if near_rows[0]:
                st |= NEAR_FILTER
        res.n_accepted[b], res.next_token[b], res.status[b] = n, nxt, st
    return res
