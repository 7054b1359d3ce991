"""Repetition / frequency / presence penalties ahead of verification (test
infrastructure).

TEST INFRASTRUCTURE ONLY: the rules of the package docstring apply (tests,
``smoke()`` and the bench's CPU legs import it; the product never does).

llmstudio.ru, "Как работает speculative decoding и MTP при инференсе LLM",
section 38: the sampling pipeline turns raw logits into the effective
distribution in the order raw logits -> penalties -> temperature -> top-k ->
top-p -> normalise, for the target (p) and alike for the draft (q);
speculative sampling works on those effective distributions.  Section 39:
stateful samplers (repetition penalties among them) keep exactness only when
their state follows the speculative branch: the state that scores position i
is the committed history plus the drafted tokens t_0..t_{i-1} the branch
assumes accepted.

Readings this file fixes:

* One token history per sequence (the caller's committed context) drives all
  three penalties.  Row i of a sequence (target row i and, for i < K_b, draft
  row i) counts ``c_i(v)`` = occurrences of ``v`` in the history plus in
  ``t_0..t_{i-1}``; tokens with ``c_i(v) = 0`` are untouched.
* For a touched logit ``x`` (the stored value, exact in f32), in f32 with one
  rounding per operation, in this order: the repetition penalty ``r``
  (``x * r`` when ``x < 0``, else ``x / r``), then ``x - freq * c`` (the
  product rounded, then the difference), then ``x - pres``; the result is
  rounded to the row's storage type (nearest, ties to even).  Neutral values
  ``r = 1, freq = 0, pres = 0`` leave the row as it is (``x / 1``, ``x - 0``
  are exact).
* A history id outside [0, V) is skipped (it names no logit); so is a draft
  id outside [0, V) (verification reports it as BAD_TOKEN at its row).
* A sequence whose parameters are unusable (``r`` not a positive finite
  number, ``freq`` or ``pres`` not finite) is reported BAD_VALUE and its rows
  are left as they are; so are rows of a sequence with out-of-range offsets
  (BAD_LAYOUT) or with more than MAX_DISTINCT distinct in-range ids in its
  history and drafts together (BAD_LAYOUT: the capacity of the per-sequence
  count table of the GPU path, part of its interface).
"""

from __future__ import annotations

from collections import Counter
from typing import Optional, Tuple

import numpy as np

BAD_VALUE = 2
BAD_LAYOUT = 64
MAX_DISTINCT = 8192
F32 = np.float32


def penalize_value(x: float, count: int, r: float, freq: float, pres: float) -> np.float32:
    """The penalised value of one logit ``x`` seen ``count`` > 0 times, in f32
    (before the rounding to the storage type)."""
    v = F32(x)
    r32, f32, p32 = F32(r), F32(freq), F32(pres)
    v = v * r32 if v < 0 else v / r32
    v = F32(v - F32(f32 * F32(count)))
    v = F32(v - p32)
    return F32(v)


def _to_storage(v: np.float32, dtype: str):
    """Round an f32 value to the row's storage (bf16 as uint16 bits)."""
    if dtype == "f32":
        return F32(v)
    if dtype == "f16":
        return np.float16(v)
    b = np.array([v], F32).view(np.uint32).astype(np.uint64)
    if np.isnan(v):
        return np.uint16(0x7FC0 | ((int(b[0]) >> 16) & 0x8000))
    b = (b + 0x7FFF + ((b >> 16) & 1)) >> 16
    return np.uint16(int(b[0]))


def _from_storage(x, dtype: str) -> float:
    if dtype == "bf16":
        return float(np.array([int(x) << 16], np.uint32).view(F32)[0])
    return float(x)


def row_counts(history, drafts, i: int, V: int) -> Counter:
    """``c_i``: occurrences in the history plus in ``t_0..t_{i-1}`` of every
    id in [0, V) (section 39: the state after accepting the first i drafts)."""
    c = Counter(int(v) for v in history if 0 <= int(v) < V)
    c.update(int(v) for v in drafts[:i] if 0 <= int(v) < V)
    return c


def penalize_rows(target: np.ndarray, draft: np.ndarray, dtype: str, hist_offsets: np.ndarray,
                  hist_tokens: np.ndarray, tokens: np.ndarray, B: int, K: int,
                  cu_k: Optional[np.ndarray], rep: np.ndarray, freq: np.ndarray,
                  pres: np.ndarray) -> Tuple[np.ndarray, np.ndarray, np.ndarray]:
    """Copies of the target and draft rows (storage layout of the verification
    calls) with every sequence's penalties applied row by row, and a status
    per sequence (BAD_LAYOUT for out-of-range offsets: its rows untouched)."""
    tg, dr = target.copy(), draft.copy()
    V = target.shape[1]
    st = np.zeros(B, np.uint32)
    sum_k = len(tokens) if cu_k is not None else B * K
    for b in range(B):
        if cu_k is None:
            k, t0, d0 = K, b * (K + 1), b * K
        else:
            lo, hi = int(cu_k[b]), int(cu_k[b + 1])
            if lo < 0 or hi < lo or hi > sum_k or hi - lo > K:
                st[b] = BAD_LAYOUT
                continue
            k, t0, d0 = hi - lo, lo + b, lo
        h0, h1 = int(hist_offsets[b]), int(hist_offsets[b + 1])
        if h0 < 0 or h1 < h0 or h1 > len(hist_tokens):
            st[b] = BAD_LAYOUT
            continue
        r_ok = np.isfinite(rep[b]) and rep[b] > 0
        if not (r_ok and np.isfinite(freq[b]) and np.isfinite(pres[b])):
            st[b] = BAD_VALUE
            continue
        hist = hist_tokens[h0:h1]
        drafts = tokens[d0:d0 + k]
        if len(row_counts(hist, drafts, k, V)) > MAX_DISTINCT:
            st[b] = BAD_LAYOUT
            continue
        for i in range(k + 1):
            for v, c in row_counts(hist, drafts, i, V).items():
                rows = [(tg, t0 + i)] + ([(dr, d0 + i)] if i < k else [])
                for arr, r in rows:
                    x = _from_storage(arr[r, v], dtype)
                    arr[r, v] = _to_storage(penalize_value(x, c, rep[b], freq[b], pres[b]), dtype)
    return tg, dr, st
