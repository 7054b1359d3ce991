"""Builders for the five synthetic verification workloads.

Every builder is deterministic in its seed (numpy's counter-based Philox bit
generator) and returns a :class:`Workload` whose arrays are laid out exactly as
the C ABI takes them:

* target rows ``[sum(K_b + 1), V]`` (probabilities f32, or logits f32 / bf16
  bits as uint16 / f16), sequence ``b`` owning rows ``cu_k[b] + b .. cu_k[b+1] + b``;
* draft rows ``[sum(K_b), V]`` (same dtype), sequence ``b`` owning rows
  ``cu_k[b] .. cu_k[b+1]``;
* draft tokens int32 ``[sum(K_b)]`` and uniforms f32 ``[sum(K_b + 1)]``
  (24-bit values ``k * 2**-24`` in ``[0, 1)``);
* ``cu_k`` int32 ``[B + 1]`` for ragged batches, ``None`` for uniform K.

Row ``i`` of a sequence scores draft token ``t_i``; the last target row is the
bonus row (spec-verify model card, section "Method"; TensorSharp
speculative_decoding.md, "The shared runtime", step 2: the verify batch is
``[last, d1..dK]`` so row ``i`` is the distribution *after* ``d_1..d_i``).

The softmax and the token draws below only synthesise inputs (the pages define
the workloads as "softmax of N(0, s^2) logits" with draft tokens drawn from the
draft distribution); none of it is the verification arithmetic.
"""

from __future__ import annotations

import dataclasses
from typing import Optional

import numpy as np

CONFIG_NAMES = ("config1", "config2", "config3", "config4", "config5", "greedy2")
SEED_BASE = 0x5EED0000

_ROW_BLOCK = 64  # rows synthesised per block, to bound host memory


@dataclasses.dataclass
class Workload:
    name: str
    mode: str  # "greedy" | "accept" | "logits" ("both" for config 1)
    dtype: str  # "f32" | "bf16" | "f16"
    B: int
    K: int  # K_max
    V: int
    target: np.ndarray
    draft: Optional[np.ndarray]
    tokens: np.ndarray
    uniforms: Optional[np.ndarray]
    cu_k: Optional[np.ndarray]
    temperature: Optional[np.ndarray]
    meta: dict

    @property
    def k_per_seq(self) -> np.ndarray:
        if self.cu_k is None:
            return np.full(self.B, self.K, np.int64)
        return np.diff(self.cu_k.astype(np.int64))

    @property
    def sum_k(self) -> int:
        return int(self.k_per_seq.sum())

    @property
    def elem_size(self) -> int:
        return 4 if self.dtype == "f32" else 2

    def formula_bytes(self) -> int:
        """Bytes per round as the benchmark formula counts them.

        Target rows always; draft rows only for sequences that sample (a
        greedy sequence reads no draft row).
        """
        kb = self.k_per_seq
        t_rows = int((kb + 1).sum())
        if self.mode == "greedy" or self.draft is None:
            d_rows = 0
        elif self.temperature is not None:
            d_rows = int(kb[self.temperature > 0].sum())
        else:
            d_rows = int(kb.sum())
        return (t_rows + d_rows) * self.V * self.elem_size


# ---------------------------------------------------------------- helpers

def _rng(seed: int) -> np.random.Generator:
    return np.random.Generator(np.random.Philox(seed))


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round finite f32 values to bf16 (nearest, ties to even); return uint16 bits."""
    b = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    b = (b + 0x7FFF + ((b >> 16) & 1)) >> 16
    return b.astype(np.uint16)


def _bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    return (bits.astype(np.uint32) << 16).view(np.float32)


def uniforms_24bit(rng: np.random.Generator, n: int) -> np.ndarray:
    """U[0,1) draws with 24 random bits: k * 2**-24, exact in f32."""
    return (rng.integers(0, 1 << 24, size=n, dtype=np.int64).astype(np.float64)
            * 2.0 ** -24).astype(np.float32)


def _softmax_rows(x: np.ndarray, scale: float = 1.0) -> np.ndarray:
    x = np.asarray(x, np.float64) * scale
    x = x - x.max(axis=-1, keepdims=True)
    e = np.exp(x)
    return e / e.sum(axis=-1, keepdims=True)


def _draw_from_rows(rng: np.random.Generator, prob: np.ndarray) -> np.ndarray:
    """One categorical draw per row of an (already normalised) fp64 matrix."""
    c = np.cumsum(prob, axis=-1)
    u = rng.random(prob.shape[0]) * c[:, -1]
    out = np.empty(prob.shape[0], np.int32)
    for r in range(prob.shape[0]):
        out[r] = min(int(np.searchsorted(c[r], u[r], side="right")), prob.shape[1] - 1)
    return out


def _layout(B: int, kb: np.ndarray):
    """Row starts of each sequence: (target_start, draft_start) arrays."""
    cu = np.zeros(B + 1, np.int64)
    cu[1:] = np.cumsum(kb)
    return cu[:-1] + np.arange(B), cu[:-1], cu


def _tune_noise(target_logits: np.ndarray, z: np.ndarray, alpha: float) -> float:
    """Noise scale s with mean sum(min(p, q)) ~= alpha, where
    q = softmax(target_logits + s * z); bisection on a few sample rows."""

    def overlap(s: float) -> float:
        p = _softmax_rows(target_logits)
        q = _softmax_rows(target_logits + s * z)
        return float(np.minimum(p, q).sum(axis=-1).mean())

    lo, hi = 0.0, 1.0
    while overlap(hi) > alpha and hi < 64.0:
        lo, hi = hi, hi * 2.0
    for _ in range(40):
        mid = 0.5 * (lo + hi)
        if overlap(mid) > alpha:
            lo = mid
        else:
            hi = mid
    return 0.5 * (lo + hi)


# ---------------------------------------------------------------- config 1

def config1_probs(seed: int = SEED_BASE + 1, rounds: int = 600, K: int = 4,
                  V: int = 32000, alpha: float = 0.68, logit_std: float = 2.0) -> Workload:
    """B=1 per round, ``rounds`` independent rounds batched as B sequences.

    Target rows: softmax of N(0, 2^2) logits.  Draft rows: softmax of the
    target logits plus N(0, s^2) noise with s tuned so sum(min(p, q)) ~ 0.68
    (the spec-verify card's "deliberately imperfect draft", sum(min) = 0.678).
    Draft tokens are drawn from q; greedy mode uses the same rows and tokens.
    """
    rng = _rng(seed)
    B = rounds
    kb = np.full(B, K, np.int64)
    t0, d0, cu = _layout(B, kb)
    n_t, n_d = int((kb + 1).sum()), int(kb.sum())

    tune_rows = rng.standard_normal((8, V)) * logit_std
    tune_z = rng.standard_normal((8, V))
    sigma = _tune_noise(tune_rows, tune_z, alpha)

    target = np.empty((n_t, V), np.float32)
    draft = np.empty((n_d, V), np.float32)
    tokens = np.empty(n_d, np.int32)
    for b0 in range(0, B, _ROW_BLOCK):
        b1 = min(B, b0 + _ROW_BLOCK)
        for b in range(b0, b1):
            tl = rng.standard_normal((K + 1, V)) * logit_std
            target[t0[b]:t0[b] + K + 1] = _softmax_rows(tl).astype(np.float32)
            if K:
                dl = tl[:K] + sigma * rng.standard_normal((K, V))
                q = _softmax_rows(dl).astype(np.float32)
                draft[d0[b]:d0[b] + K] = q
                tokens[d0[b]:d0[b] + K] = _draw_from_rows(rng, q.astype(np.float64))
    u = uniforms_24bit(rng, n_t)
    return Workload("config1", "both", "f32", B, K, V, target, draft, tokens, u,
                    None, None, {"noise_sigma": sigma, "seed": seed})


# ---------------------------------------------------------------- config 2

def config2_bf16_logits(seed: int = SEED_BASE + 2, B: int = 64, K: int = 5,
                        V: int = 128256, temperature: float = 0.8,
                        logit_std: float = 3.0, n_peaks: int = 20,
                        peak_boost: float = 8.0, draft_noise: float = 1.5,
                        draft_choice: str = "sample") -> Workload:
    """Sampling from bf16 logits with a fused temperature-0.8 softmax.

    Target logits N(0, 3^2) with 20 random "peak" ids per row raised by +8;
    draft logits = target + N(0, 1.5^2); both rounded to bf16.  Draft tokens
    are drawn from softmax(draft_bf16 / T) (``draft_choice="argmax"``: the
    argmax of the bf16 draft row instead).
    """
    rng = _rng(seed)
    kb = np.full(B, K, np.int64)
    t0, d0, cu = _layout(B, kb)
    n_t, n_d = int((kb + 1).sum()), int(kb.sum())
    target = np.empty((n_t, V), np.uint16)
    draft = np.empty((n_d, V), np.uint16)
    tokens = np.empty(n_d, np.int32)
    npk = min(n_peaks, V)
    for b in range(B):
        tl = rng.standard_normal((K + 1, V), dtype=np.float32) * np.float32(logit_std)
        for i in range(K + 1):
            ids = rng.choice(V, size=npk, replace=False)
            tl[i, ids] += np.float32(peak_boost)
        target[t0[b]:t0[b] + K + 1] = f32_to_bf16_bits(tl)
        if K:
            dl = tl[:K] + np.float32(draft_noise) * rng.standard_normal((K, V), dtype=np.float32)
            dbits = f32_to_bf16_bits(dl)
            draft[d0[b]:d0[b] + K] = dbits
            if draft_choice == "argmax":
                tokens[d0[b]:d0[b] + K] = np.argmax(_bf16_bits_to_f32(dbits), axis=-1)
            else:
                q = _softmax_rows(_bf16_bits_to_f32(dbits), 1.0 / temperature)
                tokens[d0[b]:d0[b] + K] = _draw_from_rows(rng, q)
    u = uniforms_24bit(rng, n_t)
    temp = np.full(B, temperature, np.float32)
    return Workload("config2", "logits", "bf16", B, K, V, target, draft, tokens, u,
                    None, temp, {"seed": seed})


# ---------------------------------------------------------------- config 3

def config3_greedy_probs(seed: int = SEED_BASE + 3, B: int = 256, K: int = 4,
                         V: int = 152064, logit_std: float = 2.5,
                         p_match: float = 0.8, tie_every: int = 64) -> Workload:
    """Greedy verification on f32 probability rows (softmax of N(0, 2.5^2)).

    Each draft token is the row argmax with probability 0.8, else a uniformly
    random other id.  Every 64th target row carries an exact argmax tie (the
    max value copied to a second random id), so the lowest-index rule decides;
    on half of the tie rows that are draft positions the *higher* tied id is
    drafted, which verification must reject.
    """
    rng = _rng(seed)
    kb = np.full(B, K, np.int64)
    t0, d0, cu = _layout(B, kb)
    n_t, n_d = int((kb + 1).sum()), int(kb.sum())
    target = np.empty((n_t, V), np.float32)
    tokens = np.empty(n_d, np.int32)
    tie_rows = []
    for r0 in range(0, n_t, _ROW_BLOCK):
        r1 = min(n_t, r0 + _ROW_BLOCK)
        tl = rng.standard_normal((r1 - r0, V), dtype=np.float32) * np.float32(logit_std)
        target[r0:r1] = _softmax_rows(tl).astype(np.float32)
    high_tie_draft = {}
    if V > 1:
        for r in range(0, n_t, tie_every):
            row = target[r]
            i1 = int(np.argmax(row))
            i2 = int(rng.integers(0, V - 1))
            i2 = i2 + 1 if i2 >= i1 else i2
            row[i2] = row[i1]
            tie_rows.append(r)
            high_tie_draft[r] = bool(rng.random() < 0.5)
    for b in range(B):
        for i in range(K):
            r = t0[b] + i
            row = target[r]
            win = int(np.argmax(row))  # first occurrence of the max
            if r in high_tie_draft and high_tie_draft[r]:
                ids = np.flatnonzero(row == row[win])
                tokens[d0[b] + i] = int(ids.max())
            elif rng.random() < p_match or V == 1:
                tokens[d0[b] + i] = win
            else:
                o = int(rng.integers(0, V - 1))
                tokens[d0[b] + i] = o + 1 if o >= win else o
    return Workload("config3", "greedy", "f32", B, K, V, target, None, tokens, None,
                    None, None, {"tie_rows": tie_rows, "seed": seed})


# ---------------------------------------------------------------- config 4

def config4_ragged_probs(seed: int = SEED_BASE + 4, B: int = 32, K: int = 8,
                         V: int = 129280, zipf_s: float = 1.1,
                         draft_noise: float = 1.0) -> Workload:
    """Sampling on f32 p/q given as packed ragged rows with offsets.

    K_b ~ U{0..8} per sequence (K_b = 0 is a bonus-only round).  Target logits
    are Zipf-shaped, l_v = -s ln(rank_v) with s = 1.1 and a random rank
    permutation per row; draft logits = target + N(0, 1).
    """
    rng = _rng(seed)
    kb = rng.integers(0, K + 1, size=B).astype(np.int64)
    t0, d0, cu = _layout(B, kb)
    n_t, n_d = int((kb + 1).sum()), int(kb.sum())
    target = np.empty((n_t, V), np.float32)
    draft = np.empty((max(n_d, 0), V), np.float32)
    tokens = np.empty(n_d, np.int32)
    base = -zipf_s * np.log(np.arange(1, V + 1, dtype=np.float64))
    for b in range(B):
        k = int(kb[b])
        tl = np.empty((k + 1, V))
        for i in range(k + 1):
            tl[i] = base[rng.permutation(V)]
        target[t0[b]:t0[b] + k + 1] = _softmax_rows(tl).astype(np.float32)
        if k:
            dl = tl[:k] + draft_noise * rng.standard_normal((k, V))
            q = _softmax_rows(dl).astype(np.float32)
            draft[d0[b]:d0[b] + k] = q
            tokens[d0[b]:d0[b] + k] = _draw_from_rows(rng, q.astype(np.float64))
    u = uniforms_24bit(rng, n_t)
    return Workload("config4", "accept", "f32", B, K, V, target, draft, tokens, u,
                    cu.astype(np.int32), None, {"seed": seed})


# ---------------------------------------------------------------- config 5

def config5_mixed_f16_logits(seed: int = SEED_BASE + 5, B: int = 1024, K: int = 3,
                             V: int = 32000, logit_std: float = 2.0,
                             t_lo: float = 0.5, t_hi: float = 1.2,
                             s_lo: float = 0.3, s_hi: float = 3.0) -> Workload:
    """Mixed batch on f16 logits: even sequences greedy (T = 0), odd ones
    sampled with T ~ U[0.5, 1.2].  Logits N(0, 2^2); draft = target +
    N(0, s_b^2) with s_b ~ U[0.3, 3.0] per sequence.  Greedy sequences draft
    the argmax of their draft logits; sampled ones draw from
    softmax(draft / T_b).
    """
    rng = _rng(seed)
    kb = np.full(B, K, np.int64)
    t0, d0, cu = _layout(B, kb)
    n_t, n_d = int((kb + 1).sum()), int(kb.sum())
    target = np.empty((n_t, V), np.float16)
    draft = np.empty((n_d, V), np.float16)
    tokens = np.empty(n_d, np.int32)
    temp = np.zeros(B, np.float32)
    sig = rng.uniform(s_lo, s_hi, size=B)
    for b in range(B):
        if b % 2:
            temp[b] = np.float32(rng.uniform(t_lo, t_hi))
        tl = rng.standard_normal((K + 1, V), dtype=np.float32) * np.float32(logit_std)
        target[t0[b]:t0[b] + K + 1] = tl.astype(np.float16)
        if K:
            dl = (tl[:K] + np.float32(sig[b]) * rng.standard_normal((K, V), dtype=np.float32))
            d16 = dl.astype(np.float16)
            draft[d0[b]:d0[b] + K] = d16
            if temp[b] > 0:
                q = _softmax_rows(d16.astype(np.float32), 1.0 / float(temp[b]))
                tokens[d0[b]:d0[b] + K] = _draw_from_rows(rng, q)
            else:
                tokens[d0[b]:d0[b] + K] = np.argmax(d16.astype(np.float32), axis=-1)
    u = uniforms_24bit(rng, n_t)
    return Workload("config5", "logits", "f16", B, K, V, target, draft, tokens, u,
                    None, temp, {"draft_sigma": sig, "seed": seed})


# ---------------------------------------------------------------- greedy at B=64 K=5 V=128256

def greedy2_bf16_logits(seed: int = SEED_BASE + 6, B: int = 64, K: int = 5, V: int = 128256,
                        **kw) -> Workload:
    """Greedy verification at the sampling workload's shape: bf16 target
    logits N(0, 3^2) with 20 peaks per row raised by +8, and each draft token
    the argmax of its bf16 draft row (target + N(0, 1.5^2)), the drafter's own
    greedy choice.  Only the target rows are kept: greedy verification reads
    no draft row."""
    wl = config2_bf16_logits(seed=seed, B=B, K=K, V=V, draft_choice="argmax", **kw)
    return Workload("greedy2", "greedy", "bf16", B, K, V, wl.target, None, wl.tokens, None,
                    None, None, {"seed": seed})


_BUILDERS = {
    "config1": config1_probs,
    "config2": config2_bf16_logits,
    "config3": config3_greedy_probs,
    "config4": config4_ragged_probs,
    "config5": config5_mixed_f16_logits,
    "greedy2": greedy2_bf16_logits,
}


def make_config(name: str, **overrides) -> Workload:
    """Build a workload by name; keyword overrides scale it down for tests."""
    return _BUILDERS[name](**overrides)
