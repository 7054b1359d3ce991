"""Seeded hidden states and an LM-head projection for verification from
states (llmstudio.ru section 21: logits = states times the vocabulary
projection; TensorSharp speculative_decoding.md, "DFlash and DFlash2": the
drafter borrows the target's LM head).

Data only, like the rest of this package: the matrix product and softmax
below only draw the draft tokens; none of it is the verification arithmetic.
"""

from __future__ import annotations

import dataclasses

import numpy as np

from .configs import SEED_BASE, _draw_from_rows, _rng, _softmax_rows, f32_to_bf16_bits, uniforms_24bit


@dataclasses.dataclass
class LMHeadWorkload:
    B: int
    K: int
    V: int
    d: int
    h_target: np.ndarray  # [B (K+1), d] bf16 bits (uint16)
    h_draft: np.ndarray   # [B K, d] bf16 bits
    w: np.ndarray         # [V, d] bf16 bits: row v is token v's output embedding
    tokens: np.ndarray    # [B K] int32, drawn from the draft's softmax(logits / T)
    uniforms: np.ndarray  # [B (K+1)] f32 24-bit uniforms
    temperature: np.ndarray  # [B] f32
    dtype: str = "bf16"
    cu_k: None = None


def make_lm_head(seed: int = SEED_BASE + 7, B: int = 64, K: int = 5, V: int = 128256, d: int = 4096,
                 temperature: float = 0.8, logit_std: float = 3.0, draft_noise: float = 0.5) -> LMHeadWorkload:
    """States N(0, 1); projection N(0, (logit_std^2 / d)) so the logits have
    standard deviation ``logit_std`` (the config 2 rows' spread); draft states
    = target states + N(0, draft_noise^2); all rounded to bf16.  Draft tokens
    are drawn from softmax(draft logits / T) (logits in fp32)."""
    rng = _rng(seed)
    w32 = rng.standard_normal((V, d), dtype=np.float32) * np.float32(logit_std / np.sqrt(d))
    w = f32_to_bf16_bits(w32)
    wf = (w.astype(np.uint32) << 16).view(np.float32)
    ht32 = rng.standard_normal((B * (K + 1), d), dtype=np.float32)
    ht = f32_to_bf16_bits(ht32)
    rows_d = np.array([b * (K + 1) + i for b in range(B) for i in range(K)], np.int64)
    hd32 = ht32[rows_d] + np.float32(draft_noise) * rng.standard_normal((B * K, d), dtype=np.float32)
    hd = f32_to_bf16_bits(hd32)
    tokens = np.empty(B * K, np.int32)
    for s in range(0, B * K, 64):
        hdf = (hd[s:s + 64].astype(np.uint32) << 16).view(np.float32)
        q = _softmax_rows(hdf @ wf.T, 1.0 / temperature)
        tokens[s:s + 64] = _draw_from_rows(rng, q)
    u = uniforms_24bit(rng, B * (K + 1))
    return LMHeadWorkload(B, K, V, d, ht, hd, w, tokens, u, np.full(B, temperature, np.float32))
