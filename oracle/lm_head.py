"""The LM head in front of verification (test infrastructure).

TEST INFRASTRUCTURE ONLY: the rules of the package docstring apply (tests,
``smoke()`` and the bench's CPU legs import it; the product never does).

llmstudio.ru, "Как работает speculative decoding и MTP при инференсе LLM",
section 21: the logits of the verified positions are their hidden states
times the vocabulary projection, computed for all positions of a verification
batch at once; section 22: greedy verification needs only each row's argmax,
sampled verification the whole distribution after the sampler transforms.
TensorSharp speculative_decoding.md, "DFlash and DFlash2": a drafter borrows
the target's LM head, so the draft positions use the same projection.

Readings this file fixes:

* States ``H`` are laid out like the verification rows: target states
  ``[sum(K_b + 1), d]`` (row ``i`` of a sequence is the state after the
  committed token and drafts ``0..i-1``), draft states ``[sum K_b, d]``;
  the projection ``W`` is ``[V, d]`` (row ``v`` is token ``v``'s output
  embedding) and ``logits = H W^T``.
* ``H`` and ``W`` are stored as bf16 (the storage of a served LM head, given
  here as uint16 bit patterns, or f32); the products are summed in fp64, so
  these logits are the exact dot products up to one fp64 rounding per term.
* Everything after the logits is ``spec_verify.accept_from_logits`` (or
  ``verify_greedy`` for an all-greedy batch) on those fp64 logits, with the
  per-sequence temperature and the optional top-k / top-p filters.
"""

from __future__ import annotations

from typing import Optional

import numpy as np

from .spec_verify import Result, accept_from_logits, decode_rows, verify_greedy


def lm_head_logits(h: np.ndarray, w: np.ndarray, dtype: str = "bf16") -> np.ndarray:
    """``H W^T`` in fp64 for states ``h`` ``[rows, d]`` and projection ``w``
    ``[V, d]`` stored in ``dtype``."""
    hd = decode_rows(h, dtype).reshape(h.shape)
    wd = decode_rows(w, dtype).reshape(w.shape)
    return hd @ wd.T


def accept_lm_head(h_target: np.ndarray, h_draft: np.ndarray, w: np.ndarray, dtype: str,
                   temperature: np.ndarray, tokens: np.ndarray, u: np.ndarray, B: int, K: int,
                   cu_k: Optional[np.ndarray] = None, top_k: Optional[np.ndarray] = None,
                   top_p: Optional[np.ndarray] = None) -> Result:
    """Verification of B sequences from their hidden states: the target and
    the draft rows' logits through the one LM head ``w``, then the mixed
    greedy / sampled verification of ``accept_from_logits``."""
    lt = lm_head_logits(h_target, w, dtype)
    ld = lm_head_logits(h_draft, w, dtype) if h_draft.shape[0] else np.zeros((0, w.shape[0]))
    return accept_from_logits(lt, ld, "f64", temperature, tokens, u, B, K, cu_k, top_k=top_k, top_p=top_p)


def verify_greedy_lm_head(h_target: np.ndarray, w: np.ndarray, dtype: str, tokens: np.ndarray,
                          B: int, K: int, cu_k: Optional[np.ndarray] = None) -> Result:
    """Greedy verification from hidden states (only the argmax of each row's
    logits matters, section 22)."""
    return verify_greedy(lm_head_logits(h_target, w, dtype), "f64", tokens, B, K, cu_k)
