"""Device-resident speculative decoding rounds around the verification kernel.

One round for B sequences (TensorSharp speculative_decoding.md, "The shared
runtime"; the spec-verify card, "Usage"):

1. draft K tokens, one drafter step per position (greedy: the argmax of the
   drafter's logits; sampling: an inverse-CDF draw from softmax(logits / T)
   with an explicit uniform, taken by the verification kernel as the bonus
   draw of a one-row, no-draft sequence);
2. one target pass scores the K + 1 positions (the committed prefix and each
   draft prefix);
3. verification in one kernel launch (``sv_verify_greedy`` or
   ``sv_accept_from_logits``) returns the accepted length n and the next
   token per sequence;
4. commit: drafts 0..n-1 stay where they were written, the next token goes at
   position n, the length grows by n + 1.

Nothing synchronises with the host inside a round, so a round can be captured
once as a CUDA graph and replayed.  The model callables are the caller's:

* ``draft_fn(tokens, lengths) -> [B, V]`` logits of the next token after each
  sequence's first ``lengths[b]`` tokens;
* ``target_fn(tokens, lengths, k) -> [B, k + 1, V]`` logits after each of the
  prefixes of length ``lengths[b] + j``, j = 0..k (the drafts are already
  written at ``lengths[b] .. lengths[b] + k - 1``).

Both must be deterministic and graph-capturable (device ops on the current
stream, no host synchronisation).
"""

from __future__ import annotations

from typing import Callable, Optional

import torch

from . import api


class SpeculativeDecoder:
    def __init__(self, draft_fn: Callable, target_fn: Callable, tokens: torch.Tensor,
                 lengths: torch.Tensor, k: int, vocab: int, temperature: Optional[torch.Tensor] = None,
                 seed: int = 0):
        """``tokens`` [B, max_len] int32 (the prompts in place), ``lengths``
        [B] int32; greedy when ``temperature`` is None, else per-sequence
        sampling temperatures [B] (0 = greedy for that sequence)."""
        if tokens.dim() != 2 or tokens.dtype != torch.int32 or lengths.dtype != torch.int32:
            raise ValueError("tokens must be [B, max_len] int32 and lengths [B] int32")
        self.draft_fn, self.target_fn = draft_fn, target_fn
        self.tokens, self.lengths = tokens, lengths
        self.B, self.max_len = tokens.shape
        self.k, self.vocab = int(k), int(vocab)
        self.temperature = temperature
        self.device = tokens.device
        self.seed = int(seed) & 0x7FFFFFFF
        self.counter = torch.zeros((), dtype=torch.int64, device=self.device)  # rounds so far
        self.rows = torch.arange(self.B, device=self.device)
        self.drafts = torch.zeros(self.B, self.k, dtype=torch.int32, device=self.device)
        self.draft_logits = None
        self._no_tokens = torch.zeros(0, dtype=torch.int32, device=self.device)
        self.last = None
        self.graph = None

    # ------------------------------------------------------------------ pieces
    def _uniforms(self, stream_id: int) -> torch.Tensor:
        """[B, K + 1] uniforms k * 2^-24 from a counter-based mix of (seed,
        round, stream, sequence, position): reproducible and graph-safe."""
        K1 = self.k + 1
        idx = (self.rows[:, None] * K1 + torch.arange(K1, device=self.device)[None, :]).to(torch.int64)
        x = idx + (self.counter * 4 + stream_id) * 0x100000000 + self.seed * 0x1000000000000
        for mul, sh in ((0x5851F42D4C957F2D, 33), (0x2545F4914F6CDD1D, 29), (0x14057B7EF767814F, 31)):
            x = x ^ ((x >> sh) & ((1 << (64 - sh)) - 1))   # logical shift on int64
            x = x * (mul - (1 << 64) if mul >= (1 << 63) else mul)
        bits = (x >> 40) & 0xFFFFFF
        return bits.to(torch.float32) * (1.0 / (1 << 24))

    def _draw(self, logits: torch.Tensor, u: torch.Tensor) -> torch.Tensor:
        """Greedy argmax (lowest index on ties) or an inverse-CDF draw from
        softmax(logits / T) per sequence (T = 0 rows are greedy): the
        verification kernel itself, on one row per sequence with no drafts
        (K_b = 0: the next token is the bonus draw from that row with the
        given uniform), so the drafts come from the same fp32 weights q that
        the verification later compares against.  A row the kernel cannot
        use (NaN, no finite maximum) yields -1, written as token 0."""
        empty = logits[:0]
        no_tokens = self._no_tokens
        if self.temperature is None:
            r = api.verify_greedy(logits, no_tokens)
        else:
            r = api.accept_from_logits(logits, empty, self.temperature, no_tokens, u.contiguous())
        return r.next_token.clamp(min=0)

    def round(self):
        """One draft / verify / commit round for every sequence (no host sync)."""
        B, K = self.B, self.k
        base = self.lengths.long()
        d_logits = []
        u = self._uniforms(0)
        for j in range(K):  # drafter steps, each after the previous draft
            lg = self.draft_fn(self.tokens, self.lengths + j)
            d_logits.append(lg)
            tj = self._draw(lg, u[:, j])
            self.drafts[:, j] = tj
            self.tokens[self.rows, (base + j).clamp_(max=self.max_len - 1)] = tj
        t_logits = self.target_fn(self.tokens, self.lengths, K)  # [B, K + 1, V]
        if self.temperature is None:
            res = api.verify_greedy(t_logits.reshape(B * (K + 1), -1), self.drafts.reshape(-1))
        else:
            q = torch.stack(d_logits, dim=1).to(t_logits.dtype)
            uv = self._uniforms(1)
            res = api.accept_from_logits(t_logits.reshape(B * (K + 1), -1), q.reshape(B * K, -1),
                                         self.temperature, self.drafts.reshape(-1), uv.reshape(-1))
        n = res.n_accepted.long()
        pos = (base + n).clamp_(max=self.max_len - 1)
        self.tokens[self.rows, pos] = res.next_token.clamp(min=0)
        self.lengths += (n + 1).to(torch.int32)
        self.counter += 1
        self.last = res
        return res

    # ------------------------------------------------------------------ graphs
    def capture(self):
        """Capture one round as a CUDA graph (after one eager warm-up round on
        a scratch copy of the state, which the caller's tensors do not see)."""
        saved_t, saved_l, saved_c = self.tokens.clone(), self.lengths.clone(), self.counter.clone()
        s = torch.cuda.Stream(self.device)
        s.wait_stream(torch.cuda.current_stream(self.device))
        with torch.cuda.stream(s):
            self.round()  # warm-up (allocations, library load) outside the graph
        torch.cuda.current_stream(self.device).wait_stream(s)
        torch.cuda.synchronize(self.device)
        self.tokens.copy_(saved_t)
        self.lengths.copy_(saved_l)
        self.counter.copy_(saved_c)
        self.graph = torch.cuda.CUDAGraph()
        # the library's launch queries kernel attributes: relaxed capture mode
        with torch.cuda.graph(self.graph, stream=s, capture_error_mode="relaxed"):
            self.round()
        torch.cuda.synchronize(self.device)
        return self.graph

    def run(self, rounds: int, graph: bool = True):
        """``rounds`` rounds, replaying the captured graph when ``graph``."""
        if graph and self.graph is None:
            self.capture()
        for _ in range(rounds):
            if graph:
                self.graph.replay()
            else:
                self.round()
        return self.tokens, self.lengths
