"""Speculative decoding rounds end to end (draft, verify on the GPU, commit).

Greedy: speculative decoding with any drafter reproduces plain greedy
decoding of the target exactly (spec-verify card, "Method": "all K matched
emit argmax(target_K)"; the brute-force greedy pin of the oracle, now through
the whole loop and a CUDA graph).  Sampling: the first token a round emits
follows the target's distribution whatever the drafter (llmstudio.ru,
sections 15-17: the accept / resample rule preserves p).
"""

import numpy as np
import pytest

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():  # pragma: no cover - CPU-only runs
    pytestmark = pytest.mark.skip("needs a GPU")
else:
    pytestmark = pytest.mark.gpu

import __graft_entry__  # noqa: E402

DEV = torch.device("cuda", 0)


@pytest.fixture(scope="module", autouse=True)
def built():
    __graft_entry__.build()


class TableModel:
    """Next-token logits as a fixed function of the last two tokens (a table
    row chosen by a hash of them): deterministic and graph-capturable."""

    def __init__(self, V, H, seed, scale=2.0, table=None):
        g = torch.Generator().manual_seed(seed)
        self.table = (torch.randn(H, V, generator=g) * scale if table is None else table).to(DEV)
        self.H = H

    def next_logits(self, tokens, lengths):
        B = tokens.shape[0]
        rows = torch.arange(B, device=DEV)
        t1 = tokens[rows, (lengths.long() - 1).clamp(min=0)].long()
        t2 = tokens[rows, (lengths.long() - 2).clamp(min=0)].long()
        return self.table[(t1 * 1000003 + t2 * 7919) % self.H]

    def rows(self, tokens, lengths, k):
        return torch.stack([self.next_logits(tokens, lengths + j) for j in range(k + 1)], dim=1)


def plain_greedy(model, prompt, plen, n):
    tok = prompt.clone()
    lens = torch.full((tok.shape[0],), plen, dtype=torch.int32, device=DEV)
    rows = torch.arange(tok.shape[0], device=DEV)
    for _ in range(n):
        t = model.next_logits(tok, lens).argmax(dim=-1).to(torch.int32)
        tok[rows, lens.long()] = t
        lens += 1
    return tok


def _prompts(B, L, V, seed, plen=3):
    g = torch.Generator().manual_seed(seed)
    tok = torch.zeros(B, L, dtype=torch.int32)
    tok[:, :plen] = torch.randint(0, V, (B, plen), generator=g, dtype=torch.int32)
    return tok.to(DEV), torch.full((B,), plen, dtype=torch.int32, device=DEV)


@pytest.mark.parametrize("drafter", ["perfect", "noisy", "unrelated"])
@pytest.mark.parametrize("graph,K", [(False, 4), (True, 4), (True, 9)])
def test_speculative_greedy_reproduces_plain_greedy(drafter, graph, K):
    """K = 9 takes the row-parallel plan (long drafts), inside the graph."""
    from speculative_decoding_verification_decode_gb300.decoder import SpeculativeDecoder
    V, H, B, R = 97, 211, 48, 10
    target = TableModel(V, H, seed=1)
    if drafter == "perfect":
        draft = target
    elif drafter == "noisy":
        g = torch.Generator().manual_seed(2)
        draft = TableModel(V, H, seed=0, table=target.table.cpu() + torch.randn(H, V, generator=g) * 1.5)
    else:
        draft = TableModel(V, H, seed=3)
    L = 3 + R * (K + 1) + 1
    tok, lens = _prompts(B, L, V, seed=4)
    ref = plain_greedy(target, tok, 3, R * (K + 1))
    dec = SpeculativeDecoder(draft.next_logits, target.rows, tok, lens, K, V)
    dec.run(R, graph=graph)
    out, ln = dec.tokens.cpu().numpy(), dec.lengths.cpu().numpy()
    ref = ref.cpu().numpy()
    assert (ln >= 3 + R).all() and (ln <= 3 + R * (K + 1)).all()
    if drafter == "perfect":
        assert (ln == 3 + R * (K + 1)).all()  # every draft accepted, every round
    for b in range(B):
        assert np.array_equal(out[b, :ln[b]], ref[b, :ln[b]]), b


def test_speculative_sampling_first_token_law():
    from speculative_decoding_verification_decode_gb300.decoder import SpeculativeDecoder
    V, H, B, K = 12, 5, 16384, 3
    target = TableModel(V, H, seed=11, scale=1.5)
    draft = TableModel(V, H, seed=12, scale=1.5)  # a poor drafter: many rejections
    tok = torch.zeros(B, 16, dtype=torch.int32, device=DEV)
    tok[:, :2] = torch.tensor([5, 7], dtype=torch.int32, device=DEV)  # one shared prompt
    lens = torch.full((B,), 2, dtype=torch.int32, device=DEV)
    T = torch.full((B,), 0.9, dtype=torch.float32, device=DEV)
    dec = SpeculativeDecoder(draft.next_logits, target.rows, tok, lens, K, V, temperature=T, seed=5)
    dec.run(1, graph=True)
    first = dec.tokens[:, 2].cpu().numpy()
    logit = target.next_logits(tok[:1].clone(), torch.tensor([2], dtype=torch.int32, device=DEV))[0]
    p = torch.softmax(logit.double().cpu() / 0.9, dim=-1).numpy()
    counts = np.bincount(first, minlength=V)
    exp = p * B
    chi2 = float(((counts - exp) ** 2 / exp).sum())
    from scipy.stats import chi2 as chi2_dist
    pval = 1.0 - chi2_dist.cdf(chi2, V - 1)
    assert pval > 1e-3, (chi2, counts, exp)
    # and the drafter was poor enough that the resample path was exercised
    assert (dec.last.n_accepted.cpu().numpy() == 0).mean() > 0.2


def test_mixed_temperatures_keep_greedy_rows_exact():
    from speculative_decoding_verification_decode_gb300.decoder import SpeculativeDecoder
    V, H, B, K, R = 61, 101, 32, 3, 6
    target = TableModel(V, H, seed=21)
    draft = TableModel(V, H, seed=22)
    L = 3 + R * (K + 1) + 1
    tok, lens = _prompts(B, L, V, seed=23)
    ref = plain_greedy(target, tok, 3, R * (K + 1)).cpu().numpy()
    T = torch.where(torch.arange(B, device=DEV) % 2 == 0, 0.0, 0.8).to(torch.float32)
    dec = SpeculativeDecoder(draft.next_logits, target.rows, tok, lens, K, V, temperature=T, seed=7)
    dec.run(R, graph=True)
    out, ln = dec.tokens.cpu().numpy(), dec.lengths.cpu().numpy()
    for b in range(0, B, 2):  # temperature 0: greedy verification of greedy drafts
        assert np.array_equal(out[b, :ln[b]], ref[b, :ln[b]]), b
