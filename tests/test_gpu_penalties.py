"""Penalties ahead of verification (llmstudio.ru sections 38-39) on the GPU
against the oracle: the rewritten rows bit for bit (an integer-valued
comparison of the stored bits), the per-sequence statuses, and the
verification that follows them."""

import numpy as np
import pytest

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():  # pragma: no cover
    pytestmark = pytest.mark.skip("needs a GPU")
else:
    pytestmark = pytest.mark.gpu

import __graft_entry__  # noqa: E402
import oracle  # noqa: E402
import workloads  # noqa: E402
from oracle import penalties as pen  # noqa: E402

F32 = np.float32


@pytest.fixture(scope="module", autouse=True)
def built():
    __graft_entry__.build()


def sv():
    import speculative_decoding_verification_decode_gb300 as m
    return m


def H():
    import gpu_helpers
    return gpu_helpers


def _histories(rng, B, V, lo=0, hi=400):
    lens = rng.integers(lo, hi, B)
    off = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    # repeats (a small pool per sequence) and a few ids outside [0, V)
    tok = np.concatenate([rng.choice(rng.integers(-3, V + 3, 60), n) for n in lens]).astype(np.int32)
    return off, tok


def _params(rng, B):
    return (rng.uniform(1.0, 1.8, B).astype(F32), rng.uniform(0.0, 0.6, B).astype(F32),
            rng.uniform(0.0, 1.5, B).astype(F32))


def _run(wl, off, htok, rep, fr, pr):
    tg = H().to_dev(wl.target, wl.dtype).clone()
    dr = H().to_dev(wl.draft, wl.dtype).clone()
    st = sv().apply_penalties(tg, dr, H().to_dev(wl.tokens), *(torch.from_numpy(x).cuda() for x in (rep, fr, pr)),
                              hist_offsets=None if off is None else torch.from_numpy(off).cuda(),
                              hist_tokens=None if htok is None else torch.from_numpy(htok).cuda(),
                              cu_k=H().to_dev(wl.cu_k), k=wl.K if wl.cu_k is not None else None)
    torch.cuda.synchronize()
    bits = lambda t: t.view(torch.int16 if t.element_size() == 2 else torch.int32).cpu().numpy()
    return tg, dr, bits(tg), bits(dr), st.cpu().numpy().astype(np.uint32)


def _storage_bits(a):
    return np.ascontiguousarray(a).view(np.int16 if a.dtype.itemsize == 2 else np.int32)


@pytest.mark.parametrize("name,kw", [("config2", dict(B=10, K=5, V=3001)),    # bf16
                                     ("config5", dict(B=12, V=2003)),          # f16
                                     ("config4", dict(B=9, V=4001)),           # f32 probabilities as rows, ragged
                                     ("config1", dict(rounds=8, V=1000))])     # f32
def test_rows_bit_exact(name, kw):
    wl = workloads.make_config(name, **kw)
    rng = np.random.default_rng(len(name) + wl.B)
    off, htok = _histories(rng, wl.B, wl.V)
    rep, fr, pr = _params(rng, wl.B)
    rep[0], fr[0], pr[0] = 1.0, 0.0, 0.0  # a neutral sequence
    rep[1] = np.nan                      # an unusable parameter
    off[3] = off[2] - 1 if off[2] > 0 else off[3]  # sequence 2's history ends before it starts
    _, _, tbits, dbits, st = _run(wl, off, htok, rep, fr, pr)
    dtype = wl.dtype if wl.mode != "accept" and wl.mode != "both" else "f32"
    rt, rd, rst = pen.penalize_rows(wl.target, wl.draft, dtype, off, htok, wl.tokens, wl.B, wl.K, wl.cu_k,
                                    rep, fr, pr)
    assert np.array_equal(st, rst)
    assert np.array_equal(tbits, _storage_bits(rt))
    assert np.array_equal(dbits, _storage_bits(rd))
    assert (st == 0).sum() >= wl.B - 3


def test_no_history_and_capacity():
    wl = workloads.make_config("config2", B=3, K=5, V=20011)
    rng = np.random.default_rng(9)
    rep, fr, pr = _params(rng, wl.B)
    _, _, tbits, dbits, st = _run(wl, None, None, rep, fr, pr)  # drafts only
    empty = np.zeros(wl.B + 1, np.int32)
    rt, rd, rst = pen.penalize_rows(wl.target, wl.draft, "bf16", empty, np.zeros(0, np.int32), wl.tokens, wl.B,
                                    wl.K, None, rep, fr, pr)
    assert np.array_equal(st, rst) and np.array_equal(tbits, _storage_bits(rt))
    assert np.array_equal(dbits, _storage_bits(rd))
    # sequence 1 holds 8192 distinct history ids plus new drafts: over capacity
    big = np.arange(pen.MAX_DISTINCT, dtype=np.int32)
    off = np.array([0, 5, 5 + len(big), 10 + len(big)], np.int32)
    htok = np.concatenate([big[:5], big, big[:5]]).astype(np.int32)
    tok = wl.tokens.copy()
    tok[5:10] = pen.MAX_DISTINCT + np.arange(5)  # new ids for sequence 1
    wl.tokens = tok
    _, _, tbits, dbits, st = _run(wl, off, htok, rep, fr, pr)
    rt, rd, rst = pen.penalize_rows(wl.target, wl.draft, "bf16", off, htok, tok, wl.B, wl.K, None, rep, fr, pr)
    assert list(rst) == [0, pen.BAD_LAYOUT, 0]
    assert np.array_equal(st, rst) and np.array_equal(tbits, _storage_bits(rt))


def test_verification_after_penalties():
    """Penalties then the logits verification on the GPU, against the oracle's
    penalties then its verification: rows equal, decisions equal outside the
    softmax band, draws outside the boundary band."""
    wl = workloads.make_config("config2", B=16, K=5, V=9001)
    rng = np.random.default_rng(10)
    off, htok = _histories(rng, wl.B, wl.V)
    # strong penalties on the drafted ids so that decisions move
    hist = [np.concatenate([htok[off[b]:off[b + 1]], wl.tokens[b * wl.K:(b + 1) * wl.K]]) for b in range(wl.B)]
    off = np.concatenate([[0], np.cumsum([len(h) for h in hist])]).astype(np.int32)
    htok = np.concatenate(hist).astype(np.int32)
    rep, fr, pr = (np.full(wl.B, 1.5, F32), np.full(wl.B, 0.3, F32), np.full(wl.B, 1.0, F32))
    tg, dr, tbits, _, st = _run(wl, off, htok, rep, fr, pr)
    assert (st == 0).all()
    r = sv().accept_from_logits(tg, dr, torch.from_numpy(wl.temperature).cuda(), H().to_dev(wl.tokens),
                                H().to_dev(wl.uniforms))
    torch.cuda.synchronize()
    res = oracle.Result(r.n_accepted.cpu().numpy(), r.next_token.cpu().numpy(),
                        r.status.cpu().numpy().astype(np.uint32))
    rt, rd, _ = pen.penalize_rows(wl.target, wl.draft, "bf16", off, htok, wl.tokens, wl.B, wl.K, None, rep, fr, pr)
    assert np.array_equal(tbits, _storage_bits(rt))
    ref = oracle.accept_from_logits(rt, rd, "bf16", wl.temperature, wl.tokens, wl.uniforms, wl.B, wl.K)
    H().assert_softmax_agreement(res, ref, "after penalties")
    plain = oracle.accept_from_logits(wl.target, wl.draft, "bf16", wl.temperature, wl.tokens, wl.uniforms,
                                      wl.B, wl.K)
    print(f"accepted length changed by the penalties on {int((plain.n_accepted != ref.n_accepted).sum())} "
          f"of {wl.B} sequences")
