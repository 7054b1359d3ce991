"""Pins of the oracle's top-k / top-p filters (llmstudio.ru section 38: the
sampling pipeline is temperature, then top-k, then top-p, then
normalisation, applied alike to the target's p and the draft's q).

Each pin comes from outside the oracle: brute force over every subset of a
tiny vocabulary (the nucleus is the smallest set of tokens whose probability
reaches p), a closed form in the temperature, hand-worked rows with ties, and
the reduction of top-k = 1 to greedy verification.  The planted mistakes at
the bottom show that the pins catch a wrong comparison, a dropped
renormalisation, a swapped order or a missing temperature.
"""

import inspect
import itertools
import math
import textwrap

import numpy as np
import pytest

import oracle
import oracle.sampler_filter as sf
import oracle.spec_verify as spv

F32 = np.float32


def kept(x, floor):
    return set(np.flatnonzero(np.asarray(x, np.float64) >= floor).tolist())


# ------------------------------------------------------------------ top-k

def test_top_k_keeps_exactly_k_distinct_and_all_ties():
    rng = np.random.default_rng(1)
    for _ in range(50):
        V = int(rng.integers(2, 40))
        x = rng.permutation(V).astype(np.float64) - V / 2  # distinct
        k = int(rng.integers(1, V))
        f = sf.top_k_floor(x, k)
        assert kept(x, f) == set(np.argsort(-x)[:k].tolist())
    x = np.array([5.0, 3.0, 3.0, 1.0])
    assert sf.top_k_floor(x, 2) == 3.0 and kept(x, 3.0) == {0, 1, 2}  # the tie at the boundary stays
    assert sf.top_k_floor(x, 1) == 5.0
    for k in (None, 0, -3, 4, 9):
        assert sf.top_k_floor(x, k) == -math.inf  # disabled, or k covers the row
    y = np.array([np.nan, 2.0, 1.0])
    assert sf.top_k_floor(y, 1) == 2.0
    assert sf.top_k_floor(np.array([np.nan, np.nan, 1.0]), 2) == -math.inf  # one non-NaN logit


# ------------------------------------------------------------------ top-p

def _nucleus_brute_force(x, T, p):
    """The smallest set of tokens whose probability reaches p, by trying every
    subset (distinct logits: the largest-mass set of that size is unique)."""
    w = np.exp((x - x.max()) / T)
    prob = w / w.sum()
    V = len(x)
    for size in range(1, V + 1):
        best = None
        for S in itertools.combinations(range(V), size):
            m = prob[list(S)].sum()
            if m >= p and (best is None or m > best[0]):
                best = (m, set(S))
        if best is not None:
            return best[1]
    return set(range(V))


def test_top_p_is_the_nucleus_by_brute_force():
    rng = np.random.default_rng(2)
    checked = 0
    for _ in range(300):
        V = int(rng.integers(1, 8))
        x = rng.normal(0, 2, V)
        T = float(rng.choice([0.5, 1.0, 1.7]))
        p = float(rng.uniform(0.05, 0.99))
        f, near, bad = sf.filter_floor(x, T, None, p)
        assert not bad
        if near:
            continue
        assert kept(x, f) == _nucleus_brute_force(x, T, p), (x, T, p)
        checked += 1
    assert checked > 250


def test_top_p_closed_form_in_the_temperature():
    # two tokens, logits 0 and -d: the second is kept iff 1 < p (1 + e^(-d/T)),
    # i.e. iff T > d / ln(p / (1 - p))
    d, p = 2.0, 0.8
    t_star = d / math.log(p / (1 - p))
    x = np.array([0.0, -d])
    for T in (0.5, 1.0, t_star * 0.99):
        assert sf.filter_floor(x, T, None, p)[0] == 0.0
    for T in (t_star * 1.01, 2.0, 5.0):
        assert sf.filter_floor(x, T, None, p)[0] == -d


def test_top_p_ties_are_kept_or_dropped_together():
    x = np.array([2.0, 2.0, 0.0])  # weights 1, 1, e^-2 at T = 1
    assert sf.filter_floor(x, 1.0, None, 0.3)[0] == 2.0  # both 2s, though one reaches 0.3
    assert sf.filter_floor(x, 1.0, None, 0.99)[0] == 0.0  # mass above 0 is 2 < 0.99 (2 + e^-2)
    assert sf.filter_floor(np.zeros(6), 1.0, None, 1e-3)[0] == 0.0  # one group: all kept
    # every equal logit carries its own weight: three tokens at 0 hold 3/e of
    # the mass 1 + 3/e = 2.10, so the top token alone is under half of it
    assert sf.filter_floor(np.array([1.0, 0.0, 0.0, 0.0]), 1.0, None, 0.5)[0] == 0.0


def test_mass_above_exactly_p_drops_the_token():
    # the nucleus is the smallest prefix whose mass reaches p: once the
    # tokens above a token already carry exactly p Z, that token is not needed
    x = np.array([0.0, -1.0, -2.0])
    w = np.exp(x)
    Z, above2 = math.fsum(w), float(np.cumsum(w)[1])
    p = above2 / Z
    for _ in range(8):  # the p whose product with Z is exactly the mass above token 2
        if p * Z == above2:
            break
        p = np.nextafter(p, 1.0 if p * Z < above2 else 0.0)
    assert p * Z == above2
    assert sf.filter_floor(x, 1.0, None, float(p))[0] == -1.0
    assert sf.filter_floor(x, 1.0, None, float(np.nextafter(p, 1.0)))[0] == -2.0


def test_top_k_then_top_p_on_the_renormalised_set():
    # probabilities 0.5, 0.3, 0.2 (T = 1): top-p 0.6 alone keeps two tokens;
    # after top-k 2 the kept mass is 0.8, and 0.6 of it (0.48) is reached by
    # the first token alone
    x = np.log(np.array([0.5, 0.3, 0.2]))
    assert sf.filter_floor(x, 1.0, None, 0.6)[0] == x[1]
    assert sf.filter_floor(x, 1.0, 2, 0.6)[0] == x[0]
    assert sf.filter_floor(x, 1.0, 2, None)[0] == x[1]
    assert sf.filter_floor(x, 1.0, 3, 0.6)[0] == x[1]  # k covers the row: top-p alone


def test_disabled_invalid_and_degenerate_rows():
    x = np.array([1.0, 0.0, -1.0])
    assert sf.filter_floor(x, 1.0, None, None) == (-math.inf, False, False)
    assert sf.filter_floor(x, 1.0, None, 1.0)[0] == -math.inf
    assert sf.filter_floor(x, 1.0, None, 1.5)[0] == -math.inf
    for p in (0.0, -0.5, math.nan):
        f, near, bad = sf.filter_floor(x, 1.0, 5, p)
        assert bad and math.isnan(f)
    assert sf.filter_floor(np.array([math.inf, 1.0]), 1.0, 1, 0.5)[0] == -math.inf
    assert sf.filter_floor(np.array([math.nan, math.nan]), 1.0, 1, 0.5)[0] == -math.inf
    assert sf.filter_floor(np.array([-math.inf, -math.inf]), 1.0, 1, 0.5)[0] == -math.inf
    # NaN takes no part: the same floor as without it
    y = np.array([1.0, math.nan, 0.0, -1.0])
    assert sf.filter_floor(y, 1.0, 2, 0.9)[0] == sf.filter_floor(x, 1.0, 2, 0.9)[0]
    # -inf logits count for top-k but weigh nothing
    z = np.array([0.0, -math.inf, -math.inf])
    assert sf.filter_floor(z, 1.0, 2, None)[0] == -math.inf
    assert sf.filter_floor(z, 1.0, None, 0.999)[0] == 0.0


def test_near_flag_and_both_floors_valid_at_the_boundary():
    # weights 1 and 1/3 (T = 1): with p = 3/4, p Z = 1 = the mass above the
    # second token, so either answer is correct to within rounding
    x = np.array([0.0, -math.log(3.0)])
    f, near, _ = sf.filter_floor(x, 1.0, None, 0.75)
    assert near
    assert sf.floor_is_valid(x, 1.0, None, 0.75, 0.0)
    assert sf.floor_is_valid(x, 1.0, None, 0.75, x[1])
    f, near, _ = sf.filter_floor(x, 1.0, None, 0.5)
    assert not near and f == 0.0
    assert not sf.floor_is_valid(x, 1.0, None, 0.5, x[1])
    assert not sf.floor_is_valid(x, 1.0, None, 0.5, 0.5)  # not a value of the row


# ------------------------------------------------------------------ verification with filters

def _logit_case(B, K, V, seed, T=0.9, distinct=True):
    rng = np.random.default_rng(seed)
    tgt = rng.normal(0, 2, (B * (K + 1), V)).astype(F32)
    drf = (tgt[np.arange(B * (K + 1)) % (K + 1) != K] + rng.normal(0, 1, (B * K, V))).astype(F32)
    tok = rng.integers(0, V, B * K).astype(np.int32)
    u = rng.random(B * (K + 1)).astype(F32)
    temp = np.full(B, T, F32)
    return tgt, drf, tok, u, temp


def test_disabled_filters_change_nothing():
    B, K, V = 20, 3, 40
    tgt, drf, tok, u, temp = _logit_case(B, K, V, 3)
    a = oracle.accept_from_logits(tgt, drf, "f32", temp, tok, u, B, K)
    b = oracle.accept_from_logits(tgt, drf, "f32", temp, tok, u, B, K,
                                  top_k=np.full(B, V, np.int32), top_p=np.ones(B, F32))
    for f in ("n_accepted", "next_token", "status"):
        assert np.array_equal(getattr(a, f), getattr(b, f))


def test_top_k_one_is_greedy_verification():
    # with top-k 1 every sampled row is a point mass on its argmax: a draft is
    # accepted iff it is the target's argmax and the emitted token is the
    # target argmax at the stopping row, whatever the uniforms
    B, K, V = 40, 4, 30
    tgt, drf, tok, u, temp = _logit_case(B, K, V, 4)
    for b in range(B):  # make about half the drafts the target argmax
        for i in range(K):
            if (b + i) % 2 == 0:
                tok[b * K + i] = int(np.argmax(tgt[b * (K + 1) + i]))
    s = oracle.accept_from_logits(tgt, drf, "f32", temp, tok, u, B, K, top_k=np.ones(B, np.int32))
    g = oracle.verify_greedy(tgt, "f32", tok, B, K)
    assert np.array_equal(s.n_accepted, g.n_accepted)
    assert np.array_equal(s.next_token, g.next_token)
    assert (s.n_accepted > 0).any() and (s.n_accepted < K).any()


def test_invalid_top_p_is_a_bad_value_at_row_zero():
    B, K, V = 3, 2, 10
    tgt, drf, tok, u, temp = _logit_case(B, K, V, 5)
    r = oracle.accept_from_logits(tgt, drf, "f32", temp, tok, u, B, K,
                                  top_p=np.array([0.5, 0.0, np.nan], F32))
    assert r.status[1] == oracle.BAD_VALUE and r.status[2] == oracle.BAD_VALUE
    assert r.next_token[1] == -1 and r.n_accepted[1] == 0
    assert r.status[0] & oracle.BAD_VALUE == 0


def _filtered_probs(x, T, k, p):
    f, _, _ = sf.filter_floor(x, T, k, p)
    w = np.where(x >= f, np.exp((x - x.max()) / T), 0.0)
    return w / w.sum()


def test_first_token_law_with_filters():
    """Drafts drawn from the filtered q, verified against the filtered p: the
    first emitted token follows the filtered p (llmstudio.ru sections 15-17
    with section 38's effective distributions)."""
    from scipy.stats import chi2
    rng = np.random.default_rng(6)
    V, T, k, p = 12, 1.0, 6, 0.8
    tl = rng.normal(0, 1.5, V)
    dl = tl + rng.normal(0, 1.5, V)
    pt = _filtered_probs(tl, T, k, p)
    qt = _filtered_probs(dl, T, k, p)
    N = 20000
    tgt = np.tile(np.stack([tl, tl]).astype(F32), (N, 1))
    drf = np.tile(dl.astype(F32)[None], (N, 1))
    tok = rng.choice(V, size=N, p=qt).astype(np.int32)
    u = rng.random(2 * N).astype(F32)
    r = oracle.accept_from_logits(tgt, drf, "f32", np.full(N, T, F32), tok, u, N, 1,
                                  top_k=np.full(N, k, np.int32), top_p=np.full(N, p, F32))
    first = np.where(r.n_accepted > 0, tok, r.next_token)
    counts = np.bincount(first, minlength=V).astype(float)
    keep = pt > 0
    assert counts[~keep].sum() == 0  # filtered-out tokens never come out
    exp = pt[keep] * N
    stat = float(((counts[keep] - exp) ** 2 / exp).sum())
    assert 1.0 - chi2.cdf(stat, keep.sum() - 1) > 1e-3


def pin_brute_force():
    test_top_p_is_the_nucleus_by_brute_force()


def pin_order():
    test_top_k_then_top_p_on_the_renormalised_set()


def pin_ties():
    test_mass_above_exactly_p_drops_the_token()
    test_top_p_ties_are_kept_or_dropped_together()
    test_top_k_keeps_exactly_k_distinct_and_all_ties()


def pin_temperature():
    test_top_p_closed_form_in_the_temperature()


def pin_law():
    test_first_token_law_with_filters()


FILTER_MUTATIONS = [
    # (module, function, original text, planted mistake, pins expected to catch it)
    (sf, "filter_floor", "np.flatnonzero(above < pz)", "np.flatnonzero(above <= pz)", [pin_ties]),
    (sf, "filter_floor", "keep = vals >= floor", "keep = vals >= -math.inf", [pin_order]),
    (sf, "top_k_floor", "if seen >= k:", "if seen > k:", [pin_ties, pin_order]),
    (sf, "_weights", "np.exp((vals - vals[0]) / T)", "np.exp(vals - vals[0])", [pin_temperature]),
    (sf, "_weights", "counts * np.exp(", "np.exp(", [pin_ties]),
    (sf, "filter_floor", "J = int(np.flatnonzero(above < pz)[-1])",
     "J = int(np.flatnonzero(above < pz)[-1]) + (1 if int(np.flatnonzero(above < pz)[-1]) + 1 < vals.size else 0)",
     [pin_brute_force]),
    (spv, "accept_from_logits", "getter(draft, d0, T, fk, fp, \"q\")", "getter(draft, d0, T, tag=\"q\")", [pin_law]),
]


@pytest.mark.parametrize("mod,fn_name,old,new,catchers", FILTER_MUTATIONS,
                         ids=[f"{m[1]}:{i}" for i, m in enumerate(FILTER_MUTATIONS)])
def test_planted_filter_mistake_is_caught(monkeypatch, mod, fn_name, old, new, catchers):
    src = textwrap.dedent(inspect.getsource(getattr(mod, fn_name)))
    assert src.count(old) >= 1, (fn_name, old)
    ns = dict(vars(mod))
    exec(compile(src.replace(old, new, 1), f"<mutant {fn_name}>", "exec"), ns)
    monkeypatch.setattr(mod, fn_name, ns[fn_name])
    if hasattr(oracle, fn_name):
        monkeypatch.setattr(oracle, fn_name, ns[fn_name])
    caught = []
    for pin in catchers:
        try:
            pin()
        except AssertionError:
            caught.append(pin.__name__)
    assert caught, f"no pin caught the mutation of {fn_name}: {old!r} -> {new!r}"
