"""Pins of the draft-length gate oracle (PocketLLM docs/dspark.md, the gate).

Each pin comes from something other than the oracle itself: the page's cost
figures, the geometric-series closed form, a brute-force search written
with whole products, limits the page states, and the statistics of the
online estimate under censoring.
"""

import math

import numpy as np
import pytest

import oracle
from oracle import GateParams

EDGES = [-0.5, 0.5, 1.5, 3.0, 6.0]  # the page's six confidence buckets


def test_cost_matches_the_page():
    prm = GateParams()
    # "At n=5 that is 1041ms to produce accepted + 1 tokens, against 303ms for
    # a plain single-token decode": draft 196 + verify(5) = 300 + 109 * 5
    assert oracle.round_cost(5, prm) == 1041.0
    assert oracle.round_cost(0, prm) == 303.0
    # "a round that gets nothing accepted is a ~740ms loss"
    assert oracle.round_cost(5, prm) - oracle.round_cost(0, prm) == pytest.approx(740.0, abs=5.0)


@pytest.mark.parametrize("p", [0.0, 0.2, 0.5, 0.678, 0.9, 1.0])
def test_expected_tokens_closed_form(p):
    prm = GateParams()
    r32 = oracle.ratios_f32([p] * 8, 8, prm)
    for n in range(0, 9):
        closed = float(n + 1) if p == 1.0 else 1.0 + p * (1.0 - p ** n) / (1.0 - p)
        assert oracle.expected_tokens([p] * n, n) == pytest.approx(closed, rel=1e-14, abs=1e-14)
        # the gate's fp32 ratio of the same E(n) over cost(n)
        cost = 303.0 if n == 0 else 196.0 + 300.0 + 109.0 * n
        assert float(r32[n]) == pytest.approx(closed / cost, rel=3e-6)


def _brute(p, k_b, prm, logit_margin=None):
    """The gate's rule with each E(n) as 1 + sum of whole products."""
    if prm.margin_threshold > 0 and logit_margin is not None and logit_margin < prm.margin_threshold:
        return 0
    ratios = []
    for n in range(k_b + 1):
        e = 1.0 + sum(math.prod(p[:i + 1]) for i in range(n))
        c = prm.plain_ms if n == 0 else prm.draft_ms + prm.verify_base_ms + prm.verify_slope_ms * n
        ratios.append(e / c)
    lo = min(prm.min_draft, k_b)
    cand = list(range(lo, k_b + 1))
    best = max(cand, key=lambda n: (ratios[n], -n))
    if best < k_b and ratios[best] >= prm.margin * ratios[k_b] * (1 - 1e-12):
        return best
    return k_b


def test_gate_matches_brute_force():
    rng = np.random.default_rng(7)
    for trial in range(400):
        k_b = int(rng.integers(0, 9))
        hits = rng.integers(0, 20, size=6).astype(np.float64)
        total = hits + rng.integers(0, 20, size=6)
        conf = rng.normal(1.5, 2.5, size=8).astype(np.float32)
        prm = GateParams(min_draft=int(rng.integers(0, 3)), margin=float(rng.choice([1.0, 1.15, 1.5])))
        p = [oracle.match_prob(hits[oracle.bucket_of(c, EDGES)], total[oracle.bucket_of(c, EDGES)])
             for c in conf[:k_b]]
        got = oracle.gate_length(conf, k_b, None, EDGES, hits, total, prm)
        want = _brute(p, k_b, prm)
        # the gate decides in fp32: only near-ties (within its rounding) may differ
        if got != want:
            e = lambda n: 1.0 + sum(math.prod(p[:i + 1]) for i in range(n))
            c = lambda n: prm.plain_ms if n == 0 else prm.draft_ms + prm.verify_base_ms + prm.verify_slope_ms * n
            rg, rw, rf = e(got) / c(got), e(want) / c(want), prm.margin * e(k_b) / c(k_b)
            assert abs(rg - rw) <= 1e-5 * rw or abs(rg - rf) <= 1e-5 * rf or abs(rw - rf) <= 1e-5 * rf


def test_limits_the_page_states():
    prm = GateParams()
    full = np.zeros(6), np.zeros(6)  # cold gate: no observations anywhere
    # cold gate (and confident drafts) keep the whole block
    assert oracle.gate_length([7.0] * 5, 5, None, EDGES, *full, prm) == 5
    # certain misses: a plain decode step beats any verify
    hits, total = np.zeros(6), np.full(6, 10.0)
    assert oracle.gate_length([0.0] * 5, 5, None, EDGES, hits, total, prm) == 0
    # certain matches: the full block
    assert oracle.gate_length([0.0] * 5, 5, None, EDGES, total.copy(), total, prm) == 5


def test_buckets_are_half_open_and_nan_is_lowest():
    assert oracle.bucket_of(-0.6, EDGES) == 0
    assert oracle.bucket_of(-0.5, EDGES) == 1
    assert oracle.bucket_of(0.49, EDGES) == 1
    assert oracle.bucket_of(0.5, EDGES) == 2
    assert oracle.bucket_of(6.0, EDGES) == 5
    assert oracle.bucket_of(float("nan"), EDGES) == 0
    assert oracle.bucket_of(float("inf"), EDGES) == 5


def test_margin_rule():
    prm = GateParams()
    # p = 0.6 everywhere: truncating to 1 draft beats 5 by less than 1.15?
    hits, total = np.full(6, 6.0), np.full(6, 10.0)
    p = [0.6] * 5
    r = [(1.0 + sum(math.prod(p[:i + 1]) for i in range(n))) /
         (prm.plain_ms if n == 0 else 496.0 + 109.0 * n) for n in range(6)]
    best = int(np.argmax(r))
    got = oracle.gate_length([1.0] * 5, 5, None, EDGES, hits, total, prm)
    assert got == (best if r[best] >= 1.15 * r[5] else 5)
    # with no margin the argmax is taken
    assert oracle.gate_length([1.0] * 5, 5, None, EDGES, hits, total, GateParams(margin=1.0)) == best


def test_min_draft_and_pre_draft_skip():
    hits, total = np.zeros(6), np.full(6, 10.0)  # certain misses
    assert oracle.gate_length([0.0] * 5, 5, None, EDGES, hits, total, GateParams(min_draft=2)) == 2
    assert oracle.gate_length([0.0] * 3, 2, None, EDGES, hits, total, GateParams(min_draft=4)) == 2
    ok = total.copy()  # certain matches
    prm = GateParams(margin_threshold=4.0, min_draft=3)
    assert oracle.gate_length([7.0] * 5, 5, 3.9, EDGES, ok, total, prm) == 0
    assert oracle.gate_length([7.0] * 5, 5, 4.0, EDGES, ok, total, prm) == 5


def test_update_records_only_uncensored_positions():
    conf = np.array([[7.0, 7.0, 0.0, 0.0, 0.0],    # n = 2 of 5: hits at 0, 1; miss at 2
                     [0.0, 7.0, 7.0, 7.0, 7.0],    # n = 5 of 5: five hits, no miss
                     [7.0, 0.0, 0.0, 0.0, 0.0]],   # n = 0 of 3: one miss at position 0
                    dtype=np.float32)
    h, t = oracle.update_table(conf, [5, 5, 3], [2, 5, 0], EDGES, np.zeros(6), np.zeros(6), 0.9)
    b_hi, b_lo = oracle.bucket_of(7.0, EDGES), oracle.bucket_of(0.0, EDGES)
    want_h = np.zeros(6); want_t = np.zeros(6)
    want_h[b_hi] = 2 + 4; want_t[b_hi] = 2 + 4 + 1      # row 2's miss is at 7.0
    want_h[b_lo] = 1; want_t[b_lo] = 1 + 1               # row 0's miss at 0.0, row 1's hit
    assert np.array_equal(h, want_h) and np.array_equal(t, want_t)
    h2, t2 = oracle.update_table(conf[:0], [], [], EDGES, h, t, 0.9)
    assert np.allclose(h2, 0.9 * want_h, rtol=0, atol=1e-15) and np.allclose(t2, 0.9 * want_t, rtol=0, atol=1e-15)


def test_online_estimate_is_unbiased_under_censoring():
    """Per-position matches are Bernoulli(p_true[bucket]); a round stops at the
    first miss.  Recording only positions 0..n keeps every bucket's estimate
    unbiased; counting the censored tail as misses would pull it down."""
    rng = np.random.default_rng(11)
    p_true = np.array([0.2, 0.65, 0.79, 0.89, 0.95, 1.0])  # the page's table, roughly
    h, t = np.zeros(6), np.zeros(6)
    K = 5
    for rnd in range(4000):
        conf = rng.uniform(-1.5, 7.5, size=(8, K)).astype(np.float32)
        n_acc = np.zeros(8, dtype=np.int32)
        for b in range(8):
            n = 0
            while n < K and rng.random() < p_true[oracle.bucket_of(conf[b, n], EDGES)]:
                n += 1
            n_acc[b] = n
        h, t = oracle.update_table(conf, [K] * 8, n_acc, EDGES, h, t, 1.0)
    est = h / np.maximum(t, 1)
    sd = np.sqrt(p_true * (1 - p_true) / np.maximum(t, 1))
    assert np.all(np.abs(est - p_true) <= 4 * sd + 1e-9), (est, p_true, t)


def test_ties_go_to_smaller_n():
    # every verify costs the same and no draft ever matches: n = 1..5 tie
    prm = GateParams(verify_slope_ms=0.0, plain_ms=1e9, margin=1.0)
    hits, total = np.zeros(6), np.full(6, 10.0)
    assert oracle.gate_length([0.0] * 5, 5, None, EDGES, hits, total, prm) == 1


def test_margin_between_one_and_its_factor():
    # p = 0.8 everywhere: 4 drafts beat 5 by about 1.8 %, so only a margin of
    # 1.0 truncates (E(4)/932 = 0.003607 > E(5)/1041 = 0.003544)
    hits, total = np.full(6, 8.0), np.full(6, 10.0)
    assert oracle.gate_length([1.0] * 5, 5, None, EDGES, hits, total, GateParams()) == 5
    assert oracle.gate_length([1.0] * 5, 5, None, EDGES, hits, total, GateParams(margin=1.0)) == 4


# ---------------------------------------------------------------- planted mistakes
import inspect  # noqa: E402
import textwrap  # noqa: E402

import oracle.draft_gate as dg  # noqa: E402

def _closed_form_pin():
    test_expected_tokens_closed_form(0.678)


GATE_MUTATIONS = [
    ("update_table", "if na < ks:\n            new_t[bucket_of(conf[b, na], edges)] += 1",
     "for i in range(na, ks):\n            new_t[bucket_of(conf[b, i], edges)] += 1",
     [test_update_records_only_uncensored_positions, test_online_estimate_is_unbiased_under_censoring]),
    ("update_table", "d * float(hits[k]) + float(new_h[k])", "float(hits[k]) + float(new_h[k])",
     [test_update_records_only_uncensored_positions]),
    ("gate_length", "if r[n] > r[best_n]:", "if r[n] >= r[best_n]:", [test_ties_go_to_smaller_n]),
    ("gate_length", "r[best_n] >= np.float32(np.float32(prm.margin) * r[k_b])", "r[best_n] >= r[k_b]",
     [test_margin_between_one_and_its_factor]),
    ("ratios_f32", "prod = f(prod * f(p[n - 1]))", "prod = f(prod * f(p[0]))",
     [test_gate_matches_brute_force, _closed_form_pin]),
    ("round_cost", "float(prm.verify_slope_ms) * float(n)", "float(prm.verify_slope_ms) * float(n + 1)",
     [test_cost_matches_the_page]),
    ("ratios_f32", "f(f(prm.verify_slope_ms) * f(n))", "f(f(prm.verify_slope_ms) * f(n + 1))",
     [_closed_form_pin]),
    ("match_prob", "if t > 0.0 else 1.0", "if t > 0.0 else 0.0", [test_limits_the_page_states]),
    ("bucket_of", "if c >= float(e):", "if c > float(e):", [test_buckets_are_half_open_and_nan_is_lowest]),
    ("gate_length", "n_lo = min(int(prm.min_draft), k_b)", "n_lo = 0", [test_min_draft_and_pre_draft_skip]),
]


@pytest.mark.parametrize("fn_name,old,new,catchers", GATE_MUTATIONS,
                         ids=[f"{m[0]}:{i}" for i, m in enumerate(GATE_MUTATIONS)])
def test_planted_gate_mistake_is_caught(monkeypatch, fn_name, old, new, catchers):
    src = textwrap.dedent(inspect.getsource(getattr(dg, fn_name)))
    assert src.count(old) >= 1, (fn_name, old)
    ns = dict(vars(dg))
    exec(compile(src.replace(old, new, 1), f"<mutant {fn_name}>", "exec"), ns)
    monkeypatch.setattr(dg, fn_name, ns[fn_name])
    monkeypatch.setattr(oracle, fn_name, ns[fn_name])  # callers look helpers up in dg's namespace
    caught = []
    for pin in catchers:
        try:
            pin()
        except AssertionError:
            caught.append(pin.__name__)
    assert caught, f"no pin caught the mutation of {fn_name}: {old!r} -> {new!r}"
