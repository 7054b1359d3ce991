"""Pins of the draft-length gate oracle (PocketLLM docs/dspark.md, the gate).

Each pin comes from something other than the oracle itself: the page's cost
figures, the geometric-series closed form, a brute-force search written
with whole products, limits the page states, and the statistics of the
online estimate under censoring.
"""

import math
from fractions import Fraction

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
    q = Fraction(p)  # the exact value of the double
    r = oracle.gate_ratios([q] * 8, 8, prm)
    for n in range(0, 9):
        # geometric series: 1 + q (1 - q^n) / (1 - q), or n + 1 at q = 1
        closed = Fraction(n + 1) if q == 1 else 1 + q * (1 - q ** n) / (1 - q)
        assert oracle.expected_tokens([q] * n, n) == closed
        cost = Fraction(303) if n == 0 else Fraction(196 + 300 + 109 * n)
        assert r[n] == closed / cost


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
        p = [float(oracle.match_prob(hits[oracle.bucket_of(c, EDGES)], total[oracle.bucket_of(c, EDGES)]))
             for c in conf[:k_b]]
        got = oracle.gate_length(conf, k_b, None, EDGES, hits, total, prm)
        want = _brute(p, k_b, prm)
        # the brute force's fp64 sums round differently; only exact near-ties may differ
        if got != want:
            e = lambda n: 1.0 + sum(math.prod(p[:i + 1]) for i in range(n))
            c = lambda n: prm.plain_ms if n == 0 else prm.draft_ms + prm.verify_base_ms + prm.verify_slope_ms * n
            assert abs(e(got) / c(got) - e(want) / c(want)) < 1e-12 or \
                abs(e(got) / c(got) - prm.margin * e(k_b) / c(k_b)) < 1e-12


def _fp32_gate(conf_row, k_b, edges, hits, total, prm):
    """An fp32 evaluation of the gate's rule (one rounding per operation, the
    order of ratio_error_bound's derivation): a model of a fast evaluation,
    used to check that the oracle's near-tie flag covers every disagreement."""
    f = np.float32
    p = []
    for c in conf_row[:k_b]:
        k = oracle.bucket_of(c, edges)
        p.append(f(hits[k] / total[k]) if total[k] > 0 else f(1.0))
    fixed = f(f(prm.draft_ms) + f(prm.verify_base_ms))
    e, prod, r = f(1.0), f(1.0), []
    for n in range(k_b + 1):
        if n > 0:
            prod = f(prod * p[n - 1])
            e = f(e + prod)
        cost = f(prm.plain_ms) if n == 0 else f(fixed + f(f(prm.verify_slope_ms) * f(n)))
        r.append(f(e / cost))
    n_lo = min(prm.min_draft, k_b)
    best = n_lo
    for n in range(n_lo + 1, k_b + 1):
        if r[n] > r[best]:
            best = n
    if best < k_b and r[best] >= f(f(prm.margin) * r[k_b]):
        return best
    return k_b


def test_near_tie_flag_covers_fp32_disagreements():
    """Wherever an fp32 evaluation picks another length than the exact rule,
    the oracle has flagged the sequence as a near-tie; and the flag is rare
    on random inputs (it marks ties, not ordinary decisions)."""
    rng = np.random.default_rng(17)
    flagged = differ = 0
    n_cases = 3000
    for trial in range(n_cases):
        k_b = int(rng.integers(0, 17))
        total = rng.integers(1, 40, size=6).astype(np.float64)
        hits = np.minimum(total, rng.integers(0, 40, size=6)).astype(np.float64)
        if trial % 3 == 0:  # steep tables: near-ties between lengths are common there
            hits = total.copy()
            hits[rng.integers(0, 6)] -= 1
        conf = rng.normal(1.5, 2.5, size=16).astype(np.float32)
        prm = GateParams(min_draft=int(rng.integers(0, 3)), margin=float(rng.choice([1.0, 1.15, 1.5])),
                         verify_slope_ms=float(rng.choice([109.0, 0.0, 1e-3])))
        n, near = oracle.gate_decision(conf, k_b, None, EDGES, hits, total, prm)
        n32 = _fp32_gate(conf, k_b, EDGES, hits, total, prm)
        flagged += near
        if n32 != n:
            differ += 1
            assert near, (trial, n, n32)
    assert differ <= flagged < n_cases // 5, (differ, flagged)


def test_exact_ties_are_flagged():
    # equal costs and no matches: n = 1..5 tie exactly, the rule takes 1
    prm = GateParams(verify_slope_ms=0.0, plain_ms=1e9, margin=1.0)
    hits, total = np.zeros(6), np.full(6, 10.0)
    assert oracle.gate_decision([0.0] * 5, 5, None, EDGES, hits, total, prm) == (1, True)
    # far from any tie: the page's confident and hopeless drafts
    assert oracle.gate_decision([7.0] * 5, 5, None, EDGES, hits.copy() + 10, total, GateParams()) == (5, False)
    assert oracle.gate_decision([0.0] * 5, 5, None, EDGES, hits, total, GateParams()) == (0, False)


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
    ("gate_decision", "if r[n] > r[best_n]:", "if r[n] >= r[best_n]:", [test_ties_go_to_smaller_n]),
    ("gate_decision", "full = r[k_b] * m if", "full = r[k_b] if", [test_margin_between_one_and_its_factor]),
    ("expected_tokens", "prod = prod * (p[i]", "prod = prod * (p[0]",
     [test_gate_matches_brute_force, _closed_form_pin]),
    ("round_cost", "Fraction(float(prm.verify_base_ms))", "Fraction(float(prm.verify_slope_ms))",
     [test_cost_matches_the_page]),
    ("round_cost", "Fraction(float(prm.verify_slope_ms)) * n", "Fraction(float(prm.verify_slope_ms)) * (n + 1)",
     [_closed_form_pin]),
    ("gate_decision", "ratio_error_bound(n) + ratio_error_bound(best_n))", "0)",
     [test_exact_ties_are_flagged, test_near_tie_flag_covers_fp32_disagreements]),
    ("match_prob", "if t > 0 else Fraction(1)", "if t > 0 else Fraction(0)", [test_limits_the_page_states]),
    ("bucket_of", "if c >= float(e):", "if c > float(e):", [test_buckets_are_half_open_and_nan_is_lowest]),
    ("gate_decision", "n_lo = min(int(prm.min_draft), k_b)", "n_lo = 0", [test_min_draft_and_pre_draft_skip]),
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
