"""Pins of the penalty oracle (llmstudio.ru sections 38-39): hand-computed
values, neutral parameters, the section 39 state rule checked against a
separately written sampler that appends accepted tokens and rolls back, and
monotonicity.  Planted mistakes at the end must each fail a pin."""

import inspect
import textwrap
from collections import Counter

import numpy as np
import pytest

import oracle
from oracle import penalties as pen

F32 = np.float32


def test_hand_values():
    assert pen.penalize_value(3.0, 1, 2.0, 0.0, 0.0) == F32(1.5)
    assert pen.penalize_value(-3.0, 1, 2.0, 0.0, 0.0) == F32(-6.0)
    assert pen.penalize_value(0.0, 1, 2.0, 0.0, 0.0) == F32(0.0)
    # r = 1: then 3 - 0.25 * 2 - 0.5 = 2
    assert pen.penalize_value(3.0, 2, 1.0, 0.25, 0.5) == F32(2.0)
    # r = 1.5 on 3 -> 2, frequency 0.5 x 3 -> 0.5, presence 1 -> -0.5
    assert pen.penalize_value(3.0, 3, 1.5, 0.5, 1.0) == F32(-0.5)
    # one f32 rounding per step: 1 / 3 rounds before the subtraction
    want = F32(F32(F32(1.0) / F32(3.0)) - F32(0.1))
    assert pen.penalize_value(1.0, 1, 3.0, 0.0, 0.1) == want


def _rows(rng, B, K, V, dtype):
    x = rng.normal(0, 3, (B * (K + 1), V)).astype(F32)
    y = rng.normal(0, 3, (B * K, V)).astype(F32)
    if dtype == "bf16":
        from workloads.configs import f32_to_bf16_bits
        return f32_to_bf16_bits(x), f32_to_bf16_bits(y)
    if dtype == "f16":
        return x.astype(np.float16), y.astype(np.float16)
    return x, y


@pytest.mark.parametrize("dtype", ["f32", "bf16", "f16"])
def test_neutral_parameters_change_nothing(dtype):
    rng = np.random.default_rng(1)
    B, K, V = 5, 3, 40
    tg, dr = _rows(rng, B, K, V, dtype)
    tok = rng.integers(0, V, B * K).astype(np.int32)
    hist = rng.integers(0, V, 30).astype(np.int32)
    off = np.array([0, 6, 6, 15, 22, 30], np.int32)
    one = np.ones(B, F32)
    zero = np.zeros(B, F32)
    t2, d2, st = pen.penalize_rows(tg, dr, dtype, off, hist, tok, B, K, None, one, zero, zero)
    assert (st == 0).all()
    assert np.array_equal(t2.view(np.uint8), tg.view(np.uint8))
    assert np.array_equal(d2.view(np.uint8), dr.view(np.uint8))


class RollingSampler:
    """A stateful sampler as an engine keeps it: token counts that grow as
    tokens are appended, with checkpoints to roll back to (section 39)."""

    def __init__(self, history, V):
        self.counts = {}
        self.V = V
        self.stack = []
        for t in history:
            self.append(t)

    def append(self, t):
        t = int(t)
        self.stack.append(t)
        if 0 <= t < self.V:
            self.counts[t] = self.counts.get(t, 0) + 1

    def rollback(self, n):
        for _ in range(n):
            t = self.stack.pop()
            if 0 <= t < self.V:
                self.counts[t] -= 1
                if self.counts[t] == 0:
                    del self.counts[t]

    def apply(self, row, r, f, p):
        out = row.astype(F32).copy()
        for t, c in self.counts.items():
            x = F32(out[t])
            x = F32(x * F32(r)) if x < 0 else F32(x / F32(r))
            x = F32(x - F32(F32(f) * F32(c)))
            out[t] = F32(x - F32(p))
        return out


def test_branch_state_rule_against_a_rolling_sampler():
    """Row i is penalised with the state after appending t_0..t_{i-1}; after
    the branch is verified the sampler rolls back to the history."""
    rng = np.random.default_rng(2)
    B, K, V = 6, 5, 12
    tg, dr = _rows(rng, B, K, V, "f32")
    tok = rng.integers(0, V, B * K).astype(np.int32)
    hist = rng.integers(-2, V + 2, 50).astype(np.int32)  # a few ids out of range
    off = np.sort(rng.integers(0, 51, B + 1)).astype(np.int32)
    off[0] = 0
    rep = rng.uniform(1.0, 2.0, B).astype(F32)
    fr = rng.uniform(0.0, 0.5, B).astype(F32)
    pr = rng.uniform(0.0, 1.0, B).astype(F32)
    t2, d2, st = pen.penalize_rows(tg, dr, "f32", off, hist, tok, B, K, None, rep, fr, pr)
    assert (st == 0).all()
    for b in range(B):
        s = RollingSampler(hist[off[b]:off[b + 1]], V)
        for i in range(K + 1):
            assert np.array_equal(t2[b * (K + 1) + i], s.apply(tg[b * (K + 1) + i], rep[b], fr[b], pr[b]))
            if i < K:
                assert np.array_equal(d2[b * K + i], s.apply(dr[b * K + i], rep[b], fr[b], pr[b]))
                s.append(tok[b * K + i])
        s.rollback(K)
        assert s.counts == dict(Counter(int(v) for v in hist[off[b]:off[b + 1]] if 0 <= v < V))


def test_rows_do_not_see_their_own_or_later_drafts():
    rng = np.random.default_rng(3)
    B, K, V = 1, 4, 30
    tg, dr = _rows(rng, B, K, V, "f32")
    tok = np.array([3, 7, 7, 9], np.int32)
    hist = np.array([1, 2], np.int32)
    off = np.array([0, 2], np.int32)
    a = [np.full(1, 1.7, F32), np.full(1, 0.3, F32), np.full(1, 0.2, F32)]
    t2, d2, _ = pen.penalize_rows(tg, dr, "f32", off, hist, tok, B, K, None, *a)
    tok_b = tok.copy()
    tok_b[2:] = [11, 12]  # change t_2, t_3: rows 0..2 must not move
    t3, d3, _ = pen.penalize_rows(tg, dr, "f32", off, hist, tok_b, B, K, None, *a)
    assert np.array_equal(t2[:3], t3[:3]) and np.array_equal(d2[:3], d3[:3])
    assert not np.array_equal(t2[3], t3[3])
    # row 0 touches only the history ids; row 3 counts token 7 twice
    changed0 = np.flatnonzero(t2[0] != tg[0])
    assert set(changed0) <= {1, 2}
    assert t2[3, 7] == pen.penalize_value(tg[3, 7], 2, 1.7, 0.3, 0.2)


def test_penalties_only_lower_logits():
    rng = np.random.default_rng(4)
    B, K, V = 4, 3, 25
    for dtype in ("f32", "bf16", "f16"):
        tg, dr = _rows(rng, B, K, V, dtype)
        tok = rng.integers(0, V, B * K).astype(np.int32)
        hist = rng.integers(0, V, 40).astype(np.int32)
        off = np.array([0, 10, 20, 30, 40], np.int32)
        t2, d2, _ = pen.penalize_rows(tg, dr, dtype, off, hist, tok, B, K, None, np.full(B, 1.3, F32),
                                      np.full(B, 0.2, F32), np.full(B, 0.4, F32))
        dec = lambda a: oracle.decode_rows(a, dtype).reshape(a.shape)
        assert (dec(t2) <= dec(tg)).all() and (dec(d2) <= dec(dr)).all()
        assert (dec(t2) < dec(tg)).any()


def test_bad_offsets_leave_rows_alone():
    rng = np.random.default_rng(5)
    B, K, V = 3, 2, 10
    tg, dr = _rows(rng, B, K, V, "f32")
    tok = rng.integers(0, V, B * K).astype(np.int32)
    hist = rng.integers(0, V, 9).astype(np.int32)
    off = np.array([0, 5, 3, 9], np.int32)  # sequence 1: end before start
    a = [np.full(B, 2.0, F32), np.zeros(B, F32), np.zeros(B, F32)]
    t2, d2, st = pen.penalize_rows(tg, dr, "f32", off, hist, tok, B, K, None, *a)
    assert list(st) == [0, pen.BAD_LAYOUT, 0]
    assert np.array_equal(t2[3:6], tg[3:6]) and np.array_equal(d2[2:4], dr[2:4])


def test_unusable_parameters_are_bad_values():
    rng = np.random.default_rng(6)
    B, K, V = 4, 2, 10
    tg, dr = _rows(rng, B, K, V, "f32")
    tok = rng.integers(0, V, B * K).astype(np.int32)
    hist = rng.integers(0, V, 8).astype(np.int32)
    off = np.array([0, 2, 4, 6, 8], np.int32)
    rep = np.array([0.0, np.nan, 1.5, 1.5], F32)
    fr = np.array([0.0, 0.0, np.inf, 0.1], F32)
    pr = np.zeros(B, F32)
    t2, d2, st = pen.penalize_rows(tg, dr, "f32", off, hist, tok, B, K, None, rep, fr, pr)
    assert list(st) == [pen.BAD_VALUE] * 3 + [0]
    assert np.array_equal(t2[:9], tg[:9]) and not np.array_equal(t2[9:], tg[9:])


def test_distinct_id_capacity():
    B, K, V = 2, 1, 20000
    tg = np.zeros((B * (K + 1), V), F32)
    dr = np.zeros((B * K, V), F32)
    tok = np.array([5, 6], np.int32)
    h = np.concatenate([np.arange(pen.MAX_DISTINCT - 1), np.arange(pen.MAX_DISTINCT)]).astype(np.int32)
    off = np.array([0, pen.MAX_DISTINCT - 1, len(h)], np.int32)
    # sequence 0: 8191 history ids + draft 5 (already counted) -> 8191 distinct;
    # sequence 1: 8192 history ids + draft 6 (already there) -> 8192: both fit
    a = [np.full(B, 1.0, F32), np.full(B, 0.5, F32), np.zeros(B, F32)]
    _, _, st = pen.penalize_rows(tg, dr, "f32", off, h, tok, B, K, None, *a)
    assert list(st) == [0, 0]
    tok2 = np.array([9000, 9001], np.int32)  # a new id each: 8192 fits, 8193 does not
    _, _, st = pen.penalize_rows(tg, dr, "f32", off, h, tok2, B, K, None, *a)
    assert list(st) == [0, pen.BAD_LAYOUT]


MUTATIONS = [
    ("row_counts", "drafts[:i]", "drafts[:i + 1]", [test_branch_state_rule_against_a_rolling_sampler]),
    ("penalize_value", "v * r32 if v < 0 else v / r32", "v / r32 if v < 0 else v * r32", [test_hand_values]),
    ("penalize_value", "F32(f32 * F32(count))", "F32(f32)", [test_hand_values]),
]


@pytest.mark.parametrize("fn,old,new,catchers", MUTATIONS, ids=[f"{m[0]}:{i}" for i, m in enumerate(MUTATIONS)])
def test_planted_mistake_is_caught(monkeypatch, fn, old, new, catchers):
    src = textwrap.dedent(inspect.getsource(getattr(pen, fn)))
    assert old in src
    ns = dict(vars(pen))
    exec(compile(src.replace(old, new, 1), f"<mutant {fn}>", "exec"), ns)
    monkeypatch.setattr(pen, fn, ns[fn])
    for catcher in catchers:
        with pytest.raises(AssertionError):
            catcher()
