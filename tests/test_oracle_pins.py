"""Pins of the CPU oracle to facts the pages and mathematics fix.

Each ``pin_*`` function asserts one fact; ``test_*`` run them, and
``tests/test_oracle_mutations.py`` re-runs them against deliberately broken
copies of oracle functions to show each plausible mistake is caught.
"""

import math
from fractions import Fraction

import numpy as np
import pytest

import oracle as o
from conftest import load_golden

F32 = np.float32
GRID24 = 1 << 24


# ------------------------------------------------------------------ helpers

def run_one(p_rows, q_rows, tokens, u):
    p = np.asarray(p_rows, F32).reshape(len(tokens) + 1, -1)
    q = np.asarray(q_rows, F32).reshape(len(tokens), p.shape[1])
    r = o.accept(p, q, np.asarray(tokens, np.int32), np.asarray(u, F32), 1, len(tokens))
    return int(r.n_accepted[0]), int(r.next_token[0]), int(r.status[0])


def accept_fraction(p_row, q_row, t):
    """Fraction of the 24-bit uniform grid k * 2**-24 on which the oracle
    accepts ``t`` (bisection: acceptance is monotone in u)."""
    V = len(p_row)
    rows_p = np.stack([p_row, np.full(V, 1.0 / V)])
    lo, hi = 0, GRID24  # accept at lo (if any), reject at hi
    if run_one(rows_p, [q_row], [t], [0.0, 0.5])[0] == 0:
        return 0.0
    while hi - lo > 1:
        mid = (lo + hi) // 2
        if run_one(rows_p, [q_row], [t], [mid / GRID24, 0.5])[0] == 1:
            lo = mid
        else:
            hi = mid
    return hi / GRID24


# ------------------------------------------------------------------ worked examples

def pin_s15_accept_ratio():
    g = load_golden("llmstudio_s15_accept_ratio.txt")
    p_row = [g["p_token"], 1.0 - g["p_token"]]
    q_row = [g["q_token"], 1.0 - g["q_token"]]
    a = accept_fraction(p_row, q_row, 0)
    assert abs(a - g["accept_probability"]) < 1e-6, a
    assert round(a, 3) == g["printed_accept_probability"]
    assert abs(g["q_token"] * a - g["printed_output_mass"]) < 1e-6


def pin_s16_always_accept():
    g = load_golden("llmstudio_s16_always_accept.txt")
    p_row = [g["p_token"], 1.0 - g["p_token"]]
    q_row = [g["q_token"], 1.0 - g["q_token"]]
    assert accept_fraction(p_row, q_row, 0) == g["accept_probability"]
    for u in (0.0, 0.5, 1.0 - 2.0 ** -24):
        assert run_one([p_row, [0.5, 0.5]], [q_row], [0], [u, 0.25])[0] == 1


def pin_s18_acceptance_and_residual():
    g = load_golden("llmstudio_s18_four_tokens.txt")
    p_row, q_row = g["target"], g["draft"]
    alpha = sum(q_row[t] * accept_fraction(p_row, q_row, t) for t in range(4))
    assert abs(alpha - g["acceptance"]) < 2e-6, alpha
    # residual: reject token 2 (p=.10, q=.70) with u0 = 0.5, then walk u1.
    rows_p = [p_row, [0.25] * 4]
    emitted = lambda u1: run_one(rows_p, [q_row], [2], [0.5, u1])
    assert emitted(0.0)[0] == 0
    seen = {emitted(k / 512.0)[1] for k in range(512)}
    assert seen == {0, 1}, seen  # zero-residual tokens 2 and 3 never emitted
    lo, hi = 0, GRID24  # token 0 at lo, token 1 at hi
    while hi - lo > 1:
        mid = (lo + hi) // 2
        if emitted(mid / GRID24)[1] == 0:
            lo = mid
        else:
            hi = mid
    assert abs(hi / GRID24 - g["residual"][0]) < 2e-6, hi / GRID24


def pin_zero_target_mass_never_accepted():
    # min(1, 0/q) = 0: a token the target gives zero mass is rejected for every u.
    for u in (0.0, 2.0 ** -24, 0.5):
        n, nxt, st = run_one([[0.0, 1.0], [0.5, 0.5]], [[0.5, 0.5]], [0], [u, 0.3])
        assert (n, nxt, st) == (0, 1, 0)


def pin_zero_draft_mass_accepted():
    # q(t) = 0 < p(t): min(1, p/0) = 1 (the exact predicate 0 < p*Zq holds).
    for u in (0.0, 0.999):
        assert run_one([[0.5, 0.5], [0.5, 0.5]], [[0.0, 1.0]], [0], [u, 0.3])[0] == 1


# ------------------------------------------------------------------ exact enumeration

def _dyadic_case(rng, V, m=2):
    """p, q on V tokens with q powers of two, every accept threshold p/q and
    every residual CDF step a multiple of 2**-8 (so a midpoint grid of 2**-10
    cells measures each outcome exactly)."""
    qs = [2.0 ** -(i + 1) for i in range(V - 1)]
    qs.append(qs[-1])
    q = np.array(rng.permutation(qs))
    R = 2.0 ** -m
    order = rng.permutation(V)
    A = set(order[: max(1, V // 3)].tolist())
    s = np.zeros(V)
    need = R
    for v in sorted(set(range(V)) - A, key=lambda v: -q[v]):
        take = min(need, q[v])
        take = math.floor(take * 256 * rng.uniform(0.5, 1.0)) / 256 if take < need else take
        s[v] = take
        need -= take
        if need <= 0:
            break
    assert need == 0
    r = np.zeros(V)
    left = int(R * 256)
    Al = sorted(A)
    for j, v in enumerate(Al):
        k = left if j == len(Al) - 1 else int(rng.integers(0, left + 1))
        r[v] = k / 256.0
        left -= k
    p = q - s + r
    assert abs(p.sum() - 1) < 1e-15 and (p >= 0).all()
    return p, q


def first_token_marginal(p_rows, q_rows, t_later, u_later_fixed, G=1024):
    """Exact law of the first emitted token of one round, enumerating the
    draft token t_0 (weight qhat_0) and the midpoint grids of u_0 and of the
    final uniform u_K (the only two uniforms it depends on)."""
    K = len(q_rows)
    V = len(p_rows[0])
    mids = [(k + 0.5) / G for k in range(G)]
    q0 = [Fraction(float(F32(x))) for x in q_rows[0]]
    Zq = sum(q0)
    law = [Fraction(0)] * V
    reject_at = None
    for t in range(V):
        if q0[t] == 0:
            continue
        acc = 0
        for u0 in mids:
            u = [u0] + list(u_later_fixed[: K - 1]) + [0.5]
            n, nxt, _ = run_one(p_rows, q_rows, [t] + list(t_later), u)
            if n >= 1:
                acc += 1
            elif reject_at is None:
                reject_at = (t, u0)
        law[t] += q0[t] / Zq * Fraction(acc, G)
        law_rej = q0[t] / Zq * Fraction(G - acc, G)
        if G - acc:
            law_t_rej = law_rej
            # residual draw: walk u_K with a rejecting (t, u0)
            u0r = next(u0 for u0 in mids
                       if run_one(p_rows, q_rows, [t] + list(t_later),
                                  [u0] + list(u_later_fixed[: K - 1]) + [0.5])[0] == 0)
            counts = [0] * V
            for uk in mids:
                n, nxt, _ = run_one(p_rows, q_rows, [t] + list(t_later),
                                    [u0r] + list(u_later_fixed[: K - 1]) + [uk])
                assert n == 0
                counts[nxt] += 1
            for v in range(V):
                law[v] += law_t_rej * Fraction(counts[v], G)
    return law


def pin_enumeration_marginal_equals_target():
    rng = np.random.default_rng(7)
    for V in (2, 3, 4, 6, 8):
        p, q = _dyadic_case(rng, V)
        law = first_token_marginal([p, np.full(V, 1.0 / V)], [q], [], [], G=256)
        exp = [Fraction(float(x)) for x in p]
        assert law == exp, (V, law, exp)


def pin_enumeration_degenerate_cases():
    # p == q: never rejects; disjoint supports: always rejects, residual = p.
    same = np.array([0.5, 0.25, 0.25, 0.0])
    law = first_token_marginal([same, same], [same], [], [], G=64)
    assert law == [Fraction(float(x)) for x in same]
    p = np.array([0.0, 0.0, 0.5, 0.5])
    q = np.array([0.5, 0.5, 0.0, 0.0])
    law = first_token_marginal([p, p], [q], [], [], G=64)
    assert law == [Fraction(float(x)) for x in p]


def pin_enumeration_bonus_law():
    # all accepted: the bonus token follows p_K exactly (p = q makes row 0 accept).
    row0 = np.array([0.5, 0.25, 0.25, 0.0])
    pk = np.array([0.125, 0.375, 0.0, 0.5])
    G = 256
    counts = [0] * 4
    for k in range(G):
        n, nxt, _ = run_one([row0, pk], [row0], [1], [0.7, (k + 0.5) / G])
        assert n == 1
        counts[nxt] += 1
    assert [Fraction(c, G) for c in counts] == [Fraction(float(x)) for x in pk]


def pin_enumeration_k2_first_token():
    rng = np.random.default_rng(11)
    p0, q0 = _dyadic_case(rng, 4)
    p1, q1 = _dyadic_case(rng, 4)
    law = first_token_marginal([p0, p1, np.full(4, 0.25)], [q0, q1], [1], [0.3], G=128)
    assert law == [Fraction(float(x)) for x in p0]


# ------------------------------------------------------------------ greedy

def pin_argmax_rules():
    cases = [
        ([1.0, 3.0, 3.0, 2.0], 1, False),
        ([np.nan, 1.0, np.nan], 1, True),
        ([np.nan, np.nan], 0, True),
        ([-np.inf, -np.inf], 0, False),
        ([np.nan, -np.inf], 1, True),
        ([-0.0, 0.0], 0, False),
        ([0.0, -0.0], 0, False),
        ([np.inf, np.inf], 0, False),
        ([1.0, np.inf, np.nan], 1, True),
        ([5.0], 0, False),
    ]
    for row, idx, nan in cases:
        assert o.argmax_lowest(np.array(row)) == (idx, nan), row


def _table_model(rng, V, ties):
    t = rng.standard_normal((V, V, V)).astype(F32)
    return np.round(t) if ties else t


def pin_greedy_reproduces_plain_decoding():
    """A tiny table "model" (next-token logits a seeded function of the last
    two tokens): speculative greedy decoding with any drafter must emit the
    same stream as plain greedy decoding (card, "Method" and "Correctness")."""
    rng = np.random.default_rng(3)
    for V, ties in ((5, False), (7, True), (16, False), (16, True)):
        table = _table_model(rng, V, ties)
        row = lambda s: table[s[-2], s[-1]]
        prompt = [int(rng.integers(V)), int(rng.integers(V))]
        N = 40
        plain = list(prompt)
        while len(plain) < N + 2:
            plain.append(int(np.argmax(row(plain))))  # numpy: first maximal index
        for K in range(0, 7):
            for drafter in ("perfect", "random", "wrong", "half"):
                seq = list(prompt)
                while len(seq) < N + 2:
                    ctx = list(seq)
                    draft = []
                    for i in range(K):
                        good = int(np.argmax(row(ctx)))
                        if drafter == "perfect" or (drafter == "half" and i < K // 2):
                            d = good
                        elif drafter == "wrong":
                            d = (good + 1) % V
                        else:
                            d = int(rng.integers(V))
                        draft.append(d)
                        ctx.append(d)
                    rows = np.stack([row(seq + draft[:i]) for i in range(K + 1)])
                    r = o.verify_greedy(rows, "f32", np.array(draft, np.int32), 1, K)
                    n, nxt = int(r.n_accepted[0]), int(r.next_token[0])
                    if drafter == "perfect":
                        assert n == K
                    if drafter == "wrong" and K:
                        assert n == 0
                    seq += draft[:n] + [nxt]
                assert seq[: N + 2] == plain, (V, ties, K, drafter)


def pin_greedy_error_codes():
    rows = np.array([[0.1, 0.7, 0.2], [0.5, 0.2, 0.3], [0.3, 0.3, 0.4]], F32)
    r = o.verify_greedy(rows, "f32", np.array([1, 0], np.int32), 1, 2)
    assert (r.n_accepted[0], r.next_token[0], r.status[0]) == (2, 2, 0)
    r = o.verify_greedy(rows, "f32", np.array([1, 3], np.int32), 1, 2)
    assert (r.n_accepted[0], r.next_token[0], r.status[0]) == (1, 0, o.BAD_TOKEN)
    bad = rows.copy()
    bad[0, 2] = np.nan
    r = o.verify_greedy(bad, "f32", np.array([1, 2], np.int32), 1, 2)
    assert (r.n_accepted[0], r.next_token[0], r.status[0]) == (1, 0, o.BAD_VALUE)
    # a NaN in a row the walk never reaches is not reported
    bad = rows.copy()
    bad[2, 0] = np.nan
    r = o.verify_greedy(bad, "f32", np.array([0, 0], np.int32), 1, 2)
    assert (r.n_accepted[0], r.next_token[0], r.status[0]) == (0, 1, 0)


# ------------------------------------------------------------------ masses

def pin_exact_mass_vs_fsum():
    rng = np.random.default_rng(5)
    for trial in range(60):
        n = int(rng.integers(1, 3000))
        kind = trial % 4
        if kind == 0:
            row = rng.random(n).astype(F32)
        elif kind == 1:
            row = np.exp(rng.uniform(-103, 88, n)).astype(F32)  # subnormal .. huge
        elif kind == 2:
            row = (rng.integers(0, 1 << 23, n) * 2.0 ** -149).astype(F32)  # subnormals
        else:
            row = (rng.random(n) * 3e38).astype(F32)
        exact = o.exact_mass(row)
        assert float(exact) == math.fsum(row.astype(np.float64))
        perm = row[rng.permutation(n)]
        assert o.exact_mass_int(perm) == o.exact_mass_int(row)


def pin_exact_mass_vs_fraction_sum():
    rng = np.random.default_rng(6)
    for trial in range(20):
        row = np.exp(rng.uniform(-100, 80, int(rng.integers(1, 60)))).astype(F32)
        row[rng.random(row.size) < 0.2] = 0.0
        assert o.exact_mass(row) == sum(Fraction(float(x)) for x in row)
    assert o.exact_mass(np.array([-0.0, 0.0], F32)) == 0


def pin_accept_decision_exact_ties():
    # u * q * Zp == p * Zq exactly: strict '<' rejects; one ulp lower accepts.
    p = np.array([0.25, 0.75], F32)  # Zp = 1
    q = np.array([0.5, 0.5], F32)  # Zq = 1, threshold p/q = 0.5
    assert not o.accept_decision(0.5, p[0], q[0], o.exact_mass_int(p), o.exact_mass_int(q))
    below = float(np.nextafter(F32(0.5), F32(0)))
    assert o.accept_decision(below, p[0], q[0], o.exact_mass_int(p), o.exact_mass_int(q))


def pin_scale_invariance():
    rng = np.random.default_rng(9)
    K, V = 4, 50
    for trial in range(30):
        p = rng.random((K + 1, V)).astype(F32)
        q = rng.random((K, V)).astype(F32)
        t = rng.integers(0, V, K).astype(np.int32)
        u = rng.random(K + 1).astype(F32)
        base = o.accept(p, q, t, u, 1, K)
        sp, sq = 2.0 ** int(rng.integers(-60, 60)), 2.0 ** int(rng.integers(-60, 60))
        sc = o.accept((p * sp).astype(F32), (q * sq).astype(F32), t, u, 1, K)
        assert (base.n_accepted[0], base.next_token[0]) == (sc.n_accepted[0], sc.next_token[0])


# ------------------------------------------------------------------ inverse CDF

def pin_inverse_cdf_closed_form():
    w = np.array([0.0, 0.25, 0.0, 0.5, 0.25])
    # steps at 0.25, 0.75, 1.0: u*R in [0, .25) -> 1, [.25, .75) -> 3, [.75, 1) -> 4
    for u, want in ((0.0, 1), (0.2, 1), (0.25, 3), (0.74, 3), (0.75, 4), (0.999, 4)):
        assert o.inverse_cdf_draw(w, u)[0] == want, u
    assert o.inverse_cdf_draw(w, 0.25)[1] is True
    assert o.inverse_cdf_draw(w, 0.5)[1] is False


def _fixed_point_bonus_draw(p, u, z_rel, signs):
    """A bonus draw as an fp32 implementation with 64-bit fixed point may take
    it: normalise by a mass off by ``z_rel`` (relative), perturb each weight
    by one rounding (``signs`` in {-1, 0, 1} times 2^-24, relative), floor to
    fixed point with a total near 2^(62 - bitlen V), and search the integer
    CDF for floor(u R).  Exact rationals throughout."""
    V = len(p)
    S = 62 - V.bit_length()
    z = sum(Fraction(float(x)) for x in p) * (1 + Fraction(z_rel))
    w = [math.floor(Fraction(float(x)) / z * (1 + int(sg) * Fraction(1, 1 << 24)) * (1 << S))
         for x, sg in zip(p, signs)]
    R = sum(w)
    tau = math.floor(Fraction(float(np.float32(u))) * R)
    c = 0
    for j, x in enumerate(w):
        c += x
        if c > tau:
            return j
    raise AssertionError("unreachable")


def pin_certified_bonus_draws():
    """DRAW_CERTIFIED is sound: a certified bonus draw names the same id under
    every perturbation its error model allows (any normaliser, one rounding
    per weight in either direction, the fixed-point floor), and a draw that a
    one-rounding perturbation does move is not certified."""
    rng = np.random.default_rng(21)
    certified = 0
    for trial in range(60):
        V = int(rng.integers(2, 200))
        p = (rng.random(V) ** 3).astype(F32)
        u = np.float32(int(rng.integers(0, 1 << 24)) * 2.0 ** -24)
        res = o.accept(p[None], np.zeros((0, V), F32), np.zeros(0, np.int32), np.array([u], F32), 1, 0)
        if not res.status[0] & o.DRAW_CERTIFIED:
            continue
        certified += 1
        cdf = np.cumsum(p.astype(np.float64))
        j = int(res.next_token[0])
        for signs in (np.ones(V), -np.ones(V), np.where(np.arange(V) <= j, 1, -1),
                      np.where(np.arange(V) <= j, -1, 1), rng.integers(-1, 2, V)):
            for z_rel in (0.0, 1e-3, -1e-3):
                assert _fixed_point_bonus_draw(p, u, z_rel, signs) == j, (trial, cdf[j] / cdf[-1])
    assert certified >= 50  # the flag is not vacuous: most uniforms are far from a step
    # F_0 = 1 / (2 - 2^-24) lies 2^-26 above u = 0.5: lowering weight 0 and
    # raising weight 1 by one rounding each moves the draw from 0 to 1
    p = np.array([1.0, 1.0 - 2.0 ** -24], F32)
    res = o.accept(p[None], np.zeros((0, 2), F32), np.zeros(0, np.int32), np.array([0.5], F32), 1, 0)
    assert res.next_token[0] == 0
    assert _fixed_point_bonus_draw(p, 0.5, 0.0, np.array([-1, 1])) == 1
    assert not res.status[0] & o.DRAW_CERTIFIED
    assert res.status[0] & o.NEAR_BOUNDARY


# ------------------------------------------------------------------ logits

def pin_softmax_closed_form():
    x = np.log(np.array([1.0, 2.0, 3.0]))
    pr, err = o.softmax_fp64(x, 1.0)
    assert err == 0 and np.allclose(pr, [1 / 6, 2 / 6, 3 / 6], rtol=1e-14, atol=0)
    pr2, _ = o.softmax_fp64(x * 2, 2.0)
    assert np.allclose(pr, pr2, rtol=1e-14, atol=0)
    pr3, _ = o.softmax_fp64(np.array([0.0, -np.inf, 0.0]), 0.7)
    assert list(pr3) == [0.5, 0.0, 0.5]
    assert o.softmax_fp64(np.array([1.0, np.nan]), 1.0)[1] == o.BAD_VALUE
    assert o.softmax_fp64(np.array([1.0, np.inf]), 1.0)[1] == o.BAD_VALUE
    assert o.softmax_fp64(np.array([-np.inf, -np.inf]), 1.0)[1] == o.ZERO_MASS


def pin_bf16_decode():
    bits = np.array([0x3F80, 0xC000, 0x7F80, 0x0001, 0x8000, 0x4049], np.uint16)
    got = o.decode_rows(bits, "bf16")
    assert list(got[:5]) == [1.0, -2.0, np.inf, 2.0 ** -133, 0.0]
    assert got[5] == 3.140625


def pin_mixed_logits_consistency():
    rng = np.random.default_rng(12)
    B, K, V = 6, 3, 40
    tl = rng.normal(0, 2, (B * (K + 1), V)).astype(np.float16)
    dl = (tl[: B * K].astype(F32) + rng.normal(0, 1, (B * K, V))).astype(np.float16)
    T = np.array([0, 0.7, 0, 1.1, 0.5, 0], F32)
    tok = rng.integers(0, V, B * K).astype(np.int32)
    u = rng.random(B * (K + 1)).astype(F32)
    res = o.accept_from_logits(tl, dl, "f16", T, tok, u, B, K)
    for b in range(B):
        sl_t, sl_d = slice(b * (K + 1), (b + 1) * (K + 1)), slice(b * K, (b + 1) * K)
        if T[b] == 0:
            ref = o.verify_greedy(tl[sl_t], "f16", tok[sl_d], 1, K)
        else:
            ref = o.accept(o.warped_rows_f32(tl[sl_t], "f16", T[b]),
                           o.warped_rows_f32(dl[sl_d], "f16", T[b]), tok[sl_d], u[sl_t], 1, K)
        assert (res.n_accepted[b], res.next_token[b], res.status[b]) == \
            (ref.n_accepted[0], ref.next_token[0], ref.status[0])


# ------------------------------------------------------------------ layout & errors

def pin_ragged_equals_single_sequences():
    rng = np.random.default_rng(13)
    B, Kmax, V = 9, 5, 30
    kb = rng.integers(0, Kmax + 1, B)
    cu = np.concatenate([[0], np.cumsum(kb)]).astype(np.int32)
    nt, nd = int((kb + 1).sum()), int(kb.sum())
    p = rng.random((nt, V)).astype(F32)
    q = rng.random((nd, V)).astype(F32)
    tok = rng.integers(0, V, nd).astype(np.int32)
    u = rng.random(nt).astype(F32)
    res = o.accept(p, q, tok, u, B, Kmax, cu)
    for b in range(B):
        k, t0, d0 = int(kb[b]), int(cu[b]) + b, int(cu[b])
        one = o.accept(p[t0:t0 + k + 1], q[d0:d0 + k], tok[d0:d0 + k], u[t0:t0 + k + 1], 1, k)
        assert (res.n_accepted[b], res.next_token[b]) == (one.n_accepted[0], one.next_token[0])
        if k == 0:
            assert res.n_accepted[b] == 0 and res.next_token[b] >= 0
    bad = cu.copy()
    bad[3] = bad[4] + 1  # K_2 < 0 and K_3 > bad
    r2 = o.accept(p, q, tok, u, B, Kmax, bad)
    assert r2.status[2] == o.BAD_LAYOUT and r2.next_token[2] == -1


def pin_sampling_error_codes():
    p = np.array([[0.5, 0.5], [0.5, 0.5], [0.5, 0.5]], F32)
    q = np.array([[0.5, 0.5], [0.5, 0.5]], F32)
    ok = dict(tokens=[0, 1], u=[0.1, 0.1, 0.5])
    assert run_one(p, q, **ok)[0] == 2
    assert run_one(p, q, [0, 2], ok["u"]) == (1, -1, o.BAD_TOKEN)
    bad = p.copy(); bad[1, 0] = np.nan
    assert run_one(bad, q, **ok) == (1, -1, o.BAD_VALUE)
    bad = p.copy(); bad[0, 1] = -1e-30
    assert run_one(bad, q, **ok) == (0, -1, o.BAD_VALUE)
    badq = q.copy(); badq[1, 1] = np.inf
    assert run_one(p, badq, **ok) == (1, -1, o.BAD_VALUE)
    assert run_one(p, q, [0, 1], [0.1, 1.0, 0.5]) == (1, -1, o.BAD_VALUE)
    zero = p.copy(); zero[1] = 0
    assert run_one(zero, q, **ok) == (1, -1, o.ZERO_MASS)
    zero = p.copy(); zero[2] = 0
    assert run_one(zero, q, **ok) == (2, -1, o.ZERO_MASS)
    # errors in rows past the first rejection are never read
    late = p.copy(); late[2, 0] = np.nan
    r = run_one(np.array([[1.0, 0.0], [0.5, 0.5], [np.nan, 0]], F32), q, [1, 0], [0.5, 0.5, 0.5])
    assert r == (0, 0, 0)


def pin_near_empty_residual():
    """After a rejection the residual mass is q(t) - p(t) summed the other
    way: with p = (1/2, 1/2) and q = (1/2 + d, 1/2 - d), rejecting token 0
    leaves the residual (0, d), whose mass d is flagged NEAR_EMPTY (with
    NEAR_BOUNDARY) exactly when d is inside the fp32 band; the draw still
    names token 1, the only one with residual weight."""
    p = [[0.5, 0.5], [0.5, 0.5]]
    u = [1.0 - 2.0 ** -24, 0.5]  # u q(0) > p(0) for any d >= 2^-23: a rejection
    for d, flagged in ((2.0 ** -23, True), (2.0 ** -21, True), (2.0 ** -19, False), (0.0625, False)):
        assert run_one(p, [[0.5 + d, 0.5 - d]], [0], u) == (
            0, 1, (o.NEAR_EMPTY | o.NEAR_BOUNDARY) if flagged else 0), d
    assert o.EMPTY_PROB_TOL == 2.0 ** -20
    # warped rows: the band is the row pair's softmax band (about 4.4e-5 for
    # logits near 0 at T = 1), against sigmoid(x) - 1/2 ~ x / 4
    tgt = np.zeros((2, 2), F32)
    for x, flagged in ((1e-6, True), (1e-4, True), (1e-3, False), (0.5, False)):
        dft = np.array([[x, 0.0]], F32)
        r = o.accept_from_logits(tgt, dft, "f32", np.ones(1, F32), np.zeros(1, np.int32),
                                 np.array(u, F32), 1, 1)
        assert (int(r.n_accepted[0]), int(r.next_token[0])) == (0, 1), x
        assert bool(r.status[0] & o.NEAR_EMPTY) == flagged, (x, r.status[0])
        assert not flagged or r.status[0] & o.NEAR_BOUNDARY


PINS = [v for k, v in sorted(globals().items()) if k.startswith("pin_")]


@pytest.mark.parametrize("pin", PINS, ids=[p.__name__ for p in PINS])
def test_pin(pin):
    pin()
