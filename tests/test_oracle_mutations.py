"""Planted mistakes: each test breaks one oracle function on the CPU (a
textual mutation of its source, applied to a private copy) and checks that
at least one pin from ``test_oracle_pins.py`` then fails.  This is the
evidence that the pins would catch a dropped term, a wrong sign, a wrong
index or a transposed operand in the oracle itself."""

import inspect
import textwrap

import pytest

import oracle
import oracle.spec_verify as sv
import test_oracle_pins as pins

MUTATIONS = [
    # (function, original text, planted mistake, pins expected to catch it)
    ("accept_decision", "return lhs < rhs", "return lhs <= rhs",
     ["pin_zero_target_mass_never_accepted", "pin_accept_decision_exact_ties"]),
    ("accept_decision", "Fraction(float(np.float32(q_t))) * zp_int",
     "Fraction(float(np.float32(p_t))) * zp_int", ["pin_s15_accept_ratio"]),
    ("accept_decision", "* zp_int", "* 1", ["pin_s15_accept_ratio"]),
    ("accept_decision", "rhs = Fraction(float(np.float32(p_t))) * zq_int",
     "rhs = Fraction(float(np.float32(p_t))) * zp_int", ["pin_scale_invariance"]),
    ("_accept_sequence", "np.maximum(0.0, phat - qhat)", "np.maximum(0.0, qhat - phat)",
     ["pin_s18_acceptance_and_residual"]),
    ("_accept_sequence", "inverse_cdf_draw(resid, u[k])", "inverse_cdf_draw(resid, u[i])",
     ["pin_enumeration_marginal_equals_target"]),
    ("_accept_sequence", "w = p.astype(np.float64) / _frac_to_f64(zp)",
     "w = p.astype(np.float64)[::-1] / _frac_to_f64(zp)", ["pin_enumeration_bonus_law"]),
    ("_accept_sequence", "inverse_cdf_draw(w, u[i], TIGHT_BONUS_REL)", "inverse_cdf_draw(w, u[i], 2.0 ** -30)",
     ["pin_certified_bonus_draws"]),
    ("_accept_sequence", "if not resid.sum() > band:", "if not resid.sum() > 0.0:",
     ["pin_near_empty_residual"]),
    ("_greedy_sequence", "return i, a, status\n", "return i, (a + 1) % V, status\n",
     ["pin_greedy_reproduces_plain_decoding"]),
    ("argmax_lowest", "int(cand[0])", "int(cand[-1])",
     ["pin_argmax_rules", "pin_greedy_reproduces_plain_decoding"]),
    ("exact_mass_int", "np.where(expo > 0, frac | 0x800000, frac)",
     "np.where(expo > 0, frac | 0x800000, 0)", ["pin_exact_mass_vs_fsum"]),
    ("inverse_cdf_draw", 'side="right"', 'side="left"', ["pin_inverse_cdf_closed_form"]),
    ("softmax_fp64", "(x - m) / float(temperature)", "(x - m) * float(temperature)",
     ["pin_softmax_closed_form"]),
]


def _mutated(fn_name, old, new):
    src = textwrap.dedent(inspect.getsource(getattr(sv, fn_name)))
    assert src.count(old) >= 1, (fn_name, old)
    src = src.replace(old, new, 1)
    ns = dict(vars(sv))
    exec(compile(src, f"<mutant {fn_name}>", "exec"), ns)
    return ns[fn_name]


@pytest.mark.parametrize("fn_name,old,new,catchers", MUTATIONS,
                         ids=[f"{m[0]}:{i}" for i, m in enumerate(MUTATIONS)])
def test_planted_mistake_is_caught(monkeypatch, fn_name, old, new, catchers):
    mutant = _mutated(fn_name, old, new)
    monkeypatch.setattr(sv, fn_name, mutant)
    if hasattr(oracle, fn_name):  # the package re-exports public functions
        monkeypatch.setattr(oracle, fn_name, mutant)
    caught = []
    for name in catchers:
        try:
            getattr(pins, name)()
        except AssertionError:
            caught.append(name)
    assert caught, f"no pin caught the mutation of {fn_name}: {old!r} -> {new!r}"
