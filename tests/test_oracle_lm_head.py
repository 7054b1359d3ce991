"""Pins of the oracle's LM head in front of verification (llmstudio.ru
section 21: logits = states times the vocabulary projection; section 22:
greedy needs the argmax, sampling the whole distribution; TensorSharp
speculative_decoding.md, "DFlash and DFlash2": the drafter borrows the
target's LM head).

The pins come from outside the oracle: an identity projection reduces the
path to the pinned logits verification; one-hot states pick out columns of
the projection; every logit is recomputed by brute force (an exactly rounded
sum of the d products) and the whole path re-run on those logits; doubling
the projection and the temperature (exact in bf16) changes nothing.  Planted
mistakes at the bottom are each caught.
"""

import inspect
import math
import textwrap

import numpy as np
import pytest

import oracle
import oracle.lm_head as lmh
import workloads
from workloads import f32_to_bf16_bits

F32 = np.float32


def _bits_to_f64(bits):
    return (np.asarray(bits, np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def _brute_logits(h_bits, w_bits):
    h, w = _bits_to_f64(h_bits), _bits_to_f64(w_bits)
    return np.array([[math.fsum(h[r] * w[v]) for v in range(w.shape[0])] for r in range(h.shape[0])])


def _small(seed=0, B=6, K=3, V=23, d=17, T=0.9):
    wl = workloads.make_lm_head(seed=seed, B=B, K=K, V=V, d=d, temperature=T)
    return wl


def test_logits_match_brute_force_sums():
    wl = _small()
    ref = _brute_logits(wl.h_target, wl.w)
    got = oracle.lm_head_logits(wl.h_target, wl.w, "bf16")
    assert got.shape == (wl.B * (wl.K + 1), wl.V)
    assert np.allclose(got, ref, rtol=1e-12, atol=1e-12)


def test_whole_path_on_brute_force_logits():
    for seed in range(4):
        wl = _small(seed=seed)
        r = oracle.accept_lm_head(wl.h_target, wl.h_draft, wl.w, "bf16", wl.temperature, wl.tokens,
                                  wl.uniforms, wl.B, wl.K)
        lt, ld = _brute_logits(wl.h_target, wl.w), _brute_logits(wl.h_draft, wl.w)
        ref = oracle.accept_from_logits(lt, ld, "f64", wl.temperature, wl.tokens, wl.uniforms, wl.B, wl.K)
        assert np.array_equal(r.n_accepted, ref.n_accepted)
        assert np.array_equal(r.next_token, ref.next_token)
        g = oracle.verify_greedy_lm_head(wl.h_target, wl.w, "bf16", wl.tokens, wl.B, wl.K)
        gref = oracle.verify_greedy(lt, "f64", wl.tokens, wl.B, wl.K)
        assert np.array_equal(g.n_accepted, gref.n_accepted) and np.array_equal(g.next_token, gref.next_token)


def test_identity_projection_is_logits_verification():
    # V = d and W = I: the logits are the states themselves
    rng = np.random.default_rng(3)
    B, K, d = 8, 3, 40
    w = f32_to_bf16_bits(np.eye(d, dtype=F32))
    ht = f32_to_bf16_bits(rng.normal(0, 2, (B * (K + 1), d)).astype(F32))
    hd = f32_to_bf16_bits(rng.normal(0, 2, (B * K, d)).astype(F32))
    tok = rng.integers(0, d, B * K).astype(np.int32)
    u = rng.random(B * (K + 1)).astype(F32)
    T = np.full(B, 0.7, F32)
    T[::3] = 0.0  # some greedy sequences too
    r = oracle.accept_lm_head(ht, hd, w, "bf16", T, tok, u, B, K)
    ref = oracle.accept_from_logits(ht, hd, "bf16", T, tok, u, B, K)
    for f in ("n_accepted", "next_token", "status"):
        assert np.array_equal(getattr(r, f), getattr(ref, f))


def test_one_hot_states_read_columns_of_the_projection():
    # h = e_j gives the logits W[:, j]; greedy then emits argmax_v W[v, j]
    rng = np.random.default_rng(4)
    V, d, B = 31, 9, 5
    w32 = rng.normal(0, 1, (V, d)).astype(F32)
    w = f32_to_bf16_bits(w32)
    wf = _bits_to_f64(w)
    cols = rng.integers(0, d, B)
    h = np.zeros((B, d), F32)
    h[np.arange(B), cols] = 1.0
    g = oracle.verify_greedy_lm_head(f32_to_bf16_bits(h), w, "bf16", np.zeros(0, np.int32), B, 0)
    assert np.array_equal(g.n_accepted, np.zeros(B))
    assert np.array_equal(g.next_token, np.array([int(np.argmax(wf[:, c])) for c in cols]))


def test_doubling_projection_and_temperature_changes_nothing():
    wl = _small(seed=9, B=10)
    w2 = f32_to_bf16_bits((_bits_to_f64(wl.w) * 2.0).astype(F32))  # exact: one more in the exponent
    a = oracle.accept_lm_head(wl.h_target, wl.h_draft, wl.w, "bf16", wl.temperature, wl.tokens,
                              wl.uniforms, wl.B, wl.K)
    b = oracle.accept_lm_head(wl.h_target, wl.h_draft, w2, "bf16", wl.temperature * 2, wl.tokens,
                              wl.uniforms, wl.B, wl.K)
    for f in ("n_accepted", "next_token"):
        assert np.array_equal(getattr(a, f), getattr(b, f))


def pin_brute():
    test_logits_match_brute_force_sums()
    test_whole_path_on_brute_force_logits()


def pin_identity():
    test_identity_projection_is_logits_verification()


LM_MUTATIONS = [
    ("lm_head_logits", "return hd @ wd.T", "return 0.5 * (hd @ wd.T)", [pin_brute]),
    ("lm_head_logits", "wd = decode_rows(w, dtype).reshape(w.shape)",
     "wd = np.asarray(w, np.float64)", [pin_brute, pin_identity]),
    ("accept_lm_head", "ld = lm_head_logits(h_draft, w, dtype)",
     "ld = lm_head_logits(h_target[:h_draft.shape[0]], w, dtype)", [pin_brute, pin_identity]),
]


@pytest.mark.parametrize("fn_name,old,new,catchers", LM_MUTATIONS,
                         ids=[f"{m[0]}:{i}" for i, m in enumerate(LM_MUTATIONS)])
def test_planted_lm_head_mistake_is_caught(monkeypatch, fn_name, old, new, catchers):
    src = textwrap.dedent(inspect.getsource(getattr(lmh, fn_name)))
    assert src.count(old) >= 1, (fn_name, old)
    ns = dict(vars(lmh))
    exec(compile(src.replace(old, new, 1), f"<mutant {fn_name}>", "exec"), ns)
    monkeypatch.setattr(lmh, fn_name, ns[fn_name])
    monkeypatch.setattr(oracle, fn_name, ns[fn_name])  # callers look it up in the module
    caught = []
    for pin in catchers:
        try:
            pin()
        except AssertionError:
            caught.append(pin.__name__)
    assert caught, f"no pin caught the mutation of {fn_name}: {old!r} -> {new!r}"
