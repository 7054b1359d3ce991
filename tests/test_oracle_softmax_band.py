"""Pin of the oracle's NEAR_DECISION band for verification from logits.

An fp32 evaluation of the warp (weights 2^(l k - m k) with the argument
rounded once, as one FMA does, and an exp2 of relative error up to 2^-21)
decides the accept tests on weights that differ slightly from the oracle's
fp64 softmax.  Wherever the two decide differently the oracle must have
flagged the sequence; and on ordinary inputs the flag must be rare.
"""

import numpy as np

import oracle

F32 = np.float32
LOG2E = 1.4426950408889634


def _fp32_weights(logits64, T, rng):
    """fp32 weights of one row: k = fp32(log2(e)/T), mk = fp32(m k), the
    argument l k - mk rounded once to fp32 (exact f64 product of two f32
    values minus an f32), 2^x rounded to f32 and then perturbed by a relative
    error in [-2^-21, 2^-21] (a model of a hardware exp2)."""
    k = float(F32(LOG2E / T))
    m = float(np.max(logits64))
    mk = float(F32(m * k))
    x = (logits64.astype(np.float64) * k - mk).astype(F32).astype(np.float64)
    w = np.exp2(x).astype(F32).astype(np.float64)
    w *= 1.0 + rng.uniform(-1, 1, w.shape) * oracle.spec_verify.EX2_REL
    w = w.astype(F32)
    w[x < -126] = 0  # flushed
    return w


def test_near_decision_band_covers_fp32_warps():
    rng = np.random.default_rng(23)
    B, K, V = 300, 3, 600
    T = np.where(rng.random(B) < 0.5, 0.8, rng.uniform(0.5, 1.2, B)).astype(F32)
    tl = (rng.normal(0, 3.0, (B * (K + 1), V)) + 8.0 * (rng.random((B * (K + 1), V)) < 0.03)).astype(F32)
    dl = np.empty((B * K, V), F32)
    for b in range(B):
        dl[b * K:(b + 1) * K] = tl[b * (K + 1):b * (K + 1) + K] + rng.normal(0, 1.5, (K, V)).astype(F32)
    tok = np.empty(B * K, np.int32)
    u = rng.integers(0, 1 << 24, B * (K + 1)).astype(np.float64) * 2.0 ** -24
    wt = np.empty_like(tl)
    wd = np.empty_like(dl)
    for b in range(B):
        for i in range(K + 1):
            wt[b * (K + 1) + i] = _fp32_weights(tl[b * (K + 1) + i].astype(np.float64), float(T[b]), rng)
        for i in range(K):
            r = b * K + i
            wd[r] = _fp32_weights(dl[r].astype(np.float64), float(T[b]), rng)
            q = wd[r].astype(np.float64) / wd[r].astype(np.float64).sum()
            tok[r] = rng.choice(V, p=q)
            if b % 2 == 0:  # put u_i within a few 1e-6 of the accept threshold
                p = wt[b * (K + 1) + i].astype(np.float64)
                ratio = (p[tok[r]] / p.sum()) / q[tok[r]]
                if ratio < 1:
                    u[b * (K + 1) + i] = ratio * (1 + rng.uniform(-4e-6, 4e-6))
    u = u.astype(F32)
    ref = oracle.accept_from_logits(tl, dl, "f32", T, tok, u, B, K)
    fast = oracle.accept(wt, wd, tok, u, B, K)
    near = (ref.status & oracle.NEAR_DECISION) > 0
    differ = ref.n_accepted != fast.n_accepted
    assert not (differ & ~near).any(), np.flatnonzero(differ & ~near)[:5]
    assert differ.any()  # the planted near-threshold uniforms do cross
    # ordinary (odd) sequences: u drawn freely, almost never near a threshold
    assert near[1::2].mean() < 0.02, near[1::2].mean()


def test_decision_band_formula():
    # the bound grows with |m k| and covers the exp2 error and two roundings
    t0 = oracle.softmax_weight_tol(0.0, 1.0)
    assert t0 > oracle.spec_verify.EX2_REL
    assert oracle.softmax_weight_tol(100.0, 0.5) > oracle.softmax_weight_tol(100.0, 1.0) > t0
    assert oracle.softmax_decision_tol(t0, t0) == 4 * t0 + 2 * 2.0 ** -24
