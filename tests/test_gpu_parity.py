"""GPU path vs the CPU oracle, element by element, through the C ABI.

Greedy outputs, accepted lengths and every sampled accept/reject decision
must be bit-identical to the oracle; resampled / bonus ids must match except
where the oracle flags u*R within 1e-5*R of a CDF step (counted and printed).
Sizes span several 16 KB shared-memory chunks, several CTAs per cluster and a
ragged tail; the full benchmark sizes are in test_gpu_fullsize.py.
"""

import numpy as np
import pytest

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():  # pragma: no cover - CPU-only runs
    pytestmark = pytest.mark.skip("needs a GPU")
else:
    pytestmark = pytest.mark.gpu

import __graft_entry__  # noqa: E402
import oracle  # noqa: E402
import workloads  # noqa: E402
from workloads.configs import Workload  # noqa: E402

F32 = np.float32


@pytest.fixture(scope="module", autouse=True)
def built():
    __graft_entry__.build()


def H():
    import gpu_helpers
    return gpu_helpers


def adhoc(mode, target, draft, tokens, uniforms, B, K, dtype="f32", cu_k=None, temperature=None):
    return Workload("adhoc", mode, dtype, B, K, target.shape[1], target, draft, tokens, uniforms,
                    cu_k, temperature, {})


# ------------------------------------------------------------------ greedy

@pytest.mark.parametrize("V", [1, 3, 8, 1000, 4099, 40961])
def test_greedy_probs_shapes(V):
    wl = workloads.make_config("config3", B=24, K=4, V=V, tie_every=3)
    H().compare(H().run_gpu(wl), H().run_oracle(wl), exact_tokens=True)


@pytest.mark.parametrize("dtype", ["f32", "bf16", "f16"])
def test_greedy_on_logits(dtype):
    rng = np.random.default_rng(1)
    B, K, V = 40, 3, 5001
    x = rng.normal(0, 2, (B * (K + 1), V)).astype(F32)
    x[::7, 17] = x[::7].max(axis=1)  # ties with the row max
    if dtype == "bf16":
        tgt = workloads.f32_to_bf16_bits(x)
        dec = oracle.decode_rows(tgt, "bf16")
    elif dtype == "f16":
        tgt = x.astype(np.float16)
        dec = tgt.astype(np.float64)
    else:
        tgt, dec = x, x.astype(np.float64)
    am = np.array([oracle.argmax_lowest(r)[0] for r in dec])
    tok = np.where(rng.random(B * K) < 0.8, am.reshape(B, K + 1)[:, :K].reshape(-1),
                   rng.integers(0, V, B * K)).astype(np.int32)
    wl = adhoc("greedy", tgt, None, tok, None, B, K, dtype)
    H().compare(H().run_gpu(wl), H().run_oracle(wl), exact_tokens=True)


def test_greedy_special_values():
    B, K, V = 6, 2, 700
    rows = np.random.default_rng(2).random((B * (K + 1), V)).astype(F32)
    rows[0, :] = np.nan                      # all NaN -> index 0, BAD_VALUE
    rows[3, :] = -np.inf                     # all -inf -> index 0
    rows[4, 5::9] = np.nan                   # NaN never wins
    rows[6, :] = -np.inf
    rows[6, 600] = np.nan
    rows[6, 333] = -np.inf                   # first non-NaN -inf
    rows[7, 10] = np.inf
    rows[7, 650] = np.inf                    # +inf tie -> lower index
    rows[9, 0] = -0.0
    rows[9, 1:] = -1.0
    rows[9, 500] = 0.0                       # -0 == +0 tie -> index 0
    tok = np.array([0, 0, 0, 3, 0, 333, 10, 0, 0, 0, 5, 0], np.int32)
    tok[1] = -1                              # out of range -> BAD_TOKEN
    wl = adhoc("greedy", rows, None, tok, None, B, K)
    H().compare(H().run_gpu(wl), H().run_oracle(wl), exact_tokens=True)


def test_greedy_ragged_unaligned_and_strided():
    rng = np.random.default_rng(3)
    B, Kmax, V = 13, 6, 3001
    kb = rng.integers(0, Kmax + 1, B)
    kb[0] = 0
    cu = np.concatenate([[0], np.cumsum(kb)]).astype(np.int32)
    rows = rng.random((int((kb + 1).sum()), V + 3)).astype(F32)  # row stride V + 3
    am = rows[:, :V].argmax(axis=1)
    tok = np.empty(int(kb.sum()), np.int32)
    for b in range(B):
        for i in range(kb[b]):
            tok[cu[b] + i] = am[cu[b] + b + i] if rng.random() < 0.85 else rng.integers(V)
    import torch as T
    gpu = H()
    dev = T.from_numpy(rows).to(gpu.DEV)[:, :V]  # strided view, not 16-byte aligned rows
    r = __import__("speculative_decoding_verification_decode_gb300").verify_greedy(
        dev, T.from_numpy(tok).to(gpu.DEV), T.from_numpy(cu).to(gpu.DEV), Kmax)
    got = oracle.Result(r.n_accepted.cpu().numpy(), r.next_token.cpu().numpy(),
                        r.status.cpu().numpy().astype(np.uint32))
    ref = oracle.verify_greedy(np.ascontiguousarray(rows[:, :V]), "f32", tok, B, Kmax, cu)
    gpu.compare(got, ref, exact_tokens=True)
    # misaligned base pointer (offset by one element)
    flat = T.from_numpy(np.ascontiguousarray(rows[:, :V]).reshape(-1)).to(gpu.DEV)
    buf = T.empty(flat.numel() + 1, device=gpu.DEV)
    buf[1:] = flat
    r2 = __import__("speculative_decoding_verification_decode_gb300").verify_greedy(
        buf[1:].view(-1, V), T.from_numpy(tok).to(gpu.DEV), T.from_numpy(cu).to(gpu.DEV), Kmax)
    assert np.array_equal(r2.next_token.cpu().numpy(), ref.next_token)


def test_greedy_bad_layout():
    rng = np.random.default_rng(4)
    B, K, V = 4, 3, 100
    cu = np.array([0, 2, 1, 5, 9], np.int32)  # K_1 < 0; K_3 = 4 > K
    rows = rng.random((9 + B, V)).astype(F32)
    tok = rng.integers(0, V, 9).astype(np.int32)
    wl = adhoc("greedy", rows, None, tok, None, B, K, cu_k=cu)
    H().compare(H().run_gpu(wl), H().run_oracle(wl), exact_tokens=True)


# ------------------------------------------------------------------ sampling from probabilities

def test_accept_config1_full_600_rounds():
    wl = workloads.make_config("config1")  # B=600 rounds, K=4, V=32000
    near, diff = H().compare(H().run_gpu(wl, "accept"), H().run_oracle(wl, "accept"))
    print(f"config1 sampled: {near} boundary-flagged draws, {diff} differ")
    g = H().run_gpu(wl, "greedy")
    H().compare(g, H().run_oracle(wl, "greedy"), exact_tokens=True)


@pytest.mark.parametrize("V", [2, 7, 64, 4099, 20011])
def test_accept_ragged_shapes(V):
    wl = workloads.make_config("config4", B=24, V=V)
    near, diff = H().compare(H().run_gpu(wl), H().run_oracle(wl))
    print(f"V={V}: {near} flagged, {diff} differ")


def test_accept_force_exact_agrees():
    wl = workloads.make_config("config4", B=32, V=5003)
    a = H().run_gpu(wl)
    b = H().run_gpu(wl, flags=1)
    assert np.array_equal(a.n_accepted, b.n_accepted)
    assert np.array_equal(a.next_token, b.next_token)
    assert (b.status & 16).all() or (b.n_accepted == 0).any()
    H().compare(b, H().run_oracle(wl))


def test_accept_exact_ties_and_dyadic_thresholds():
    """u * q(t) * Zp == p(t) * Zq exactly on dyadic rows: strict '<' rejects;
    the filter cannot decide these, so they exercise the exact path."""
    rng = np.random.default_rng(5)
    V, K = 16, 3
    B = 300
    p = np.zeros((B * (K + 1), V), F32)
    q = np.zeros((B * K, V), F32)
    tok = np.zeros(B * K, np.int32)
    u = np.zeros(B * (K + 1), F32)
    for b in range(B):
        for i in range(K + 1):
            p[b * (K + 1) + i] = rng.integers(0, 64, V) / 64.0
            p[b * (K + 1) + i, 0] = 1.0
        for i in range(K):
            qr = rng.integers(1, 64, V) / 64.0
            q[b * K + i] = qr
            t = int(rng.integers(V))
            tok[b * K + i] = t
            pr = p[b * (K + 1) + i]
            ratio = (pr[t] / pr.sum()) / (qr[t] / qr.sum())
            # threshold exactly, one ulp below, one ulp above, or random
            choice = rng.integers(4)
            uu = F32(min(ratio, 0.999))
            if choice == 1:
                uu = np.nextafter(uu, F32(0))
            elif choice == 2:
                uu = np.nextafter(uu, F32(1))
            elif choice == 3:
                uu = F32(rng.random())
            u[b * (K + 1) + i] = min(uu, F32(0.99999994))
        u[b * (K + 1) + K] = F32(rng.random())
    wl = adhoc("accept", p, q, tok, u, B, K)
    for flags in (0, 1):
        H().compare(H().run_gpu(wl, flags=flags), H().run_oracle(wl))


def test_accept_error_cases():
    rng = np.random.default_rng(6)
    B, K, V = 10, 2, 300
    p = rng.random((B * (K + 1), V)).astype(F32)
    q = rng.random((B * K, V)).astype(F32)
    tok = rng.integers(0, V, B * K).astype(np.int32)
    u = (rng.random(B * (K + 1)) * 0.01).astype(F32)  # mostly accept
    tok[0] = V                       # seq 0: bad token at row 0
    p[3, 7] = np.nan                 # seq 1: NaN in target row 0
    q[4, 8] = -1e-20                 # seq 2: negative draft value at row 0
    p[9, :] = 0                      # seq 3: zero target row 0
    q[8, :] = 0                      # seq 4: zero draft row 0
    u[15] = 1.0                      # seq 5: uniform out of range
    p[20, 3] = np.inf                # seq 6: +Inf in the target row 2 (bonus)
    p[21:24] *= 2.0 ** 100           # seq 7: huge unnormalised rows (exact scaling)
    q[14:16] *= 2.0 ** -110
    p[24:27] = (p[24:27] * 2.0 ** -126).astype(F32)  # seq 8: tiny (partly subnormal) rows
    p[27, :] = 3.0e38                # seq 9: finite values whose fp32 partial sums overflow
    wl = adhoc("accept", p, q, tok, u, B, K)
    H().compare(H().run_gpu(wl), H().run_oracle(wl))


def test_accept_scale_invariance():
    wl = workloads.make_config("config4", B=16, V=3001)
    a = H().run_gpu(wl)
    wl.target = (wl.target * F32(2.0 ** 70)).astype(F32)
    wl.draft = (wl.draft * F32(2.0 ** -50)).astype(F32)
    b = H().run_gpu(wl)
    assert np.array_equal(a.n_accepted, b.n_accepted)
    ref = H().run_oracle(wl)
    H().compare(b, ref)


def test_accept_determinism():
    wl = workloads.make_config("config4", B=16, V=20000)
    a, b = H().run_gpu(wl), H().run_gpu(wl)
    for x, y in zip((a.n_accepted, a.next_token, a.status), (b.n_accepted, b.next_token, b.status)):
        assert np.array_equal(x, y)


# ------------------------------------------------------------------ logits

def _warped_parity(wl, res, warped, rtol):
    """Warped rows vs the oracle's fp64 softmax (normalised by the exact sum
    of the kernel's own weights), and decisions vs the oracle run on the
    kernel's own warped rows (bit-exact)."""
    wt, wd = warped
    K = wl.K
    worst = 0.0
    for b in range(wl.B):
        T = float(wl.temperature[b])
        if T == 0:
            continue
        n = int(res.n_accepted[b])
        for i in range(min(n, K) + 1):
            for rows, warp, idx in ((wl.target, wt, b * (K + 1) + i), (wl.draft, wd, b * K + i)):
                if rows is wl.draft and i >= K:
                    continue
                w = warp[idx].astype(np.float64)
                assert np.isfinite(w).all(), (b, i)
                pg = w / float(oracle.exact_mass(warp[idx]))
                pr, err = oracle.softmax_fp64(oracle.decode_rows(rows[idx], wl.dtype), T)
                big = pr >= 1e-30
                rel = np.abs(pg[big] - pr[big]) / pr[big]
                worst = max(worst, float(rel.max()))
                assert rel.max() <= rtol, (b, i, rel.max())
                assert np.all(np.abs(pg[~big] - pr[~big]) <= 1e-30)
    # decisions on the kernel's own weights: bit-exact
    samp = wl.temperature > 0
    ref = oracle.accept(np.nan_to_num(wt, nan=0.0), np.nan_to_num(wd, nan=0.0), wl.tokens,
                        wl.uniforms, wl.B, wl.K)
    assert np.array_equal(res.n_accepted[samp], ref.n_accepted[samp])
    near = (ref.status & oracle.NEAR_BOUNDARY) > 0
    ok = (res.next_token == ref.next_token) | near
    assert ok[samp].all()
    return worst


@pytest.mark.parametrize("dtype,rtol", [("bf16", 2e-3), ("f16", 2e-3), ("f32", 1e-6)])
def test_logits_warp_and_decisions(dtype, rtol):
    wl = workloads.make_config("config2", B=12, K=5, V=9001)
    if dtype != "bf16":
        x = oracle.decode_rows(wl.target, "bf16").astype(F32)
        y = oracle.decode_rows(wl.draft, "bf16").astype(F32)
        if dtype == "f16":
            wl.target, wl.draft = x.astype(np.float16), y.astype(np.float16)
        else:
            rng = np.random.default_rng(8)
            wl.target = (x + rng.normal(0, 1e-3, x.shape)).astype(F32)
            wl.draft = (y + rng.normal(0, 1e-3, y.shape)).astype(F32)
        wl.dtype = dtype
    res, warped = H().run_gpu(wl, warped=True)
    worst = _warped_parity(wl, res, warped, rtol)
    print(f"{dtype}: worst relative error of the fused softmax {worst:.3g}")
    ref = H().run_oracle(wl)
    H().assert_softmax_agreement(res, ref, f"{dtype}")


def test_logits_mixed_config5_scaled():
    wl = workloads.make_config("config5", B=64, V=7001)
    res, warped = H().run_gpu(wl, warped=True)
    _warped_parity(wl, res, warped, 2e-3)
    ref = H().run_oracle(wl)
    g = wl.temperature == 0
    assert np.array_equal(res.n_accepted[g], ref.n_accepted[g])
    assert np.array_equal(res.next_token[g], ref.next_token[g])
    assert np.array_equal(res.status[g], ref.status[g])
    H().assert_softmax_agreement(res, ref, "config5 (scaled) sampled half", mask=~g)


def test_logits_error_cases():
    rng = np.random.default_rng(9)
    B, K, V = 6, 2, 500
    tl = rng.normal(0, 2, (B * (K + 1), V)).astype(F32)
    dl = (tl[: B * K] + rng.normal(0, 1, (B * K, V))).astype(F32)
    T = np.array([0.7, -1.0, np.nan, 0.9, 0.8, 1.0], F32)
    tl[9, 4] = np.inf       # seq 3: +Inf logit in target row 0
    dl[8, :] = -np.inf      # seq 4: draft row 0 all -inf -> zero mass
    tl[15, 2] = np.nan      # seq 5: NaN in target row 0
    tok = rng.integers(0, V, B * K).astype(np.int32)
    u = rng.random(B * (K + 1)).astype(F32)
    wl = adhoc("logits", tl.astype(np.float16), dl.astype(np.float16), tok, u, B, K, "f16",
               temperature=T)
    H().compare(H().run_gpu(wl), H().run_oracle(wl))


# ------------------------------------------------------------------ laws on the GPU

def test_gpu_accepted_length_law():
    from scipy import stats
    rng = np.random.default_rng(20240601)
    K, V, R = 4, 16, 100_000
    tl = rng.normal(0, 1.5, (K + 1, V))
    p = np.exp(tl).astype(F32)
    q = np.exp(tl[:K] + rng.normal(0, 1.0, (K, V))).astype(F32)
    qh = q.astype(np.float64) / q.astype(np.float64).sum(1, keepdims=True)
    cdf = np.cumsum(qh, 1)
    tok = np.stack([np.minimum(np.searchsorted(cdf[i], rng.random(R) * cdf[i, -1], "right"), V - 1)
                    for i in range(K)], 1).astype(np.int32)
    u = (rng.integers(0, 1 << 24, (R, K + 1)) * 2.0 ** -24).astype(F32)
    wl = adhoc("accept", np.tile(p, (R, 1)), np.tile(q, (R, 1)), tok.reshape(-1), u.reshape(-1),
               R, K)
    res = H().run_gpu(wl)
    ph = p.astype(np.float64) / p.astype(np.float64).sum(1, keepdims=True)
    alpha = np.minimum(ph[:K], qh).sum(1)
    surv = np.concatenate([[1.0], np.cumprod(alpha)])
    probs = np.concatenate([surv[:-1] - surv[1:], [surv[-1]]])
    counts = np.bincount(res.n_accepted, minlength=K + 1)
    pv = stats.chisquare(counts, probs * R).pvalue
    assert pv > 0.01, (counts, probs * R)
    # the emitted token after a rejection / the bonus follows p exactly in law:
    # compare with the oracle on a sample of the same rounds
    sub = slice(0, 2000)
    ref = oracle.accept(wl.target[: 2000 * (K + 1)], wl.draft[: 2000 * K], wl.tokens[: 2000 * K],
                        wl.uniforms[: 2000 * (K + 1)], 2000, K)
    assert np.array_equal(res.n_accepted[sub], ref.n_accepted)


def test_host_buffers_roundtrip():
    import speculative_decoding_verification_decode_gb300 as sv
    wl = workloads.make_config("config4", B=8, V=4001)
    import torch as T
    r = sv.accept(T.from_numpy(wl.target).pin_memory(), T.from_numpy(wl.draft).pin_memory(),
                  T.from_numpy(wl.tokens), T.from_numpy(wl.uniforms), T.from_numpy(wl.cu_k), wl.K)
    assert r.n_accepted.device.type == "cpu"
    ref = H().run_gpu(wl)
    assert np.array_equal(r.n_accepted.numpy(), ref.n_accepted)
    assert np.array_equal(r.next_token.numpy(), ref.next_token)
