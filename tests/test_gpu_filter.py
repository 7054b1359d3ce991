"""Top-k / top-p sampler filters on the GPU against the oracle
(llmstudio.ru section 38: temperature, then top-k, then top-p, applied alike
to the target's p and the draft's q before verification).

Floors: top-k floors are integers in disguise (a value of the row picked by a
count) and must be bit-identical; top-p floors must equal the oracle's except
on rows the oracle itself flags ``near`` (its fp64 boundary within 1e-5 of
p Z), where the kernel's floor must still be a valid one.  Verification with
floors: decisions are bit-exact against the oracle run on the kernel's own
warped (and cut) rows, the cut matches the floors exactly, and top-k 1 turns
sampled verification into the GPU's own greedy verification.
"""

import math

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

F32 = np.float32
DEV = torch.device("cuda", 0)


@pytest.fixture(scope="module", autouse=True)
def built():
    __graft_entry__.build()


def H():
    import gpu_helpers
    return gpu_helpers


def sv():
    import speculative_decoding_verification_decode_gb300 as m
    return m


def _rows_of(wl):
    """Sequence of every target row and every draft row."""
    kb = wl.k_per_seq
    st = np.concatenate([np.full(k + 1, b) for b, k in enumerate(kb)]) if wl.B else np.zeros(0, int)
    sd = np.concatenate([np.full(k, b) for b, k in enumerate(kb)]) if wl.B else np.zeros(0, int)
    return st.astype(int), sd.astype(int)


def _filters(rng, B, V):
    top_k = rng.choice([0, 1, 2, 5, 50, V // 3, V - 1, V, V + 5], size=B).astype(np.int32)
    top_p = rng.choice([1.0, 0.5, 0.9, 0.95, 0.999, 1e-4, 1.5], size=B).astype(F32)
    return top_k, top_p


def _gpu_floors(wl, top_k, top_p):
    ft, fd = sv().sampler_floors(H().to_dev(wl.target, wl.dtype), H().to_dev(wl.draft, wl.dtype),
                                 H().to_dev(wl.temperature), H().to_dev(top_k), H().to_dev(top_p),
                                 H().to_dev(wl.cu_k), k=wl.K, sum_k=int(wl.tokens.size))
    torch.cuda.synchronize()
    return ft.cpu().numpy(), fd.cpu().numpy()


def _check_floors(wl, top_k, top_p, ft_g, fd_g, rows=None):
    """Floors equal the oracle's, or (on rows the oracle flags near) are valid.
    Returns the number of near rows whose floors differ."""
    dec = lambda r: oracle.decode_rows(r, wl.dtype)
    st, sd = _rows_of(wl)
    differ = 0
    for arr, g, seq in ((wl.target, ft_g, st), (wl.draft, fd_g, sd)):
        idx = range(arr.shape[0]) if rows is None else [r for r in rows if r < arr.shape[0]]
        for r in idx:
            b = seq[r]
            T = float(np.float32(wl.temperature[b]))
            if not T > 0:
                assert g[r] == -np.inf, (r, g[r])
                continue
            k = None if top_k is None else int(top_k[b])
            p = None if top_p is None else float(np.float32(top_p[b]))
            x = dec(arr[r])
            f, near, bad = oracle.filter_floor(x, T, k, p)
            if bad:
                assert math.isnan(g[r]), (r, g[r])
                continue
            if g[r] == f:
                continue
            assert near and oracle.floor_is_valid(x, T, k, p, float(g[r])), (r, b, k, p, g[r], f)
            differ += 1
    return differ


@pytest.mark.parametrize("name,dtype,V", [("config2", "bf16", 9001), ("config5", "f16", 7001),
                                          ("config2", "f32", 4099), ("config4", "f32", 12007)])
def test_floors_match_the_oracle(name, dtype, V):
    kw = dict(B=12, K=5, V=V) if name == "config2" else (dict(B=24, V=V) if name == "config5" else dict(B=10, V=V))
    wl = workloads.make_config(name, **kw)
    if wl.temperature is None:  # probabilities workload: use its logs as logits at T = 0.9
        wl.target = np.log(np.maximum(wl.target, 1e-30)).astype(F32)
        wl.draft = np.log(np.maximum(wl.draft, 1e-30)).astype(F32)
        wl.temperature = np.full(wl.B, 0.9, F32)
        wl.dtype = "f32"
    elif dtype == "f32" and wl.dtype != "f32":
        wl.target = oracle.decode_rows(wl.target, wl.dtype).astype(F32)
        wl.draft = oracle.decode_rows(wl.draft, wl.dtype).astype(F32)
        wl.dtype = "f32"
    rng = np.random.default_rng(V)
    top_k, top_p = _filters(rng, wl.B, wl.V)
    ft, fd = _gpu_floors(wl, top_k, top_p)
    d = _check_floors(wl, top_k, top_p, ft, fd)
    print(f"{name} {dtype}: {d} near-boundary rows took the other valid floor")
    # top-k alone, and top-p alone
    ft, fd = _gpu_floors(wl, top_k, None)
    _check_floors(wl, top_k, None, ft, fd)
    ft, fd = _gpu_floors(wl, None, top_p)
    _check_floors(wl, None, top_p, ft, fd)


def test_floors_ties_special_values_and_unaligned_rows():
    rng = np.random.default_rng(3)
    B, K, V = 6, 2, 1001
    rows = B * (K + 1) + B * K
    x = (np.round(rng.normal(0, 2, (rows, V)) * 4) / 4).astype(F32)  # quarter steps: many ties
    x[0, :7] = np.nan
    x[1, 5:400] = -np.inf
    x[2, 3] = np.inf                      # no finite maximum: no filter
    x[3, :] = 0.0
    x[3, ::2] = -0.0                      # -0 ties +0
    x[4, :] = -np.inf
    x[4, 17] = 1.0                        # one finite logit
    x[5, :] = np.nan                      # nothing to rank
    # stored with a row stride of V + 2 (4012 bytes: rows not 16-byte aligned)
    buf = np.zeros((rows, V + 2), F32)
    buf[:, :V] = x
    tgt_t = torch.from_numpy(buf[:B * (K + 1)]).to(DEV)[:, :V]
    drf_t = torch.from_numpy(buf[B * (K + 1):]).to(DEV)[:, :V]
    T = np.full(B, 1.3, F32)
    T[5] = 0.0
    for top_k, top_p in ((np.array([1, 2, 3, 500, 7, 1], np.int32), None),
                         (None, np.array([0.3, 0.9, 0.5, 0.99, 0.7, 0.5], F32)),
                         (np.array([3, 40, 2, 900, 1, 4], np.int32), np.array([0.6, 0.9, 0.5, 0.2, 0.7, 0.5], F32))):
        ft, fd = sv().sampler_floors(tgt_t, drf_t, torch.from_numpy(T).to(DEV),
                                     None if top_k is None else torch.from_numpy(top_k).to(DEV),
                                     None if top_p is None else torch.from_numpy(top_p).to(DEV))
        torch.cuda.synchronize()
        from workloads.configs import Workload
        wl = Workload("ties", "logits", "f32", B, K, V, x[:B * (K + 1)], x[B * (K + 1):],
                      np.zeros(B * K, np.int32), None, None, T, {})
        _check_floors(wl, top_k, top_p, ft.cpu().numpy(), fd.cpu().numpy())


def test_invalid_top_p_gives_nan_floors_and_bad_value():
    wl = workloads.make_config("config2", B=6, K=3, V=2003)
    top_p = np.array([0.9, 0.0, -1.0, np.nan, 1.0, 0.5], F32)
    ft, fd = _gpu_floors(wl, None, top_p)
    st, _ = _rows_of(wl)
    assert np.isnan(ft[np.isin(st, [1, 2, 3])]).all()
    assert not np.isnan(ft[np.isin(st, [0, 4, 5])]).any()
    r = sv().accept_from_logits(H().to_dev(wl.target, wl.dtype), H().to_dev(wl.draft, wl.dtype),
                                H().to_dev(wl.temperature), H().to_dev(wl.tokens), H().to_dev(wl.uniforms),
                                top_p=H().to_dev(top_p))
    torch.cuda.synchronize()
    ref = oracle.accept_from_logits(wl.target, wl.draft, wl.dtype, wl.temperature, wl.tokens, wl.uniforms,
                                    wl.B, wl.K, top_p=top_p)
    n, nxt, s = (x.cpu().numpy() for x in r)
    for b in (1, 2, 3):
        assert s[b] == sv().SEQ_BAD_VALUE and nxt[b] == -1 and n[b] == 0
        assert ref.status[b] == oracle.BAD_VALUE and ref.next_token[b] == -1


def _run_filtered(wl, top_k, top_p, warped=True):
    out = None
    if warped:
        out = (torch.full(wl.target.shape, float("nan"), device=DEV),
               torch.full(wl.draft.shape, float("nan"), device=DEV))
    r = sv().accept_from_logits(H().to_dev(wl.target, wl.dtype), H().to_dev(wl.draft, wl.dtype),
                                H().to_dev(wl.temperature), H().to_dev(wl.tokens), H().to_dev(wl.uniforms),
                                H().to_dev(wl.cu_k), wl.K if wl.cu_k is not None else None, warped_out=out,
                                top_k=None if top_k is None else H().to_dev(top_k),
                                top_p=None if top_p is None else H().to_dev(top_p))
    torch.cuda.synchronize()
    res = oracle.Result(*(x.cpu().numpy() for x in r))
    res.status = res.status.astype(np.uint32)
    if warped:
        return res, (out[0].cpu().numpy(), out[1].cpu().numpy())
    return res


@pytest.mark.parametrize("name,dtype", [("config2", "bf16"), ("config5", "f16"), ("config4", "f32")])
def test_filtered_verification(name, dtype):
    if name == "config2":
        wl = workloads.make_config(name, B=16, K=5, V=9001)
    elif name == "config5":
        wl = workloads.make_config(name, B=32, V=7001)
    else:  # ragged: logits from the probability workload
        wl = workloads.make_config(name, B=12, V=5003)
        wl.target = np.log(np.maximum(wl.target, 1e-30)).astype(F32)
        wl.draft = np.log(np.maximum(wl.draft, 1e-30)).astype(F32)
        wl.temperature = np.full(wl.B, 0.7, F32)
        wl.dtype, wl.mode = "f32", "logits"
    rng = np.random.default_rng(11)
    top_k, top_p = _filters(rng, wl.B, wl.V)
    top_p[top_p < 0.01] = 0.3  # keep every parameter valid here
    res, (wt, wd) = _run_filtered(wl, top_k, top_p)
    ft, fd = _gpu_floors(wl, top_k, top_p)
    _check_floors(wl, top_k, top_p, ft, fd)
    samp = wl.temperature > 0
    # the cut: on every row the kernel warped, weights below the floor are 0
    st, sd = _rows_of(wl)
    dec = lambda r: oracle.decode_rows(r, wl.dtype)
    for arr, w, f, seq in ((wl.target, wt, ft, st), (wl.draft, wd, fd, sd)):
        for r in range(arr.shape[0]):
            if np.isnan(w[r]).all() or not samp[seq[r]]:
                continue
            x = dec(arr[r])
            assert (w[r][x < f[r]] == 0).all(), r
            assert (w[r][x >= f[r]] > 0).any(), r
    # decisions on the kernel's own cut weights: bit-exact
    ref_w = oracle.accept(np.nan_to_num(wt, nan=0.0), np.nan_to_num(wd, nan=0.0), wl.tokens, wl.uniforms,
                          wl.B, wl.K, wl.cu_k)
    assert np.array_equal(res.n_accepted[samp], ref_w.n_accepted[samp])
    near = (ref_w.status & oracle.NEAR_BOUNDARY) > 0
    assert ((res.next_token == ref_w.next_token) | near)[samp].all()
    # and against the oracle's own filtered fp64 softmax
    ref = oracle.accept_from_logits(wl.target, wl.draft, wl.dtype, wl.temperature, wl.tokens, wl.uniforms,
                                    wl.B, wl.K, wl.cu_k, top_k=top_k, top_p=top_p)
    import gpu_helpers
    gpu_helpers.assert_softmax_agreement(res, ref, f"{name} filtered")
    g = wl.temperature == 0  # greedy sequences ignore the filters
    if g.any():
        plain = oracle.accept_from_logits(wl.target, wl.draft, wl.dtype, wl.temperature, wl.tokens,
                                          wl.uniforms, wl.B, wl.K, wl.cu_k)
        assert np.array_equal(res.n_accepted[g], plain.n_accepted[g])
        assert np.array_equal(res.next_token[g], plain.next_token[g])


def test_top_k_one_equals_greedy_verification_on_the_gpu():
    wl = workloads.make_config("config2", B=48, K=5, V=6007)
    rng = np.random.default_rng(12)
    x = oracle.decode_rows(wl.target, "bf16").astype(F32)
    wl.target = (x + rng.normal(0, 1e-3, x.shape)).astype(F32)  # distinct maxima
    wl.draft = (oracle.decode_rows(wl.draft, "bf16") + rng.normal(0, 1e-3, x[:wl.draft.shape[0]].shape)).astype(F32)
    wl.dtype = "f32"
    K1 = wl.K + 1
    for b in range(wl.B):  # about half the drafts are the target's argmax
        for i in range(wl.K):
            if rng.random() < 0.6:
                wl.tokens[b * wl.K + i] = int(np.argmax(wl.target[b * K1 + i]))
    res = _run_filtered(wl, np.ones(wl.B, np.int32), None, warped=False)
    g = sv().verify_greedy(H().to_dev(wl.target), H().to_dev(wl.tokens))
    torch.cuda.synchronize()
    assert np.array_equal(res.n_accepted, g.n_accepted.cpu().numpy())
    assert np.array_equal(res.next_token, g.next_token.cpu().numpy())
    assert (res.n_accepted > 0).any()


def test_filters_at_full_vocabulary():
    """B = 64, K = 5, V = 128256 bf16 at T = 0.8 with top-k 50 / top-p 0.9:
    floors on sampled rows, and decisions on the kernel's cut rows."""
    wl = workloads.make_config("config2")
    rng = np.random.default_rng(13)
    top_k = rng.choice([0, 50, 1000], size=wl.B).astype(np.int32)
    top_p = rng.choice([1.0, 0.9, 0.95], size=wl.B).astype(F32)
    ft, fd = _gpu_floors(wl, top_k, top_p)
    rows = sorted(rng.choice(wl.target.shape[0], size=24, replace=False).tolist())
    _check_floors(wl, top_k, top_p, ft, fd, rows=rows)
    res, (wt, wd) = _run_filtered(wl, top_k, top_p)
    assert (res.status & ~np.uint32(sv().SEQ_EXACT_PATH | sv().SEQ_NEAR_BOUNDARY) == 0).all()
    ref_w = oracle.accept(np.nan_to_num(wt, nan=0.0), np.nan_to_num(wd, nan=0.0), wl.tokens, wl.uniforms,
                          wl.B, wl.K)
    assert np.array_equal(res.n_accepted, ref_w.n_accepted)
