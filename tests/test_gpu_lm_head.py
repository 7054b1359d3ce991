"""The LM head in front of verification (llmstudio.ru sections 21-22): the
tensor-core product against the oracle's fp64 logits, and verification from
hidden states against the oracle run on the logits the kernel wrote (decisions
equal outside the oracle's softmax band, draws outside its boundary band), with
the agreement against the oracle's own fp64 logits reported."""

import numpy as np
import pytest

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():  # pragma: no cover
    pytestmark = pytest.mark.skip("needs a GPU")
else:
    pytestmark = pytest.mark.gpu

import __graft_entry__  # noqa: E402
import oracle  # noqa: E402
from workloads.configs import f32_to_bf16_bits  # noqa: E402
from workloads.lm_head import make_lm_head  # noqa: E402

DEV = torch.device("cuda", 0)
# |logit - exact| <= REL * sum_k |h_k w_k|: fp32 accumulation of d bf16
# products in any order stays far inside 2^-13 of that sum for d <= 2^13
REL = 2.0 ** -13


@pytest.fixture(scope="module", autouse=True)
def built():
    __graft_entry__.build()


def sv():
    import speculative_decoding_verification_decode_gb300 as m
    return m


def H():
    import gpu_helpers
    return gpu_helpers


def bf16_dev(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to(DEV).view(torch.bfloat16)


def as_f64(bits):
    return oracle.decode_rows(bits, "bf16").reshape(bits.shape)


def check_logits(got, h_bits, w_bits, label):
    ref = oracle.lm_head_logits(h_bits, w_bits, "bf16")
    scale = np.abs(as_f64(h_bits)) @ np.abs(as_f64(w_bits)).T
    err = np.abs(got.astype(np.float64) - ref)
    ratio = float((err / np.maximum(scale, 1e-300)).max())
    print(f"{label}: max |logit - exact| / sum|h w| = {ratio:.3e}")
    assert np.isfinite(got).all()
    assert (err <= REL * scale).all(), ratio


@pytest.mark.parametrize("rows,V,d", [(1, 256, 64), (130, 1000, 136), (300, 4097, 512), (257, 2048, 1024),
                                      (704, 8192, 4096)])
def test_logits_against_exact_products(rows, V, d):
    """Ragged M tiles (rows not a multiple of 128), V not a multiple of the
    256-column tile (a partial last tile, stores masked), d not a multiple of
    the 64-element K step (the tensor map's zero fill)."""
    rng = np.random.default_rng(rows * 7 + V + d)
    h = f32_to_bf16_bits(rng.standard_normal((rows, d), dtype=np.float32))
    w = f32_to_bf16_bits(rng.standard_normal((V, d), dtype=np.float32) * np.float32(3.0 / np.sqrt(d)))
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    out = sv().lm_head_logits(bf16_dev(h), bf16_dev(w), err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    check_logits(out.cpu().numpy(), h, w, f"rows={rows} V={V} d={d}")


def test_logits_leave_padding_and_other_rows_alone():
    """Only [rows, V] of the output is written: the padding columns of each
    row and the rows after the last stay as they were."""
    rng = np.random.default_rng(5)
    rows, V, d = 200, 1001, 128
    h = f32_to_bf16_bits(rng.standard_normal((rows, d), dtype=np.float32))
    w = f32_to_bf16_bits(rng.standard_normal((V, d), dtype=np.float32) * np.float32(0.1))
    buf = torch.full((rows + 3, 1004), 7.0, device=DEV)
    sv().lm_head_logits(bf16_dev(h), bf16_dev(w), out=buf[:rows, :V])
    torch.cuda.synchronize()
    b = buf.cpu().numpy()
    assert (b[:rows, V:] == 7.0).all() and (b[rows:] == 7.0).all()
    check_logits(b[:rows, :V], h, w, "padded output")


def _verify(wl, flags=0):
    T = torch.from_numpy(wl.temperature).to(DEV)
    r = sv().lm_head_verify(bf16_dev(wl.h_target), bf16_dev(wl.h_draft), bf16_dev(wl.w), T,
                            torch.from_numpy(wl.tokens).to(DEV), torch.from_numpy(wl.uniforms).to(DEV),
                            flags=flags)
    torch.cuda.synchronize()
    res = oracle.Result(r.n_accepted.cpu().numpy(), r.next_token.cpu().numpy(),
                        r.status.cpu().numpy().astype(np.uint32))
    return res, r.target_logits.cpu().numpy(), r.draft_logits.cpu().numpy()


def _against_own_logits(wl, res, lt, ld, label):
    """Decisions and draws against the oracle run on the kernel's own fp32
    logits; then the agreement with the oracle's fp64 logits."""
    T = wl.temperature
    ref = oracle.accept_from_logits(lt, ld, "f32", T, wl.tokens, wl.uniforms, wl.B, wl.K)
    g = T == 0
    # greedy sequences: the argmax of the written logits, bit-exact
    assert np.array_equal(res.n_accepted[g], ref.n_accepted[g])
    assert np.array_equal(res.next_token[g], ref.next_token[g])
    H().assert_softmax_agreement(res, ref, f"{label} (kernel logits)", mask=~g)
    same_dec = (res.n_accepted == ref.n_accepted) & ~g
    near = (ref.status & np.uint32(oracle.NEAR_BOUNDARY)) > 0
    assert ((res.next_token == ref.next_token) | near | ~same_dec | g).all()
    own = oracle.accept_lm_head(wl.h_target, wl.h_draft, wl.w, "bf16", T, wl.tokens, wl.uniforms, wl.B, wl.K)
    agree = float((own.n_accepted == res.n_accepted).mean())
    print(f"{label}: accepted lengths equal to the oracle on fp64 logits for {agree:.4f} of sequences")
    return ref


@pytest.mark.parametrize("B,K,V,d,T", [(8, 5, 4096, 256, 0.8), (12, 3, 5000, 512, 1.0), (6, 4, 3000, 128, 0.0)])
def test_verify_from_states(B, K, V, d, T):
    wl = make_lm_head(B=B, K=K, V=V, d=d, temperature=T if T > 0 else 1.0)
    if T == 0:
        wl.temperature[:] = 0.0
    res, lt, ld = _verify(wl)
    check_logits(lt, wl.h_target, wl.w, "target logits")
    check_logits(ld, wl.h_draft, wl.w, "draft logits")
    _against_own_logits(wl, res, lt, ld, f"B={B} K={K} V={V} d={d} T={T}")


def test_verify_mixed_temperatures():
    wl = make_lm_head(B=10, K=4, V=2600, d=192)
    wl.temperature[::2] = 0.0
    wl.temperature[1::4] = 1.2
    res, lt, ld = _verify(wl)
    _against_own_logits(wl, res, lt, ld, "mixed temperatures")


def test_verify_full_size():
    """B=64, K=5, V=128256, d=4096 (the benchmark's shape): every decision
    against the oracle on the kernel's logits, and 4096 sampled logits
    against exact dot products."""
    wl = make_lm_head()
    res, lt, ld = _verify(wl)
    rng = np.random.default_rng(0)
    for logits, states in ((lt, wl.h_target), (ld, wl.h_draft)):
        r = rng.integers(0, logits.shape[0], 2048)
        c = rng.integers(0, logits.shape[1], 2048)
        hs, ws = as_f64(states[r]), as_f64(wl.w[c])
        exact = (hs * ws).sum(1)
        scale = (np.abs(hs) * np.abs(ws)).sum(1)
        assert (np.abs(logits[r, c] - exact) <= REL * scale).all()
    _against_own_logits(wl, res, lt, ld, "full size")


def test_whole_sampling_pipeline_from_states():
    """llmstudio.ru section 38's pipeline end to end on the GPU: the LM head's
    logits, penalties (section 39's branch state), then the temperature,
    top-k and top-p (the floors) and the verification; against the oracle
    running the same pipeline on the kernel's logits: penalised rows bit for
    bit, decisions equal outside the oracle's flagged bands."""
    from oracle import penalties as pen
    wl = make_lm_head(B=6, K=4, V=3000, d=256)
    B, K, V = wl.B, wl.K, wl.V
    hist = np.random.default_rng(3).integers(0, V, 60).astype(np.int32)
    off = np.array([0, 10, 20, 30, 40, 50, 60], np.int32)
    rep, fr, pr = (np.full(B, 1.3, np.float32), np.full(B, 0.2, np.float32), np.full(B, 0.5, np.float32))
    top_k = np.array([50, 0, 5, 50, 200, 1], np.int32)
    top_p = np.array([0.9, 0.8, 1.0, 0.95, 0.9, 0.5], np.float32)
    lt = sv().lm_head_logits(bf16_dev(wl.h_target), bf16_dev(wl.w))
    ld = sv().lm_head_logits(bf16_dev(wl.h_draft), bf16_dev(wl.w))
    raw_t, raw_d = lt.cpu().numpy().copy(), ld.cpu().numpy().copy()
    dev = lambda a: torch.from_numpy(a).to(DEV)
    st = sv().apply_penalties(lt, ld, dev(wl.tokens), dev(rep), dev(fr), dev(pr), hist_offsets=dev(off),
                              hist_tokens=dev(hist))
    T = dev(wl.temperature)
    r = sv().accept_from_logits(lt, ld, T, dev(wl.tokens), dev(wl.uniforms), top_k=dev(top_k), top_p=dev(top_p))
    torch.cuda.synchronize()
    assert (st.cpu().numpy() == 0).all()
    pt, pd, _ = pen.penalize_rows(raw_t, raw_d, "f32", off, hist, wl.tokens, B, K, None, rep, fr, pr)
    assert np.array_equal(lt.cpu().numpy(), pt) and np.array_equal(ld.cpu().numpy(), pd)
    ref = oracle.accept_from_logits(pt, pd, "f32", wl.temperature, wl.tokens, wl.uniforms, B, K,
                                    top_k=top_k, top_p=top_p)
    res = oracle.Result(r.n_accepted.cpu().numpy(), r.next_token.cpu().numpy(),
                        r.status.cpu().numpy().astype(np.uint32))
    H().assert_softmax_agreement(res, ref, "states -> penalties -> filters -> verification")
    same = res.n_accepted == ref.n_accepted
    near = (ref.status & np.uint32(oracle.NEAR_BOUNDARY | oracle.NEAR_FILTER | oracle.NEAR_DECISION)) > 0
    assert ((res.next_token == ref.next_token) | near | ~same).all()
