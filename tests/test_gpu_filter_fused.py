"""The one-call filtered verification (`sv_accept_from_logits_filtered`)
with the fused plan requested (SV_FLAG_PLAN_ROWS) against the two-call path
it replaces (`sv_sampler_floors`, then
`sv_accept_from_logits_floored`): the fused top-k plan decides the
sequences its candidate lists hold and hands the rest (top-k outside
[1, 64], top-p alone, a list or kept set over capacity) to the floors and the
floored verification.  Accepted lengths and statuses must equal the two-call
path's bit for bit (the exact-path and near-boundary bits aside), drawn ids
outside either path's boundary band; and the decisions must agree with the
oracle's filtered sampler as the other filter tests require."""

import numpy as np
import pytest

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():  # pragma: no cover
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


def sv():
    import speculative_decoding_verification_decode_gb300 as m
    return m


def H():
    import gpu_helpers
    return gpu_helpers


def _run(wl, top_k, top_p, two_calls, flags=0):
    tg, dr = H().to_dev(wl.target, wl.dtype), H().to_dev(wl.draft, wl.dtype)
    T, tok, u = H().to_dev(wl.temperature), H().to_dev(wl.tokens), H().to_dev(wl.uniforms)
    cu = H().to_dev(wl.cu_k)
    k = wl.K if wl.cu_k is not None else None
    tk = None if top_k is None else torch.from_numpy(top_k).to(DEV)
    tp = None if top_p is None else torch.from_numpy(top_p).to(DEV)
    if two_calls:
        floors = sv().sampler_floors(tg, dr, T, tk, tp, cu, k, int(wl.tokens.size))
        r = sv().accept_from_logits(tg, dr, T, tok, u, cu, k, floors=floors, flags=flags)
    else:  # the one call, with the fused plan requested
        r = sv().accept_from_logits(tg, dr, T, tok, u, cu, k, top_k=tk, top_p=tp,
                                    flags=flags | sv().FLAG_PLAN_ROWS)
    torch.cuda.synchronize()
    return oracle.Result(r.n_accepted.cpu().numpy(), r.next_token.cpu().numpy(),
                         r.status.cpu().numpy().astype(np.uint32))


def _check(wl, top_k, top_p, label, oracle_check=True):
    one = _run(wl, top_k, top_p, False)
    two = _run(wl, top_k, top_p, True)
    assert np.array_equal(one.n_accepted, two.n_accepted), H()._first_diff(one.n_accepted, two.n_accepted)
    mask = np.uint32(~np.uint32(sv().SEQ_EXACT_PATH | sv().SEQ_NEAR_BOUNDARY))
    assert np.array_equal(one.status & mask, two.status & mask), H()._first_diff(one.status & mask,
                                                                                  two.status & mask)
    near = ((one.status | two.status) & np.uint32(sv().SEQ_NEAR_BOUNDARY)) > 0
    assert ((one.next_token == two.next_token) | near).all(), H()._first_diff(one.next_token, two.next_token)
    if oracle_check:
        ref = oracle.accept_from_logits(wl.target, wl.draft, wl.dtype, wl.temperature, wl.tokens, wl.uniforms,
                                        wl.B, wl.K, wl.cu_k, top_k=top_k, top_p=top_p)
        H().assert_softmax_agreement(one, ref, label)
        same = one.n_accepted == ref.n_accepted
        flagged = (ref.status & np.uint32(oracle.NEAR_BOUNDARY | oracle.NEAR_FILTER | oracle.NEAR_DECISION
                                          | oracle.NEAR_EMPTY)) > 0
        assert ((one.next_token == ref.next_token) | flagged | ~same).all()
    return one


@pytest.mark.parametrize("V", [20011, 128256])
def test_config2_rows_top_k_top_p(V):
    wl = workloads.make_config("config2", B=16, K=5, V=V)
    B = wl.B
    _check(wl, np.full(B, 50, np.int32), np.full(B, 0.9, F32), f"fused top-k 50 top-p 0.9 V={V}", V < 100000)
    _check(wl, np.full(B, 50, np.int32), None, f"fused top-k 50 V={V}", V < 100000)


def test_mixed_parameters_and_fallbacks():
    """Per-sequence top-k in and out of the fused range, top-p valid,
    invalid, absent; greedy and invalid temperatures among them."""
    wl = workloads.make_config("config2", B=24, K=4, V=9001)
    B = wl.B
    top_k = np.array([1, 2, 50, 64, 65, 0, -3, 9001, 9002, 7, 50, 64] * 2, np.int32)
    top_p = np.array([0.9, 0.5, 1.0, 0.95, 0.9, 0.8, 0.9, 0.3, 1.5, np.nan, 0.0, -1.0] * 2, F32)
    wl.temperature = wl.temperature.copy()
    wl.temperature[12] = 0.0
    wl.temperature[13] = -1.0
    wl.temperature[14] = np.nan
    wl.temperature[15:18] = [0.5, 1.0, 2.0]
    _check(wl, top_k, top_p, "mixed filters")
    _check(wl, top_k, None, "mixed top-k alone")


def test_ties_special_values_and_f16():
    """Logits tied at the k-th value (a list or kept set over capacity hands
    the row to the fallback), NaN / +Inf / all -Inf rows, f16 rows, ragged
    layouts with bonus-only sequences."""
    rng = np.random.default_rng(11)
    wl = workloads.make_config("config2", B=12, K=3, V=5003)
    tgt = wl.target.copy()
    from workloads.configs import _bf16_bits_to_f32, f32_to_bf16_bits
    vals = _bf16_bits_to_f32(tgt)
    vals[0, rng.choice(5003, 300, replace=False)] = vals[0].max() + 1.0   # 300 ties above the rest
    vals[4, rng.choice(5003, 40, replace=False)] = vals[4].max() + 1.0    # 40 ties: within capacity
    vals[8, 17] = np.nan
    vals[9, 3] = np.inf
    vals[10, :] = -np.inf
    wl.target = f32_to_bf16_bits(vals)
    B = wl.B
    _check(wl, np.full(B, 50, np.int32), np.full(B, 0.9, F32), "ties and special values")
    f16 = workloads.make_config("config5", B=32, V=4001)
    _check(f16, np.full(f16.B, 20, np.int32), np.full(f16.B, 0.8, F32), "f16 mixed")
    rag = workloads.make_config("config2", B=10, K=6, V=3001)
    kb = rng.integers(0, 7, rag.B)
    kb[:3] = 0
    cu = np.concatenate([[0], np.cumsum(kb)]).astype(np.int32)
    t_rows = np.concatenate([np.arange(b * 7, b * 7 + kb[b] + 1) for b in range(rag.B)])
    d_rows = np.concatenate([np.arange(b * 6, b * 6 + kb[b]) for b in range(rag.B)])
    rag.target, rag.draft = rag.target[t_rows], rag.draft[d_rows]
    rag.tokens, rag.uniforms, rag.cu_k = rag.tokens[d_rows], rag.uniforms[t_rows], cu
    _check(rag, np.full(rag.B, 30, np.int32), np.full(rag.B, 0.9, F32), "ragged")


def test_f32_rows_take_the_two_call_path():
    wl = workloads.make_config("config2", B=6, K=3, V=4001)
    from workloads.configs import _bf16_bits_to_f32
    wl.target = _bf16_bits_to_f32(wl.target).astype(F32)
    wl.draft = _bf16_bits_to_f32(wl.draft).astype(F32)
    wl.dtype = "f32"
    _check(wl, np.full(wl.B, 40, np.int32), np.full(wl.B, 0.9, F32), "f32 rows")


def test_repeated_calls_and_force_exact():
    """The scratch is put back by every call (three calls agree), and with
    every accept test forced through the exact masses both paths still agree
    and mark the exact path on every sequence that decided a row."""
    wl = workloads.make_config("config2", B=20, K=5, V=12007)
    B = wl.B
    tk, tp = np.full(B, 50, np.int32), np.full(B, 0.9, F32)
    first = _run(wl, tk, tp, False)
    for _ in range(2):
        again = _run(wl, tk, tp, False)
        assert np.array_equal(first.n_accepted, again.n_accepted)
        assert np.array_equal(first.next_token, again.next_token)
        assert np.array_equal(first.status, again.status)
    one = _run(wl, tk, tp, False, sv().FLAG_FORCE_EXACT)
    two = _run(wl, tk, tp, True, sv().FLAG_FORCE_EXACT)
    assert np.array_equal(one.n_accepted, two.n_accepted)
    assert np.array_equal(one.n_accepted, first.n_accepted)
    ok = (one.status & np.uint32(sv().SEQ_BAD_TOKEN | sv().SEQ_BAD_VALUE | sv().SEQ_ZERO_MASS)) == 0
    assert ((one.status[ok] & np.uint32(sv().SEQ_EXACT_PATH)) > 0).all()


@pytest.mark.parametrize("V", [200, 257])
def test_small_vocab_takes_the_two_steps(V):
    """Vocabularies too short for the fused plan (rank 0's receive area, the
    gathered lists and its work space, must fit where its two slices were:
    about 3700 16-bit logits per row): the one call falls back to the two
    steps and must match them; top-k up to 64 and 1, top-p on and off."""
    wl = workloads.make_config("config2", B=12, K=3, V=V)
    top_k = np.array([64, 1, 2, 50, 63, 10] * 2, np.int32)
    top_p = np.array([0.5, 1.0, 0.9, 0.95, 0.3, 1.0] * 2, F32)
    _check(wl, top_k, top_p, f"small vocab {V}")
    _check(wl, top_k, None, f"small vocab {V}, top-k alone")


def test_f16_full_vocab_and_ties_across_slices():
    """Eight slices per row: f16 rows, and bf16 rows whose largest logits are
    tied across every slice (600 ties: a top-k set over 64 and a kept set over
    256, handed to the general path; 2100 ties: a slice's list over its
    capacity) beside ordinary rows."""
    f16 = workloads.make_config("config5", B=8, K=3, V=128256)
    _check(f16, np.full(f16.B, 50, np.int32), np.full(f16.B, 0.9, F32), "f16 V=128256", False)
    rng = np.random.default_rng(23)
    wl = workloads.make_config("config2", B=4, K=3, V=128256)
    from workloads.configs import _bf16_bits_to_f32, f32_to_bf16_bits
    vals = _bf16_bits_to_f32(wl.target.copy())
    vals[0, rng.choice(128256, 600, replace=False)] = vals[0].max() + 1.0
    vals[4, rng.choice(128256, 2100, replace=False)] = vals[4].max() + 1.0
    wl.target = f32_to_bf16_bits(vals)
    B = wl.B
    _check(wl, np.full(B, 50, np.int32), np.full(B, 0.9, F32), "ties across slices", False)
    _check(wl, np.full(B, 50, np.int32), None, "ties across slices, top-k alone", False)
