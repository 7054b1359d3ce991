"""Parity at the full benchmark sizes, in the launch configuration bench.py
times (same entry points, same default flags, one launch per round)."""

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


@pytest.fixture(scope="module", autouse=True)
def built():
    __graft_entry__.build()


def H():
    import gpu_helpers
    return gpu_helpers


def test_config2_full_bf16_logits():
    wl = workloads.make_config("config2")  # B=64, K=5, V=128256, T=0.8
    res, warped = H().run_gpu(wl, warped=True)
    # decisions bit-exact against the oracle on the kernel's own warped rows
    wt, wd = warped
    ref = oracle.accept(np.nan_to_num(wt, nan=0.0), np.nan_to_num(wd, nan=0.0), wl.tokens,
                        wl.uniforms, wl.B, wl.K)
    assert np.array_equal(res.n_accepted, ref.n_accepted)
    near = (ref.status & oracle.NEAR_BOUNDARY) > 0
    assert ((res.next_token == ref.next_token) | near).all()
    # and against the oracle's own fp64 softmax: agreement rate
    own = H().run_oracle(wl)
    print(f"config2: {int(near.sum())} flagged draws")
    H().assert_softmax_agreement(res, own, "config2")


def test_config3_full_greedy():
    wl = workloads.make_config("config3")  # B=256, K=4, V=152064
    H().compare(H().run_gpu(wl), H().run_oracle(wl), exact_tokens=True)


def test_greedy2_full_bf16_logits():
    """Greedy at B=64, K=5, V=128256 on bf16 logits (the sampling workload's
    shape): every accepted length and emitted token bit-exact."""
    wl = workloads.make_config("greedy2")
    H().compare(H().run_gpu(wl), H().run_oracle(wl), exact_tokens=True)


def test_config1_rounds_as_single_calls():
    """Config 1 as the benchmark's per-round latency line runs it: one B=1
    call per round (sampled, then greedy on the same rows); each equals the
    oracle on that round alone."""
    wl = workloads.make_config("config1", rounds=40)
    x = [H().to_dev(a) for a in (wl.target, wl.draft, wl.tokens, wl.uniforms)]
    import speculative_decoding_verification_decode_gb300 as sv
    K = wl.K
    n_s, t_s, n_g, t_g = [], [], [], []
    for r in range(wl.B):
        tg, dr = x[0][r * (K + 1):(r + 1) * (K + 1)], x[1][r * K:(r + 1) * K]
        tok, u = x[2][r * K:(r + 1) * K], x[3][r * (K + 1):(r + 1) * (K + 1)]
        a = sv.accept(tg, dr, tok, u)
        g = sv.verify_greedy(tg, tok)
        n_s.append(int(a.n_accepted[0])); t_s.append(int(a.next_token[0]))
        n_g.append(int(g.n_accepted[0])); t_g.append(int(g.next_token[0]))
    ref_s = H().run_oracle(wl, "accept")
    ref_g = H().run_oracle(wl, "greedy")
    assert n_s == ref_s.n_accepted.tolist()
    near = (ref_s.status & oracle.NEAR_BOUNDARY) > 0
    assert ((np.array(t_s) == ref_s.next_token) | near).all()
    assert n_g == ref_g.n_accepted.tolist() and t_g == ref_g.next_token.tolist()


def test_config4_full_ragged():
    wl = workloads.make_config("config4")  # B=32, K_b ~ U{0..8}, V=129280
    near, diff = H().compare(H().run_gpu(wl), H().run_oracle(wl))
    print(f"config4: {near} flagged draws, {diff} differ")


def test_config5_full_mixed():
    wl = workloads.make_config("config5")  # B=1024, K=3, V=32000, f16
    res = H().run_gpu(wl)
    ref = H().run_oracle(wl)
    g = wl.temperature == 0
    assert np.array_equal(res.n_accepted[g], ref.n_accepted[g])
    assert np.array_equal(res.next_token[g], ref.next_token[g])
    H().assert_softmax_agreement(res, ref, "config5 sampled half", mask=~g)
