"""Edge cases of the verification kernel against the oracle: drafts longer
than the rows whose decision inputs are prefetched at start (K = 40 > 32),
a 262144-token vocabulary, a draft identical to the target (every draft
accepted, then the bonus), a batch of bonus-only sequences, a large batch over
a tiny vocabulary, and an empty batch."""

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


def sv():
    import speculative_decoding_verification_decode_gb300 as m
    return m


def test_long_drafts_past_the_prefetched_rows():
    """K = 40 with a near-perfect draft: most sequences reach rows past the
    32 whose token, uniform and probabilities the kernel prefetches."""
    wl = workloads.make_config("config1", rounds=12, K=40, V=3001, alpha=0.995)
    for mode in ("accept", "greedy"):
        res = H().run_gpu(wl, mode)
        ref = H().run_oracle(wl, mode)
        H().compare(res, ref, exact_tokens=mode == "greedy")
    assert (H().run_oracle(wl, "accept").n_accepted > 32).sum() >= 3


def test_vocabulary_of_262144():
    wl = workloads.make_config("config2", B=4, K=3, V=262144)
    res, warped = H().run_gpu(wl, warped=True)
    wt, wd = warped
    ref = oracle.accept(np.nan_to_num(wt, nan=0.0), np.nan_to_num(wd, nan=0.0), wl.tokens, wl.uniforms,
                        wl.B, wl.K)
    assert np.array_equal(res.n_accepted, ref.n_accepted)
    near = (ref.status & oracle.NEAR_BOUNDARY) > 0
    assert ((res.next_token == ref.next_token) | near).all()
    H().assert_softmax_agreement(res, H().run_oracle(wl), "V=262144")
    g = workloads.make_config("greedy2", B=4, K=3, V=262144)
    H().compare(H().run_gpu(g), H().run_oracle(g), exact_tokens=True)


def test_identical_draft_accepts_every_token():
    """q = p on every row: u q(t) Zp < p(t) Zq holds for every u < 1, so every
    draft is accepted and the bonus comes from p_K."""
    wl = workloads.make_config("config4", B=16, V=5003)
    t0 = np.concatenate([[0], np.cumsum(wl.k_per_seq + 1)])[:-1]
    for b in range(wl.B):
        k = int(wl.k_per_seq[b])
        d0 = int(wl.cu_k[b])
        wl.draft[d0:d0 + k] = wl.target[t0[b]:t0[b] + k]
    res = H().run_gpu(wl)
    ref = H().run_oracle(wl)
    H().compare(res, ref)
    assert np.array_equal(res.n_accepted, wl.k_per_seq.astype(np.int32))


def test_bonus_only_batch():
    """Every K_b = 0: one target row per sequence, the bonus drawn from it."""
    wl = workloads.make_config("config4", B=20, V=4099)
    B = wl.B
    t0 = np.concatenate([[0], np.cumsum(wl.k_per_seq + 1)])[:-1]
    wl.target = np.ascontiguousarray(wl.target[t0])
    wl.uniforms = np.ascontiguousarray(wl.uniforms[t0])
    wl.draft = np.zeros((0, wl.V), np.float32)
    wl.tokens = np.zeros(0, np.int32)
    wl.cu_k = np.zeros(B + 1, np.int32)
    res = H().run_gpu(wl)
    ref = H().run_oracle(wl)
    H().compare(res, ref)
    assert (res.n_accepted == 0).all() and (res.next_token >= 0).all()


def test_large_batch_tiny_vocabulary():
    wl = workloads.make_config("config1", rounds=4096, K=2, V=64)
    for mode in ("accept", "greedy"):
        H().compare(H().run_gpu(wl, mode), H().run_oracle(wl, mode), exact_tokens=mode == "greedy")


def test_empty_batch():
    dev = torch.device("cuda", 0)
    r = sv().accept(torch.zeros(0, 10, device=dev), torch.zeros(0, 10, device=dev),
                    torch.zeros(0, dtype=torch.int32, device=dev), torch.zeros(0, device=dev))
    assert r.n_accepted.numel() == 0
    g = sv().verify_greedy(torch.zeros(0, 10, device=dev), torch.zeros(0, dtype=torch.int32, device=dev))
    assert g.next_token.numel() == 0
