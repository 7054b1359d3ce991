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
