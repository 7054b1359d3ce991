"""The give-up path of the bounded cluster waits.  With the testing flag
FLAG_EXPIRE_EXCHANGE every wait for the records of the sequence's cluster
gives up at once, as a wait on a stalled peer would after its poll limit: each
sequence must end with SEQ_TIMEOUT, n = 0 and next_token = -1, the launch must
return normally (the CTAs still drain their own copies and meet before they
exit), and the next ordinary call on the same inputs must equal the oracle."""

import time

import numpy as np
import pytest

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():  # pragma: no cover
    pytestmark = pytest.mark.skip("needs a GPU")
else:
    pytestmark = pytest.mark.gpu

import __graft_entry__  # noqa: E402
import workloads  # noqa: E402


@pytest.fixture(scope="module", autouse=True)
def built():
    __graft_entry__.build()


def H():
    import gpu_helpers
    return gpu_helpers


CASES = [
    ("config1", dict(rounds=6, V=4001), "accept"),
    ("config1", dict(rounds=6, V=4001), "greedy"),
    ("config2", dict(B=5, K=5, V=9001), None),
    ("config4", dict(B=6, V=20011), None),  # ragged, K_b = 0 bonus-only sequences among them
    ("config5", dict(B=8, V=3001), None),  # greedy and sampled sequences in one launch
]


@pytest.mark.parametrize("name,kw,mode", CASES, ids=[f"{c[0]}-{c[2] or 'own'}" for c in CASES])
def test_expired_exchange_reports_timeout(name, kw, mode):
    import speculative_decoding_verification_decode_gb300 as sv
    wl = workloads.make_config(name, **kw)
    t = time.perf_counter()
    res = H().run_gpu(wl, mode, flags=sv.FLAG_EXPIRE_EXCHANGE)  # synchronises
    elapsed = time.perf_counter() - t
    assert (res.status & sv.SEQ_TIMEOUT).all(), res.status
    assert (res.next_token == -1).all()
    assert (res.n_accepted == 0).all()
    assert elapsed < 10.0  # no wait ran to its full limit
    # the context is intact: an ordinary call equals the oracle
    ok = H().run_gpu(wl, mode)
    ref = H().run_oracle(wl, mode)
    if wl.mode == "logits":
        g = wl.temperature == 0
        assert np.array_equal(ok.n_accepted[g], ref.n_accepted[g])
        H().assert_softmax_agreement(ok, ref, name, mask=~g)
    else:
        H().compare(ok, ref, exact_tokens=(mode or wl.mode) == "greedy")
