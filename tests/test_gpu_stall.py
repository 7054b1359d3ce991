"""No launch may stall on the producer/consumer hand-over.

When the shared-memory ring holds fewer chunks than one target/draft row
pair, the producer warp can be waiting for a slot whose chunk belongs to a
row the consumers cut short after a rejection.  Such a wait must end as soon
as the cut is visible; before that was so, a launch finished with correct
outputs but only after its bounded wait expired (seconds).  The shapes below
give single-CTA clusters with 3 to 8 chunks per row, so the cut lands on
every chunk position over the repetitions.
"""

import time

import numpy as np
import pytest

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():  # pragma: no cover - CPU-only runs
    pytestmark = pytest.mark.skip("needs a GPU")
else:
    pytestmark = pytest.mark.gpu

import __graft_entry__  # noqa: E402
import workloads  # noqa: E402

REPS = 12
LIMIT_S = 0.25  # a healthy launch of these shapes takes well under a millisecond


@pytest.fixture(scope="module", autouse=True)
def built():
    __graft_entry__.build()


def _timed(fn):
    torch.cuda.synchronize()
    worst = 0.0
    for _ in range(REPS):
        t = time.perf_counter()
        r = fn()
        torch.cuda.synchronize()
        worst = max(worst, time.perf_counter() - t)
    return r, worst


@pytest.mark.parametrize("V", [12000, 16000, 20000, 24000, 28000, 32000])
def test_probs_small_ring_no_stall(V):
    import gpu_helpers as H
    wl = workloads.make_config("config1", rounds=320, K=4, V=V)
    args = [H.to_dev(a) for a in (wl.target, wl.draft, wl.tokens, wl.uniforms)]
    import speculative_decoding_verification_decode_gb300 as sv
    r, worst = _timed(lambda: sv.accept(*args))
    st = r.status.cpu().numpy().astype(np.uint32)
    assert not (st & sv.SEQ_TIMEOUT).any()
    assert worst < LIMIT_S, f"slowest launch {worst * 1e3:.1f} ms"


@pytest.mark.parametrize("V", [16000, 32000])
def test_logits_small_ring_no_stall(V):
    import gpu_helpers as H
    wl = workloads.make_config("config5", B=320, K=3, V=V)
    args = [H.to_dev(wl.target, wl.dtype), H.to_dev(wl.draft, wl.dtype), H.to_dev(wl.temperature),
            H.to_dev(wl.tokens), H.to_dev(wl.uniforms)]
    import speculative_decoding_verification_decode_gb300 as sv
    r, worst = _timed(lambda: sv.accept_from_logits(*args))
    st = r.status.cpu().numpy().astype(np.uint32)
    assert not (st & sv.SEQ_TIMEOUT).any()
    assert worst < LIMIT_S, f"slowest launch {worst * 1e3:.1f} ms"
