"""The row-parallel plan (one cluster per row of a sequence, a last-arriver
combine) against the oracle and against the chain plan, on every mode and
element type: decisions and statuses equal to the chain's bit for bit (both
take the exact predicate on the same defined weights; the exact-path and
near-boundary bits depend on each plan's approximate masses), drawn ids
equal outside either plan's boundary band; repeated launches on one stream,
launches on a second stream, forced exact decisions, the give-up path, long
drafts, and the seeded shape fuzz."""

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


def sv():
    import speculative_decoding_verification_decode_gb300 as m
    return m


def H():
    import gpu_helpers
    return gpu_helpers


def plans(wl, mode=None, flags=0, ref=None):
    """Both plans on one workload: the row-parallel result, after checking
    it against the chain's."""
    rows = H().run_gpu(wl, mode, flags=flags | sv().FLAG_PLAN_ROWS)
    chain = H().run_gpu(wl, mode, flags=flags | sv().FLAG_PLAN_CHAIN)
    assert np.array_equal(rows.n_accepted, chain.n_accepted), H()._first_diff(rows.n_accepted, chain.n_accepted)
    mask = np.uint32(~np.uint32(sv().SEQ_EXACT_PATH | sv().SEQ_NEAR_BOUNDARY))
    rs, cs = rows.status & mask, chain.status & mask
    if ref is not None:  # a residual within the fp32 band of zero may come out empty in either plan
        empty = (ref.status & np.uint32(oracle.NEAR_EMPTY)) > 0
        zm = np.uint32(~np.uint32(oracle.ZERO_MASS))
        rs, cs = np.where(empty, rs & zm, rs), np.where(empty, cs & zm, cs)
    assert np.array_equal(rs, cs), H()._first_diff(rs, cs)
    near = ((rows.status | chain.status) & np.uint32(sv().SEQ_NEAR_BOUNDARY)) > 0
    if ref is not None:
        near |= (ref.status & np.uint32(oracle.NEAR_EMPTY)) > 0
    same = rows.next_token == chain.next_token
    assert (same | near).all(), H()._first_diff(np.where(near, chain.next_token, rows.next_token), chain.next_token)
    return rows


@pytest.mark.parametrize("name,kw", [("config2", dict(B=16, K=5, V=20011)),
                                     ("config2", dict(B=64, K=5, V=128256)),
                                     ("config5", dict(B=64, V=32000)),
                                     ("config2", dict(B=8, K=3, V=262144))])
def test_logits(name, kw):
    wl = workloads.make_config(name, **kw)
    ref = H().run_oracle(wl)
    res = plans(wl, ref=ref)
    g = wl.temperature == 0
    assert np.array_equal(res.n_accepted[g], ref.n_accepted[g])
    assert np.array_equal(res.next_token[g], ref.next_token[g])
    H().assert_softmax_agreement(res, ref, f"rows {name} {kw}", mask=~g)


@pytest.mark.parametrize("name,kw,mode", [("config4", dict(B=32, V=30011), "accept"),
                                          ("config1", dict(rounds=64, V=32000), "accept"),
                                          ("config1", dict(rounds=64, V=32000), "greedy"),
                                          ("config3", dict(B=16, K=4, V=20000), "greedy"),
                                          ("greedy2", dict(B=16, K=5, V=128256), "greedy")])
def test_probs_and_greedy(name, kw, mode):
    wl = workloads.make_config(name, **kw)
    ref = H().run_oracle(wl, mode)
    res = plans(wl, mode, ref=ref)
    H().compare(res, ref, exact_tokens=mode == "greedy")


def test_force_exact():
    for name, kw in (("config4", dict(B=16, V=5003)), ("config2", dict(B=8, K=5, V=9001))):
        wl = workloads.make_config(name, **kw)
        res = plans(wl, flags=sv().FLAG_FORCE_EXACT)
        ref = H().run_oracle(wl)
        if wl.mode == "accept":
            H().compare(res, ref)
        else:
            H().assert_softmax_agreement(res, ref, f"rows forced exact {name}")
        decided = (res.status & np.uint32(sv().SEQ_BAD_TOKEN | sv().SEQ_BAD_VALUE)) == 0
        assert ((res.status[decided & (res.n_accepted > 0)] & np.uint32(sv().SEQ_EXACT_PATH)) > 0).all()


def test_repeated_launches_and_a_second_stream():
    """The scratch words are put back by each sequence's last item: the same
    call three times on one stream, then on another stream, gives the same
    outputs each time."""
    wl = workloads.make_config("config2", B=24, K=5, V=30011)
    first = H().run_gpu(wl, flags=sv().FLAG_PLAN_ROWS)
    for _ in range(2):
        again = H().run_gpu(wl, flags=sv().FLAG_PLAN_ROWS)
        assert np.array_equal(first.n_accepted, again.n_accepted)
        assert np.array_equal(first.next_token, again.next_token)
        assert np.array_equal(first.status, again.status)
    side = torch.cuda.Stream()
    with torch.cuda.stream(side):
        other = H().run_gpu(wl, flags=sv().FLAG_PLAN_ROWS)
    torch.cuda.synchronize()
    assert np.array_equal(first.n_accepted, other.n_accepted)
    assert np.array_equal(first.next_token, other.next_token)


def test_give_up_path():
    """Every exchange wait expires at once: each sequence that exchanges
    reports SV_SEQ_TIMEOUT with n = 0 and next = -1, and the launch returns;
    a normal launch right after it is unaffected (the scratch was put back)."""
    wl = workloads.make_config("config2", B=12, K=4, V=20011)
    res = H().run_gpu(wl, flags=sv().FLAG_PLAN_ROWS | sv().FLAG_EXPIRE_EXCHANGE)
    assert (res.status == sv().SEQ_TIMEOUT).all()
    assert (res.n_accepted == 0).all() and (res.next_token == -1).all()
    after = plans(wl)
    ref = H().run_oracle(wl)
    H().assert_softmax_agreement(after, ref, "rows after a give-up")


def test_long_drafts_and_bad_layout():
    wl = workloads.make_config("config1", rounds=12, K=40, V=3001, alpha=0.995)
    for mode in ("accept", "greedy"):
        ref = H().run_oracle(wl, mode)
        H().compare(plans(wl, mode, ref=ref), ref, exact_tokens=mode == "greedy")
    wl = workloads.make_config("config4", B=12, V=4001)
    wl.cu_k = wl.cu_k.copy()
    wl.cu_k[5] = wl.cu_k[6] + 1  # sequence 5 ends before it starts; sequence 4 runs past its K
    ref = H().run_oracle(wl)
    H().compare(plans(wl, ref=ref), ref)


@pytest.mark.parametrize("seed", list(range(0, 160, 4)))
def test_fuzz(seed):
    import test_gpu_fuzz as fz
    wl = fz._case(1000 + seed)
    ref = H().run_oracle(wl)
    res = plans(wl, ref=ref)
    if wl.mode == "logits":
        g = wl.temperature == 0
        assert np.array_equal(res.n_accepted[g], ref.n_accepted[g])
        assert np.array_equal(res.next_token[g], ref.next_token[g])
        H().assert_softmax_agreement(res, ref, f"rows fuzz {seed}", mask=~g)
    else:
        H().compare(res, ref, exact_tokens=wl.mode == "greedy")
