"""sv_lm_head_verify_static (the library's fixed scratch, no workspace)
against sv_lm_head_verify with a caller workspace: the same results on two
calls in a row, and calls larger than the scratch refused before any device
work.  Named to be collected last; it needs no state from other tests."""

import numpy as np
import pytest

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():  # pragma: no cover
    pytestmark = pytest.mark.skip("needs a GPU")
else:
    pytestmark = pytest.mark.gpu

import __graft_entry__  # noqa: E402
from workloads.lm_head import make_lm_head  # noqa: E402

DEV = torch.device("cuda", 0)


@pytest.fixture(scope="module", autouse=True)
def built():
    __graft_entry__.build()


def sv():
    import speculative_decoding_verification_decode_gb300 as m
    return m


def _dev(wl):
    bf = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(DEV).view(torch.bfloat16)
    return (bf(wl.h_target), bf(wl.h_draft), bf(wl.w), torch.from_numpy(wl.temperature).to(DEV),
            torch.from_numpy(wl.tokens).to(DEV), torch.from_numpy(wl.uniforms).to(DEV))


def _host(r):
    return tuple(x.cpu().numpy() for x in (r.n_accepted, r.next_token, r.status))


def test_static_scratch_equals_workspace_call_twice_in_a_row():
    a = make_lm_head(seed=11, B=6, K=5, V=20000, d=512)
    b = make_lm_head(seed=12, B=4, K=3, V=30011, d=256)
    b.temperature[::2] = 0.0  # greedy and sampled sequences
    for wl in (a, b, a):
        x = _dev(wl)
        ref = _host(sv().lm_head_verify(*x))
        got = _host(sv().lm_head_verify_static(*x))
        torch.cuda.synchronize()
        for r, g in zip(ref, got):
            assert np.array_equal(r, g)
    # two calls in a row on one stream, no synchronisation between them
    xa, xb = _dev(a), _dev(b)
    ra, rb = sv().lm_head_verify_static(*xa), sv().lm_head_verify_static(*xb)
    ga, gb = _host(ra), _host(rb)
    for r, g in zip(_host(sv().lm_head_verify(*xa)), ga):
        assert np.array_equal(r, g)
    for r, g in zip(_host(sv().lm_head_verify(*xb)), gb):
        assert np.array_equal(r, g)


def test_static_scratch_limit():
    """A call whose workspace would exceed SV_STATIC_SCRATCH_BYTES (64 MiB) is
    refused with SV_ERR_UNSUPPORTED; nothing is enqueued."""
    lib = sv()._lib.load()
    limit = 64 << 20
    assert lib.sv_lm_head_workspace_size(64, 320, 128256) > limit
    assert lib.sv_lm_head_workspace_size(8, 40, 128256) <= limit
    P = 1 << 12
    rc = lib.sv_lm_head_verify_static(P, P, P, 4096, P, P, P, None, 64, 5, 320, 128256, P, P, P, 0, None)
    assert rc == sv()._lib.SV_ERR_UNSUPPORTED
    assert b"static scratch" in lib.sv_last_error()
