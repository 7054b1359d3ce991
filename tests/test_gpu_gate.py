"""Draft-length gate on the GPU vs the oracle (PocketLLM dspark.md, the gate).

The oracle takes the length decision in exact rational arithmetic; the
kernel takes it in fp32.  Lengths must be identical on every sequence the
oracle does not flag as a near-tie (two compared ratios within the fp32
evaluation's error bound), and cu_k must be the prefix sum of the kernel's
lengths (equal to the oracle's when no flagged length differs).  The updated
calibration counts are bit-identical: integers tallied before the one fp64
decay-and-add.
"""

import numpy as np
import pytest

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():  # pragma: no cover - CPU-only runs
    pytestmark = pytest.mark.skip("needs a GPU")
else:
    pytestmark = pytest.mark.gpu

import __graft_entry__  # noqa: E402
import oracle  # noqa: E402
from oracle import GateParams  # noqa: E402

DEV = torch.device("cuda", 0)
EDGES = np.array([-0.5, 0.5, 1.5, 3.0, 6.0], dtype=np.float32)


@pytest.fixture(scope="module", autouse=True)
def built():
    __graft_entry__.build()


def sv():
    import speculative_decoding_verification_decode_gb300 as m
    return m


def _inputs(rng, B, K, cold=False, specials=True):
    conf = rng.normal(1.5, 3.0, size=(B, K)).astype(np.float32)
    if specials and B * K:
        flat = conf.reshape(-1)
        idx = rng.choice(flat.size, size=max(1, flat.size // 50), replace=False)
        flat[idx] = rng.choice([np.nan, np.inf, -np.inf, -0.5, 0.5, 6.0], size=idx.size)
    nb = EDGES.size + 1
    if cold:
        hits, total = np.zeros(nb), np.zeros(nb)
    else:
        total = rng.uniform(0, 40, size=nb).round(3)
        total[rng.integers(0, nb)] = 0.0
        hits = (total * rng.uniform(0, 1, size=nb)).round(3)
    return conf, hits, total


def _params(rng):
    return GateParams(margin=float(rng.choice([1.0, 1.15, 1.5])), min_draft=int(rng.integers(0, 4)),
                      margin_threshold=float(rng.choice([0.0, 4.0])),
                      verify_slope_ms=float(rng.choice([109.0, 40.0, 0.0])))


def _gpu_gate(conf, hits, total, prm, k_drafted=None, logit_margin=None):
    g = sv().gate_draft_lengths(torch.from_numpy(conf).to(DEV), torch.from_numpy(EDGES).to(DEV),
                                torch.from_numpy(hits).to(DEV), torch.from_numpy(total).to(DEV),
                                None if k_drafted is None else torch.from_numpy(k_drafted).to(DEV),
                                None if logit_margin is None else torch.from_numpy(logit_margin).to(DEV),
                                margin=prm.margin, draft_ms=prm.draft_ms, verify_base_ms=prm.verify_base_ms,
                                verify_slope_ms=prm.verify_slope_ms, plain_ms=prm.plain_ms,
                                margin_threshold=prm.margin_threshold, min_draft=prm.min_draft)
    torch.cuda.synchronize()
    return g.n_submit.cpu().numpy(), g.cu_k.cpu().numpy()


NEAR_SEEN = {"flagged": 0, "differ": 0}


def _check_lengths(n_g, cu_g, n_o, cu_o, near, prm=None):
    """Equal lengths outside the oracle's near-ties; cu_k the kernel's own
    prefix sum (the oracle's when every length agrees)."""
    differ = n_g != n_o
    assert not (differ & ~near).any(), (np.flatnonzero(differ & ~near)[:5], prm)
    want_cu = np.zeros(n_g.size + 1, dtype=np.int64)
    want_cu[1:] = np.cumsum(n_g)
    assert np.array_equal(cu_g, want_cu)
    if not differ.any():
        assert np.array_equal(cu_g, cu_o)
    NEAR_SEEN["flagged"] += int(near.sum())
    NEAR_SEEN["differ"] += int(differ.sum())


@pytest.mark.parametrize("B,K", [(0, 5), (1, 0), (1, 5), (7, 5), (64, 5), (300, 16), (1025, 8), (40, 64)])
def test_gate_lengths_match_outside_near_ties(B, K):
    rng = np.random.default_rng(1000 + B * 7 + K)
    for trial in range(3):
        conf, hits, total = _inputs(rng, B, K, cold=(trial == 0))
        prm = _params(rng)
        kd = rng.integers(0, K + 1, size=B).astype(np.int32) if trial == 2 else None
        lm = rng.uniform(0, 8, size=B).astype(np.float32) if prm.margin_threshold > 0 else None
        n_g, cu_g = _gpu_gate(conf, hits, total, prm, kd, lm)
        _check_lengths(n_g, cu_g, *oracle.gate_batch(conf, kd, lm, EDGES, hits, total, prm, with_near=True),
                       prm)


def test_gate_page_defaults():
    # the page's setting: six buckets, defaults; confident drafts keep the
    # block, hopeless ones skip the verify
    nb = EDGES.size + 1
    total = np.full(nb, 20.0)
    hits = np.array([4.0, 13.0, 15.8, 17.8, 20.0, 20.0])  # 20 % .. 100 %, the page's table
    conf = np.array([[7.0] * 5, [-1.0] * 5, [2.0, 1.0, 0.0, -1.0, -1.0]], dtype=np.float32)
    n_g, cu_g = _gpu_gate(conf, hits, total, GateParams())
    n_o, cu_o, near = oracle.gate_batch(conf, None, None, EDGES, hits, total, GateParams(), with_near=True)
    assert not near.any()
    assert np.array_equal(n_g, n_o) and np.array_equal(cu_g, cu_o)
    assert n_g[0] == 5 and n_g[1] == 0


def test_gate_near_ties_reported():
    """How many sequences the oracle flagged as near-ties over the length
    tests, and how many of them the kernel decided the other way (printed)."""
    print(f"gate near-ties: {NEAR_SEEN['flagged']} flagged, {NEAR_SEEN['differ']} decided differently")
    assert NEAR_SEEN["differ"] <= NEAR_SEEN["flagged"]


def test_gate_update_bit_exact_over_rounds():
    rng = np.random.default_rng(5)
    nb = EDGES.size + 1
    hits_o, total_o = np.zeros(nb), np.zeros(nb)
    hits_g = torch.zeros(nb, dtype=torch.float64, device=DEV)
    total_g = torch.zeros(nb, dtype=torch.float64, device=DEV)
    for rnd in range(12):
        B, K = int(rng.integers(0, 300)), 5
        conf, _, _ = _inputs(rng, B, K)
        ns = rng.integers(0, K + 1, size=B).astype(np.int32)
        na = (ns * rng.uniform(0, 1, size=B)).astype(np.int32)
        decay = float(rng.choice([0.9, 1.0, 0.5]))
        hits_o, total_o = oracle.update_table(conf, ns, na, EDGES, hits_o, total_o, decay)
        sv().gate_update(torch.from_numpy(conf).to(DEV), torch.from_numpy(ns).to(DEV),
                         torch.from_numpy(na).to(DEV), torch.from_numpy(EDGES).to(DEV), hits_g, total_g, decay)
        torch.cuda.synchronize()
        assert np.array_equal(hits_g.cpu().numpy(), hits_o), rnd
        assert np.array_equal(total_g.cpu().numpy(), total_o), rnd


def test_gate_then_ragged_verify():
    """The gate's cu_k drives a ragged verification launch."""
    import gpu_helpers as H
    import workloads
    rng = np.random.default_rng(9)
    B, K, V = 24, 6, 3000
    conf, hits, total = _inputs(rng, B, K, specials=False)
    n, cu = _gpu_gate(conf, hits, total, GateParams(margin=1.0))
    wl = workloads.make_config("config4", B=B, K=K, V=V)
    # keep the first n_b drafts (and rows 0..n_b) of each sequence
    kb = wl.k_per_seq
    t_rows, d_rows, toks, us = [], [], [], []
    for b in range(B):
        nb_ = int(min(n[b], kb[b]))
        t0, d0 = int(wl.cu_k[b]) + b, int(wl.cu_k[b])
        t_rows.append(wl.target[t0:t0 + nb_ + 1]); d_rows.append(wl.draft[d0:d0 + nb_])
        toks.append(wl.tokens[d0:d0 + nb_]); us.append(wl.uniforms[t0:t0 + nb_ + 1])
    cu_k = np.zeros(B + 1, dtype=np.int32)
    cu_k[1:] = np.cumsum([len(t) for t in toks])
    target, draft = np.concatenate(t_rows), np.concatenate(d_rows) if cu_k[-1] else np.zeros((0, V), np.float32)
    tokens, uni = np.concatenate(toks).astype(np.int32), np.concatenate(us).astype(np.float32)
    from workloads.configs import Workload
    w2 = Workload("gated", "accept", "f32", B, int(max(1, (cu_k[1:] - cu_k[:-1]).max())), V, target, draft, tokens,
                  uni, cu_k, None, {})
    H.compare(H.run_gpu(w2), H.run_oracle(w2))
