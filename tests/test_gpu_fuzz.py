"""Seeded random shapes against the oracle: batch sizes from 1 to 300, K_b
from 0 to 12 (ragged or not), vocabularies from 1 to 70000 (so that cluster
sizes from 1 to 16 and slices down to a few elements come up), every mode
and element type, mixed temperatures, and a sprinkling of special values
(NaN, +-Inf, zero rows, out-of-range tokens).  Each case must match the
oracle under the rules of the other parity tests."""

import numpy as np
import pytest

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():  # pragma: no cover
    pytestmark = pytest.mark.skip("needs a GPU")
else:
    pytestmark = pytest.mark.gpu

import __graft_entry__  # noqa: E402
import oracle  # noqa: E402
from workloads.configs import Workload, f32_to_bf16_bits, uniforms_24bit  # noqa: E402

F32 = np.float32


@pytest.fixture(scope="module", autouse=True)
def built():
    __graft_entry__.build()


def H():
    import gpu_helpers
    return gpu_helpers


def _case(seed):
    rng = np.random.default_rng(seed)
    B = int(rng.choice([1, 2, 3, 7, 16, 33, 64, 100, 300]))
    K = int(rng.integers(0, 13))
    V = int(rng.choice([1, 2, 5, 31, 100, 1000, 3001, 8192, 20011, 70000]))
    if B * (K + 1) * V > 6_000_000:  # keep the oracle quick
        V = max(1, 6_000_000 // (B * (K + 1)))
    ragged = bool(rng.random() < 0.5)
    kb = rng.integers(0, K + 1, B) if ragged else np.full(B, K)
    cu = np.concatenate([[0], np.cumsum(kb)]).astype(np.int32)
    nt, nd = int((kb + 1).sum()), int(kb.sum())
    mode = str(rng.choice(["greedy", "accept", "logits"]))
    dtype = "f32" if mode == "accept" else str(rng.choice(["f32", "bf16", "f16"]))
    x = rng.normal(0, 2.5, (nt, V)).astype(F32)
    y = (np.concatenate([x[cu[b] + b:cu[b] + b + int(kb[b])] for b in range(B)]) if nd else np.zeros((0, V), F32))
    y = (y + rng.normal(0, 1.0, y.shape)).astype(F32)
    if mode == "accept":
        x = np.exp(x - x.max(1, keepdims=True)).astype(F32)
        y = np.exp(y - (y.max(1, keepdims=True) if nd else 0)).astype(F32)
    tok = rng.integers(0, V, nd).astype(np.int32)
    # special values on a few rows
    for _ in range(int(rng.integers(0, 3))):
        r = int(rng.integers(0, nt))
        x[r, int(rng.integers(0, V))] = rng.choice([np.nan, np.inf, -np.inf, 0.0])
    if nd and rng.random() < 0.3:
        tok[int(rng.integers(0, nd))] = V + 3  # a token out of range
    if mode == "accept" and rng.random() < 0.2:
        x[int(rng.integers(0, nt))] = 0.0  # a zero-mass row
    u = uniforms_24bit(rng, nt)
    T = None
    if mode == "logits":
        T = np.where(rng.random(B) < 0.3, 0.0, rng.uniform(0.3, 1.5, B)).astype(F32)
    store = {"f32": lambda a: a, "f16": lambda a: a.astype(np.float16), "bf16": f32_to_bf16_bits}[dtype]
    wl = Workload("fuzz", mode, dtype, B, K, V, store(x), store(y), tok, u,
                  cu if ragged else None, T, {"seed": seed})
    return wl


@pytest.mark.parametrize("seed", list(range(160)))
def test_random_case(seed):
    wl = _case(1000 + seed)
    res = H().run_gpu(wl)
    ref = H().run_oracle(wl)
    if wl.mode == "logits":
        g = wl.temperature == 0
        assert np.array_equal(res.n_accepted[g], ref.n_accepted[g]), seed
        assert np.array_equal(res.next_token[g], ref.next_token[g]), seed
        H().assert_softmax_agreement(res, ref, f"seed {seed}", mask=~g)
        # error bits where both took the same decisions (a sequence decided
        # differently inside the band may reach rows the other never reads)
        errs = np.uint32(oracle.BAD_TOKEN | oracle.BAD_VALUE | oracle.ZERO_MASS | oracle.BAD_LAYOUT)
        same = (res.n_accepted == ref.n_accepted) & ~g
        empty = (ref.status & np.uint32(oracle.NEAR_EMPTY)) > 0
        for sel, bits in ((same & ~empty, errs), (same & empty, errs & ~np.uint32(oracle.ZERO_MASS))):
            assert np.array_equal(res.status[sel] & bits, ref.status[sel] & bits), seed
    else:
        H().compare(res, ref, exact_tokens=wl.mode == "greedy")
