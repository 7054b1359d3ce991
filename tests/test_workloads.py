"""Synthetic inputs: determinism, layout and the distribution facts the
configurations promise (they carry none of the verification arithmetic)."""

import numpy as np

import workloads as w


def test_deterministic_and_shaped():
    a = w.make_config("config4", B=6, V=257)
    b = w.make_config("config4", B=6, V=257)
    assert np.array_equal(a.target, b.target) and np.array_equal(a.cu_k, b.cu_k)
    kb = a.k_per_seq
    assert a.target.shape == (int((kb + 1).sum()), 257)
    assert a.draft.shape == (int(kb.sum()), 257)
    assert a.tokens.shape == (int(kb.sum()),) and a.uniforms.shape == (int((kb + 1).sum()),)
    assert kb.min() >= 0 and kb.max() <= 8 and a.cu_k[0] == 0


def test_config1_overlap_near_068():
    wl = w.make_config("config1", rounds=20, V=4000)
    ph = wl.target[: 5].astype(np.float64)
    alphas = []
    for b in range(20):
        for i in range(4):
            p = wl.target[b * 5 + i].astype(np.float64)
            q = wl.draft[b * 4 + i].astype(np.float64)
            alphas.append(np.minimum(p / p.sum(), q / q.sum()).sum())
    assert abs(np.mean(alphas) - 0.68) < 0.03


def test_config3_ties_and_match_rate():
    wl = w.make_config("config3", B=64, V=3001)
    for r in wl.meta["tie_rows"]:
        row = wl.target[r]
        assert (row == row.max()).sum() >= 2
    assert len(wl.meta["tie_rows"]) == (64 * 5 + 63) // 64


def test_config5_mixed_temperatures_and_uniform_grid():
    wl = w.make_config("config5", B=16, V=300)
    assert (wl.temperature[0::2] == 0).all()
    assert ((wl.temperature[1::2] >= 0.5) & (wl.temperature[1::2] <= 1.2)).all()
    u = wl.uniforms.astype(np.float64)
    assert (u >= 0).all() and (u < 1).all() and np.array_equal(u * 2 ** 24, np.floor(u * 2 ** 24))


def test_bf16_rounding():
    x = np.array([1.0, 1.00390625, 1.01171875, -2.5, 3.0e38], np.float32)
    bits = w.f32_to_bf16_bits(x)
    assert list(bits[:4]) == [0x3F80, 0x3F80, 0x3F82, 0xC020]


def test_lm_head_workload_shapes_and_determinism():
    import workloads as W
    a = W.make_lm_head(B=3, K=2, V=50, d=16)
    b = W.make_lm_head(B=3, K=2, V=50, d=16)
    assert a.h_target.shape == (9, 16) and a.h_draft.shape == (6, 16) and a.w.shape == (50, 16)
    assert a.h_target.dtype == np.uint16 and a.w.dtype == np.uint16
    assert ((a.tokens >= 0) & (a.tokens < 50)).all() and a.uniforms.shape == (9,)
    for x, y in ((a.h_target, b.h_target), (a.w, b.w), (a.tokens, b.tokens), (a.uniforms, b.uniforms)):
        assert np.array_equal(x, y)
    # logits of the projection have about the requested spread
    h = (a.h_target.astype(np.uint32) << 16).view(np.float32)
    w = (a.w.astype(np.uint32) << 16).view(np.float32)
    assert 1.5 < float((h @ w.T).std()) < 5.0
