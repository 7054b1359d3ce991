"""The C ABI library loads without a GPU, exports every symbol include/sv.h
declares, and rejects bad arguments on the host before touching CUDA."""

import ctypes

import pytest

import __graft_entry__
from speculative_decoding_verification_decode_gb300 import _lib


@pytest.fixture(scope="module")
def lib():
    __graft_entry__.build()
    return _lib.load()


def test_exports_every_declared_symbol(lib):
    declared = _lib.header_symbols()
    assert set(declared) == set(_lib.SIGNATURES), declared
    for name in declared:
        assert hasattr(lib, name), name


def test_status_strings_and_version(lib):
    for code in range(4):
        assert lib.sv_status_string(code).startswith(b"SV_")
    assert lib.sv_status_string(99) == b"unknown sv_status"
    assert lib.sv_version() >= 100


NULL = None


def greedy(lib, **kw):
    args = dict(target=1 << 12, dtype=0, stride=16, tok=1 << 12, cu=NULL, B=2, K=3, sum_k=6, V=16,
                n=1 << 12, nxt=1 << 12, st=1 << 12, flags=0, stream=NULL)
    args.update(kw)
    return lib.sv_verify_greedy(*args.values())


@pytest.mark.parametrize("kw,frag", [
    (dict(B=-1), b"batch"),
    (dict(K=-2), b"k must"),
    (dict(V=0), b"vocab"),
    (dict(stride=8), b"row_stride"),
    (dict(sum_k=5), b"sum_k must equal"),
    (dict(flags=16), b"flag"),
    (dict(target=NULL), b"target"),
    (dict(tok=NULL), b"draft_tokens"),
    (dict(n=NULL), b"output"),
    (dict(dtype=7), b"dtype"),
])
def test_greedy_argument_errors(lib, kw, frag):
    assert greedy(lib, **kw) == _lib.SV_ERR_ARG
    assert frag in lib.sv_last_error()


def test_empty_batch_is_a_noop(lib):
    assert greedy(lib, B=0, sum_k=0, target=NULL, tok=NULL, n=NULL, nxt=NULL, st=NULL) == _lib.SV_OK
    # both testing flags pass the host checks
    for f in (_lib.FLAG_FORCE_EXACT, _lib.FLAG_EXPIRE_EXCHANGE, _lib.FLAG_FORCE_EXACT | _lib.FLAG_EXPIRE_EXCHANGE,
              _lib.FLAG_PLAN_ROWS, _lib.FLAG_PLAN_CHAIN, _lib.FLAG_PLAN_ROWS | _lib.FLAG_PLAN_CHAIN):
        assert greedy(lib, B=0, sum_k=0, target=NULL, tok=NULL, n=NULL, nxt=NULL, st=NULL, flags=f) == _lib.SV_OK


def test_workspace_size_is_zero(lib):
    """The verification calls need no scratch in global memory (partials stay
    in the cluster's distributed shared memory): the query answers 0 for the
    benchmark shapes of every mode, and for degenerate ones."""
    for mode in (_lib.SV_MODE_GREEDY, _lib.SV_MODE_PROBS, _lib.SV_MODE_LOGITS):
        for B, K, V in ((64, 5, 128256), (256, 4, 152064), (1, 4, 32000), (0, 0, 1), (1024, 16, 262144)):
            assert lib.sv_workspace_size(B, K, V, mode) == 0


def test_accept_argument_errors(lib):
    rc = lib.sv_accept(1 << 12, NULL, 16, 1 << 12, 1 << 12, NULL, 2, 3, 6, 16,
                       1 << 12, 1 << 12, 1 << 12, 0, NULL)
    assert rc == _lib.SV_ERR_ARG and b"draft_probs" in lib.sv_last_error()
    rc = lib.sv_accept(1 << 12, 1 << 12, 16, 1 << 12, NULL, NULL, 2, 3, 6, 16,
                       1 << 12, 1 << 12, 1 << 12, 0, NULL)
    assert rc == _lib.SV_ERR_ARG and b"uniforms" in lib.sv_last_error()


def test_logits_argument_errors(lib):
    rc = lib.sv_accept_from_logits(1 << 12, 1 << 12, 1, 16, NULL, 1 << 12, 1 << 12, NULL, 2, 3, 6,
                                   16, 1 << 12, 1 << 12, 1 << 12, NULL, NULL, 0, NULL)
    assert rc == _lib.SV_ERR_ARG and b"temperature" in lib.sv_last_error()


def test_binding_fails_loudly_without_library(monkeypatch, tmp_path):
    monkeypatch.setattr(_lib, "_lib", None)
    monkeypatch.setattr(_lib, "LIB_PATH", str(tmp_path / "missing.so"))
    with pytest.raises(ImportError):
        _lib.load()


# ---------------------------------------------------------------- draft-length gate (host checks)

def gate(lib, params=True, **kw):
    prm = _lib.GateParams(1.15, 196.0, 300.0, 109.0, 303.0, 0.0, 0)
    for k in ("margin", "plain_ms", "min_draft", "verify_slope_ms"):
        if k in kw:
            setattr(prm, k, kw.pop(k))
    args = dict(conf=1 << 12, kd=NULL, lm=NULL, edges=1 << 12, hits=1 << 12, total=1 << 12, nb=6, B=4, K=5,
                prm=ctypes.byref(prm) if params else NULL, n=1 << 12, cu=1 << 12, stream=NULL)
    args.update(kw)
    return lib.sv_gate_draft_lengths(*args.values())


@pytest.mark.parametrize("kw,frag", [
    (dict(B=-1), b"batch"),
    (dict(K=65), b"k must"),
    (dict(nb=0), b"n_buckets"),
    (dict(nb=33), b"n_buckets"),
    (dict(conf=NULL), b"confidence"),
    (dict(edges=NULL), b"edges"),
    (dict(hits=NULL), b"hits"),
    (dict(cu=NULL), b"output"),
    (dict(plain_ms=0.0), b"gate params"),
    (dict(margin=-1.0), b"gate params"),
    (dict(min_draft=-1), b"gate params"),
    (dict(verify_slope_ms=float("nan")), b"gate params"),
])
def test_gate_argument_errors(lib, kw, frag):
    assert gate(lib, **kw) == _lib.SV_ERR_ARG
    assert frag in lib.sv_last_error()


def test_gate_params_pointer_required(lib):
    assert gate(lib, params=False) == _lib.SV_ERR_ARG
    assert b"params" in lib.sv_last_error()


@pytest.mark.parametrize("kw,frag", [
    (dict(decay=1.5), b"decay"),
    (dict(decay=float("nan")), b"decay"),
    (dict(ns=NULL), b"length"),
    (dict(K=-1), b"k must"),
])
def test_gate_update_argument_errors(lib, kw, frag):
    args = dict(conf=1 << 12, ns=1 << 12, na=1 << 12, edges=1 << 12, hits=1 << 12, total=1 << 12, nb=6, B=4,
                K=5, decay=0.9, stream=NULL)
    args.update(kw)
    assert lib.sv_gate_update(*args.values()) == _lib.SV_ERR_ARG
    assert frag in lib.sv_last_error()


# ---------------------------------------------------------------- sampler filters (host checks)

def floors(lib, **kw):
    args = dict(target=1 << 12, draft=1 << 12, dtype=1, stride=16, temp=1 << 12, top_k=1 << 12,
                top_p=1 << 12, cu=NULL, B=2, K=3, sum_k=6, V=16, ft=1 << 12, fd=1 << 12, stream=NULL)
    args.update(kw)
    return lib.sv_sampler_floors(*args.values())


@pytest.mark.parametrize("kw,frag", [
    (dict(B=-1), b"batch"),
    (dict(K=-1), b"k must"),
    (dict(V=0), b"vocab"),
    (dict(stride=8), b"row_stride"),
    (dict(sum_k=5), b"sum_k"),
    (dict(dtype=7), b"dtype"),
    (dict(target=NULL), b"target"),
    (dict(temp=NULL), b"temperature"),
    (dict(draft=NULL), b"draft_logits"),
])
def test_floors_argument_errors(lib, kw, frag):
    assert floors(lib, **kw) == _lib.SV_ERR_ARG
    assert frag in lib.sv_last_error()


def test_floors_without_filters_or_rows_launch_nothing(lib):
    # no CUDA call happens on these paths, so they run without a GPU
    assert floors(lib, top_k=NULL, top_p=NULL) == _lib.SV_OK
    assert floors(lib, B=0, sum_k=0) == _lib.SV_OK
    assert floors(lib, ft=NULL, fd=NULL) == _lib.SV_OK


def test_floored_logits_argument_errors(lib):
    args = [1 << 12, 1 << 12, 9, 16, 1 << 12, 1 << 12, 1 << 12, NULL, 2, 3, 6, 16, NULL, NULL,
            1 << 12, 1 << 12, 1 << 12, NULL, NULL, 0, NULL]
    assert lib.sv_accept_from_logits_floored(*args) == _lib.SV_ERR_ARG
    assert b"dtype" in lib.sv_last_error()


def test_floors_binding_checks_row_counts_before_any_device_work():
    import torch
    from speculative_decoding_verification_decode_gb300 import sampler_floors
    T = torch.full((4,), 0.8)
    with pytest.raises(ValueError, match="B\\*\\(K\\+1\\)"):
        sampler_floors(torch.zeros(4 * 3 + 1, 8), torch.zeros(8, 8), T, torch.ones(4, dtype=torch.int32))
    with pytest.raises(ValueError, match="B\\*\\(K\\+1\\)"):
        sampler_floors(torch.zeros(12, 8), torch.zeros(7, 8), T, torch.ones(4, dtype=torch.int32))
    with pytest.raises(ValueError, match="cu_k needs"):
        sampler_floors(torch.zeros(5, 8), torch.zeros(2, 8), T, None, torch.full((4,), 0.9),
                       torch.tensor([0, 1, 2, 3, 4], dtype=torch.int32), k=1, sum_k=4)


def test_lm_head_host_checks(lib):
    """Host-side argument checks of the LM head (nothing is launched)."""
    P = 1 << 12
    assert lib.sv_lm_head_logits(P, P, 4, 100, 12, P, 100, NULL, NULL) == _lib.SV_ERR_ARG  # dim % 8
    assert b"dim" in lib.sv_last_error()
    assert lib.sv_lm_head_logits(P, P, 4, 100, 64, P, 98, NULL, NULL) == _lib.SV_ERR_ARG  # ld < vocab
    assert lib.sv_lm_head_logits(P, P, 4, 100, 64, P, 102, NULL, NULL) == _lib.SV_ERR_ARG  # ld % 4
    assert lib.sv_lm_head_logits(P + 8, P, 4, 100, 64, P, 100, NULL, NULL) == _lib.SV_ERR_ARG  # alignment
    assert lib.sv_lm_head_logits(P, P, 0, 100, 64, P, 100, NULL, NULL) == _lib.SV_OK  # nothing to do
    # workspace: 256 flag bytes, then (2 sum_k + B) rows of ceil4(V) floats
    assert lib.sv_lm_head_workspace_size(64, 320, 128256) == 256 + 704 * 128256 * 4
    assert lib.sv_lm_head_workspace_size(3, 6, 1001) == 256 + 15 * 1004 * 4
    need = lib.sv_lm_head_workspace_size(2, 6, 100)
    args = [P, P, P, 64, P, P, P, NULL, 2, 3, 6, 100, P, P, P]
    assert lib.sv_lm_head_verify(*args, P, need - 4, 0, NULL) == _lib.SV_ERR_ARG
    assert b"workspace_bytes" in lib.sv_last_error()
    assert lib.sv_lm_head_verify(*args, P, need, 16, NULL) == _lib.SV_ERR_ARG  # unknown flag
    assert lib.sv_lm_head_verify(*args, P + 8, need, 0, NULL) == _lib.SV_ERR_ARG  # workspace alignment
    assert lib.sv_lm_head_verify(P, P, P, 64, P, P, P, NULL, 2, 3, 5, 100, P, P, P, P, need, 0,
                                 NULL) == _lib.SV_ERR_ARG  # sum_k != B * K without cu_k


def test_penalties_host_checks(lib):
    P = 1 << 12
    base = dict(t=P, d=P, dt=1, stride=100, ho=P, ht=P, hn=10, tok=P, cu=NULL, B=2, K=3, sk=6, V=100,
                r=P, f=P, p=P, st=P, stream=NULL)

    def call(**kw):
        a = dict(base)
        a.update(kw)
        return lib.sv_apply_penalties(*a.values())

    assert call(K=1025, sk=2050) == _lib.SV_ERR_UNSUPPORTED
    assert call(ho=NULL) == _lib.SV_ERR_ARG and b"hist" in lib.sv_last_error()
    assert call(ho=NULL, ht=NULL, hn=3) == _lib.SV_ERR_ARG
    assert call(sk=5) == _lib.SV_ERR_ARG
    assert call(stride=99) == _lib.SV_ERR_ARG
    assert call(dt=5) == _lib.SV_ERR_ARG
    assert call(st=NULL) == _lib.SV_ERR_ARG
    assert call(B=0, sk=0, t=NULL, d=NULL, tok=NULL, st=NULL) == _lib.SV_OK
