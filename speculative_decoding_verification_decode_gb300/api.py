"""PyTorch binding of libsv: argument marshalling only.

Every step of verification runs in the CUDA kernel behind the C ABI; these
functions only check shapes, pick the current CUDA stream and pass device
pointers.  When the inputs live in host memory the call copies them to the
GPU (from pinned memory when they are pinned), runs the kernel and copies the
results back, which is how an end-to-end caller with host buffers uses it.
"""

from __future__ import annotations

import ctypes
from typing import NamedTuple, Optional

import torch

from . import _lib

_DTYPES = {torch.float32: _lib.SV_F32, torch.bfloat16: _lib.SV_BF16, torch.float16: _lib.SV_F16}


class VerifyResult(NamedTuple):
    n_accepted: torch.Tensor  # int32 [B]
    next_token: torch.Tensor  # int32 [B]; -1 when the sequence's inputs are invalid
    status: torch.Tensor  # int32 [B]; OR of SV_SEQ_* bits


class SVError(RuntimeError):
    pass


def _check(rc: int):
    if rc != _lib.SV_OK:
        lib = _lib.load()
        raise SVError(f"{lib.sv_status_string(rc).decode()}: {lib.sv_last_error().decode()}")


def _rows(x: torch.Tensor) -> torch.Tensor:
    """[rows, V] view of a 2-D or 3-D ([B, rows_per_seq, V]) input with unit
    stride along V."""
    if x.dim() == 3:
        x = x.reshape(-1, x.shape[-1])
    if x.dim() != 2:
        raise ValueError("rows must be 2-D [rows, V] or 3-D [B, rows, V]")
    if x.stride(1) != 1:
        x = x.contiguous()
    return x


def _layout(n_target_rows: int, tokens: torch.Tensor, cu_k, k):
    sum_k = int(tokens.numel())
    if cu_k is None:
        B = n_target_rows - sum_k
        if B < 0 or (B and sum_k % B):
            raise ValueError("target rows must be B*(K+1) for B*K draft tokens")
        K = sum_k // B if B else 0
        return B, K, sum_k
    B = int(cu_k.numel()) - 1
    if k is None:
        raise ValueError("k (the largest K_b) is required with cu_k")
    if n_target_rows < sum_k + B:
        raise ValueError("target must hold sum(K_b) + B rows")
    return B, int(k), sum_k


class _Marshal:
    """Moves host inputs to the device (and results back) for one call."""

    def __init__(self, ref: torch.Tensor):
        self.host = ref.device.type != "cuda"
        self.device = torch.device("cuda", torch.cuda.current_device()) if self.host else ref.device

    def dev(self, t: Optional[torch.Tensor], dtype=None) -> Optional[torch.Tensor]:
        if t is None:
            return None
        if dtype is not None and t.dtype != dtype:
            t = t.to(dtype)
        if t.device != self.device:
            t = t.to(self.device, non_blocking=True)
        return t.contiguous() if t.dim() == 1 else t

    def outputs(self, B: int):
        mk = lambda: torch.empty(B, dtype=torch.int32, device=self.device)
        return mk(), mk(), mk()

    def finish(self, res: VerifyResult) -> VerifyResult:
        if not self.host:
            return res
        return VerifyResult(*(x.to("cpu") for x in res))

    def stream(self):
        return ctypes_ptr(torch.cuda.current_stream(self.device).cuda_stream)


def ctypes_ptr(v):
    return None if v is None else int(v)


def _p(t: Optional[torch.Tensor]):
    return None if t is None else t.data_ptr()


def verify_greedy(target: torch.Tensor, draft_tokens: torch.Tensor,
                  cu_k: Optional[torch.Tensor] = None, k: Optional[int] = None,
                  flags: int = 0) -> VerifyResult:
    """Greedy verification (spec-verify card, "Method"): ``target`` holds the
    K_b + 1 rows of every sequence (probabilities or logits, f32/bf16/f16)."""
    m = _Marshal(target)
    tg = _rows(m.dev(target))
    tok = m.dev(draft_tokens.reshape(-1), torch.int32)
    cu = m.dev(cu_k, torch.int32)
    B, K, sum_k = _layout(tg.shape[0], tok, cu, k)
    n, nxt, st = m.outputs(B)
    lib = _lib.load()
    with torch.cuda.device(m.device):
        _check(lib.sv_verify_greedy(_p(tg), _DTYPES[tg.dtype], tg.stride(0), _p(tok), _p(cu), B, K,
                                    sum_k, tg.shape[1], _p(n), _p(nxt), _p(st), flags, m.stream()))
    return m.finish(VerifyResult(n, nxt, st))


def accept(target_probs: torch.Tensor, draft_probs: torch.Tensor, draft_tokens: torch.Tensor,
           uniforms: torch.Tensor, cu_k: Optional[torch.Tensor] = None, k: Optional[int] = None,
           flags: int = 0) -> VerifyResult:
    """Speculative sampling on f32 probability rows with explicit uniforms
    (``K_b + 1`` per sequence; the last one draws the correction or bonus)."""
    m = _Marshal(target_probs)
    tg = _rows(m.dev(target_probs, torch.float32))
    dr = _rows(m.dev(draft_probs, torch.float32))
    if dr.stride(0) != tg.stride(0):
        dr = dr.contiguous()
        tg = tg.contiguous()
    tok = m.dev(draft_tokens.reshape(-1), torch.int32)
    u = m.dev(uniforms.reshape(-1), torch.float32)
    cu = m.dev(cu_k, torch.int32)
    B, K, sum_k = _layout(tg.shape[0], tok, cu, k)
    n, nxt, st = m.outputs(B)
    lib = _lib.load()
    with torch.cuda.device(m.device):
        _check(lib.sv_accept(_p(tg), _p(dr), tg.stride(0), _p(tok), _p(u), _p(cu), B, K, sum_k,
                             tg.shape[1], _p(n), _p(nxt), _p(st), flags, m.stream()))
    return m.finish(VerifyResult(n, nxt, st))


def accept_from_logits(target_logits: torch.Tensor, draft_logits: torch.Tensor,
                       temperature: torch.Tensor, draft_tokens: torch.Tensor,
                       uniforms: torch.Tensor, cu_k: Optional[torch.Tensor] = None,
                       k: Optional[int] = None, warped_out: Optional[tuple] = None,
                       flags: int = 0, top_k: Optional[torch.Tensor] = None,
                       top_p: Optional[torch.Tensor] = None,
                       floors: Optional[tuple] = None) -> VerifyResult:
    """Mixed greedy / sampled verification from logits with a fused
    per-sequence temperature softmax (``temperature[b] == 0`` is greedy).

    ``warped_out``: optional pair of f32 device tensors ``[target_rows, V]``
    and ``[draft_rows, V]`` that receive the warped weights of every row the
    kernel reached (a testing aid).

    ``top_k`` (int32 ``[B]``) / ``top_p`` (f32 ``[B]``): the sampler filters of
    include/sv_filter.h, applied alike to target and draft rows, in one call of
    ``sv_accept_from_logits_filtered`` (the fused top-k plan where it applies,
    the floors and the floored verification for the rest; with ``warped_out``
    the two calls instead).  ``floors``: a pair of f32 device tensors
    ``[target_rows]``, ``[draft_rows]`` of precomputed floors (used instead of
    top_k / top_p; either may be None)."""
    m = _Marshal(target_logits)
    tg = _rows(m.dev(target_logits))
    dr = _rows(m.dev(draft_logits, tg.dtype))
    if dr.stride(0) != tg.stride(0):
        dr = dr.contiguous()
        tg = tg.contiguous()
    tok = m.dev(draft_tokens.reshape(-1), torch.int32)
    u = m.dev(uniforms.reshape(-1), torch.float32)
    T = m.dev(temperature.reshape(-1), torch.float32)
    cu = m.dev(cu_k, torch.int32)
    B, K, sum_k = _layout(tg.shape[0], tok, cu, k)
    wt, wd = (None, None) if warped_out is None else warped_out
    n, nxt, st = m.outputs(B)
    lib = _lib.load()
    if floors is None and (top_k is not None or top_p is not None):
        tk, tp = m.dev(top_k, torch.int32), m.dev(top_p, torch.float32)
        if warped_out is None:
            with torch.cuda.device(m.device):
                _check(lib.sv_accept_from_logits_filtered(_p(tg), _p(dr), _DTYPES[tg.dtype], tg.stride(0), _p(T),
                                                          _p(tk), _p(tp), _p(tok), _p(u), _p(cu), B, K, sum_k,
                                                          tg.shape[1], _p(n), _p(nxt), _p(st), flags, m.stream()))
            return m.finish(VerifyResult(n, nxt, st))
        floors = _floors(lib, m, tg, dr, T, tk, tp, cu, B, K, sum_k)
    with torch.cuda.device(m.device):
        if floors is None:
            _check(lib.sv_accept_from_logits(_p(tg), _p(dr), _DTYPES[tg.dtype], tg.stride(0), _p(T),
                                             _p(tok), _p(u), _p(cu), B, K, sum_k, tg.shape[1], _p(n),
                                             _p(nxt), _p(st), _p(wt), _p(wd), flags, m.stream()))
        else:
            ft, fd = (m.dev(f, torch.float32) for f in floors)
            _check(lib.sv_accept_from_logits_floored(_p(tg), _p(dr), _DTYPES[tg.dtype], tg.stride(0),
                                                     _p(T), _p(tok), _p(u), _p(cu), B, K, sum_k,
                                                     tg.shape[1], _p(ft), _p(fd), _p(n), _p(nxt),
                                                     _p(st), _p(wt), _p(wd), flags, m.stream()))
    return m.finish(VerifyResult(n, nxt, st))


def _floors(lib, m, tg, dr, T, tk, tp, cu, B, K, sum_k, out=None):
    if out is not None:
        ft, fd = out
    else:
        ft = torch.full((sum_k + B,), float("-inf"), dtype=torch.float32, device=m.device)
        fd = torch.full((sum_k,), float("-inf"), dtype=torch.float32, device=m.device)
    with torch.cuda.device(m.device):
        _check(lib.sv_sampler_floors(_p(tg), _p(dr), _DTYPES[tg.dtype], tg.stride(0), _p(T), _p(tk),
                                     _p(tp), _p(cu), B, K, sum_k, tg.shape[1], _p(ft), _p(fd),
                                     m.stream()))
    return ft, fd


def sampler_floors(target_logits: torch.Tensor, draft_logits: torch.Tensor,
                   temperature: torch.Tensor, top_k: Optional[torch.Tensor] = None,
                   top_p: Optional[torch.Tensor] = None, cu_k: Optional[torch.Tensor] = None,
                   k: Optional[int] = None, sum_k: Optional[int] = None, out: Optional[tuple] = None):
    """Per-row floors of the top-k / top-p filters (include/sv_filter.h):
    ``(floor_target [target_rows], floor_draft [draft_rows])`` f32; the rows a
    filter keeps are those with logit >= floor (-inf keeps all, NaN marks an
    invalid top-p).  Without ``cu_k`` the layout is B*(K+1) target rows and
    B*K draft rows with ``k`` = K.  ``out``: optional preallocated f32 device
    tensors for the two results (device inputs only; rows the kernel does not
    reach keep their values)."""
    n_t = target_logits.reshape(-1, target_logits.shape[-1]).shape[0]
    n_d = draft_logits.reshape(-1, draft_logits.shape[-1]).shape[0]
    if cu_k is None:
        B = int(temperature.numel())
        K = (n_t - B) // B if B else 0
        sk = B * K
        if n_t != B * (K + 1) or n_d != sk:
            raise ValueError(f"without cu_k the rows must be B*(K+1) target and B*K draft rows for "
                             f"B = {B} temperatures (got {n_t} and {n_d})")
    else:
        B = int(cu_k.numel()) - 1
        if k is None or sum_k is None:
            raise ValueError("k and sum_k are required with cu_k")
        K, sk = int(k), int(sum_k)
        if n_t < sk + B or n_d < sk:
            raise ValueError(f"cu_k needs {sk + B} target and {sk} draft rows (got {n_t} and {n_d})")
    m = _Marshal(target_logits)
    tg = _rows(m.dev(target_logits))
    dr = _rows(m.dev(draft_logits, tg.dtype))
    if dr.stride(0) != tg.stride(0):
        dr = dr.contiguous()
        tg = tg.contiguous()
    T = m.dev(temperature.reshape(-1), torch.float32)
    cu = m.dev(cu_k, torch.int32)
    ft, fd = _floors(_lib.load(), m, tg, dr, T, m.dev(top_k, torch.int32), m.dev(top_p, torch.float32),
                     cu, B, K, sk, None if m.host else out)
    if m.host:
        return ft.cpu(), fd.cpu()
    return ft, fd


# ---------------------------------------------------------------- draft-length gate

class GateResult(NamedTuple):
    n_submit: torch.Tensor  # int32 [B]: drafts each sequence submits
    cu_k: torch.Tensor  # int32 [B+1]: their exclusive prefix sum (the verify calls' cu_k)


def gate_draft_lengths(confidence: torch.Tensor, edges: torch.Tensor, hits: torch.Tensor,
                       total: torch.Tensor, k_drafted: Optional[torch.Tensor] = None,
                       logit_margin: Optional[torch.Tensor] = None, margin: float = 1.15,
                       draft_ms: float = 196.0, verify_base_ms: float = 300.0,
                       verify_slope_ms: float = 109.0, plain_ms: float = 303.0,
                       margin_threshold: float = 0.0, min_draft: int = 0) -> GateResult:
    """Draft-length gate (include/sv_gate.h; PocketLLM dspark.md): ``confidence``
    is ``[B, K]`` f32; ``edges`` ``[n_buckets - 1]`` f32; ``hits`` / ``total``
    ``[n_buckets]`` f64 calibration counts.  Defaults are the page's."""
    if confidence.dim() != 2:
        raise ValueError("confidence must be [B, K]")
    dev = confidence.device
    if dev.type != "cuda":
        raise ValueError("gate inputs must be CUDA tensors")
    conf = confidence.to(torch.float32).contiguous()
    B, K = conf.shape
    e = edges.to(device=dev, dtype=torch.float32).contiguous()
    h = hits.to(device=dev, dtype=torch.float64).contiguous()
    t = total.to(device=dev, dtype=torch.float64).contiguous()
    kd = None if k_drafted is None else k_drafted.to(device=dev, dtype=torch.int32).contiguous()
    lm = None if logit_margin is None else logit_margin.to(device=dev, dtype=torch.float32).contiguous()
    n = torch.empty(B, dtype=torch.int32, device=dev)
    cu = torch.empty(B + 1, dtype=torch.int32, device=dev)
    prm = _lib.GateParams(margin, draft_ms, verify_base_ms, verify_slope_ms, plain_ms,
                          margin_threshold, min_draft)
    lib = _lib.load()
    with torch.cuda.device(dev):
        stream = torch.cuda.current_stream(dev).cuda_stream
        _check(lib.sv_gate_draft_lengths(_p(conf), _p(kd), _p(lm), _p(e), _p(h), _p(t), h.numel(), B, K,
                                         ctypes.byref(prm), _p(n), _p(cu), stream))
    return GateResult(n, cu)


def gate_update(confidence: torch.Tensor, n_submitted: torch.Tensor, n_accepted: torch.Tensor,
                edges: torch.Tensor, hits: torch.Tensor, total: torch.Tensor, decay: float = 0.9) -> None:
    """One round of calibration, in place on ``hits`` / ``total`` (f64 CUDA
    tensors, contiguous): positions before the accepted length are hits, the
    first rejected position is a miss, later ones are not recorded."""
    if confidence.dim() != 2:
        raise ValueError("confidence must be [B, K]")
    dev = confidence.device
    for x in (hits, total):
        if x.device != dev or x.dtype != torch.float64 or not x.is_contiguous():
            raise ValueError("hits / total must be contiguous f64 tensors on the confidence's device")
    conf = confidence.to(torch.float32).contiguous()
    B, K = conf.shape
    e = edges.to(device=dev, dtype=torch.float32).contiguous()
    ns = n_submitted.to(device=dev, dtype=torch.int32).contiguous()
    na = n_accepted.to(device=dev, dtype=torch.int32).contiguous()
    lib = _lib.load()
    with torch.cuda.device(dev):
        stream = torch.cuda.current_stream(dev).cuda_stream
        _check(lib.sv_gate_update(_p(conf), _p(ns), _p(na), _p(e), _p(hits), _p(total), hits.numel(), B, K,
                                  float(decay), stream))



# ---------------------------------------------------------------- LM head in front of verification

def _bf16_rows(x: torch.Tensor, m: "_Marshal") -> torch.Tensor:
    x = m.dev(x)
    if x.dtype != torch.bfloat16:
        raise ValueError("states and projection must be bfloat16")
    return x.reshape(-1, x.shape[-1]).contiguous()


def lm_head_logits(states: torch.Tensor, proj: torch.Tensor, out: Optional[torch.Tensor] = None,
                   err: Optional[torch.Tensor] = None) -> torch.Tensor:
    """``states [rows, d] . proj[V, d]^T`` in fp32 on the tensor cores
    (include/sv_lm_head.h).  ``out``: optional f32 ``[rows, >= V]`` device
    tensor with unit stride along V; ``err``: optional int32 ``[1]`` device
    word that receives bit 0 if a device wait gave up."""
    m = _Marshal(states)
    h = _bf16_rows(states, m)
    w = _bf16_rows(proj, m)
    if h.shape[1] != w.shape[1]:
        raise ValueError("states and projection must have the same last dimension")
    rows, V = h.shape[0], w.shape[0]
    if out is None:
        out = torch.empty(rows, (V + 3) // 4 * 4, dtype=torch.float32, device=m.device)[:, :V]
    lib = _lib.load()
    with torch.cuda.device(m.device):
        _check(lib.sv_lm_head_logits(_p(h), _p(w), rows, V, h.shape[1], _p(out), out.stride(0), _p(err),
                                     m.stream()))
    return out.cpu() if m.host else out


class LMHeadResult(NamedTuple):
    n_accepted: torch.Tensor
    next_token: torch.Tensor
    status: torch.Tensor
    target_logits: Optional[torch.Tensor]  # f32 [target rows, V] the verification read (views of the workspace)
    draft_logits: Optional[torch.Tensor]


def lm_head_workspace(batch: int, sum_k: int, vocab: int, device=None) -> torch.Tensor:
    """A workspace for sv_lm_head_verify of this size (uninitialised bytes)."""
    n = int(_lib.load().sv_lm_head_workspace_size(batch, sum_k, vocab))
    return torch.empty(n, dtype=torch.uint8, device=device or torch.device("cuda", torch.cuda.current_device()))


def lm_head_verify(target_states: torch.Tensor, draft_states: torch.Tensor, proj: torch.Tensor,
                   temperature: torch.Tensor, draft_tokens: torch.Tensor, uniforms: torch.Tensor,
                   cu_k: Optional[torch.Tensor] = None, k: Optional[int] = None, flags: int = 0,
                   workspace: Optional[torch.Tensor] = None) -> LMHeadResult:
    """Verification from hidden states (include/sv_lm_head.h): the target and
    draft positions' logits through the one bf16 projection ``proj [V, d]``,
    then the mixed greedy / sampled verification of accept_from_logits.
    Returns the verification results and, for device inputs, the fp32 logits
    it read (views of the workspace, valid until it is reused)."""
    m = _Marshal(target_states)
    ht = _bf16_rows(target_states, m)
    hd = _bf16_rows(draft_states, m)
    w = _bf16_rows(proj, m)
    tok = m.dev(draft_tokens.reshape(-1), torch.int32)
    u = m.dev(uniforms.reshape(-1), torch.float32)
    T = m.dev(temperature.reshape(-1), torch.float32)
    cu = m.dev(cu_k, torch.int32)
    B, K, sum_k = _layout(ht.shape[0], tok, cu, k)
    V, d = w.shape
    if ht.shape[1] != d or (hd.numel() and hd.shape[1] != d):
        raise ValueError("states and projection must have the same last dimension")
    lib = _lib.load()
    need = int(lib.sv_lm_head_workspace_size(B, sum_k, V))
    if workspace is None or workspace.numel() * workspace.element_size() < need:
        workspace = lm_head_workspace(B, sum_k, V, m.device)
    n, nxt, st = m.outputs(B)
    with torch.cuda.device(m.device):
        _check(lib.sv_lm_head_verify(_p(ht), _p(hd), _p(w), d, _p(T), _p(tok), _p(u), _p(cu), B, K, sum_k, V,
                                     _p(n), _p(nxt), _p(st), _p(workspace),
                                     workspace.numel() * workspace.element_size(), flags, m.stream()))
    res = m.finish(VerifyResult(n, nxt, st))
    lt = ld = None
    if not m.host:
        ldv = (V + 3) // 4 * 4
        f = workspace[256:256 + (2 * sum_k + B) * ldv * 4].view(torch.float32).view(-1, ldv)
        lt, ld = f[:sum_k + B, :V], f[sum_k + B:, :V]
    return LMHeadResult(res.n_accepted, res.next_token, res.status, lt, ld)


def lm_head_verify_static(target_states: torch.Tensor, draft_states: torch.Tensor, proj: torch.Tensor,
                          temperature: torch.Tensor, draft_tokens: torch.Tensor, uniforms: torch.Tensor,
                          cu_k: Optional[torch.Tensor] = None, k: Optional[int] = None,
                          flags: int = 0) -> VerifyResult:
    """lm_head_verify on the library's own fixed device scratch
    (sv_lm_head_verify_static, include/sv_lm_head.h): no workspace is
    allocated or passed.  Calls larger than the scratch raise SVError; calls
    that overlap on the GPU race on the scratch (issue them on one stream)."""
    m = _Marshal(target_states)
    ht = _bf16_rows(target_states, m)
    hd = _bf16_rows(draft_states, m)
    w = _bf16_rows(proj, m)
    tok = m.dev(draft_tokens.reshape(-1), torch.int32)
    u = m.dev(uniforms.reshape(-1), torch.float32)
    T = m.dev(temperature.reshape(-1), torch.float32)
    cu = m.dev(cu_k, torch.int32)
    B, K, sum_k = _layout(ht.shape[0], tok, cu, k)
    V, d = w.shape
    n, nxt, st = m.outputs(B)
    lib = _lib.load()
    with torch.cuda.device(m.device):
        _check(lib.sv_lm_head_verify_static(_p(ht), _p(hd), _p(w), d, _p(T), _p(tok), _p(u), _p(cu), B, K, sum_k,
                                            V, _p(n), _p(nxt), _p(st), flags, m.stream()))
    return m.finish(VerifyResult(n, nxt, st))


# ---------------------------------------------------------------- penalties (in place)

def apply_penalties(target_logits: torch.Tensor, draft_logits: torch.Tensor, draft_tokens: torch.Tensor,
                    repetition: torch.Tensor, frequency: torch.Tensor, presence: torch.Tensor,
                    hist_offsets: Optional[torch.Tensor] = None, hist_tokens: Optional[torch.Tensor] = None,
                    cu_k: Optional[torch.Tensor] = None, k: Optional[int] = None) -> torch.Tensor:
    """Repetition / frequency / presence penalties on the raw logits rows, in
    place (include/sv_penalties.h): row i of a sequence sees its history plus
    the drafts before position i.  The rows must be CUDA tensors with unit
    stride along V.  Returns the per-sequence status (int32 [B])."""
    for x in (target_logits, draft_logits):
        if x.device.type != "cuda" or x.stride(-1) != 1:
            raise ValueError("the rows must be CUDA tensors with unit stride along V (modified in place)")
    dev = target_logits.device
    tg = target_logits.reshape(-1, target_logits.shape[-1])
    dr = draft_logits.reshape(-1, draft_logits.shape[-1])
    if tg.data_ptr() != target_logits.data_ptr() or dr.data_ptr() != draft_logits.data_ptr():
        raise ValueError("the rows must be addressable as [rows, V] in place")
    if dr.numel() and dr.stride(0) != tg.stride(0):
        raise ValueError("target and draft rows must have the same row stride")
    m = _Marshal(target_logits)
    tok = m.dev(draft_tokens.reshape(-1), torch.int32)
    cu = m.dev(cu_k, torch.int32)
    B, K, sum_k = _layout(tg.shape[0], tok, cu, k)
    f = lambda x: m.dev(x.reshape(-1), torch.float32)
    r, fr, pr = f(repetition), f(frequency), f(presence)
    ho = m.dev(hist_offsets, torch.int32)
    ht = m.dev(hist_tokens, torch.int32)
    st = torch.empty(B, dtype=torch.int32, device=dev)
    lib = _lib.load()
    with torch.cuda.device(dev):
        _check(lib.sv_apply_penalties(_p(tg), _p(dr), _DTYPES[tg.dtype], tg.stride(0), _p(ho), _p(ht),
                                      0 if ht is None else ht.numel(), _p(tok), _p(cu), B, K, sum_k, tg.shape[1],
                                      _p(r), _p(fr), _p(pr), _p(st), m.stream()))
    return st
