"""ctypes declarations of the C ABI in include/sv.h and include/sv_gate.h (loads lib/libsv.so)."""

import ctypes
import os
import re

from ._build import LIB_PATH, PKG_DIR

HEADERS = [os.path.join(os.path.dirname(PKG_DIR), "include", h) for h in ("sv.h", "sv_gate.h", "sv_filter.h", "sv_lm_head.h", "sv_penalties.h")]

SV_F32, SV_BF16, SV_F16 = 0, 1, 2
SV_OK, SV_ERR_ARG, SV_ERR_CUDA, SV_ERR_UNSUPPORTED = 0, 1, 2, 3
SEQ_BAD_TOKEN, SEQ_BAD_VALUE, SEQ_ZERO_MASS, SEQ_NEAR_BOUNDARY = 1, 2, 4, 8
SEQ_EXACT_PATH, SEQ_TIMEOUT, SEQ_BAD_LAYOUT = 16, 32, 64
FLAG_FORCE_EXACT = 1
FLAG_EXPIRE_EXCHANGE = 2  # testing aid: exchange waits give up at once (SV_SEQ_TIMEOUT)
FLAG_PLAN_ROWS = 4  # the row-parallel plan where the shape allows it
FLAG_PLAN_CHAIN = 8  # the chain plan (wins over FLAG_PLAN_ROWS)

_vp = ctypes.c_void_p
_i32, _i64, _u32 = ctypes.c_int32, ctypes.c_int64, ctypes.c_uint32
_f64 = ctypes.c_double
SV_MODE_GREEDY, SV_MODE_PROBS, SV_MODE_LOGITS = 0, 1, 2


class GateParams(ctypes.Structure):
    """sv_gate_params (include/sv_gate.h)."""
    _fields_ = [("margin", ctypes.c_double), ("draft_ms", ctypes.c_double),
                ("verify_base_ms", ctypes.c_double), ("verify_slope_ms", ctypes.c_double),
                ("plain_ms", ctypes.c_double), ("margin_threshold", ctypes.c_float),
                ("min_draft", ctypes.c_int32)]


SIGNATURES = {
    "sv_verify_greedy": (_i32, [_vp, _i32, _i64, _vp, _vp, _i32, _i32, _i32, _i32,
                                _vp, _vp, _vp, _u32, _vp]),
    "sv_accept": (_i32, [_vp, _vp, _i64, _vp, _vp, _vp, _i32, _i32, _i32, _i32,
                         _vp, _vp, _vp, _u32, _vp]),
    "sv_accept_from_logits": (_i32, [_vp, _vp, _i32, _i64, _vp, _vp, _vp, _vp, _i32, _i32,
                                     _i32, _i32, _vp, _vp, _vp, _vp, _vp, _u32, _vp]),
    "sv_workspace_size": (ctypes.c_size_t, [_i32, _i32, _i32, _i32]),
    "sv_sampler_floors": (_i32, [_vp, _vp, _i32, _i64, _vp, _vp, _vp, _vp, _i32, _i32, _i32, _i32,
                                 _vp, _vp, _vp]),
    "sv_accept_from_logits_floored": (_i32, [_vp, _vp, _i32, _i64, _vp, _vp, _vp, _vp, _i32, _i32,
                                             _i32, _i32, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _u32,
                                             _vp]),
    # target, draft, dtype, stride, temperature, top_k, top_p, tokens, uniforms, cu_k, B, K, sum_k, V,
    # n, next, status, flags, stream
    "sv_accept_from_logits_filtered": (_i32, [_vp, _vp, _i32, _i64, _vp, _vp, _vp, _vp, _vp, _vp, _i32, _i32,
                                              _i32, _i32, _vp, _vp, _vp, _u32, _vp]),
    "sv_gate_draft_lengths": (_i32, [_vp, _vp, _vp, _vp, _vp, _vp, _i32, _i32, _i32,
                                     ctypes.POINTER(GateParams), _vp, _vp, _vp]),
    "sv_gate_update": (_i32, [_vp, _vp, _vp, _vp, _vp, _vp, _i32, _i32, _i32, _f64, _vp]),
    "sv_lm_head_logits": (_i32, [_vp, _vp, _i32, _i32, _i32, _vp, _i64, _vp, _vp]),
    "sv_lm_head_workspace_size": (ctypes.c_size_t, [_i32, _i32, _i32]),
    "sv_lm_head_verify": (_i32, [_vp, _vp, _vp, _i32, _vp, _vp, _vp, _vp, _i32, _i32, _i32, _i32,
                                 _vp, _vp, _vp, _vp, ctypes.c_size_t, _u32, _vp]),
    "sv_lm_head_verify_static": (_i32, [_vp, _vp, _vp, _i32, _vp, _vp, _vp, _vp, _i32, _i32, _i32, _i32,
                                        _vp, _vp, _vp, _u32, _vp]),
    "sv_apply_penalties": (_i32, [_vp, _vp, _i32, _i64, _vp, _vp, _i32, _vp, _vp, _i32, _i32, _i32, _i32,
                                  _vp, _vp, _vp, _vp, _vp]),
    "sv_status_string": (ctypes.c_char_p, [_i32]),
    "sv_last_error": (ctypes.c_char_p, []),
    "sv_version": (_i32, []),
}

_lib = None


def header_symbols():
    """Function names declared in the headers under include/."""
    text = "".join(open(h).read() for h in HEADERS)
    return sorted(set(re.findall(r"\b(sv_[a-z_]+)\s*\(", text)))


def load():
    """Load libsv.so; raise (never fall back) if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise ImportError(
            f"{LIB_PATH} is missing: build it first with "
            "`python -c 'import __graft_entry__ as g; g.build()'`")
    lib = ctypes.CDLL(LIB_PATH)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib
