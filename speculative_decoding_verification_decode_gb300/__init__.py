"""GB300-native verification step of speculative decoding.

Greedy verification and Leviathan/Chen rejection sampling for B sequences in
one kernel launch (libsv.so, C ABI in include/sv.h); this package is the thin
PyTorch binding.  See the spec-verify model card, sections "Method" and
"Correctness", for what is computed.
"""

from ._lib import (  # noqa: F401
    FLAG_EXPIRE_EXCHANGE,
    FLAG_FORCE_EXACT,
    FLAG_PLAN_CHAIN,
    FLAG_PLAN_ROWS,
    SEQ_BAD_LAYOUT,
    SEQ_BAD_TOKEN,
    SEQ_BAD_VALUE,
    SEQ_EXACT_PATH,
    SEQ_NEAR_BOUNDARY,
    SEQ_TIMEOUT,
    SEQ_ZERO_MASS,
    load as load_library,
)
from .api import (  # noqa: F401
    GateResult,
    LMHeadResult,
    SVError,
    VerifyResult,
    accept,
    accept_from_logits,
    apply_penalties,
    gate_draft_lengths,
    gate_update,
    lm_head_logits,
    lm_head_verify,
    lm_head_verify_static,
    lm_head_workspace,
    sampler_floors,
    verify_greedy,
)
from ._build import build  # noqa: F401
from .decoder import SpeculativeDecoder  # noqa: F401,E402
