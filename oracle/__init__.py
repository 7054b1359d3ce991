"""CPU oracle for speculative-decoding verification.  TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` /
``--impl reference`` legs of ``bench.py`` may import this package.  The
product path (the CUDA library and its Python binding) never imports, calls
or links anything here, and this package imports nothing from it: the two
share no code, constants or helpers.  Inputs come from ``workloads`` (data
only) or from the tests themselves.

``lm_head`` puts the LM head (logits = H W^T, llmstudio.ru section 21) in
front of the verification.  ``sampler_filter`` holds the top-k / top-p filters applied to p and q
before verification (llmstudio.ru section 38); ``penalties`` the repetition,
frequency and presence penalties ahead of them, with the sampler state of
each row following the speculative branch (sections 38-39).  ``draft_gate`` is the
draft-length gate that produces the ragged ``cu_k``
(PocketLLM docs/dspark.md, the draft-length gate section).

What it computes follows the spec-verify model card (sections "Method",
"Correctness", "Requirements and limits") and the llmstudio.ru explainer
"Как работает speculative decoding и MTP при инференсе LLM" (sections 13,
15-17, 38, 47, 48).  Every function is pinned by ``tests/test_oracle_*.py``
against values the pages print, closed forms, exact enumeration or brute
force; none is "parity unpinned".
"""

from .spec_verify import (  # noqa: F401
    BAD_TOKEN,
    BAD_VALUE,
    ZERO_MASS,
    NEAR_BOUNDARY,
    BAD_LAYOUT,
    NEAR_FILTER,
    NEAR_DECISION,
    DRAW_CERTIFIED,
    NEAR_EMPTY,
    EMPTY_PROB_TOL,
    TIGHT_BONUS_REL,
    TIGHT_BONUS_MAX_V,
    softmax_weight_tol,
    softmax_decision_tol,
    BOUNDARY_REL_TOL,
    Result,
    decode_rows,
    exact_mass_int,
    exact_mass,
    argmax_lowest,
    accept_decision,
    inverse_cdf_draw,
    verify_greedy,
    accept,
    accept_from_logits,
    softmax_fp64,
    warped_rows_f32,
)
from .sampler_filter import (  # noqa: F401
    FILTER_REL_TOL,
    top_k_floor,
    filter_floor,
    floor_is_valid,
    apply_floor,
    floors_batch,
)
from .lm_head import (  # noqa: F401
    lm_head_logits,
    accept_lm_head,
    verify_greedy_lm_head,
)
from .penalties import (  # noqa: F401
    penalize_value,
    penalize_rows,
)
from .draft_gate import (  # noqa: F401
    GateParams,
    bucket_of,
    match_prob,
    round_cost,
    expected_tokens,
    gate_ratios,
    ratio_error_bound,
    gate_decision,
    gate_length,
    gate_batch,
    update_table,
)
