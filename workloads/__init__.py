"""Seeded synthetic inputs for the verification step.

This package only *makes data*: target/draft rows, draft tokens, uniforms,
ragged offsets and temperatures shaped like the workloads on the spec-verify
model card (section "Measured": V=32000 K=4 and V=128256 K=5 rows, a
deliberately imperfect draft with sum(min(p, q)) about 0.68) and the five
benchmark configurations of this library.  It holds none of the verification
arithmetic (no argmax, no accept test, no residual): both the CPU oracle and
the CUDA path consume the arrays it returns, and neither imports the other.
"""

from .configs import (  # noqa: F401
    Workload,
    CONFIG_NAMES,
    make_config,
    config1_probs,
    config2_bf16_logits,
    config3_greedy_probs,
    config4_ragged_probs,
    config5_mixed_f16_logits,
    f32_to_bf16_bits,
    uniforms_24bit,
)
from .lm_head import LMHeadWorkload, make_lm_head  # noqa: F401,E402
