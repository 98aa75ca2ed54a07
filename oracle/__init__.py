"""CPU oracle for the grouped expert MLP (test infrastructure only).

Only the tests, the smoke check and the benchmark's CPU-baseline arm may import
this package. The CUDA library never calls into it and it never calls into the
CUDA library.
"""

from .moe_oracle import (  # noqa: F401
    bf16_bits_to_f64,
    round_to_bf16,
    route,
    permute,
    grouped_linear,
    grouped_linear_t,
    GLU_ALPHA,
    PROB_MODES,
    glu,
    glu_backward,
    swiglu,
    swiglu_backward,
    combine,
    prob_grad,
    moe_forward,
    moe_backward,
    token_forward,
    token_backward,
    token_prob_grad,
)
