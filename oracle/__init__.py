"""CPU oracle (test infrastructure only; see dspark_oracle.py)."""

from .dspark_oracle import (  # noqa: F401
    confidence,
    draft_distribution,
    draft_sample,
    final_weights,
    first_argmax,
    inverse_cdf,
    markov_bias,
    schedule,
    softmax_rows,
    to_fixed,
    verify,
)
