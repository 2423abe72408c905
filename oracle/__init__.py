"""CPU oracles (TEST INFRASTRUCTURE ONLY): the numpy restatement in
dspark_oracle.py (its functions are re-exported here) and the plain C++ one
in dspark_oracle.cpp behind the same API in ``oracle.native``."""

from . import native  # noqa: F401
from .dspark_oracle import (  # noqa: F401
    confidence,
    draft_distribution,
    draft_distribution_rows,
    draft_sample,
    draft_sample_rnn,
    fma32,
    final_weights,
    first_argmax,
    inverse_cdf,
    markov_bias,
    rnn_state,
    rnn_states,
    round_to,
    schedule,
    schedule_capacity,
    softmax_rows,
    to_fixed,
    verify,
)
