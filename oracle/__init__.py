"""CPU oracle (test infrastructure only; see spec_oracle's header)."""
from .spec_oracle import (  # noqa: F401
    accept_probability, acceptance_rate, argmax_lowest, inverse_cdf, lm_head, residual,
    softmax_t, spec_verify, verify_greedy, verify_sampling,
)
from . import draft_head, kv_commit, ngram_drafter, tree_verify  # noqa: F401,E402
