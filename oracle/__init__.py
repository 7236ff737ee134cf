"""fp64 CPU oracle for selected-token log-probabilities (test infrastructure).

TEST INFRASTRUCTURE ONLY: only the tests, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg may import or call anything in this package.  The
CUDA library never links, imports or calls it, and the two share no code.
"""

from .logprob import (  # noqa: F401
    linear_logits,
    linear_selected_logprob,
    linear_selected_logprob_backward,
    logsumexp_rows,
    selected_logprob,
    selected_logprob_grad_logits,
)
