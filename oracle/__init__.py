"""FP64 CPU oracle (test infrastructure only; see ``oracle.linear_logp``)."""
from .linear_logp import (  # noqa: F401
    decode,
    grad_logits,
    linear_backward,
    linear_forward,
    linear_forward_backward,
    linear_logits,
    linear_rows,
    logits_backward,
    logits_forward,
    logp_from_logits,
    logsumexp_rows,
)
