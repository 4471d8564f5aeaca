"""FP64 CPU oracle (test infrastructure only; see ``oracle/linear_logp.py``)."""
from .linear_logp import (  # noqa: F401
    ROW_CHUNK,
    backward,
    dlogits,
    forward,
    grad_weight_rows,
    logits,
    valid_rows,
)
