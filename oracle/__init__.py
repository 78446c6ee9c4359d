"""CPU oracle (test infrastructure only; never imported by the product path)."""
from .attention import (  # noqa: F401
    backward,
    delta,
    forward,
    sequences,
    sink_grad,
    sparse_backward,
    sparse_forward,
    visible,
)
