"""CPU oracle (test infrastructure only; see ``oracle.attention``)."""
from .attention import (  # noqa: F401
    backward,
    causal_mask,
    credited_flops,
    forward,
    head_backward,
    head_forward,
    kv_head,
    preprocess_D,
)
