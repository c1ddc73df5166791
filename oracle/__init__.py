"""fp64 CPU oracle (test infrastructure only; the product path never imports it)."""
from .mlp_oracle import (  # noqa: F401
    ACTIVATIONS, GATED, act_fn, act_grad, flops, is_gated, mlp_backward,
    mlp_forward, rel_err, sampled_inter_units, sampled_token_rows,
)
