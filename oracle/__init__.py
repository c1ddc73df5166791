"""fp64 CPU oracle (test infrastructure only; the product path never imports it)."""
from .mlp_oracle import (  # noqa: F401
    ACTIVATIONS, GATED, act_fn, act_grad, block_backward, block_forward, flops, is_gated,
    mlp_backward, mlp_forward, rel_err, rms_norm, sampled_inter_units, sampled_token_rows,
)
from .fp8_oracle import E4M3_MAX, e4m3, fp8_relu_sq_forward, quantize, weight_scale  # noqa: F401,E402
