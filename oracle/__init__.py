"""fp64 CPU oracle (test infrastructure only; the product path never imports it)."""
from .mlp_oracle import (  # noqa: F401
    ACTIVATIONS, GATED, act_fn, act_grad, block_backward, block_forward, block_sampled, flops,
    is_gated,
    mlp_backward, mlp_forward, rel_err, rms_norm, sampled_inter_units, sampled_token_rows,
)
from .fp8_oracle import (  # noqa: F401,E402
    E4M3_MAX, E5M2_MAX, e4m3, e5m2, fp8_relu_sq_backward, fp8_relu_sq_forward,
    fp8_relu_sq_sampled, quantize, quantize_e5m2, weight_scale,
)
