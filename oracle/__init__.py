"""fp64 CPU oracle for TriMul (test infrastructure only; never on the product path)."""
from .trimul_oracle import (  # noqa: F401
    INCOMING, OUTGOING, PARAM_KEYS, gated_projection, gemm_flops, layer_norm,
    output_projection, sigmoid, triangle, trimul_forward, trimul_forward_sampled,
)
