"""Float64 CPU oracle of the fused dense layer (test infrastructure only).

Imported only by tests/, the smoke check and the benchmark's CPU baseline;
never by the product path.
"""
from .fusedlin_oracle import (  # noqa: F401
    ACTIVATIONS, PATTERNS, fused_pattern, gelu_tanh, gemm_epilogue, input_bias_gemm, layer_norm, linear,
    norm_gemm, relu, rms_norm, round_to_dtype, silu, swiglu_ffn, swiglu_hidden,
)
