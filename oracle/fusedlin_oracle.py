"""Float64 CPU oracle for the fused transformer dense layer.

TEST INFRASTRUCTURE ONLY. Only the test suite, the smoke check and the
benchmark's CPU-baseline / reference leg may import this module. The
product path (the CUDA library and its Python binding) never imports or
calls it, and this module imports nothing from the product.

What it computes is the plain definition of each fused pattern: a fused
kernel reaches, up to rounding order, exactly the result of the unfused op
chain (the "Fusion Compiler" glossary page, "fused kernel": fusion changes
the schedule, not the mathematics). So every function below is that
definition written out in float64 NumPy, with a matmul as the one library
step and no blocking, fusion or reordering.

Inputs are the same fp16/bf16-rounded values the GPU receives, widened
exactly to float64. Outputs are float64 and unrounded, except for the one
rounding point the SwiGLU block has by construction (its hidden activation
h is stored in the block dtype between the two GEMMs).

Layouts: A/x [M, K] row-major; W [N, K] row-major (the linear-layer layout);
bias [N]; residual/out [M, N]; gamma, beta [K].

Readings of the pages where they are silent or ambiguous:
  * GeLU is the tanh form ("fast approximation" of the llm-fusion-compiler
    pattern table, whose stated 0.000473 gap to torch.gelu is the tanh form's
    float64 maximum gap to erf-GeLU).
  * RMS puts eps inside the root, 1/sqrt(mean(x^2) + eps), as the generated
    RMSNorm kernel of the hackable-compiler page and the LLMBoost CUDA kernel
    ("rsqrtf(ss / d_in + epsilon)") both do.
  * LayerNorm uses the biased variance (divide by K); the pages give no
    formula, this is the standard definition.
  * Epilogue order is accumulate, + bias, activation, + residual. None of
    the nine patterns has both an activation and a residual.
  * The SwiGLU residual is the pre-norm input x; bias_down may be absent.

Parity pins live in tests/test_oracle_pins.py: brute force on tiny shapes,
PyTorch float64 library routines, identity and zero weights, the GeLU gap
closed form and invariants (row permutation, K split, scale invariance).
"""
from __future__ import annotations

import math

import numpy as np

# The nine fused patterns, in the order of the llm-fusion-compiler pattern
# table ("Pattern / Operations fused").
PATTERNS = (
    "gemm_bias_gelu",
    "gemm_bias_silu",
    "gemm_bias_relu",
    "gemm_bias",
    "gemm_bias_residual",
    "gemm_gelu",
    "gemm_silu",
    "layernorm_gemm",
    "rmsnorm_gemm",
)

# IEEE-style binary formats: (significand bits including the implicit one,
# minimum normal exponent, maximum exponent).
_FORMATS = {"f16": (11, -14, 15), "bf16": (8, -126, 127)}


def round_to_dtype(v, dtype: str) -> np.ndarray:
    """Round float64 values to fp16 or bf16, round-to-nearest-even, as float64.

    Written from the definition of the binary formats: the quantum of a value
    in [2^e, 2^(e+1)) is 2^(e - p + 1); below the smallest normal exponent the
    quantum stays at that of the smallest normal (gradual underflow). Values
    whose rounded magnitude exceeds the largest finite number become +-inf.
    """
    p, emin, emax = _FORMATS[dtype]
    v = np.asarray(v, dtype=np.float64)
    _, ex = np.frexp(np.abs(v))  # |v| = m * 2^ex with 0.5 <= m < 1
    e = np.maximum(ex.astype(np.int64) - 1, emin)
    q = np.ldexp(1.0, e - (p - 1))
    r = np.rint(v / q) * q  # np.rint rounds halves to even
    max_finite = (2.0 - 2.0 ** (1 - p)) * 2.0 ** emax
    r = np.where(np.abs(r) > max_finite, np.copysign(np.inf, v), r)
    return np.where(np.isnan(v), v, r)


# --- activations (llm-fusion-compiler pattern table) ----------------------

def gelu_tanh(v):
    """GeLU, tanh form: 0.5 v (1 + tanh(sqrt(2/pi) (v + 0.044715 v^3)))."""
    v = np.asarray(v, dtype=np.float64)
    return 0.5 * v * (1.0 + np.tanh(math.sqrt(2.0 / math.pi) * (v + 0.044715 * v * v * v)))


def silu(v):
    """SiLU: v * sigmoid(v) = v / (1 + exp(-v))."""
    v = np.asarray(v, dtype=np.float64)
    with np.errstate(over="ignore"):
        return v / (1.0 + np.exp(-v))


def relu(v):
    """ReLU: max(0, v)."""
    v = np.asarray(v, dtype=np.float64)
    return np.maximum(v, 0.0)


ACTIVATIONS = {"none": lambda v: np.asarray(v, dtype=np.float64),
               "gelu": gelu_tanh, "silu": silu, "relu": relu}


# --- norms ----------------------------------------------------------------

def rms_norm(x, gamma, eps: float):
    """RMSNorm of each row: x * gamma / sqrt(mean_k(x^2) + eps).

    Follows the RMSNorm loop nest of the hackable-compiler page (sum of
    squares, times 1/K, plus eps, rsqrt, times x, times the weight) and the
    LLMBoost CUDA kernel section.
    """
    x = np.asarray(x, dtype=np.float64)
    ms = np.mean(x * x, axis=1, keepdims=True)
    return x / np.sqrt(ms + eps) * np.asarray(gamma, dtype=np.float64)[None, :]


def layer_norm(x, gamma, beta, eps: float):
    """LayerNorm of each row: (x - mean) / sqrt(var + eps) * gamma + beta, biased var."""
    x = np.asarray(x, dtype=np.float64)
    mu = np.mean(x, axis=1, keepdims=True)
    d = x - mu
    var = np.mean(d * d, axis=1, keepdims=True)
    y = d / np.sqrt(var + eps) * np.asarray(gamma, dtype=np.float64)[None, :]
    if beta is not None:
        y = y + np.asarray(beta, dtype=np.float64)[None, :]
    return y


# --- the contraction --------------------------------------------------------

def linear(A, W):
    """GEMM in the linear-layer layout: out[m, n] = sum_k A[m, k] W[n, k]."""
    return np.asarray(A, dtype=np.float64) @ np.asarray(W, dtype=np.float64).T


def _epilogue(acc, bias, act: str, residual):
    y = acc
    if bias is not None:
        y = y + np.asarray(bias, dtype=np.float64)[None, :]
    y = ACTIVATIONS[act](y)
    if residual is not None:
        y = y + np.asarray(residual, dtype=np.float64)
    return y


# --- the nine fused patterns ------------------------------------------------

_GEMM_FIRST = {
    # pattern: (uses bias, activation, uses residual)
    "gemm_bias_gelu": (True, "gelu", False),
    "gemm_bias_silu": (True, "silu", False),
    "gemm_bias_relu": (True, "relu", False),
    "gemm_bias": (True, "none", False),
    "gemm_bias_residual": (True, "none", True),
    "gemm_gelu": (False, "gelu", False),
    "gemm_silu": (False, "silu", False),
}


def gemm_epilogue(A, W, bias, residual, pattern: str):
    """One of the seven GEMM-first patterns of the llm-fusion-compiler table.

    gemm_bias_{gelu,silu,relu}: act(A W^T + bias); gemm_bias: A W^T + bias;
    gemm_bias_residual: A W^T + bias + residual; gemm_{gelu,silu}: act(A W^T).
    """
    uses_bias, act, uses_res = _GEMM_FIRST[pattern]
    if uses_bias and bias is None:
        raise ValueError(f"{pattern} needs a bias")
    if uses_res and residual is None:
        raise ValueError(f"{pattern} needs a residual")
    return _epilogue(linear(A, W), bias if uses_bias else None, act,
                     residual if uses_res else None)


def norm_gemm(x, gamma, beta, W, bias, eps: float, norm: str, act: str = "none"):
    """Norm prologue, GEMM, optional bias and activation.

    norm = "rms": RMSNorm(x; gamma, eps) W^T  (rmsnorm_gemm pattern; the
    LLMBoost fused_rmsnorm_linear op computes the same thing).
    norm = "layer": LayerNorm(x; gamma, beta, eps) W^T  (layernorm_gemm).
    beta is ignored for RMS and means zero when absent for LayerNorm.
    """
    if norm == "rms":
        xh = rms_norm(x, gamma, eps)
    elif norm == "layer":
        xh = layer_norm(x, gamma, beta, eps)
    else:
        raise ValueError(norm)
    return _epilogue(linear(xh, W), bias, act, None)


def input_bias_gemm(A, bias_in, W, bias, residual, act: str = "none"):
    """Elementwise input prologue: act((A + bias_in) W^T + bias) (+ residual).

    The hackable-compiler page's example torch.relu(torch.matmul(x + bias, w))
    adds a bias along K to the activation inside the reduction loop (its
    Loop IR "prologue (inside reduce)"); this is that prologue followed by
    the usual epilogue. bias_in has K entries; bias and residual may be absent.
    """
    Ab = np.asarray(A, dtype=np.float64) + np.asarray(bias_in, dtype=np.float64)[None, :]
    return _epilogue(linear(Ab, W), bias, act, residual)


def fused_pattern(pattern: str, A, W, bias=None, residual=None, gamma=None, beta=None,
                  eps: float = 1e-6):
    """Any of the nine patterns by name (norm patterns: no bias, no activation)."""
    if pattern == "rmsnorm_gemm":
        return norm_gemm(A, gamma, None, W, None, eps, "rms")
    if pattern == "layernorm_gemm":
        return norm_gemm(A, gamma, beta, W, None, eps, "layer")
    return gemm_epilogue(A, W, bias, residual, pattern)


def swiglu_hidden(x, gamma, Wg, Wu, eps: float):
    """Unrounded SwiGLU hidden activation silu(xh Wg^T) * (xh Wu^T), xh = RMSNorm(x)."""
    xh = rms_norm(x, gamma, eps)
    return silu(linear(xh, Wg)) * linear(xh, Wu)


def swiglu_ffn(x, gamma, Wg, Wu, Wd, bias_down, eps: float, h_dtype: str):
    """Llama-style SwiGLU FFN block with the pre-norm input as residual.

    The llm-fusion-compiler FFN block: three GEMMs, one activation, one
    elementwise product, one bias, one residual, computed as
        h   = round_dtype(silu(xh Wg^T) * (xh Wu^T)),   xh = RMSNorm(x)
        out = h Wd^T (+ bias_down) + x.
    h is rounded to the block dtype because it is the one tensor that
    crosses between the two fused kernels in that dtype.
    """
    h = round_to_dtype(swiglu_hidden(x, gamma, Wg, Wu, eps), h_dtype)
    return _epilogue(linear(h, Wd), bias_down, "none", x)
