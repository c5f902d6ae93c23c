"""Seeded synthetic inputs for the fused dense-layer workloads.

This module only draws random numbers and rounds them to the storage dtype
(fp16 or bf16). It holds none of the fused layer's arithmetic, so both the
CUDA path and the float64 oracle may consume what it produces: the oracle
reads the same dtype-rounded bytes, widened exactly to float64.

Distributions follow the workloads of the fused-layer pages:
  activations A / x        ~ N(0, 1)
  weights W[N, K]          ~ N(0, 1/K)   (1/K is a variance: O(1) outputs)
  bias, beta               ~ N(0, 0.1)   (0.1 is a standard deviation)
  residual                 ~ N(0, 1)
  gamma                    ~ N(1, 0.1)   (0.1 is a standard deviation)
  FFN down weight Wd[D, F] ~ N(0, 1/F)

Draw order inside one generator: A/x, W (Wg, Wu, Wd), bias, residual, gamma,
beta. Every tensor is drawn in float64 with NumPy's PCG64 and rounded to the
dtype by PyTorch's round-to-nearest-even conversion.
"""
from __future__ import annotations

import math

import numpy as np
import torch

DTYPES = {"f16": torch.float16, "bf16": torch.bfloat16}
DTYPE_IDS = {"f16": 0, "bf16": 1}

# Pattern names in the order of the fused-pattern table of the
# llm-fusion-compiler page ("Pattern / Operations fused").
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


def rng_for(*key: int) -> np.random.Generator:
    """A PCG64 generator seeded by a tuple of non-negative integers."""
    return np.random.default_rng([int(k) for k in key])


def _draw(rng: np.random.Generator, shape, mean: float, std: float, dtype: str) -> torch.Tensor:
    v = rng.standard_normal(size=shape, dtype=np.float64)
    if std != 1.0:
        v *= std
    if mean != 0.0:
        v += mean
    return torch.from_numpy(v).to(DTYPES[dtype])


def pattern_uses(pattern: str) -> dict:
    """Which optional operands a fused pattern reads."""
    return {
        "bias": "bias" in pattern,
        "residual": pattern.endswith("residual"),
        "gamma": pattern in ("layernorm_gemm", "rmsnorm_gemm"),
        "beta": pattern == "layernorm_gemm",
    }


def gemm_inputs(M: int, N: int, K: int, pattern: str, dtype: str, seed=None) -> dict:
    """Inputs of one fused-pattern call: A[M,K], W[N,K] and what the pattern reads.

    `seed` defaults to the tuple (pattern id, dtype id, M, N, K). Returned
    tensors live on the CPU in the storage dtype.
    """
    if seed is None:
        seed = (PATTERNS.index(pattern), DTYPE_IDS[dtype], M, N, K)
    rng = rng_for(*(seed if isinstance(seed, (tuple, list)) else (seed,)))
    use = pattern_uses(pattern)
    out = {"A": _draw(rng, (M, K), 0.0, 1.0, dtype),
           "W": _draw(rng, (N, K), 0.0, 1.0 / math.sqrt(K), dtype)}
    out["bias"] = _draw(rng, (N,), 0.0, 0.1, dtype) if use["bias"] else None
    out["residual"] = _draw(rng, (M, N), 0.0, 1.0, dtype) if use["residual"] else None
    out["gamma"] = _draw(rng, (K,), 1.0, 0.1, dtype) if use["gamma"] else None
    out["beta"] = _draw(rng, (K,), 0.0, 0.1, dtype) if use["beta"] else None
    return out


def norm_gemm_inputs(M: int, N: int, K: int, norm: str, dtype: str, with_bias=False,
                     with_beta=None, seed=None) -> dict:
    """Inputs of one norm-prologue call: x[M,K], W[N,K], gamma[K], beta[K], bias[N]."""
    pattern = "layernorm_gemm" if norm == "layer" else "rmsnorm_gemm"
    if seed is None:
        seed = (PATTERNS.index(pattern), DTYPE_IDS[dtype], M, N, K, int(with_bias))
    rng = rng_for(*(seed if isinstance(seed, (tuple, list)) else (seed,)))
    if with_beta is None:
        with_beta = norm == "layer"
    out = {"x": _draw(rng, (M, K), 0.0, 1.0, dtype),
           "W": _draw(rng, (N, K), 0.0, 1.0 / math.sqrt(K), dtype)}
    out["bias"] = _draw(rng, (N,), 0.0, 0.1, dtype) if with_bias else None
    out["gamma"] = _draw(rng, (K,), 1.0, 0.1, dtype)
    out["beta"] = _draw(rng, (K,), 0.0, 0.1, dtype) if with_beta else None
    return out


def swiglu_inputs(M: int, D: int, F: int, dtype: str, with_bias=False, seed=None) -> dict:
    """Inputs of one SwiGLU FFN block: x[M,D], gamma[D], Wg/Wu[F,D], Wd[D,F], bias_down[D]."""
    if seed is None:
        seed = (100, DTYPE_IDS[dtype], M, D, F, int(with_bias))
    rng = rng_for(*(seed if isinstance(seed, (tuple, list)) else (seed,)))
    out = {"x": _draw(rng, (M, D), 0.0, 1.0, dtype),
           "Wg": _draw(rng, (F, D), 0.0, 1.0 / math.sqrt(D), dtype),
           "Wu": _draw(rng, (F, D), 0.0, 1.0 / math.sqrt(D), dtype),
           "Wd": _draw(rng, (D, F), 0.0, 1.0 / math.sqrt(F), dtype)}
    out["bias_down"] = _draw(rng, (D,), 0.0, 0.1, dtype) if with_bias else None
    out["gamma"] = _draw(rng, (D,), 1.0, 0.1, dtype)
    return out


def as_f64(t):
    """Exact widening of a dtype-rounded CPU tensor to a float64 NumPy array (None passes through)."""
    if t is None:
        return None
    return t.detach().cpu().to(torch.float64).numpy()


def dense_layer_inputs(M: int, N: int, K: int, dtype: str, seed=None) -> dict:
    """Every operand any of the nine patterns reads, for sweeping all patterns on one draw.

    Draw order A, W, bias, residual, gamma, beta; seed defaults to (3, dtype id, M, N, K).
    """
    if seed is None:
        seed = (3, DTYPE_IDS[dtype], M, N, K)
    rng = rng_for(*(seed if isinstance(seed, (tuple, list)) else (seed,)))
    return {"A": _draw(rng, (M, K), 0.0, 1.0, dtype),
            "W": _draw(rng, (N, K), 0.0, 1.0 / math.sqrt(K), dtype),
            "bias": _draw(rng, (N,), 0.0, 0.1, dtype),
            "residual": _draw(rng, (M, N), 0.0, 1.0, dtype),
            "gamma": _draw(rng, (K,), 1.0, 0.1, dtype),
            "beta": _draw(rng, (K,), 0.0, 0.1, dtype)}


def multi_inputs(M: int, Ns, K: int, norm: str, dtype: str, seed=None) -> dict:
    """Inputs of one multi-consumer norm call: x[M,K], gamma[K], beta[K] (LayerNorm),
    then W_i[N_i,K] and bias_i[N_i] per output (keys W0, bias0, W1, bias1, ...)."""
    if seed is None:
        seed = (41, DTYPE_IDS[dtype], M, K, *Ns)
    rng = rng_for(*(seed if isinstance(seed, (tuple, list)) else (seed,)))
    out = {"x": _draw(rng, (M, K), 0.0, 1.0, dtype)}
    for i, N in enumerate(Ns):
        out[f"W{i}"] = _draw(rng, (N, K), 0.0, 1.0 / math.sqrt(K), dtype)
        out[f"bias{i}"] = _draw(rng, (N,), 0.0, 0.1, dtype)
    out["gamma"] = _draw(rng, (K,), 1.0, 0.1, dtype)
    out["beta"] = _draw(rng, (K,), 0.0, 0.1, dtype) if norm == "layer" else None
    return out


def input_bias_inputs(M: int, N: int, K: int, dtype: str, seed=None) -> dict:
    """Inputs of one input-prologue call: A[M,K], bias_in[K] ~ N(0, 0.5), W[N,K], bias[N], residual[M,N]."""
    if seed is None:
        seed = (42, DTYPE_IDS[dtype], M, N, K)
    rng = rng_for(*(seed if isinstance(seed, (tuple, list)) else (seed,)))
    return {"A": _draw(rng, (M, K), 0.0, 1.0, dtype),
            "W": _draw(rng, (N, K), 0.0, 1.0 / math.sqrt(K), dtype),
            "bias_in": _draw(rng, (K,), 0.0, 0.5, dtype),
            "bias": _draw(rng, (N,), 0.0, 0.1, dtype),
            "residual": _draw(rng, (M, N), 0.0, 1.0, dtype)}


def layer_inputs(M: int, D: int, Dkv: int, F: int, dtype: str, seed=None) -> dict:
    """Inputs of one decoder layer's dense part: x[M,D], gamma_attn[D], Wq[D,D],
    Wk/Wv[Dkv,D], attn[M,D] (stands in for the attention output), Wo[D,D],
    gamma_ffn[D], Wg/Wu[F,D], Wd[D,F]."""
    if seed is None:
        seed = (43, DTYPE_IDS[dtype], M, D, Dkv, F)
    rng = rng_for(*(seed if isinstance(seed, (tuple, list)) else (seed,)))
    s = 1.0 / math.sqrt(D)
    return {"x": _draw(rng, (M, D), 0.0, 1.0, dtype), "gamma_attn": _draw(rng, (D,), 1.0, 0.1, dtype),
            "Wq": _draw(rng, (D, D), 0.0, s, dtype), "Wk": _draw(rng, (Dkv, D), 0.0, s, dtype),
            "Wv": _draw(rng, (Dkv, D), 0.0, s, dtype), "attn": _draw(rng, (M, D), 0.0, 1.0, dtype),
            "Wo": _draw(rng, (D, D), 0.0, s, dtype), "gamma_ffn": _draw(rng, (D,), 1.0, 0.1, dtype),
            "Wg": _draw(rng, (F, D), 0.0, s, dtype), "Wu": _draw(rng, (F, D), 0.0, s, dtype),
            "Wd": _draw(rng, (D, F), 0.0, 1.0 / math.sqrt(F), dtype)}
