"""Element-wise comparison of a CUDA result with the float64 oracle.

Tolerance, against the unrounded float64 oracle on outputs of O(1) scale:
  fp16: max |err| <= 1e-2 and mean |err| <= 1e-3 (the stated bound).
  bf16: the same bound scaled by the ratio of the unit roundoffs,
        2^-8 / 2^-11 = 8: max <= 8e-2, mean <= 8e-3. A bf16 output rounded
        perfectly from the exact value already has a mean error near 1.1e-3
        and a maximum near 1.2e-2 at these sizes, so the unscaled bound is
        below bf16's own rounding floor. To keep that scaled bound from
        hiding a real loss of accuracy, a bf16 result must also have a mean
        error of at most 1.25 times that of the unfused bf16 op chain on the
        same inputs (`chain_*` below: every tensor an unfused sequence of
        library calls would store between its ops, rounded to bf16), checked
        wherever the output has enough elements (>= 4096) for the mean to be
        a stable statistic.

The chain model is test infrastructure built from the oracle's own
primitives (definitions plus round-to-nearest-even to the dtype); the CUDA
path never sees it.

With FL_PARITY_LOG=<path> in the environment every comparison appends one
JSON line (what, dtype, elements, max, mean, chain mean) to that file, so a
GPU run records the literal errors of every case.
"""
import json
import os

import numpy as np

import oracle

TOL = {"f16": (1e-2, 1e-3), "bf16": (8e-2, 8e-3)}
CHAIN_RATIO = 1.25
CHAIN_MIN_ELEMENTS = 4096


def errors(got, ref):
    g = got.detach().float().cpu().double().numpy()
    r = np.asarray(ref, dtype=np.float64)
    assert g.shape == r.shape, (g.shape, r.shape)
    assert np.isfinite(g).all(), "non-finite values in the CUDA result"
    e = np.abs(g - r)
    return float(e.max()), float(e.mean())


def _log(record):
    path = os.environ.get("FL_PARITY_LOG")
    if path:
        with open(path, "a") as f:
            f.write(json.dumps(record) + "\n")


def assert_close(got, ref, dtype, what="", chain=None):
    """got (a tensor) against the float64 oracle ref; for bf16, against the
    unfused chain `chain` (float64 array of the chain's rounded output) too."""
    mx, mean = errors(got, ref)
    tmax, tmean = TOL[dtype]
    n = int(np.asarray(ref).size)
    chain_mean = None
    if chain is not None:
        chain_mean = float(np.abs(np.asarray(chain, dtype=np.float64) - np.asarray(ref, dtype=np.float64)).mean())
    _log({"what": what, "dtype": dtype, "elements": n, "max": mx, "mean": mean, "chain_mean": chain_mean})
    assert mx <= tmax and mean <= tmean, f"{what}: max|err| {mx:.3e} (<= {tmax}), mean {mean:.3e} (<= {tmean})"
    if dtype == "bf16" and chain_mean is not None and n >= CHAIN_MIN_ELEMENTS:
        assert mean <= CHAIN_RATIO * chain_mean, (
            f"{what}: mean|err| {mean:.3e} above {CHAIN_RATIO} x the unfused bf16 chain's {chain_mean:.3e}")
    return mx, mean


def sample_rows(M, n=256, seed=0):
    """Sorted sample of n rows, always with the first and the last."""
    if M <= n:
        return np.arange(M)
    rng = np.random.default_rng([seed, M])
    mid = rng.choice(np.arange(1, M - 1), size=n - 2, replace=False)
    return np.sort(np.concatenate([[0, M - 1], mid]))


# ---------------------------------------------------------------------------
# the unfused op chain, rounded to the dtype wherever it would be stored
# ---------------------------------------------------------------------------
_GEMM_FIRST = {
    # pattern: (bias, activation, residual)
    "gemm_bias_gelu": (True, "gelu", False),
    "gemm_bias_silu": (True, "silu", False),
    "gemm_bias_relu": (True, "relu", False),
    "gemm_bias": (True, "none", False),
    "gemm_bias_residual": (True, "none", True),
    "gemm_gelu": (False, "gelu", False),
    "gemm_silu": (False, "silu", False),
}


def _r(v, dtype):
    return oracle.round_to_dtype(v, dtype)


def _bias_add(y, bias):
    return y if bias is None else y + np.asarray(bias, dtype=np.float64)[None, :]


def chain_gemm_epilogue(A, W, bias, residual, pattern, dtype):
    """linear(A, W, bias) stored in the dtype, then the activation or the
    residual add as a second stored op (the unfused library sequence)."""
    uses_bias, act, uses_res = _GEMM_FIRST[pattern]
    y = _r(_bias_add(oracle.linear(A, W), bias if uses_bias else None), dtype)
    if act != "none":
        y = _r(oracle.ACTIVATIONS[act](y), dtype)
    if uses_res:
        y = _r(y + np.asarray(residual, dtype=np.float64), dtype)
    return y


def chain_norm_gemm(x, gamma, beta, W, bias, eps, norm, act, dtype):
    """The normalised activation stored in the dtype, then linear (+ bias)
    stored, then the activation stored."""
    xh = oracle.rms_norm(x, gamma, eps) if norm == "rms" else oracle.layer_norm(x, gamma, beta, eps)
    y = _r(_bias_add(oracle.linear(_r(xh, dtype), W), bias), dtype)
    if act != "none":
        y = _r(oracle.ACTIVATIONS[act](y), dtype)
    return y


def chain_pattern(pattern, A, W, bias, residual, gamma, beta, eps, dtype):
    if pattern == "rmsnorm_gemm":
        return chain_norm_gemm(A, gamma, None, W, None, eps, "rms", "none", dtype)
    if pattern == "layernorm_gemm":
        return chain_norm_gemm(A, gamma, beta, W, None, eps, "layer", "none", dtype)
    return chain_gemm_epilogue(A, W, bias, residual, pattern, dtype)


def chain_swiglu_ffn(x, gamma, Wg, Wu, Wd, bias_down, eps, dtype):
    """RMSNorm, gate and up projections, SiLU, product, down projection (+
    bias) and residual add, each result stored in the dtype."""
    xh = _r(oracle.rms_norm(x, gamma, eps), dtype)
    g = _r(oracle.linear(xh, Wg), dtype)
    u = _r(oracle.linear(xh, Wu), dtype)
    h = _r(_r(oracle.silu(g), dtype) * u, dtype)
    d = _r(_bias_add(oracle.linear(h, Wd), bias_down), dtype)
    return _r(d + np.asarray(x, dtype=np.float64), dtype)


def chain_input_bias_gemm(A, bias_in, W, bias, residual, act, dtype):
    """A + bias_in stored in the dtype, then linear (+ bias) stored, then the
    activation and the residual add, each stored."""
    Ab = _r(np.asarray(A, dtype=np.float64) + np.asarray(bias_in, dtype=np.float64)[None, :], dtype)
    y = _r(_bias_add(oracle.linear(Ab, W), bias), dtype)
    if act != "none":
        y = _r(oracle.ACTIVATIONS[act](y), dtype)
    if residual is not None:
        y = _r(y + np.asarray(residual, dtype=np.float64), dtype)
    return y
