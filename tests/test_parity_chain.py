"""Host checks of the unfused-chain model that guards the bf16 parity gate.

The chain model (tests/parity.py) rounds every intermediate an unfused
sequence of library calls would store. These checks pin it to things fixed
independently of it: with rounding taken out it is the oracle's definition;
with identity weights its rounding points are visible one by one; and its
mean error sits between that of one final rounding and the scaled bf16 bound.
"""
import numpy as np
import pytest

import oracle
import parity
from gemm_epilogue_tma_gb300 import synthetic as syn


def f64(t):
    return syn.as_f64(t)


@pytest.fixture
def no_rounding(monkeypatch):
    monkeypatch.setattr(parity, "_r", lambda v, dtype: np.asarray(v, dtype=np.float64))


@pytest.mark.parametrize("pattern", syn.PATTERNS)
def test_chain_without_rounding_is_the_definition(no_rounding, pattern):
    t = syn.dense_layer_inputs(9, 16, 24, "bf16", seed=(7,))
    args = (f64(t["A"]), f64(t["W"]), f64(t["bias"]), f64(t["residual"]), f64(t["gamma"]), f64(t["beta"]))
    want = oracle.fused_pattern(pattern, *args, eps=1e-5)
    got = parity.chain_pattern(pattern, *args, 1e-5, "bf16")
    np.testing.assert_allclose(got, want, rtol=0, atol=1e-12)


def test_swiglu_chain_without_rounding_is_the_definition(no_rounding):
    t = syn.swiglu_inputs(5, 16, 24, "bf16", with_bias=True)
    f = {k: f64(v) for k, v in t.items()}
    # the oracle rounds h once by construction; compare with that rounding undone
    h = oracle.swiglu_hidden(f["x"], f["gamma"], f["Wg"], f["Wu"], 1e-6)
    want = h @ f["Wd"].T + f["bias_down"][None, :] + f["x"]
    got = parity.chain_swiglu_ffn(f["x"], f["gamma"], f["Wg"], f["Wu"], f["Wd"], f["bias_down"], 1e-6, "bf16")
    np.testing.assert_allclose(got, want, rtol=0, atol=1e-12)


def test_chain_rounding_points_with_identity_weight():
    """W = I: linear(A) = A, so gemm_bias_gelu's chain is round(gelu(round(A + b)))."""
    K = 32
    t = syn.dense_layer_inputs(6, K, K, "bf16", seed=(8,))
    A, b = f64(t["A"]), f64(t["bias"])
    got = parity.chain_gemm_epilogue(A, np.eye(K), b, None, "gemm_bias_gelu", "bf16")
    y = oracle.round_to_dtype(A + b[None, :], "bf16")
    want = oracle.round_to_dtype(oracle.gelu_tanh(y), "bf16")
    np.testing.assert_array_equal(got, want)
    # residual pattern: round(round(A + b) + r)
    r = f64(t["residual"])
    got = parity.chain_gemm_epilogue(A, np.eye(K), b, r, "gemm_bias_residual", "bf16")
    np.testing.assert_array_equal(got, oracle.round_to_dtype(y + r, "bf16"))


def test_norm_chain_rounds_the_normalised_activation():
    """gamma = 1, W = I: the RMS chain is round(round(x / rms(x)))."""
    K = 64
    t = syn.norm_gemm_inputs(4, K, K, "rms", "bf16")
    x = f64(t["x"])
    got = parity.chain_norm_gemm(x, np.ones(K), None, np.eye(K), None, 1e-6, "rms", "none", "bf16")
    xh = oracle.round_to_dtype(x / np.sqrt(np.mean(x * x, axis=1, keepdims=True) + 1e-6), "bf16")
    np.testing.assert_array_equal(got, xh)


@pytest.mark.parametrize("pattern", ["rmsnorm_gemm", "layernorm_gemm", "gemm_bias_gelu"])
def test_chain_error_between_one_rounding_and_the_scaled_bound(pattern):
    t = syn.dense_layer_inputs(96, 256, 512, "bf16", seed=(9,))
    args = (f64(t["A"]), f64(t["W"]), f64(t["bias"]), f64(t["residual"]), f64(t["gamma"]), f64(t["beta"]))
    ref = oracle.fused_pattern(pattern, *args, eps=1e-5)
    chain = parity.chain_pattern(pattern, *args, 1e-5, "bf16")
    one = oracle.round_to_dtype(ref, "bf16")
    e_chain = np.abs(chain - ref).mean()
    e_one = np.abs(one - ref).mean()
    assert e_one < e_chain < parity.TOL["bf16"][1]


def test_gate_rejects_a_result_much_worse_than_the_chain():
    """A planted error: a bf16 result whose mean error is 2x the chain's fails the gate."""
    import torch
    t = syn.dense_layer_inputs(64, 128, 256, "bf16", seed=(10,))
    args = (f64(t["A"]), f64(t["W"]), None, None, f64(t["gamma"]), None)
    ref = oracle.fused_pattern("rmsnorm_gemm", *args, eps=1e-6)
    chain = parity.chain_pattern("rmsnorm_gemm", *args, 1e-6, "bf16")
    bad = ref + 2.0 * (chain - ref)  # twice the chain's error, still inside the scaled bound
    assert np.abs(bad - ref).mean() < parity.TOL["bf16"][1]
    with pytest.raises(AssertionError):
        parity.assert_close(torch.from_numpy(bad), ref, "bf16", "planted", chain=chain)
    parity.assert_close(torch.from_numpy(chain), ref, "bf16", "chain itself", chain=chain)
