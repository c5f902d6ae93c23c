"""Pins of the float64 oracle to things other than itself (CPU only).

Each check ties the oracle to a page value, a closed form, a brute-force
evaluation in exact rational arithmetic, a PyTorch float64 library routine
the special case reduces to, or an invariant of the mathematics. The last
section plants plausible mistakes in copies of the oracle and shows that at
least one pin catches each.
"""
import math
from fractions import Fraction

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
from oracle import fusedlin_oracle as O
from conftest import golden

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


# ----------------------------------------------------------------------------
# brute force helpers: pure Python, exact rational sums, math-module functions
# ----------------------------------------------------------------------------

def bf_linear(A, W):
    M, K = A.shape
    N = W.shape[0]
    out = np.empty((M, N))
    for m in range(M):
        for n in range(N):
            s = Fraction(0)
            for k in range(K):
                s += Fraction(float(A[m, k])) * Fraction(float(W[n, k]))
            out[m, n] = float(s)
    return out


def bf_act(name, v):
    if name == "none":
        return v
    if name == "relu":
        return v if v > 0 else 0.0
    if name == "silu":
        return v / (1.0 + math.exp(-v))
    if name == "gelu":
        c = math.sqrt(2.0 / math.pi)
        return 0.5 * v * (1.0 + math.tanh(c * (v + 0.044715 * v ** 3)))
    raise ValueError(name)


def bf_rms(x, gamma, eps):
    M, K = x.shape
    out = np.empty_like(x)
    for m in range(M):
        ss = sum((Fraction(float(x[m, k])) ** 2 for k in range(K)), Fraction(0))
        r = 1.0 / math.sqrt(float(ss / K) + eps)
        for k in range(K):
            out[m, k] = float(x[m, k]) * r * float(gamma[k])
    return out


def bf_layer(x, gamma, beta, eps):
    M, K = x.shape
    out = np.empty_like(x)
    for m in range(M):
        row = [Fraction(float(v)) for v in x[m]]
        mu = sum(row, Fraction(0)) / K
        var = sum(((v - mu) ** 2 for v in row), Fraction(0)) / K
        rstd = 1.0 / math.sqrt(float(var) + eps)
        for k in range(K):
            b = 0.0 if beta is None else float(beta[k])
            out[m, k] = float(row[k] - mu) * rstd * float(gamma[k]) + b
    return out


GEMM_FIRST = {
    "gemm_bias_gelu": (True, "gelu", False),
    "gemm_bias_silu": (True, "silu", False),
    "gemm_bias_relu": (True, "relu", False),
    "gemm_bias": (True, "none", False),
    "gemm_bias_residual": (True, "none", True),
    "gemm_gelu": (False, "gelu", False),
    "gemm_silu": (False, "silu", False),
}


def bf_gemm_epilogue(A, W, bias, res, pattern):
    uses_bias, act, uses_res = GEMM_FIRST[pattern]
    acc = bf_linear(A, W)
    M, N = acc.shape
    out = np.empty_like(acc)
    for m in range(M):
        for n in range(N):
            v = acc[m, n] + (float(bias[n]) if uses_bias else 0.0)
            v = bf_act(act, v)
            if uses_res:
                v += float(res[m, n])
            out[m, n] = v
    return out


def rand(rng, *shape, scale=1.0):
    return rng.standard_normal(shape) * scale


def dyadic(rng, *shape, bits=10):
    """Random values exactly representable in fp16 (so tiny cases mirror GPU inputs)."""
    return O.round_to_dtype(rng.standard_normal(shape), "f16")


# ----------------------------------------------------------------------------
# 1. page values and closed forms
# ----------------------------------------------------------------------------

def erf_gelu(v):
    return np.array([0.5 * t * (1.0 + math.erf(t / math.sqrt(2.0))) for t in v])


def gelu_gap(gelu_fn):
    v = np.arange(-100000, 100001) * 1e-4  # [-10, 10], step 1e-4
    return float(np.max(np.abs(gelu_fn(v) - erf_gelu(v))))


def check_gelu_gap(gelu_fn):
    g = golden("gelu_tanh_gap.txt")
    page = float(g["max_abs_gap"])
    gap = gelu_gap(gelu_fn)
    # the page prints three significant figures: 0.000473
    assert abs(gap - page) <= 0.5e-6, (gap, page)
    assert gap <= 5e-4


def test_gelu_tanh_gap_matches_page():
    check_gelu_gap(O.gelu_tanh)


def test_activation_special_values():
    assert O.gelu_tanh(0.0) == 0.0 and O.silu(0.0) == 0.0 and O.relu(0.0) == 0.0
    assert O.relu(-3.5) == 0.0 and O.relu(2.25) == 2.25
    # tails: gelu -> v for large v, -> 0 for very negative v; silu likewise
    assert abs(O.gelu_tanh(30.0) - 30.0) < 1e-12 and abs(O.gelu_tanh(-30.0)) < 1e-12
    assert abs(O.silu(40.0) - 40.0) < 1e-12 and abs(O.silu(-40.0)) < 1e-15
    # silu(v) = v * sigmoid(v); sigmoid(v) + sigmoid(-v) = 1  =>  silu(v) - silu(-v) = v
    v = np.linspace(-8, 8, 1001)
    assert np.max(np.abs(O.silu(v) - O.silu(-v) - v)) < 1e-13
    # gelu_tanh(v) - gelu_tanh(-v) = v (odd part of the tanh factor)
    assert np.max(np.abs(O.gelu_tanh(v) - O.gelu_tanh(-v) - v)) < 1e-13


def test_activations_match_torch_float64():
    v = torch.linspace(-12, 12, 20001, dtype=torch.float64)
    vn = v.numpy()
    assert np.max(np.abs(O.gelu_tanh(vn) - F.gelu(v, approximate="tanh").numpy())) < 1e-14
    assert np.max(np.abs(O.silu(vn) - F.silu(v).numpy())) < 1e-14
    assert np.array_equal(O.relu(vn), F.relu(v).numpy())


# ----------------------------------------------------------------------------
# 2. rounding to the storage dtypes (pinned to NumPy and PyTorch conversions)
# ----------------------------------------------------------------------------

def test_round_f16_matches_numpy():
    rng = np.random.default_rng(1)
    v = np.concatenate([
        rng.standard_normal(200000) * 10.0 ** rng.integers(-9, 6, size=200000),
        [0.0, -0.0, 65504.0, 65519.99, 65520.0, 1e6, -1e6, 2 ** -24, 2 ** -25, 3 * 2 ** -26,
         1 + 2 ** -11, 1 + 3 * 2 ** -11, 2 ** -14 * (1 + 2 ** -11)],
    ])
    ref = v.astype(np.float16).astype(np.float64)
    got = O.round_to_dtype(v, "f16")
    assert np.array_equal(got, ref, equal_nan=True)


def test_round_bf16_matches_torch():
    rng = np.random.default_rng(2)
    # float32-representable inputs, so torch's float32 -> bf16 conversion is a single rounding
    v = (rng.standard_normal(200000) * 10.0 ** rng.integers(-30, 30, size=200000)).astype(np.float32)
    v = np.concatenate([v, np.array([0.0, 1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, 2 ** -133, 2 ** -134,
                                     3.3895313892515355e38, 3.4e38, -3.4e38], dtype=np.float32)])
    ref = torch.from_numpy(v).to(torch.bfloat16).to(torch.float64).numpy()
    got = O.round_to_dtype(v.astype(np.float64), "bf16")
    assert np.array_equal(got, ref, equal_nan=True)


# ----------------------------------------------------------------------------
# 3. brute force on tiny shapes (exact rational GEMM sums)
# ----------------------------------------------------------------------------

TINY = [(1, 1, 1), (2, 3, 7), (3, 2, 8), (7, 16, 3), (5, 9, 9), (8, 7, 16), (16, 33, 2), (33, 8, 33)]


def check_gemm_patterns_bruteforce(gemm_epilogue):
    rng = np.random.default_rng(3)
    for (M, N, K) in TINY:
        A, W = dyadic(rng, M, K), dyadic(rng, N, K) / math.sqrt(K)
        W = O.round_to_dtype(W, "f16")
        bias, res = dyadic(rng, N) * 0.1, dyadic(rng, M, N)
        for p in GEMM_FIRST:
            got = gemm_epilogue(A, W, bias, res, p)
            ref = bf_gemm_epilogue(A, W, bias, res, p)
            np.testing.assert_allclose(got, ref, rtol=0, atol=1e-12, err_msg=f"{p} {M}x{N}x{K}")


def test_gemm_patterns_bruteforce():
    check_gemm_patterns_bruteforce(O.gemm_epilogue)


def check_norm_bruteforce(norm_gemm):
    rng = np.random.default_rng(4)
    for (M, N, K) in TINY:
        x, W = dyadic(rng, M, K) + 0.25, O.round_to_dtype(dyadic(rng, N, K) / math.sqrt(K), "f16")
        g, b = 1 + 0.1 * dyadic(rng, K), 0.1 * dyadic(rng, K)
        bias = 0.1 * dyadic(rng, N)
        for norm in ("rms", "layer"):
            for act, use_bias in (("none", False), ("gelu", True), ("silu", False), ("relu", True)):
                got = norm_gemm(x, g, b, W, bias if use_bias else None, 1e-5, norm, act)
                xh = bf_rms(x, g, 1e-5) if norm == "rms" else bf_layer(x, g, b, 1e-5)
                acc = bf_linear(xh, W)
                ref = np.vectorize(lambda v: bf_act(act, v))(acc + (bias[None, :] if use_bias else 0.0))
                np.testing.assert_allclose(got, ref, rtol=0, atol=1e-12, err_msg=f"{norm} {act} {M}x{N}x{K}")


def test_norm_gemm_bruteforce():
    check_norm_bruteforce(O.norm_gemm)


def bf_swiglu(x, g, Wg, Wu, Wd, bd, eps, dt):
    xh = bf_rms(x, g, eps)
    gate, up = bf_linear(xh, Wg), bf_linear(xh, Wu)
    h = np.vectorize(lambda a, b: bf_act("silu", a) * b)(gate, up)
    h = O.round_to_dtype(h, dt)
    out = bf_linear(h, Wd) + x
    return out + (bd[None, :] if bd is not None else 0.0)


def check_swiglu_bruteforce(swiglu_ffn):
    rng = np.random.default_rng(5)
    for (M, D, Fh) in [(1, 8, 16), (3, 16, 24), (5, 8, 40)]:
        x = dyadic(rng, M, D)
        g = 1 + 0.1 * dyadic(rng, D)
        Wg = O.round_to_dtype(dyadic(rng, Fh, D) / math.sqrt(D), "bf16")
        Wu = O.round_to_dtype(dyadic(rng, Fh, D) / math.sqrt(D), "bf16")
        Wd = O.round_to_dtype(dyadic(rng, D, Fh) / math.sqrt(Fh), "bf16")
        bd = 0.1 * dyadic(rng, D)
        for b in (None, bd):
            got = swiglu_ffn(x, g, Wg, Wu, Wd, b, 1e-6, "bf16")
            ref = bf_swiglu(x, g, Wg, Wu, Wd, b, 1e-6, "bf16")
            # h is rounded to bf16 on both sides; an unrounded h that lands on a
            # rounding tie differently would show as one bf16 ulp of h times |Wd|
            np.testing.assert_allclose(got, ref, rtol=0, atol=1e-10)


def test_swiglu_bruteforce():
    check_swiglu_bruteforce(O.swiglu_ffn)


# ----------------------------------------------------------------------------
# 4. PyTorch float64 library routines (the pages validate against PyTorch)
# ----------------------------------------------------------------------------

def test_against_torch_float64():
    rng = np.random.default_rng(6)
    M, N, K = 37, 45, 64
    A, W = rand(rng, M, K), rand(rng, N, K, scale=K ** -0.5)
    bias, res = rand(rng, N, scale=0.1), rand(rng, M, N)
    g, b = 1 + rand(rng, K, scale=0.1), rand(rng, K, scale=0.1)
    tA, tW, tb, tr = map(torch.from_numpy, (A, W, bias, res))
    tg, tbe = torch.from_numpy(g), torch.from_numpy(b)
    lin = F.linear(tA, tW, tb)
    ref = {
        "gemm_bias_gelu": F.gelu(lin, approximate="tanh"),
        "gemm_bias_silu": F.silu(lin),
        "gemm_bias_relu": F.relu(lin),
        "gemm_bias": lin,
        "gemm_bias_residual": lin + tr,
        "gemm_gelu": F.gelu(F.linear(tA, tW), approximate="tanh"),
        "gemm_silu": F.silu(F.linear(tA, tW)),
        "layernorm_gemm": F.linear(F.layer_norm(tA, (K,), tg, tbe, eps=1e-5), tW),
        "rmsnorm_gemm": F.linear(F.rms_norm(tA, (K,), tg, eps=1e-6), tW),
    }
    for p in O.PATTERNS:
        eps = 1e-5 if p == "layernorm_gemm" else 1e-6
        got = O.fused_pattern(p, A, W, bias, res, g, b, eps=eps)
        np.testing.assert_allclose(got, ref[p].numpy(), rtol=0, atol=1e-12, err_msg=p)


# ----------------------------------------------------------------------------
# 5. RMSNorm as the pages spell it out
# ----------------------------------------------------------------------------

def test_rms_follows_page_loop_nest():
    """The hackable-compiler RMSNorm loop nest, step by step, on its own shape."""
    g = golden("rmsnorm_loop_nest.txt")
    rows, cols, eps = int(g["rows"]), int(g["cols"]), float(g["eps"])
    rng = np.random.default_rng(7)
    x, w = rng.standard_normal((rows, cols)), 1 + 0.1 * rng.standard_normal(cols)
    ref = np.empty_like(x)
    v0 = 1.0 / cols
    for a0 in range(rows):
        acc0 = 0.0
        for a1 in range(cols):
            acc0 += x[a0, a1] * x[a0, a1]
        v4 = 1.0 / math.sqrt(acc0 * v0 + eps)
        for a2 in range(cols):
            ref[a0, a2] = x[a0, a2] * v4 * w[a2]
    np.testing.assert_allclose(O.rms_norm(x, w, eps), ref, rtol=1e-13, atol=0)


def test_rms_eps_inside_root_llmboost():
    """LLMBoost kernel: rsqrt(ss / d_in + epsilon); eps visible on a small-norm row."""
    g = golden("rmsnorm_cuda_kernel.txt")
    d_in, eps = int(g["d_in"]), float(g["eps"])
    x = np.full((1, d_in), 1e-3)  # mean square 1e-6, comparable to eps
    got = O.rms_norm(x, np.ones(d_in), eps)
    assert abs(got[0, 0] - 1e-3 / math.sqrt(1e-6 + eps)) < 1e-15
    # the tempting misreading 1/(sqrt(ms) + eps) gives a visibly different value
    assert abs(got[0, 0] - 1e-3 / (1e-3 + eps)) > 1e-3


# ----------------------------------------------------------------------------
# 6. identity and zero weights
# ----------------------------------------------------------------------------

def test_identity_and_zero_weights():
    rng = np.random.default_rng(8)
    M, K = 9, 24
    A, bias, res = rand(rng, M, K), rand(rng, K, scale=0.1), rand(rng, M, K)
    I, Z = np.eye(K), np.zeros((K, K))
    for p, (ub, act, ur) in GEMM_FIRST.items():
        f = O.ACTIVATIONS[act]
        y = O.gemm_epilogue(A, I, bias, res, p)
        expect = f(A + (bias if ub else 0.0)) + (res if ur else 0.0)
        assert np.array_equal(y, expect), p
        y0 = O.gemm_epilogue(A, Z, bias, res, p)
        expect0 = f(np.zeros((M, K)) + (bias if ub else 0.0)) + (res if ur else 0.0)
        assert np.array_equal(y0, expect0), p
    assert np.array_equal(O.gemm_epilogue(A, Z, None, None, "gemm_gelu"), np.zeros((M, K)))


def test_norm_rows_with_identity_weight():
    rng = np.random.default_rng(9)
    M, K, eps = 11, 64, 1e-6
    x = rand(rng, M, K) * 3 + 0.5
    ones, zeros, I = np.ones(K), np.zeros(K), np.eye(K)
    y = O.norm_gemm(x, ones, None, I, None, eps, "rms")
    ms = np.mean(x * x, axis=1)
    np.testing.assert_allclose(np.mean(y * y, axis=1), ms / (ms + eps), rtol=1e-13)
    y = O.norm_gemm(x, ones, zeros, I, None, eps, "layer")
    var = np.var(x, axis=1)
    np.testing.assert_allclose(np.mean(y, axis=1), 0.0, atol=1e-14)
    np.testing.assert_allclose(np.var(y, axis=1), var / (var + eps), rtol=1e-13)


def test_layernorm_no_cancellation():
    """A row with a large common offset normalises like the centred row."""
    rng = np.random.default_rng(10)
    K = 256
    d = rng.standard_normal((4, K))
    x = d + 1000.0
    g, b = np.ones(K), np.zeros(K)
    np.testing.assert_allclose(O.layer_norm(x, g, b, 1e-5), bf_layer(x, g, b, 1e-5), atol=1e-9)


# ----------------------------------------------------------------------------
# 7. invariants
# ----------------------------------------------------------------------------

def test_invariants():
    rng = np.random.default_rng(11)
    M, N, K = 13, 21, 48
    x, W = rand(rng, M, K), rand(rng, N, K, scale=K ** -0.5)
    g, b, bias = 1 + rand(rng, K, scale=0.1), rand(rng, K, scale=0.1), rand(rng, N, scale=0.1)
    # RMSNorm-GEMM and LayerNorm-GEMM are invariant to a row scale when eps = 0
    for norm in ("rms", "layer"):
        y1 = O.norm_gemm(x, g, b, W, bias, 0.0, norm, "silu")
        y2 = O.norm_gemm(x * 7.25, g, b, W, bias, 0.0, norm, "silu")
        np.testing.assert_allclose(y1, y2, rtol=0, atol=1e-12)
    # LayerNorm is invariant to a per-row shift
    np.testing.assert_allclose(O.norm_gemm(x, g, b, W, None, 1e-5, "layer"),
                               O.norm_gemm(x + 3.0, g, b, W, None, 1e-5, "layer"), atol=1e-12)
    # permuting rows of A permutes output rows
    perm = rng.permutation(M)
    res = rand(rng, M, N)
    for p in GEMM_FIRST:
        y = O.gemm_epilogue(x, W, bias, res, p)
        yp = O.gemm_epilogue(x[perm], W, bias, res[perm], p)
        np.testing.assert_allclose(yp, y[perm], rtol=0, atol=1e-13)
    # permuting rows of W permutes output columns (with bias and residual columns)
    pn = rng.permutation(N)
    for p in GEMM_FIRST:
        y = O.gemm_epilogue(x, W, bias, res, p)
        yq = O.gemm_epilogue(x, W[pn], bias[pn], res[:, pn], p)
        np.testing.assert_allclose(yq, y[:, pn], rtol=0, atol=1e-13)
    # a split of K into two halves adds up (the split-K decode variant relies on it)
    k1 = 20
    np.testing.assert_allclose(O.linear(x, W), O.linear(x[:, :k1], W[:, :k1]) + O.linear(x[:, k1:], W[:, k1:]),
                               atol=1e-13)


def test_swiglu_degenerate_weights():
    rng = np.random.default_rng(12)
    M, D, Fh = 6, 32, 48
    x = O.round_to_dtype(rand(rng, M, D), "bf16")
    g = 1 + rand(rng, D, scale=0.1)
    Wg, Wu, Wd = rand(rng, Fh, D, scale=D ** -0.5), rand(rng, Fh, D, scale=D ** -0.5), rand(rng, D, Fh)
    bd = rand(rng, D, scale=0.1)
    assert np.array_equal(O.swiglu_ffn(x, g, Wg, np.zeros_like(Wu), Wd, None, 1e-6, "bf16"), x)
    assert np.array_equal(O.swiglu_ffn(x, g, Wg, Wu, np.zeros_like(Wd), None, 1e-6, "bf16"), x)
    assert np.array_equal(O.swiglu_ffn(x, g, Wg, Wu, np.zeros_like(Wd), bd, 1e-6, "bf16"), x + bd[None, :])
    # gate at zero: silu(0) = 0 kills h whatever the up projection is
    assert np.array_equal(O.swiglu_ffn(x, g, np.zeros_like(Wg), Wu, Wd, None, 1e-6, "bf16"), x)


# ----------------------------------------------------------------------------
# 7b. the elementwise input prologue (x + bias along K, then the GEMM)
# ----------------------------------------------------------------------------

def check_input_bias_bruteforce(fn):
    rng = np.random.default_rng(31)
    for (M, N, K) in [(1, 1, 1), (3, 2, 7), (5, 8, 16), (4, 7, 7)]:
        A, W = dyadic(rng, M, K), dyadic(rng, N, K)
        bi, b, r = dyadic(rng, K), dyadic(rng, N), dyadic(rng, M, N)
        for act in ("none", "gelu", "silu", "relu"):
            for use_b, use_r in ((False, False), (True, False), (True, True)):
                # exact rational (A + bias_in) first: the sums are over that
                acc = bf_linear(np.array([[float(Fraction(float(A[m, k])) + Fraction(float(bi[k])))
                                           for k in range(K)] for m in range(M)]), W)
                want = np.empty_like(acc)
                for m in range(M):
                    for n in range(N):
                        v = bf_act(act, acc[m, n] + (float(b[n]) if use_b else 0.0))
                        want[m, n] = v + (float(r[m, n]) if use_r else 0.0)
                got = fn(A, bi, W, b if use_b else None, r if use_r else None, act)
                np.testing.assert_allclose(got, want, rtol=1e-12, atol=1e-12)


def test_input_bias_bruteforce():
    check_input_bias_bruteforce(O.input_bias_gemm)


def test_input_bias_page_example_against_torch():
    """The page's example relu(matmul(x + bias, w)), x (16, 64), bias (64,), w (64, 16):
    w is [K, N] there, so W = w^T in the linear-layer layout."""
    g = torch.Generator().manual_seed(5)
    x = torch.randn(16, 64, generator=g, dtype=torch.float64)
    bias = torch.randn(64, generator=g, dtype=torch.float64)
    w = torch.randn(64, 16, generator=g, dtype=torch.float64)
    want = torch.relu(torch.matmul(x + bias, w)).numpy()
    got = O.input_bias_gemm(x.numpy(), bias.numpy(), w.numpy().T, None, None, "relu")
    np.testing.assert_allclose(got, want, rtol=1e-12, atol=1e-12)
    # and with an output bias and residual, against F.linear
    ob, res = torch.randn(16, generator=g, dtype=torch.float64), torch.randn(16, 16, generator=g, dtype=torch.float64)
    want = (F.silu(F.linear(x + bias, w.T, ob)) + res).numpy()
    got = O.input_bias_gemm(x.numpy(), bias.numpy(), w.numpy().T, ob.numpy(), res.numpy(), "silu")
    np.testing.assert_allclose(got, want, rtol=1e-12, atol=1e-12)


def test_input_bias_reduces_to_gemm_patterns():
    rng = np.random.default_rng(32)
    A, W, b = rand(rng, 6, 24), rand(rng, 10, 24, scale=0.2), rand(rng, 10)
    np.testing.assert_array_equal(O.input_bias_gemm(A, np.zeros(24), W, b, None, "gelu"),
                                  O.gemm_epilogue(A, W, b, None, "gemm_bias_gelu"))
    # W = I: the output is act(A + bias_in + bias)
    bi = rand(rng, 24)
    np.testing.assert_allclose(O.input_bias_gemm(A, bi, np.eye(24), None, None, "relu"),
                               np.maximum(A + bi[None, :], 0.0), rtol=0, atol=1e-15)


# ----------------------------------------------------------------------------
# 8. planted mistakes: each plausible slip in a copy of the oracle fails a pin
# ----------------------------------------------------------------------------

def _fails(check, fn):
    try:
        check(fn)
    except AssertionError:
        return True
    return False


def test_planted_mistakes_are_caught():
    # GeLU with a mistyped cubic coefficient, or with the sigmoid approximation
    bad_coef = lambda v: 0.5 * v * (1 + np.tanh(math.sqrt(2 / math.pi) * (v + 0.0447 * v ** 3)))
    bad_sig = lambda v: v / (1 + np.exp(-1.702 * v))
    assert _fails(check_gelu_gap, bad_coef) and _fails(check_gelu_gap, bad_sig)

    # GEMM-first patterns: transposed weight, dropped bias, wrong epilogue order,
    # sign slip in SiLU
    def transposed(A, W, bias, res, p):
        # W's row-major bytes read as a [K, N] matrix (the other layout the pages use)
        K, N = A.shape[1], W.shape[0]
        Wkn = np.ascontiguousarray(W).reshape(K, N)
        ub, act, ur = GEMM_FIRST[p]
        y = O.ACTIVATIONS[act](A @ Wkn + (bias if ub else 0))
        return y + (res if ur else 0)

    def no_bias(A, W, bias, res, p):
        return O.gemm_epilogue(A, W, np.zeros_like(bias), res, p)

    def act_before_bias(A, W, bias, res, p):
        ub, act, ur = GEMM_FIRST[p]
        y = O.ACTIVATIONS[act](O.linear(A, W)) + (bias if ub else 0)
        return y + (res if ur else 0)

    def silu_sign(A, W, bias, res, p):
        y = O.gemm_epilogue(A, W, bias, res, p)
        if GEMM_FIRST[p][1] == "silu":
            v = O.linear(A, W) + (bias if GEMM_FIRST[p][0] else 0)
            y = v / (1 + np.exp(v))
        return y

    for bad in (transposed, no_bias, act_before_bias, silu_sign):
        assert _fails(check_gemm_patterns_bruteforce, bad), bad.__name__

    # norms: eps outside the root, unbiased variance, gamma dropped, missing beta
    def eps_outside(x, g, b, W, bias, eps, norm, act):
        if norm != "rms":
            return O.norm_gemm(x, g, b, W, bias, eps, norm, act)
        xh = x / (np.sqrt(np.mean(x * x, axis=1, keepdims=True)) + eps) * g
        return O._epilogue(O.linear(xh, W), bias, act, None)

    def unbiased_var(x, g, b, W, bias, eps, norm, act):
        if norm != "layer":
            return O.norm_gemm(x, g, b, W, bias, eps, norm, act)
        d = x - x.mean(axis=1, keepdims=True)
        xh = d / np.sqrt(d.var(axis=1, ddof=1, keepdims=True) + eps) * g + b
        return O._epilogue(O.linear(xh, W), bias, act, None)

    def no_gamma(x, g, b, W, bias, eps, norm, act):
        return O.norm_gemm(x, np.ones_like(g), b, W, bias, eps, norm, act)

    def no_beta(x, g, b, W, bias, eps, norm, act):
        return O.norm_gemm(x, g, None, W, bias, eps, norm, act)

    for bad in (eps_outside, unbiased_var, no_gamma, no_beta):
        assert _fails(check_norm_bruteforce, bad), bad.__name__

    # SwiGLU: h left unrounded, gate and up swapped, residual dropped
    def h_unrounded(x, g, Wg, Wu, Wd, bd, eps, dt):
        h = O.swiglu_hidden(x, g, Wg, Wu, eps)
        return O._epilogue(O.linear(h, Wd), bd, "none", x)

    def swapped(x, g, Wg, Wu, Wd, bd, eps, dt):
        return O.swiglu_ffn(x, g, Wu, Wg, Wd, bd, eps, dt)

    def no_residual(x, g, Wg, Wu, Wd, bd, eps, dt):
        return O.swiglu_ffn(x, g, Wg, Wu, Wd, bd, eps, dt) - x

    for bad in (h_unrounded, swapped, no_residual):
        assert _fails(check_swiglu_bruteforce, bad), bad.__name__

    # input prologue: bias_in dropped, or added to the output instead of the input
    def no_bias_in(A, bi, W, b, r, act):
        return O.input_bias_gemm(A, np.zeros_like(bi), W, b, r, act)

    def bias_in_after(A, bi, W, b, r, act):
        y = O._epilogue(O.linear(A, W), b, act, r)
        return y + (bi[None, :y.shape[1]] if y.shape[1] <= bi.shape[0] else 0.0)

    for bad in (no_bias_in, bias_in_after):
        assert _fails(check_input_bias_bruteforce, bad), bad.__name__
