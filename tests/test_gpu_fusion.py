"""CUDA path vs the float64 oracle for the horizontal-fusion, input-prologue
and standalone-RMSNorm entry points (needs an sm_103a GPU).

* fl_norm_gemm_multi: one normalised activation feeding several weights in one
  launch; every output is compared element by element with oracle.norm_gemm
  for its own weight, bias and activation.
* fl_input_bias_gemm: act((A + bias_in) W^T + bias) (+ residual) against
  oracle.input_bias_gemm.
* fl_rms_norm: against oracle.rms_norm.
Tolerances (and the bf16 unfused-chain guard) are in tests/parity.py.
"""
import numpy as np
import pytest
import torch

import gemm_epilogue_tma_gb300 as fl
import oracle
import parity
from gemm_epilogue_tma_gb300 import _build
from gemm_epilogue_tma_gb300 import synthetic as syn
from parity import assert_close, sample_rows

pytestmark = pytest.mark.gpu
DTYPES = ("f16", "bf16")


@pytest.fixture(scope="module", autouse=True)
def library():
    _build.build()
    fl.lib()
    torch.cuda.set_device(0)
    yield
    for k in ("tile_n", "variant", "split_k"):
        fl.set_option(k, 0)
    fl.device_status()


def f64(t):
    return syn.as_f64(t)


def dev(t):
    return None if t is None else t.cuda()


def multi_inputs(M, Ns, K, norm, dt):
    """x, gamma, beta and one (W, bias) per output, from one seeded generator."""
    t = syn.multi_inputs(M, Ns, K, norm, dt)
    return t["x"], t["gamma"], t["beta"], [t[f"W{i}"] for i in range(len(Ns))], [t[f"bias{i}"] for i in range(len(Ns))]


def run_multi(M, Ns, K, norm, dt, acts=None, with_bias=True, rows=None, opts=None):
    x, gamma, beta, Ws, biases = multi_inputs(M, Ns, K, norm, dt)
    acts = acts or ["none"] * len(Ns)
    eps = 1e-5 if norm == "layer" else 1e-6
    for k, v in (opts or {}).items():
        fl.set_option(k, v)
    try:
        outs = fl.norm_gemm_multi(dev(x), dev(gamma), [dev(W) for W in Ws], beta=dev(beta),
                                  biases=[dev(b) for b in biases] if with_bias else None, acts=acts, eps=eps,
                                  norm=norm)
        torch.cuda.synchronize()
        fl.device_status()
    finally:
        for k in (opts or {}):
            fl.set_option(k, 0)
    sel = slice(None) if rows is None else rows
    for i, (W, b, act, out) in enumerate(zip(Ws, biases, acts, outs)):
        args = (f64(x)[sel], f64(gamma), f64(beta), f64(W), f64(b) if with_bias else None, eps, norm, act)
        ref = oracle.norm_gemm(*args)
        assert_close(out[sel], ref, dt, f"multi {norm} {dt} {M}x{Ns}x{K} out{i}",
                     chain=parity.chain_norm_gemm(*args, dt))
    return outs


@pytest.mark.parametrize("dt", DTYPES)
@pytest.mark.parametrize("norm", ["rms", "layer"])
@pytest.mark.parametrize("shape", [(300, (200, 136, 72), 520), (129, (264, 8), 72), (1, (64, 32, 32, 16), 128),
                                   (512, (512, 256, 256), 1024)],
                         ids=lambda s: f"{s[0]}x{'-'.join(map(str, s[1]))}x{s[2]}")
def test_multi_ragged(dt, norm, shape):
    M, Ns, K = shape
    run_multi(M, Ns, K, norm, dt, acts=["none", "gelu", "silu", "relu"][:len(Ns)])


@pytest.mark.parametrize("dt", DTYPES)
@pytest.mark.parametrize("variant", ["tile", "splitk", "pair", "pair_ksplit"])
def test_multi_forced_variants(dt, variant):
    opts = {"tile": {"variant": 1}, "splitk": {"variant": 2, "split_k": 3}, "pair": {"variant": 3},
            "pair_ksplit": {"variant": 3, "split_k": 2}}[variant]
    run_multi(300, (264, 136, 520), 1000, "rms", dt, acts=["silu", "none", "gelu"], opts=opts)
    run_multi(200, (136, 72), 520, "layer", dt, opts=opts)


@pytest.mark.parametrize("dt", DTYPES)
@pytest.mark.parametrize("M", [1, 32, 4096])
def test_multi_qkv(dt, M):
    """Q, K, V projections of one RMSNorm'd activation: D = 4096, grouped K/V of 1024."""
    rows = sample_rows(M, n=128)
    run_multi(M, (4096, 1024, 1024), 4096, "rms", dt, with_bias=False, rows=rows)


def test_multi_output_and_single_call_agree():
    """An output of a two-output launch and the single-output call of the same
    weight both meet the bound against the oracle (the two calls may take
    different kernels: twice the tiles changes the dispatch)."""
    x, gamma, beta, Ws, biases = multi_inputs(384, (512, 512), 768, "rms", "bf16")
    outs = fl.norm_gemm_multi(dev(x), dev(gamma), [dev(W) for W in Ws], biases=[dev(b) for b in biases],
                              acts=["gelu", "none"])
    one = fl.norm_gemm(dev(x), dev(gamma), dev(Ws[1]), bias=dev(biases[1]), eps=1e-6, norm="rms")
    torch.cuda.synchronize()
    ref = oracle.norm_gemm(f64(x), f64(gamma), None, f64(Ws[1]), f64(biases[1]), 1e-6, "rms")
    assert_close(one, ref, "bf16", "single")
    assert_close(outs[1], ref, "bf16", "multi out1")


# ---------------------------------------------------------------------------
# input-bias prologue
# ---------------------------------------------------------------------------
def run_input_bias(M, N, K, dt, act, with_bias, with_res, opts=None, seed=0, rows=None):
    t = syn.input_bias_inputs(M, N, K, dt, seed=(42, seed, syn.DTYPE_IDS[dt], M, N, K))
    A, W, bi, b, r = t["A"], t["W"], t["bias_in"], t["bias"], t["residual"]
    for k, v in (opts or {}).items():
        fl.set_option(k, v)
    try:
        got = fl.input_bias_gemm(dev(A), dev(bi), dev(W), bias=dev(b) if with_bias else None,
                                 residual=dev(r) if with_res else None, act=act)
        torch.cuda.synchronize()
        fl.device_status()
    finally:
        for k in (opts or {}):
            fl.set_option(k, 0)
    sel = slice(None) if rows is None else rows
    args = (f64(A)[sel], f64(bi), f64(W), f64(b) if with_bias else None, f64(r)[sel] if with_res else None, act)
    ref = oracle.input_bias_gemm(*args)
    assert_close(got[sel], ref, dt, f"input bias {dt} {act} {M}x{N}x{K} b={with_bias} r={with_res}",
                 chain=parity.chain_input_bias_gemm(*args, dt))


@pytest.mark.parametrize("dt", DTYPES)
@pytest.mark.parametrize("act", ["none", "gelu", "silu", "relu"])
@pytest.mark.parametrize("shape", [(1, 8, 8), (200, 136, 328), (300, 520, 1000)], ids=lambda s: "x".join(map(str, s)))
def test_input_bias_ragged(dt, act, shape):
    M, N, K = shape
    run_input_bias(M, N, K, dt, act, with_bias=True, with_res=act == "none")
    run_input_bias(M, N, K, dt, act, with_bias=False, with_res=False)


@pytest.mark.parametrize("dt", DTYPES)
@pytest.mark.parametrize("variant", ["tile128", "tile256", "splitk", "pair", "pair_ksplit"])
def test_input_bias_forced_variants(dt, variant):
    opts = {"tile128": {"variant": 1, "tile_n": 128}, "tile256": {"variant": 1, "tile_n": 256},
            "splitk": {"variant": 2, "split_k": 4}, "pair": {"variant": 3},
            "pair_ksplit": {"variant": 3, "split_k": 2}}[variant]
    run_input_bias(300, 520, 1000, dt, "relu", with_bias=True, with_res=False, opts=opts)


def test_input_bias_large():
    """The plain-pattern workload size with the prologue, on sampled rows."""
    run_input_bias(2048, 4096, 4096, "f16", "gelu", with_bias=True, with_res=False, rows=sample_rows(2048))


# ---------------------------------------------------------------------------
# standalone RMSNorm
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("dt", DTYPES)
@pytest.mark.parametrize("shape", [(1, 8), (7, 264), (300, 4096), (33, 4104), (64, 11008), (4096, 4096)],
                         ids=lambda s: "x".join(map(str, s)))
def test_rms_norm(dt, shape):
    M, K = shape
    t = syn.norm_gemm_inputs(M, 8, K, "rms", dt)
    x = t["x"].clone()
    if M > 2:
        x[1] = 0.0  # a zero row normalises to zero
    got = fl.rms_norm(dev(x), dev(t["gamma"]), eps=1e-6)
    torch.cuda.synchronize()
    ref = oracle.rms_norm(f64(x), f64(t["gamma"]), 1e-6)
    assert_close(got, ref, dt, f"rms_norm {dt} {M}x{K}", chain=oracle.round_to_dtype(ref, dt))
    if M > 2:
        assert bool((got[1] == 0).all())


def test_rms_norm_in_place():
    t = syn.norm_gemm_inputs(129, 8, 4096 + 2048, "rms", "bf16")
    x = dev(t["x"])
    y = fl.rms_norm(x, dev(t["gamma"]), out=x, eps=1e-6)
    torch.cuda.synchronize()
    assert y.data_ptr() == x.data_ptr()
    ref = oracle.rms_norm(f64(t["x"]), f64(t["gamma"]), 1e-6)
    assert_close(y, ref, "bf16", "rms_norm in place")


# ---------------------------------------------------------------------------
# the weight-streaming decode kernel (1 to 8 rows), forced and automatic
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("dt", DTYPES)
@pytest.mark.parametrize("M", [1, 2, 3, 5, 8])
@pytest.mark.parametrize("NK", [(8, 8), (264, 136), (1032, 4096), (64, 5560)], ids=lambda s: "x".join(map(str, s)))
def test_decode_kernel_all_patterns(dt, M, NK):
    N, K = NK
    t = syn.dense_layer_inputs(M, N, K, dt)
    A, W = dev(t["A"]), dev(t["W"])
    fl.set_option("variant", 4)
    try:
        for pattern in syn.PATTERNS:
            eps = 1e-5 if pattern == "layernorm_gemm" else 1e-6
            if pattern == "rmsnorm_gemm":
                got = fl.norm_gemm(A, dev(t["gamma"]), W, eps=eps, norm="rms")
            elif pattern == "layernorm_gemm":
                got = fl.norm_gemm(A, dev(t["gamma"]), W, beta=dev(t["beta"]), eps=eps, norm="layer")
            else:
                got = fl.gemm_epilogue(A, W, bias=dev(t["bias"]), residual=dev(t["residual"]), pattern=pattern)
            torch.cuda.synchronize()
            args = (f64(t["A"]), f64(t["W"]), f64(t["bias"]), f64(t["residual"]), f64(t["gamma"]), f64(t["beta"]))
            ref = oracle.fused_pattern(pattern, *args, eps=eps)
            assert_close(got, ref, dt, f"decode kernel {pattern} {dt} M={M} {N}x{K}",
                         chain=parity.chain_pattern(pattern, *args, eps, dt))
        run_input_bias(M, N, K, dt, "silu", with_bias=True, with_res=True, opts={"variant": 4})
        fl.device_status()
    finally:
        fl.set_option("variant", 0)


@pytest.mark.parametrize("dt", DTYPES)
@pytest.mark.parametrize("norm", ["rms", "layer"])
def test_decode_kernel_multi_and_degenerate_rows(dt, norm):
    # QKV at one, three and eight rows, automatic choice
    for M in (1, 3, 8):
        run_multi(M, (1024, 256, 256), 1024, norm, dt, acts=["none", "gelu", "none"])
    # zero and constant rows through the in-kernel LayerNorm statistics
    t = syn.norm_gemm_inputs(7, 136, 456, norm, dt, with_bias=True)
    x = t["x"].clone()
    x[0] = 0.0
    x[1] = 40.0
    x[2] = -0.75
    x[6] = 0.0
    got = fl.norm_gemm(dev(x), dev(t["gamma"]), dev(t["W"]), beta=dev(t["beta"]), bias=dev(t["bias"]), eps=1e-5,
                       norm=norm)
    torch.cuda.synchronize()
    ref = oracle.norm_gemm(f64(x), f64(t["gamma"]), f64(t["beta"]), f64(t["W"]), f64(t["bias"]), 1e-5, norm)
    assert_close(got, ref, dt, f"decode kernel degenerate rows {norm} {dt}")
    # two rows (the register-held prologue): a constant row and a row with a
    # large offset (mean 200, unit spread: the shifted sums must not cancel)
    t2 = syn.norm_gemm_inputs(2, 264, 4096, norm, dt, with_bias=True)
    x2 = t2["x"].clone()
    x2[0] = -3.5
    x2[1] = x2[1] + 200.0
    got = fl.norm_gemm(dev(x2), dev(t2["gamma"]), dev(t2["W"]), beta=dev(t2["beta"]), bias=dev(t2["bias"]), eps=1e-5,
                       norm=norm)
    torch.cuda.synchronize()
    ref = oracle.norm_gemm(f64(x2), f64(t2["gamma"]), f64(t2["beta"]), f64(t2["W"]), f64(t2["bias"]), 1e-5, norm)
    assert_close(got, ref, dt, f"decode kernel constant and offset rows {norm} {dt}")


@pytest.mark.parametrize("dt", DTYPES)
def test_decode_ffn_repeated_and_noalloc(dt):
    """The decode FFN (gate/up and down projections on the decode kernel) twice
    in a row on one workspace, and through the allocation-free entry point:
    the same bits each time."""
    M, D, F = 2, 1024, 2816
    t = syn.swiglu_inputs(M, D, F, dt, with_bias=True)
    g = {k: dev(v) for k, v in t.items()}
    ws = torch.empty(fl.swiglu_ffn_workspace_size(M, F, dt), dtype=torch.uint8, device="cuda")
    outs = [fl.swiglu_ffn(g["x"], g["gamma"], g["Wg"], g["Wu"], g["Wd"], bias_down=g["bias_down"], eps=1e-6,
                          workspace=ws) for _ in range(2)]
    na = fl.swiglu_ffn_noalloc(g["x"], g["gamma"], g["Wg"], g["Wu"], g["Wd"], bias_down=g["bias_down"], eps=1e-6)
    torch.cuda.synchronize()
    fl.device_status()
    assert torch.equal(outs[0], outs[1]) and torch.equal(outs[0], na)
    f = {k: f64(v) for k, v in t.items()}
    ref = oracle.swiglu_ffn(f["x"], f["gamma"], f["Wg"], f["Wu"], f["Wd"], f["bias_down"], 1e-6, dt)
    assert_close(outs[0], ref, dt, f"decode ffn {dt}")


@pytest.mark.parametrize("dt", DTYPES)
def test_kernel_launch_counts(dt):
    """The library's own launch counter: one launch per fused call, plus the
    LayerNorm statistics pass on the tensor-core path (not on the decode
    kernel, which computes its rows' statistics itself); the SwiGLU block is
    two launches on either path."""
    def count(fn):
        n0 = fl.kernel_launches()
        fn()
        torch.cuda.synchronize()
        return fl.kernel_launches() - n0

    for M, ln_launches in ((4, 1), (300, 2)):
        t = syn.norm_gemm_inputs(M, 264, 512, "layer", dt, with_bias=True)
        x, g, b, W = dev(t["x"]), dev(t["gamma"]), dev(t["beta"]), dev(t["W"])
        assert count(lambda: fl.norm_gemm(x, g, W, beta=b, eps=1e-5, norm="layer")) == ln_launches
        assert count(lambda: fl.norm_gemm(x, g, W, eps=1e-6, norm="rms")) == 1
        s = syn.swiglu_inputs(M, 512, 1376, dt)
        s = {k: dev(v) for k, v in s.items()}
        assert count(lambda: fl.swiglu_ffn(s["x"], s["gamma"], s["Wg"], s["Wu"], s["Wd"], eps=1e-6)) == 2
