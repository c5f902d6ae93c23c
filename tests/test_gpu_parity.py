"""CUDA path vs the float64 oracle, element by element (needs an sm_103a GPU).

Every call goes through the C ABI (the ctypes binding). Small ragged shapes
cover partial tiles in M, N and K; the workload sizes of the fused-layer
pages are checked on every element where the oracle is quick, and on a
seeded sample of rows (always the first and the last) where it is not.
Tolerances are in tests/parity.py.
"""
import numpy as np
import pytest
import torch

import gemm_epilogue_tma_gb300 as fl
import oracle
from gemm_epilogue_tma_gb300 import _build
from gemm_epilogue_tma_gb300 import synthetic as syn
import parity
from parity import assert_close, sample_rows

pytestmark = pytest.mark.gpu

GEMM_FIRST = syn.PATTERNS[:7]
DTYPES = ("f16", "bf16")


@pytest.fixture(scope="module", autouse=True)
def library():
    _build.build()
    fl.lib()
    torch.cuda.set_device(0)
    yield
    fl.set_option("tile_n", 0)
    fl.set_option("variant", 0)
    fl.set_option("split_k", 0)
    fl.device_status()


def dev(t):
    return None if t is None else t.cuda()


def f64(t):
    return syn.as_f64(t)


def run_pattern(t, pattern, rows=None, out=None):
    """Launch one of the nine patterns on GPU copies of t; oracle and unfused
    chain on `rows` (all if None). Returns (got, ref, chain)."""
    eps = 1e-5 if pattern == "layernorm_gemm" else 1e-6
    A, W = dev(t["A"]), dev(t["W"])
    if pattern == "rmsnorm_gemm":
        got = fl.norm_gemm(A, dev(t["gamma"]), W, eps=eps, norm="rms", out=out)
    elif pattern == "layernorm_gemm":
        got = fl.norm_gemm(A, dev(t["gamma"]), W, beta=dev(t["beta"]), eps=eps, norm="layer", out=out)
    else:
        got = fl.gemm_epilogue(A, W, bias=dev(t.get("bias")), residual=dev(t.get("residual")), pattern=pattern,
                               out=out)
    torch.cuda.synchronize()
    sel = slice(None) if rows is None else rows
    res = t.get("residual")
    args = (f64(t["A"])[sel], f64(t["W"]), f64(t.get("bias")), None if res is None else f64(res)[sel],
            f64(t.get("gamma")), f64(t.get("beta")))
    ref = oracle.fused_pattern(pattern, *args, eps=eps)
    chain = parity.chain_pattern(pattern, *args, eps, syn_dtype(t))
    return (got[sel] if rows is not None else got), ref, chain


def syn_dtype(t):
    return "bf16" if t["A"].dtype == torch.bfloat16 else "f16"


# ---------------------------------------------------------------------------
# ragged shapes, every pattern, both dtypes, both tile widths
# ---------------------------------------------------------------------------
RAGGED = [(1, 8, 8), (7, 24, 40), (200, 136, 328), (129, 264, 72), (300, 520, 1000), (128, 256, 64)]


@pytest.mark.parametrize("dt", DTYPES)
@pytest.mark.parametrize("shape", RAGGED, ids=lambda s: "x".join(map(str, s)))
def test_all_patterns_ragged(dt, shape):
    M, N, K = shape
    t = syn.dense_layer_inputs(M, N, K, dt)
    for pattern in syn.PATTERNS:
        got, ref, chain = run_pattern(t, pattern)
        assert_close(got, ref, dt, f"{pattern} {dt} {M}x{N}x{K}", chain=chain)
    fl.device_status()


@pytest.mark.parametrize("tile_n", [128, 256])
@pytest.mark.parametrize("dt", DTYPES)
def test_tile_widths(tile_n, dt):
    M, N, K = 384, 776, 520
    t = syn.dense_layer_inputs(M, N, K, dt)
    fl.set_option("tile_n", tile_n)
    try:
        for pattern in ("gemm_bias_gelu", "gemm_bias_residual", "gemm_silu", "rmsnorm_gemm", "layernorm_gemm"):
            got, ref, chain = run_pattern(t, pattern)
            assert_close(got, ref, dt, f"{pattern} {dt} BN={tile_n}", chain=chain)
    finally:
        fl.set_option("tile_n", 0)


@pytest.mark.parametrize("dt", DTYPES)
@pytest.mark.parametrize("norm", ["rms", "layer"])
@pytest.mark.parametrize("act", ["none", "gelu", "silu", "relu"])
def test_norm_gemm_bias_act(dt, norm, act):
    M, N, K = 260, 200, 456
    t = syn.norm_gemm_inputs(M, N, K, norm, dt, with_bias=True)
    eps = 1e-5
    got = fl.norm_gemm(dev(t["x"]), dev(t["gamma"]), dev(t["W"]), beta=dev(t["beta"]), bias=dev(t["bias"]),
                       eps=eps, norm=norm, act=act)
    torch.cuda.synchronize()
    args = (f64(t["x"]), f64(t["gamma"]), f64(t["beta"]), f64(t["W"]), f64(t["bias"]), eps, norm, act)
    ref = oracle.norm_gemm(*args)
    assert_close(got, ref, dt, f"{norm} {act} {dt}", chain=parity.chain_norm_gemm(*args, dt))


def test_layernorm_without_beta_and_offset_rows():
    """beta = NULL means zero; rows with a large common offset normalise without cancellation."""
    M, N, K = 130, 64, 192
    t = syn.norm_gemm_inputs(M, N, K, "layer", "f16")
    x = (t["x"].double() * 0.5 + 40.0).to(torch.float16)
    got = fl.norm_gemm(dev(x), dev(t["gamma"]), dev(t["W"]), eps=1e-5, norm="layer")
    torch.cuda.synchronize()
    ref = oracle.norm_gemm(f64(x), f64(t["gamma"]), None, f64(t["W"]), None, 1e-5, "layer")
    assert_close(got, ref, "f16", "layernorm offset rows")


# ---------------------------------------------------------------------------
# degenerate rows: an all-zero row (a padding token) and constant rows
# (LayerNorm variance exactly zero). Each has one correct result the oracle
# gives exactly: RMS of a zero row scales 0 by 1/sqrt(eps), so out = 0;
# LayerNorm of a zero or constant row is beta, so out = beta W^T.
# ---------------------------------------------------------------------------
def _with_degenerate_rows(x, values):
    x = x.clone()
    for i, v in enumerate(values):
        if i < x.shape[0]:
            x[i] = v
    return x


EDGE_VARIANTS = {
    # name: (options, shape)
    "auto": ({}, (133, 200, 456)),
    "tile": ({"variant": 1}, (133, 200, 456)),
    "splitk": ({"variant": 2, "split_k": 3}, (40, 136, 1000)),
    "pair": ({"variant": 3}, (300, 264, 520)),
    "pair_ksplit": ({"variant": 3, "split_k": 2}, (300, 520, 1000)),
}


@pytest.mark.parametrize("dt", DTYPES)
@pytest.mark.parametrize("norm", ["rms", "layer"])
@pytest.mark.parametrize("variant", list(EDGE_VARIANTS))
def test_zero_and_constant_rows(dt, norm, variant):
    opts, (M, N, K) = EDGE_VARIANTS[variant]
    t = syn.norm_gemm_inputs(M, N, K, norm, dt, with_bias=True)
    # zero row, constant rows of small, negative and large magnitude, then a
    # row with a single non-zero entry
    x = _with_degenerate_rows(t["x"], [0.0, 0.75, -3.0, 40.0])
    x[4].zero_()
    x[4, K // 2] = 2.5
    eps = 1e-5
    for k, v in opts.items():
        fl.set_option(k, v)
    try:
        got = fl.norm_gemm(dev(x), dev(t["gamma"]), dev(t["W"]), beta=dev(t["beta"]), bias=dev(t["bias"]), eps=eps,
                           norm=norm, act="none")
        torch.cuda.synchronize()
        fl.device_status()
    finally:
        for k in opts:
            fl.set_option(k, 0)
    args = (f64(x), f64(t["gamma"]), f64(t["beta"]), f64(t["W"]), f64(t["bias"]), eps, norm, "none")
    ref = oracle.norm_gemm(*args)
    assert_close(got, ref, dt, f"degenerate rows {norm} {dt} {variant}", chain=parity.chain_norm_gemm(*args, dt))
    # the exact results of the zero row
    want0 = (np.zeros(N) if norm == "rms" else f64(t["beta"]) @ f64(t["W"]).T) + f64(t["bias"])
    tmax = parity.TOL[dt][0]
    assert np.abs(got[0].double().cpu().numpy() - want0).max() <= tmax, f"zero row {norm} {dt} {variant}"


@pytest.mark.parametrize("dt", DTYPES)
@pytest.mark.parametrize("norm", ["rms", "layer"])
@pytest.mark.parametrize("D", [1024, 4096])
@pytest.mark.parametrize("row", ["zero", "constant"])
def test_decode_single_degenerate_row(dt, norm, D, row):
    """M = 1 (one decode token) whose row is all zeros or constant."""
    t = syn.norm_gemm_inputs(1, D, D, norm, dt)
    x = torch.zeros_like(t["x"]) if row == "zero" else torch.full_like(t["x"], -1.5)
    eps = 1e-5
    got = fl.norm_gemm(dev(x), dev(t["gamma"]), dev(t["W"]), beta=dev(t.get("beta")), eps=eps, norm=norm)
    torch.cuda.synchronize()
    fl.device_status()
    ref = oracle.norm_gemm(f64(x), f64(t["gamma"]), f64(t.get("beta")), f64(t["W"]), None, eps, norm)
    assert_close(got, ref, dt, f"decode {row} row {norm} {dt} D={D}")
    if row == "zero" and norm == "rms":
        assert bool((got == 0).all()), "RMSNorm of a zero row must give exactly zero"


def test_residual_aliases_out():
    M, N, K = 256, 384, 512
    t = syn.gemm_inputs(M, N, K, "gemm_bias_residual", "bf16")
    res = dev(t["residual"])
    got = fl.gemm_epilogue(dev(t["A"]), dev(t["W"]), bias=dev(t["bias"]), residual=res, out=res,
                           pattern="gemm_bias_residual")
    torch.cuda.synchronize()
    assert got.data_ptr() == res.data_ptr()
    ref = oracle.gemm_epilogue(f64(t["A"]), f64(t["W"]), f64(t["bias"]), f64(t["residual"]), "gemm_bias_residual")
    assert_close(got, ref, "bf16", "residual aliasing out")


def test_no_write_outside_out():
    """A sentinel region on both sides of out stays untouched (ragged tails are clipped)."""
    M, N, K = 131, 72, 136
    t = syn.dense_layer_inputs(M, N, K, "f16")
    pad = 4096
    buf = torch.full((pad + M * N + pad,), 1234.0, dtype=torch.float16, device="cuda")
    out = buf[pad:pad + M * N].view(M, N)
    for pattern in ("gemm_bias_gelu", "gemm_bias_residual", "rmsnorm_gemm", "layernorm_gemm"):
        got, ref, chain = run_pattern(t, pattern, out=out)
        assert_close(got, ref, "f16", pattern, chain=chain)
        assert bool((buf[:pad] == 1234.0).all()) and bool((buf[pad + M * N:] == 1234.0).all()), pattern


def test_repeatable_bitwise():
    M, N, K = 384, 512, 768
    t = syn.dense_layer_inputs(M, N, K, "bf16")
    a = run_pattern(t, "rmsnorm_gemm")[0].clone()
    b = run_pattern(t, "rmsnorm_gemm")[0]
    assert torch.equal(a, b)


# ---------------------------------------------------------------------------
# the split-K variant (cluster of K ranges, reduction through distributed
# shared memory), forced on shapes it would not pick by itself too
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("dt", DTYPES)
@pytest.mark.parametrize("splits", [1, 2, 3, 8])
@pytest.mark.parametrize("shape", [(1, 64, 512), (17, 200, 1000), (128, 136, 4096), (300, 264, 520)],
                         ids=lambda s: "x".join(map(str, s)))
def test_splitk_variant_all_patterns(dt, splits, shape):
    M, N, K = shape
    t = syn.dense_layer_inputs(M, N, K, dt)
    fl.set_option("variant", 2)
    fl.set_option("split_k", splits)
    try:
        for pattern in syn.PATTERNS:
            got, ref, chain = run_pattern(t, pattern)
            assert_close(got, ref, dt, f"split-K x{splits} {pattern} {dt} {M}x{N}x{K}", chain=chain)
        fl.device_status()
    finally:
        fl.set_option("variant", 0)
        fl.set_option("split_k", 0)


@pytest.mark.parametrize("dt", DTYPES)
@pytest.mark.parametrize("splits", [4, 5, 6, 7])
def test_splitk_uneven_column_slices(dt, splits):
    # 16 eight-column chunks over 5, 6 or 7 ranks: owners of unequal width
    M, N, K = 200, 392, 2048
    t = syn.dense_layer_inputs(M, N, K, dt)
    fl.set_option("variant", 2)
    fl.set_option("tile_n", 128)
    fl.set_option("split_k", splits)
    try:
        for pattern in syn.PATTERNS:
            got, ref, chain = run_pattern(t, pattern)
            assert_close(got, ref, dt, f"split-K x{splits} BN=128 {pattern} {dt}", chain=chain)
        fl.device_status()
    finally:
        fl.set_option("variant", 0)
        fl.set_option("tile_n", 0)
        fl.set_option("split_k", 0)


@pytest.mark.parametrize("dt", DTYPES)
def test_splitk_wide_tiles_and_norm_bias_act(dt):
    M, N, K = 96, 392, 1536
    t = syn.norm_gemm_inputs(M, N, K, "layer", dt, with_bias=True)
    fl.set_option("variant", 2)
    fl.set_option("tile_n", 128)
    try:
        for norm in ("rms", "layer"):
            for act in ("gelu", "relu"):
                got = fl.norm_gemm(dev(t["x"]), dev(t["gamma"]), dev(t["W"]), beta=dev(t["beta"]),
                                   bias=dev(t["bias"]), eps=1e-5, norm=norm, act=act)
                torch.cuda.synchronize()
                args = (f64(t["x"]), f64(t["gamma"]), f64(t["beta"]), f64(t["W"]), f64(t["bias"]), 1e-5, norm, act)
                ref = oracle.norm_gemm(*args)
                assert_close(got, ref, dt, f"split-K BN=128 {norm} {act}", chain=parity.chain_norm_gemm(*args, dt))
    finally:
        fl.set_option("variant", 0)
        fl.set_option("tile_n", 0)


# ---------------------------------------------------------------------------
# the CTA-pair kernel (cta_group::2, 256 x 256 tiles on two SMs), forced
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("dt", DTYPES)
@pytest.mark.parametrize("tile_n", [128, 256])
@pytest.mark.parametrize("shape", [(1, 8, 8), (200, 136, 328), (300, 520, 1000), (512, 512, 512), (640, 264, 2056),
                                   (1536, 1280, 648)],
                         ids=lambda s: "x".join(map(str, s)))
def test_pair_variant_all_patterns(dt, tile_n, shape):
    """Includes a shape with several tiles per pair (persistent loop, buffer reuse)."""
    M, N, K = shape
    t = syn.dense_layer_inputs(M, N, K, dt)
    fl.set_option("variant", 3)
    fl.set_option("tile_n", tile_n)
    try:
        rows = sample_rows(M, n=384)
        for pattern in syn.PATTERNS:
            got, ref, chain = run_pattern(t, pattern, rows=rows)
            assert_close(got, ref, dt, f"pair BN={tile_n} {pattern} {dt} {M}x{N}x{K}", chain=chain)
        fl.device_status()
    finally:
        fl.set_option("variant", 0)
        fl.set_option("tile_n", 0)


@pytest.mark.parametrize("dt", DTYPES)
@pytest.mark.parametrize("shape", [(256, 256, 512), (300, 520, 1000), (512, 1024, 520), (777, 264, 4096)],
                         ids=lambda s: "x".join(map(str, s)))
def test_pair_split_k_all_patterns(dt, shape):
    """Two pairs per tile, one per K half, partials exchanged through distributed shared memory."""
    M, N, K = shape
    t = syn.dense_layer_inputs(M, N, K, dt)
    fl.set_option("variant", 3)
    fl.set_option("split_k", 2)
    try:
        for pattern in syn.PATTERNS:
            got, ref, chain = run_pattern(t, pattern)
            assert_close(got, ref, dt, f"pair split-K {pattern} {dt} {M}x{N}x{K}", chain=chain)
        fl.device_status()
    finally:
        fl.set_option("variant", 0)
        fl.set_option("split_k", 0)


@pytest.mark.parametrize("dt", DTYPES)
def test_pair_norm_bias_act_residual_alias(dt):
    M, N, K = 777, 520, 776
    t = syn.norm_gemm_inputs(M, N, K, "layer", dt, with_bias=True)
    fl.set_option("variant", 3)
    try:
        for norm in ("rms", "layer"):
            for act in ("silu", "gelu"):
                got = fl.norm_gemm(dev(t["x"]), dev(t["gamma"]), dev(t["W"]), beta=dev(t["beta"]),
                                   bias=dev(t["bias"]), eps=1e-5, norm=norm, act=act)
                torch.cuda.synchronize()
                args = (f64(t["x"]), f64(t["gamma"]), f64(t["beta"]), f64(t["W"]), f64(t["bias"]), 1e-5, norm, act)
                ref = oracle.norm_gemm(*args)
                assert_close(got, ref, dt, f"pair {norm} {act}", chain=parity.chain_norm_gemm(*args, dt))
        r = syn.gemm_inputs(M, N, K, "gemm_bias_residual", dt)
        res = dev(r["residual"])
        fl.gemm_epilogue(dev(r["A"]), dev(r["W"]), bias=dev(r["bias"]), residual=res, out=res,
                         pattern="gemm_bias_residual")
        torch.cuda.synchronize()
        ref = oracle.gemm_epilogue(f64(r["A"]), f64(r["W"]), f64(r["bias"]), f64(r["residual"]), "gemm_bias_residual")
        assert_close(res, ref, dt, "pair residual alias")
    finally:
        fl.set_option("variant", 0)


# ---------------------------------------------------------------------------
# the workloads of the pages, at full size
# ---------------------------------------------------------------------------
def test_gemm_bias_gelu_512x1024x1024_all_elements():
    """fp16 gemm_bias_gelu, A[512,1024], W[1024,1024], bias[1024], seed 0."""
    t = syn.gemm_inputs(512, 1024, 1024, "gemm_bias_gelu", "f16", seed=0)
    got, ref, chain = run_pattern(t, "gemm_bias_gelu")
    assert_close(got, ref, "f16", "gemm_bias_gelu 512x1024x1024", chain=chain)


def test_rmsnorm_gemm_512x4096x4096_all_elements():
    """fp16 rmsnorm_gemm, x[512,4096], gamma ~ N(1,0.1), eps 1e-6, W[4096,4096], no bias."""
    t = syn.gemm_inputs(512, 4096, 4096, "rmsnorm_gemm", "f16")
    got, ref, chain = run_pattern(t, "rmsnorm_gemm")
    assert_close(got, ref, "f16", "rmsnorm_gemm 512x4096x4096", chain=chain)


@pytest.mark.parametrize("dt", DTYPES)
@pytest.mark.parametrize("M", [512, 1024, 2048, 4096])
def test_nine_patterns_n4096_k4096_sampled_rows(dt, M):
    t = syn.dense_layer_inputs(M, 4096, 4096, dt)
    rows = sample_rows(M)
    for pattern in syn.PATTERNS:
        got, ref, chain = run_pattern(t, pattern, rows=rows)
        assert_close(got, ref, dt, f"{pattern} {dt} M={M}", chain=chain)
    fl.device_status()


def test_swiglu_ffn_4096x4096x11008_sampled_rows():
    """bf16 Llama-style FFN block: x[4096,4096], Wg/Wu[11008,4096], Wd[4096,11008], + x."""
    M, D, F = 4096, 4096, 11008
    t = syn.swiglu_inputs(M, D, F, "bf16")
    g = {k: dev(v) for k, v in t.items()}
    ws = torch.empty(fl.swiglu_ffn_workspace_size(M, F, torch.bfloat16), dtype=torch.uint8, device="cuda")
    got = fl.swiglu_ffn(g["x"], g["gamma"], g["Wg"], g["Wu"], g["Wd"], eps=1e-6, workspace=ws)
    torch.cuda.synchronize()
    rows = sample_rows(M, n=64)
    f = {k: f64(v) for k, v in t.items()}
    ref = oracle.swiglu_ffn(f["x"][rows], f["gamma"], f["Wg"], f["Wu"], f["Wd"], None, 1e-6, "bf16")
    chain = parity.chain_swiglu_ffn(f["x"][rows], f["gamma"], f["Wg"], f["Wu"], f["Wd"], None, 1e-6, "bf16")
    assert_close(got[rows], ref, "bf16", "swiglu 4096x4096x11008", chain=chain)
    # the workspace holds h: check it against the oracle's unrounded hidden activation too
    h = ws.view(torch.bfloat16).view(M, F)[rows]
    href = oracle.swiglu_hidden(f["x"][rows], f["gamma"], f["Wg"], f["Wu"], 1e-6)
    assert_close(h, href, "bf16", "swiglu hidden h")


@pytest.mark.parametrize("dt", DTYPES)
@pytest.mark.parametrize("with_bias", [False, True])
@pytest.mark.parametrize("shape", [(1, 64, 128), (136, 256, 384), (300, 264, 520)], ids=lambda s: "x".join(map(str, s)))
def test_swiglu_ffn_small_all_elements(dt, with_bias, shape):
    M, D, F = shape
    t = syn.swiglu_inputs(M, D, F, dt, with_bias=with_bias)
    g = {k: dev(v) for k, v in t.items()}
    got = fl.swiglu_ffn(g["x"], g["gamma"], g["Wg"], g["Wu"], g["Wd"], bias_down=g["bias_down"], eps=1e-6)
    torch.cuda.synchronize()
    f = {k: f64(v) for k, v in t.items()}
    ref = oracle.swiglu_ffn(f["x"], f["gamma"], f["Wg"], f["Wu"], f["Wd"], f["bias_down"], 1e-6, dt)
    chain = parity.chain_swiglu_ffn(f["x"], f["gamma"], f["Wg"], f["Wu"], f["Wd"], f["bias_down"], 1e-6, dt)
    assert_close(got, ref, dt, f"swiglu {dt} {shape}", chain=chain)


@pytest.mark.parametrize("dt", DTYPES)
@pytest.mark.parametrize("shape", [(1, 512, 1376), (3, 1024, 2816), (4, 4096, 11008), (8, 1024, 2816), (16, 1024, 2816),
                                   (77, 256, 3008), (128, 512, 1024), (32, 4096, 11008), (2, 264, 136)],
                         ids=lambda s: "x".join(map(str, s)))
def test_swiglu_ffn_decode_rows(dt, shape):
    """Decode row counts: up to 8 rows the gate/up pair and the down projection
    run on the decode kernel (where their rows fit in shared memory); up to 64 the gate/up GEMM is the split-K form
    with Wg and Wu in every stage (two accumulators exchanged together)."""
    M, D, F = shape
    t = syn.swiglu_inputs(M, D, F, dt, with_bias=M == 77)
    g = {k: dev(v) for k, v in t.items()}
    ws = torch.empty(fl.swiglu_ffn_workspace_size(M, F, dt), dtype=torch.uint8, device="cuda")
    got = fl.swiglu_ffn(g["x"], g["gamma"], g["Wg"], g["Wu"], g["Wd"], bias_down=g["bias_down"], eps=1e-6,
                        workspace=ws)
    torch.cuda.synchronize()
    fl.device_status()
    f = {k: f64(v) for k, v in t.items()}
    ref = oracle.swiglu_ffn(f["x"], f["gamma"], f["Wg"], f["Wu"], f["Wd"], f["bias_down"], 1e-6, dt)
    chain = parity.chain_swiglu_ffn(f["x"], f["gamma"], f["Wg"], f["Wu"], f["Wd"], f["bias_down"], 1e-6, dt)
    assert_close(got, ref, dt, f"swiglu decode {dt} {shape}", chain=chain)
    h = ws[:M * F * 2].view(torch.bfloat16 if dt == "bf16" else torch.float16).view(M, F)
    href = oracle.swiglu_hidden(f["x"], f["gamma"], f["Wg"], f["Wu"], 1e-6)
    assert_close(h, href, dt, f"swiglu decode hidden {dt} {shape}")


@pytest.mark.parametrize("dt", DTYPES)
@pytest.mark.parametrize("tile_n", [128, 256])
@pytest.mark.parametrize("splits", [1, 2, 3, 5, 8])
def test_swiglu_gate_up_split_k_forced(dt, tile_n, splits):
    """The split-K gate/up form at forced weight-tile widths (128; 256 selects 64)
    and cluster sizes, including uneven column slices."""
    M, D, F = 40, 2048, 1032
    t = syn.swiglu_inputs(M, D, F, dt)
    g = {k: dev(v) for k, v in t.items()}
    fl.set_option("tile_n", tile_n)
    fl.set_option("split_k", splits)
    try:
        got = fl.swiglu_ffn(g["x"], g["gamma"], g["Wg"], g["Wu"], g["Wd"], eps=1e-6)
        torch.cuda.synchronize()
        fl.device_status()
    finally:
        fl.set_option("tile_n", 0)
        fl.set_option("split_k", 0)
    f = {k: f64(v) for k, v in t.items()}
    ref = oracle.swiglu_ffn(f["x"], f["gamma"], f["Wg"], f["Wu"], f["Wd"], None, 1e-6, dt)
    assert_close(got, ref, dt, f"swiglu split-K gate/up {dt} BN={tile_n} x{splits}")


@pytest.mark.parametrize("dt", DTYPES)
@pytest.mark.parametrize("D", [1024, 2048, 4096])
@pytest.mark.parametrize("M", [1, 32, 128, 512, 1024])
def test_decode_sweep_rmsnorm_all_elements(dt, D, M):
    """rmsnorm_gemm with square W[D,D]: the decode-shape sweep of the LLMBoost page."""
    t = syn.norm_gemm_inputs(M, D, D, "rms", dt)
    got = fl.norm_gemm(dev(t["x"]), dev(t["gamma"]), dev(t["W"]), eps=1e-6, norm="rms")
    torch.cuda.synchronize()
    args = (f64(t["x"]), f64(t["gamma"]), None, f64(t["W"]), None, 1e-6, "rms", "none")
    ref = oracle.norm_gemm(*args)
    assert_close(got, ref, dt, f"decode rms {dt} M={M} D={D}", chain=parity.chain_norm_gemm(*args, dt))


@pytest.mark.parametrize("dt", DTYPES)
@pytest.mark.parametrize("with_bias", [False, True])
@pytest.mark.parametrize("shape", [(136, 256, 384), (300, 264, 520), (512, 128, 1024)], ids=lambda s: "x".join(map(str, s)))
def test_swiglu_ffn_on_cta_pairs(dt, with_bias, shape):
    """Gate/up on the CTA-pair kernel (Wg and Wu stacked in one weight tile), forced on small shapes."""
    M, D, F = shape
    t = syn.swiglu_inputs(M, D, F, dt, with_bias=with_bias)
    g = {k: dev(v) for k, v in t.items()}
    fl.set_option("variant", 3)
    try:
        got = fl.swiglu_ffn(g["x"], g["gamma"], g["Wg"], g["Wu"], g["Wd"], bias_down=g["bias_down"], eps=1e-6)
        torch.cuda.synchronize()
        fl.device_status()
    finally:
        fl.set_option("variant", 0)
    f = {k: f64(v) for k, v in t.items()}
    ref = oracle.swiglu_ffn(f["x"], f["gamma"], f["Wg"], f["Wu"], f["Wd"], f["bias_down"], 1e-6, dt)
    chain = parity.chain_swiglu_ffn(f["x"], f["gamma"], f["Wg"], f["Wu"], f["Wd"], f["bias_down"], 1e-6, dt)
    assert_close(got, ref, dt, f"swiglu pairs {dt} {shape}", chain=chain)


@pytest.mark.parametrize("dt", DTYPES)
@pytest.mark.parametrize("shape", [(200, 264, 520), (512, 512, 1024), (1, 128, 256)], ids=lambda s: "x".join(map(str, s)))
def test_layernorm_captured_in_cuda_graph(dt, shape):
    """LayerNorm takes stream-ordered scratch for its row statistics: it must
    capture into a CUDA graph and give the same result on every replay."""
    M, N, K = shape
    t = syn.norm_gemm_inputs(M, N, K, "layer", dt)
    g = {k: dev(v) for k, v in t.items()}
    out = torch.empty((M, N), dtype=g["x"].dtype, device="cuda")
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        fl.norm_gemm(g["x"], g["gamma"], g["W"], beta=g["beta"], out=out, eps=1e-5, norm="layer")
    torch.cuda.current_stream().wait_stream(side)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        fl.norm_gemm(g["x"], g["gamma"], g["W"], beta=g["beta"], out=out, eps=1e-5, norm="layer")
    ref = oracle.norm_gemm(f64(t["x"]), f64(t["gamma"]), f64(t["beta"]), f64(t["W"]), None, 1e-5, "layer")
    first = None
    for _ in range(3):
        out.zero_()
        graph.replay()
        torch.cuda.synchronize()
        assert_close(out, ref, dt, f"graph layernorm {dt} {shape}")
        if first is None:
            first = out.clone()
        else:
            assert torch.equal(out, first)
    fl.device_status()


@pytest.mark.parametrize("dt", DTYPES)
@pytest.mark.parametrize("M,D", [(1, 4096), (16, 1024), (32, 2048), (128, 1024)])
def test_weight_preload_chained_layers(dt, M, D):
    """Two decode layers back to back on one stream, the second reading the first's output.

    With weight preload the second kernel stages weight tiles before the first
    has finished; its activation (the first's output, overwritten with NaN by
    a kernel just before) must still be read after it.
    """
    t1 = syn.norm_gemm_inputs(M, D, D, "rms", dt, seed=11)
    t2 = syn.norm_gemm_inputs(M, D, D, "rms", dt, seed=12)
    g1 = {k: dev(v) for k, v in t1.items()}
    g2 = {k: dev(v) for k, v in t2.items()}
    fl.set_option("weight_preload", 1)
    try:
        y1 = torch.empty((M, D), dtype=g1["x"].dtype, device="cuda")
        for _ in range(3):
            y1.fill_(float("nan"))
            fl.norm_gemm(g1["x"], g1["gamma"], g1["W"], out=y1, eps=1e-6, norm="rms")
            y2 = fl.norm_gemm(y1, g2["gamma"], g2["W"], eps=1e-6, norm="rms")
        torch.cuda.synchronize()
        fl.device_status()
    finally:
        fl.set_option("weight_preload", 0)
    ref1 = oracle.norm_gemm(f64(t1["x"]), f64(t1["gamma"]), None, f64(t1["W"]), None, 1e-6, "rms")
    assert_close(y1, ref1, dt, f"preload layer 1 {dt} M={M} D={D}")
    ref2 = oracle.norm_gemm(f64(y1.cpu()), f64(t2["gamma"]), None, f64(t2["W"]), None, 1e-6, "rms")
    assert_close(y2, ref2, dt, f"preload layer 2 {dt} M={M} D={D}")


@pytest.mark.parametrize("dt", DTYPES)
@pytest.mark.parametrize("norm,M,D", [("rms", 512, 1024), ("rms", 4096, 2048), ("layer", 512, 1024),
                                      ("layer", 4096, 2048), (None, 512, 1024), (None, 4096, 2048)])
def test_weight_preload_chained_layers_on_cta_pairs(dt, norm, M, D):
    """The weight-preload promise on the CTA-pair kernel (one tile per K-split
    cluster at M=512, several tiles per pair at M=4096): two layers back to back,
    the second reading the first's output, which a kernel just before overwrites
    with NaN, so an activation read ahead of the dependency would show."""
    kind = norm or "plain"
    if norm is None:
        t1 = syn.gemm_inputs(M, D, D, "gemm_bias", dt, seed=21)
        t2 = syn.gemm_inputs(M, D, D, "gemm_bias", dt, seed=22)
        x1, W1, W2 = dev(t1["A"]), dev(t1["W"]), dev(t2["W"])
        b1, b2 = dev(t1["bias"]), dev(t2["bias"])
    else:
        t1 = syn.norm_gemm_inputs(M, D, D, norm, dt, seed=21)
        t2 = syn.norm_gemm_inputs(M, D, D, norm, dt, seed=22)
        x1, W1, W2 = dev(t1["x"]), dev(t1["W"]), dev(t2["W"])
        g1, g2, be1, be2 = dev(t1["gamma"]), dev(t2["gamma"]), dev(t1["beta"]), dev(t2["beta"])
    eps = 1e-5

    def layer(x, W, i, out=None):
        if norm is None:
            return fl.gemm_epilogue(x, W, bias=(b1, b2)[i], out=out, pattern="gemm_bias")
        return fl.norm_gemm(x, (g1, g2)[i], W, beta=(be1, be2)[i], out=out, eps=eps, norm=norm)

    fl.set_option("variant", 3)
    fl.set_option("weight_preload", 1)
    try:
        y1 = torch.empty((M, D), dtype=x1.dtype, device="cuda")
        for _ in range(3):
            y1.fill_(float("nan"))
            layer(x1, W1, 0, out=y1)
            y2 = layer(y1, W2, 1)
        torch.cuda.synchronize()
        fl.device_status()
    finally:
        fl.set_option("weight_preload", 0)
        fl.set_option("variant", 0)
    if norm is None:
        ref1 = oracle.gemm_epilogue(f64(t1["A"]), f64(t1["W"]), f64(t1["bias"]), None, "gemm_bias")
        ref2 = oracle.gemm_epilogue(f64(y1.cpu()), f64(t2["W"]), f64(t2["bias"]), None, "gemm_bias")
    else:
        ref1 = oracle.norm_gemm(f64(t1["x"]), f64(t1["gamma"]), f64(t1["beta"]), f64(t1["W"]), None, eps, norm)
        ref2 = oracle.norm_gemm(f64(y1.cpu()), f64(t2["gamma"]), f64(t2["beta"]), f64(t2["W"]), None, eps, norm)
    assert_close(y1, ref1, dt, f"pair preload layer 1 {kind} {dt} M={M} D={D}")
    assert_close(y2, ref2, dt, f"pair preload layer 2 {kind} {dt} M={M} D={D}")


# ---------------------------------------------------------------------------
# bounded waits
# ---------------------------------------------------------------------------
def test_bounded_wait_reports_timeout_and_context_survives():
    fl.device_status()  # clean slate
    fl.debug_wait_timeout(2000)  # a wait that nothing completes, 2 ms limit
    with pytest.raises(fl.FusedLinError) as e:
        fl.device_status()
    assert e.value.status == 6
    fl.device_status()  # cleared
    # the context still works
    t = syn.gemm_inputs(64, 64, 64, "gemm_bias", "f16")
    got, ref, chain = run_pattern(t, "gemm_bias")
    assert_close(got, ref, "f16", "after timeout", chain=chain)


def test_timeout_is_reported_on_its_own_stream_only():
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    for s in (None, s1, s2):
        fl.device_status(s)  # clean slate
    fl.debug_wait_timeout(2000, stream=s1)
    torch.cuda.synchronize()
    fl.device_status(s2)  # another stream's word stays clear
    fl.device_status()  # and so does the default stream's
    # a kernel on the other stream runs normally while s1's word is set
    t = syn.gemm_inputs(300, 512, 1024, "gemm_bias", "f16")
    A, W, b = dev(t["A"]), dev(t["W"]), dev(t["bias"])
    out = torch.empty(300, 512, dtype=torch.float16, device="cuda")
    s2.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s2):
        fl.gemm_epilogue(A, W, bias=b, out=out, pattern="gemm_bias", stream=s2)
    fl.device_status(s2)
    ref = oracle.gemm_epilogue(f64(t["A"]), f64(t["W"]), f64(t["bias"]), None, "gemm_bias")
    assert_close(out, ref, "f16", "other stream after a timeout")
    with pytest.raises(fl.FusedLinError) as e:
        fl.device_status(s1)
    assert e.value.status == 6
    fl.device_status(s1)  # read once, then clear
