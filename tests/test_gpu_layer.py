"""The decoder layer's dense part (fl_layer_*) and graph capture of library
calls (fl_capture_*), against the float64 oracle (needs an sm_103a GPU).

Each stage is compared with the oracle on the tensors it reads: q, k, v with
oracle.norm_gemm of x; h with attn Wo^T (+ bias) + x; out with
oracle.swiglu_ffn of the layer's own h (h is stored in the dtype between the
two halves, so it is the exact input of the FFN). A captured graph of two
chained layers must equal the same calls issued directly, bit for bit, and a
replay after x is rewritten in place must follow the new x.
"""
import numpy as np
import pytest
import torch

import gemm_epilogue_tma_gb300 as fl
import oracle
from gemm_epilogue_tma_gb300 import _build
from gemm_epilogue_tma_gb300 import synthetic as syn
from parity import assert_close, sample_rows

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def library():
    _build.build()
    fl.lib()
    torch.cuda.set_device(0)
    yield
    fl.device_status()


def f64(t):
    return syn.as_f64(t.cpu())


def make_layer(M, D, Dkv, F, dt, with_bias, seed=0):
    rng = syn.rng_for(43, seed, syn.DTYPE_IDS[dt], M, D, Dkv, F)
    draw = lambda shape, mean, std: syn._draw(rng, shape, mean, std, dt).cuda()
    T = {"x": draw((M, D), 0.0, 1.0), "gamma_attn": draw((D,), 1.0, 0.1),
         "Wq": draw((D, D), 0.0, 1 / np.sqrt(D)), "Wk": draw((Dkv, D), 0.0, 1 / np.sqrt(D)),
         "Wv": draw((Dkv, D), 0.0, 1 / np.sqrt(D)), "attn": draw((M, D), 0.0, 1.0),
         "Wo": draw((D, D), 0.0, 1 / np.sqrt(D)), "bias_o": draw((D,), 0.0, 0.1) if with_bias else None,
         "gamma_ffn": draw((D,), 1.0, 0.1), "Wg": draw((F, D), 0.0, 1 / np.sqrt(D)),
         "Wu": draw((F, D), 0.0, 1 / np.sqrt(D)), "Wd": draw((D, F), 0.0, 1 / np.sqrt(F))}
    dtype = T["x"].dtype
    for name, shape in (("q", (M, D)), ("k", (M, Dkv)), ("v", (M, Dkv)), ("h", (M, D)), ("out", (M, D))):
        T[name] = torch.empty(shape, dtype=dtype, device="cuda")
    return T


def check_layer(T, dt, rows, what):
    x, attn = f64(T["x"])[rows], f64(T["attn"])[rows]
    for name in ("q", "k", "v"):
        W = {"q": "Wq", "k": "Wk", "v": "Wv"}[name]
        ref = oracle.norm_gemm(x, f64(T["gamma_attn"]), None, f64(T[W]), None, 1e-6, "rms")
        assert_close(T[name][rows], ref, dt, f"{what} {name}")
    bias = np.zeros(x.shape[1]) if T["bias_o"] is None else f64(T["bias_o"])
    href = oracle.gemm_epilogue(attn, f64(T["Wo"]), bias, x, "gemm_bias_residual")
    assert_close(T["h"][rows], href, dt, f"{what} h")
    h = f64(T["h"])[rows]
    oref = oracle.swiglu_ffn(h, f64(T["gamma_ffn"]), f64(T["Wg"]), f64(T["Wu"]), f64(T["Wd"]), None, 1e-6, dt)
    assert_close(T["out"][rows], oref, dt, f"{what} out")


@pytest.mark.parametrize("dt", ["f16", "bf16"])
@pytest.mark.parametrize("shape", [(1, 1024, 256, 2816), (32, 4096, 1024, 11008), (200, 512, 128, 1376)],
                         ids=lambda s: "x".join(map(str, s)))
def test_layer_stack_graph_matches_oracle_and_direct_calls(dt, shape):
    M, D, Dkv, F = shape
    T = make_layer(M, D, Dkv, F, dt, with_bias=M == 200)
    # a second layer reading the first one's output, with its own buffers
    T2 = dict(T)
    dtype = T["x"].dtype
    T2["x"] = T["out"]
    for name, shp in (("q", (M, D)), ("k", (M, Dkv)), ("v", (M, Dkv)), ("h", (M, D)), ("out", (M, D))):
        T2[name] = torch.empty(shp, dtype=dtype, device="cuda")
    layers = [fl.DecoderLayer(eps=1e-6, **T), fl.DecoderLayer(eps=1e-6, **T2)]
    names = ("q", "k", "v", "h", "out")
    graph = None
    try:
        def step():
            for layer in layers:
                layer.issue(0)
                layer.issue(1)

        step()
        torch.cuda.synchronize()
        fl.device_status()
        rows = sample_rows(M, n=64)
        check_layer(T, dt, rows, f"layer 1 {dt} {shape}")
        check_layer(T2, dt, rows, f"layer 2 {dt} {shape}")
        direct = [{n: t[n].clone() for n in names} for t in (T, T2)]
        # one graph of both layers (captured on a side stream: the legacy
        # default stream cannot be captured): the same bits
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            graph = fl.Graph.capture(step)
        torch.cuda.current_stream().wait_stream(side)
        for t in (T, T2):
            for n in names:
                t[n].zero_()
        graph.launch()
        torch.cuda.synchronize()
        for t, d in zip((T, T2), direct):
            for n in names:
                assert torch.equal(t[n], d[n]), n
        # new x written in place: the replay follows it
        T["x"].copy_(T["x"].flip(0) * 0.5)
        graph.launch()
        torch.cuda.synchronize()
        check_layer(T, dt, rows, f"layer 1 replay {dt} {shape}")
        check_layer(T2, dt, rows, f"layer 2 replay {dt} {shape}")
    finally:
        if graph is not None:
            graph.close()
        for layer in layers:
            layer.close()
