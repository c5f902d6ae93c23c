"""The host-side launch cache (needs an sm_103a GPU): a repeated call reuses
its prepared launch, gives the same bits as a call prepared afresh, and a call
that differs in any pointer, size or option gets its own entry."""
import pytest
import torch

import gemm_epilogue_tma_gb300 as fl
import oracle
from gemm_epilogue_tma_gb300 import _build
from gemm_epilogue_tma_gb300 import synthetic as syn
from parity import assert_close

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def library():
    _build.build()
    fl.lib()
    torch.cuda.set_device(0)
    yield
    fl.set_option("launch_cache", 1)
    fl.set_option("variant", 0)


def f64(t):
    return syn.as_f64(t)


@pytest.mark.parametrize("norm", ["rms", "layer"])
@pytest.mark.parametrize("M", [16, 300])
def test_repeated_calls_hit_and_match_uncached(norm, M):
    N, K = 520, 1000
    t = syn.norm_gemm_inputs(M, N, K, norm, "bf16", with_bias=True)
    g = {k: (v.cuda() if v is not None else None) for k, v in t.items()}
    out = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")

    def call(o):
        return fl.norm_gemm(g["x"], g["gamma"], g["W"], beta=g["beta"], bias=g["bias"], out=o, eps=1e-5, norm=norm)

    fl.launch_cache_clear()
    h0, m0 = fl.launch_cache_stats()
    call(out)
    first = out.clone()
    for _ in range(3):
        out.zero_()
        call(out)
        torch.cuda.synchronize()
        assert torch.equal(out, first)
    h1, m1 = fl.launch_cache_stats()
    assert m1 - m0 == 1 and h1 - h0 == 3
    # prepared afresh: the same bits
    fl.set_option("launch_cache", 0)
    try:
        fresh = torch.empty_like(out)
        call(fresh)
        torch.cuda.synchronize()
    finally:
        fl.set_option("launch_cache", 1)
    assert torch.equal(fresh, first)
    ref = oracle.norm_gemm(f64(t["x"]), f64(t["gamma"]), f64(t["beta"]), f64(t["W"]), f64(t["bias"]), 1e-5, norm)
    assert_close(first, ref, "bf16", f"cached {norm} M={M}")
    fl.device_status()


def test_changed_pointer_or_option_is_a_new_entry():
    M, N, K = 200, 264, 520
    t = syn.gemm_inputs(M, N, K, "gemm_bias_gelu", "f16")
    A, W, b = t["A"].cuda(), t["W"].cuda(), t["bias"].cuda()
    o1 = torch.empty((M, N), dtype=torch.float16, device="cuda")
    o2 = torch.empty_like(o1)
    fl.launch_cache_clear()
    h0, m0 = fl.launch_cache_stats()
    fl.gemm_epilogue(A, W, bias=b, out=o1, pattern="gemm_bias_gelu")
    fl.gemm_epilogue(A, W, bias=b, out=o2, pattern="gemm_bias_gelu")   # other output: miss
    fl.set_option("variant", 2)
    try:
        o3 = fl.gemm_epilogue(A, W, bias=b, pattern="gemm_bias_gelu")  # other option: miss
    finally:
        fl.set_option("variant", 0)
    fl.gemm_epilogue(A, W, bias=b, out=o1, pattern="gemm_bias_gelu")   # repeat: hit
    torch.cuda.synchronize()
    h1, m1 = fl.launch_cache_stats()
    assert (h1 - h0, m1 - m0) == (1, 3)
    ref = oracle.gemm_epilogue(f64(t["A"]), f64(t["W"]), f64(t["bias"]), None, "gemm_bias_gelu")
    for o in (o1, o2, o3):
        assert_close(o, ref, "f16", "cache entries")
