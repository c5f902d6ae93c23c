"""fl_swiglu_ffn_noalloc: the FFN block for callers that may not allocate.

Some callers may not allocate device memory when they call the library (an
engine or plugin that owns a fixed memory budget). This entry point keeps the
FFN's hidden activation in a fixed array of the library instead of a
caller-provided workspace. It runs the same kernels as fl_swiglu_ffn with
only the location of h changed, so its results must equal fl_swiglu_ffn's
bit for bit, call after call, whatever the previous call left in the array.

The file sorts last so that a run stopping at its first failure has already
run every other test.
"""
import ctypes

import pytest
import torch

import gemm_epilogue_tma_gb300 as fl
import oracle
from gemm_epilogue_tma_gb300 import _build
from gemm_epilogue_tma_gb300 import synthetic as syn
from parity import assert_close

INVALID_ARG = 1
WORKSPACE = 4
LIMIT = 8 << 20


@pytest.fixture(scope="module")
def L():
    _build.build()
    return fl.lib()


def test_rejects_sizes_beyond_the_fixed_array(L):
    """Checked on the host before any device work: runs without a GPU too."""
    M, F = 512, 8200  # 8.4 MB of h > 8 MiB
    assert M * F * 2 > LIMIT
    p = ctypes.c_void_p(0x7F0000000000)
    st = L.fl_swiglu_ffn_noalloc(p, p, p, p, p, None, p, M, 64, F, 1e-6, 1, None)
    assert st == WORKSPACE
    assert "fixed" in fl.last_error()


def test_rejects_bad_arguments_before_any_device_call(L):
    """Null pointers, empty sizes and a bad dtype fail on the host (no GPU needed)."""
    p = ctypes.c_void_p(0x7F0000000000)
    assert L.fl_swiglu_ffn_noalloc(p, p, p, p, p, None, None, 4, 64, 64, 1e-6, 1, None) == INVALID_ARG
    assert L.fl_swiglu_ffn_noalloc(p, p, p, p, p, None, p, 0, 64, 64, 1e-6, 1, None) == INVALID_ARG
    assert L.fl_swiglu_ffn_noalloc(p, p, p, p, p, None, p, 4, 64, 0, 1e-6, 1, None) == INVALID_ARG
    assert L.fl_swiglu_ffn_noalloc(p, p, p, p, p, None, p, 4, 64, 64, 1e-6, 7, None) == INVALID_ARG


def _both(M, D, F, dt, bias):
    t = syn.swiglu_inputs(M, D, F, dt, with_bias=bias)
    g = {k: (v.cuda() if v is not None else None) for k, v in t.items()}
    ws = torch.empty(fl.swiglu_ffn_workspace_size(M, F, dt), dtype=torch.uint8, device="cuda")
    ref = fl.swiglu_ffn(g["x"], g["gamma"], g["Wg"], g["Wu"], g["Wd"], bias_down=g["bias_down"], eps=1e-6,
                        workspace=ws)
    got = fl.swiglu_ffn_noalloc(g["x"], g["gamma"], g["Wg"], g["Wu"], g["Wd"], bias_down=g["bias_down"], eps=1e-6)
    torch.cuda.synchronize()
    fl.device_status()
    return t, got, ref


@pytest.mark.gpu
def test_matches_workspace_entry_point_on_two_calls_in_a_row(L):
    torch.cuda.set_device(0)
    # the second call is smaller than the first, so stale h from call one sits
    # in the array around call two's h
    for (M, D, F, dt, bias) in [(300, 512, 1024, "bf16", True), (96, 256, 512, "f16", False)]:
        t, got, ref = _both(M, D, F, dt, bias)
        assert torch.equal(got, ref), (M, D, F, dt)
        f = {k: syn.as_f64(v) for k, v in t.items()}
        want = oracle.swiglu_ffn(f["x"], f["gamma"], f["Wg"], f["Wu"], f["Wd"], f["bias_down"], 1e-6, dt)
        assert_close(got, want, dt, f"noalloc swiglu {dt} {M}x{D}x{F}")


@pytest.mark.gpu
def test_call_at_the_size_limit(L):
    """h of exactly 8 MiB (M * F * 2 = 8 MiB) fits and matches the workspace entry point."""
    torch.cuda.set_device(0)
    M, D, F = 512, 256, 8192
    assert M * F * 2 == LIMIT
    _, got, ref = _both(M, D, F, "bf16", False)
    assert torch.equal(got, ref)
