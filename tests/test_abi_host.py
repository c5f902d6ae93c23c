"""The C ABI on the host (no GPU needed).

The library loads, exports every function include/fusedlin.h declares, and
rejects bad arguments with the documented status before touching CUDA.
"""
import ctypes
import os
import re

import pytest

import gemm_epilogue_tma_gb300 as fl
from gemm_epilogue_tma_gb300 import _build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
OK, INVALID, UNSUPPORTED, ALIGN, WORKSPACE, CUDA, TIMEOUT = range(7)


@pytest.fixture(scope="module")
def L():
    _build.build()
    return fl.lib()


def declared_functions():
    src = open(os.path.join(ROOT, "include", "fusedlin.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(fl_[a-z0-9_]+)\s*\(", src)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for n in ("fl_gemm_epilogue", "fl_norm_gemm", "fl_swiglu_ffn", "fl_swiglu_ffn_workspace_size",
              "fl_last_error", "fl_device_status"):
        assert n in names


def header_enum(type_name):
    """{enumerator: value} of `typedef enum { ... } type_name;` in include/fusedlin.h."""
    src = open(os.path.join(ROOT, "include", "fusedlin.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    body = re.search(r"typedef enum\s*\{([^}]*)\}\s*" + type_name + r"\s*;", src).group(1)
    return {k: int(v) for k, v in re.findall(r"(FL_[A-Z0-9_]+)\s*=\s*(\d+)", body)}


def test_binding_enums_match_header():
    pat = header_enum("fl_pattern")
    assert {k[3:].lower(): v for k, v in pat.items()} == {n: i for i, n in enumerate(fl.PATTERNS)}
    assert {k[len("FL_NORM_"):].lower(): v for k, v in header_enum("fl_norm_kind").items()} == fl.NORMS
    acts = {k[len("FL_ACT_"):].lower().replace("_tanh", ""): v for k, v in header_enum("fl_act").items()}
    assert acts == fl.ACTS
    assert {k[3:].lower(): v for k, v in header_enum("fl_dtype").items()} == fl.DTYPE_CODES
    assert {k[len("FL_OPT_"):].lower(): v for k, v in header_enum("fl_option").items()} == fl.OPTIONS


def test_every_declared_symbol_is_exported(L):
    for name in declared_functions():
        assert hasattr(L, name), name
        assert name in fl.SIGNATURES, f"binding lacks {name}"


def test_version(L):
    assert "sm_103a" in fl.version()


# Fake, well-aligned device addresses: validation never dereferences them, and
# every call below fails validation (or finds no device) before any launch.
BASE = 0x7F0000000000


def addr(i, off=0):
    return ctypes.c_void_p(BASE + i * (1 << 32) + off)


def gemm(L, A=addr(0), W=addr(1), bias=addr(2), res=addr(3), out=addr(4), M=64, N=64, K=64, p=0, dt=0):
    return L.fl_gemm_epilogue(A, W, bias, res, out, M, N, K, p, dt, None)


def test_gemm_epilogue_validation(L):
    assert gemm(L, A=None) == INVALID
    assert gemm(L, W=None) == INVALID
    assert gemm(L, out=None) == INVALID
    assert gemm(L, bias=None, p=0) == INVALID            # gemm_bias_gelu needs a bias
    assert gemm(L, res=None, p=4) == INVALID             # gemm_bias_residual needs a residual
    assert gemm(L, p=7) == INVALID and "fl_norm_gemm" in fl.last_error()
    assert gemm(L, p=8) == INVALID
    assert gemm(L, p=9) == INVALID and gemm(L, p=-1) == INVALID
    assert gemm(L, dt=2) == INVALID
    assert gemm(L, M=0) == INVALID and gemm(L, N=0) == INVALID and gemm(L, K=-8) == INVALID
    assert gemm(L, K=60) == ALIGN and gemm(L, N=12) == ALIGN
    assert gemm(L, A=addr(0, 8)) == ALIGN
    assert gemm(L, out=addr(4, 2)) == ALIGN
    assert gemm(L, bias=addr(2, 4)) == ALIGN
    # out overlapping an input; residual may alias out only exactly
    assert gemm(L, out=addr(0, 64)) == INVALID
    assert gemm(L, p=4, res=addr(4, 16)) == INVALID and "alias" in fl.last_error()
    # unused pointers are ignored (no bias for gemm_gelu, even misaligned)
    st = gemm(L, p=5, bias=addr(2, 3), res=addr(3, 1))
    assert st in (UNSUPPORTED, CUDA)  # reaches the device query: none on this machine


def test_valid_call_without_gpu_reports_unsupported(L):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    assert gemm(L) == UNSUPPORTED
    assert fl.last_error()
    assert gemm(L, p=4, res=addr(4)) == UNSUPPORTED  # exact alias of residual and out is allowed


def norm(L, x=addr(0), g=addr(1), b=addr(2), W=addr(3), bias=None, out=addr(4), M=64, N=64, K=64, eps=1e-6,
         nk=0, act=0, dt=0):
    return L.fl_norm_gemm(x, g, b, W, bias, out, M, N, K, eps, nk, act, dt, None)


def test_norm_gemm_validation(L):
    assert norm(L, x=None) == INVALID and norm(L, g=None) == INVALID and norm(L, W=None) == INVALID
    assert norm(L, nk=2) == INVALID and norm(L, act=4) == INVALID and norm(L, dt=-1) == INVALID
    assert norm(L, eps=-1.0) == INVALID and norm(L, eps=float("nan")) == INVALID
    assert norm(L, eps=float("inf")) == INVALID
    assert norm(L, K=20) == ALIGN
    assert norm(L, g=addr(1, 2)) == ALIGN
    assert norm(L, nk=1, b=addr(2, 2)) == ALIGN          # LayerNorm reads beta
    assert norm(L, nk=0, b=addr(2, 2)) != ALIGN          # RMS ignores beta
    assert norm(L, out=addr(3, 32)) == INVALID          # out overlaps W


def ffn(L, x=addr(0), g=addr(1), Wg=addr(2), Wu=addr(3), Wd=addr(4), bd=None, out=addr(5), M=16, D=64, F=128,
        eps=1e-6, ws=addr(6), wsb=None, dt=1):
    if wsb is None:
        wsb = M * F * 2
    return L.fl_swiglu_ffn(x, g, Wg, Wu, Wd, bd, out, M, D, F, eps, ws, wsb, dt, None)


def test_swiglu_validation(L):
    assert L.fl_swiglu_ffn_workspace_size(16, 128, 1) == 16 * 128 * 2
    assert L.fl_swiglu_ffn_workspace_size(1, 136, 0) == 136 * 2
    assert L.fl_swiglu_ffn_workspace_size(0, 128, 1) == 0
    assert ffn(L, ws=None) == WORKSPACE
    assert ffn(L, wsb=16 * 128 * 2 - 1) == WORKSPACE
    assert ffn(L, ws=addr(6, 8)) == ALIGN
    assert ffn(L, F=100) == ALIGN and ffn(L, D=36) == ALIGN
    assert ffn(L, Wu=None) == INVALID
    assert ffn(L, out=addr(0)) == INVALID               # out must not alias x
    assert ffn(L, ws=addr(5, 16)) == INVALID            # workspace overlaps out


def test_options(L):
    assert L.fl_set_option(0, 100) == INVALID
    assert L.fl_set_option(0, 256) == OK and L.fl_set_option(0, 0) == OK
    assert L.fl_set_option(1, 5) == INVALID and L.fl_set_option(1, 4) == OK and L.fl_set_option(1, 0) == OK
    assert L.fl_set_option(2, 0) == INVALID and L.fl_set_option(2, 2000) == OK
    assert L.fl_set_option(3, 9) == INVALID and L.fl_set_option(3, 0) == OK
    assert L.fl_set_option(4, 2) == INVALID and L.fl_set_option(4, 0) == OK and L.fl_set_option(4, 1) == OK
    assert L.fl_set_option(5, 2) == INVALID and L.fl_set_option(5, 1) == OK and L.fl_set_option(5, 0) == OK
    assert L.fl_set_option(42, 0) == INVALID
    assert L.fl_debug_wait_timeout(0, None) == INVALID


def test_binding_fails_loudly_without_library(monkeypatch, tmp_path):
    monkeypatch.setattr(fl, "_lib", None)
    monkeypatch.setattr(fl, "LIB_PATH", str(tmp_path / "missing.so"))
    with pytest.raises(ImportError):
        fl.lib()


def multi(L, x=addr(0), g=addr(1), b=None, n=3, Ws=None, biases=None, outs=None, Ns=None, acts=None, M=64, K=64,
          eps=1e-6, nk=0, dt=0):
    Ws = Ws if Ws is not None else [addr(10 + i) for i in range(n)]
    outs = outs if outs is not None else [addr(20 + i) for i in range(n)]
    Ns = Ns if Ns is not None else [64] * n
    arr = ctypes.c_void_p * max(n, 1)
    W_arr = arr(*Ws[:max(n, 1)]) if Ws else None
    o_arr = arr(*outs[:max(n, 1)]) if outs else None
    b_arr = arr(*biases) if biases is not None else None
    N_arr = (ctypes.c_int * max(n, 1))(*Ns[:max(n, 1)])
    a_arr = (ctypes.c_int * max(n, 1))(*acts) if acts is not None else None
    return L.fl_norm_gemm_multi(x, g, b, n, W_arr, b_arr, o_arr, N_arr, a_arr, M, K, eps, nk, dt, None)


def test_norm_gemm_multi_validation(L):
    assert multi(L, n=0) == INVALID and multi(L, n=5, Ws=[addr(10 + i) for i in range(5)],
                                              outs=[addr(20 + i) for i in range(5)], Ns=[64] * 5) == INVALID
    assert multi(L, x=None) == INVALID and multi(L, g=None) == INVALID
    assert multi(L, Ws=[addr(10), None, addr(12)]) == INVALID
    assert multi(L, outs=[addr(20), addr(21), None]) == INVALID
    assert multi(L, Ns=[64, 60, 64]) == ALIGN
    assert multi(L, Ns=[64, 0, 64]) == INVALID
    assert multi(L, acts=[0, 4, 0]) == INVALID
    assert multi(L, nk=3) == INVALID and multi(L, dt=2) == INVALID and multi(L, eps=-1.0) == INVALID
    assert multi(L, biases=[None, addr(30, 2), None]) == ALIGN
    # outputs overlapping each other or an input
    assert multi(L, outs=[addr(20), addr(20, 64), addr(22)]) == INVALID and "out[" in fl.last_error()
    assert multi(L, outs=[addr(20), addr(11), addr(22)]) == INVALID   # out[1] is W[1]
    assert multi(L, outs=[addr(0, 32), addr(21), addr(22)]) == INVALID  # out[0] overlaps x
    st = multi(L)  # valid: reaches the device query
    assert st in (OK, UNSUPPORTED, CUDA)


def test_input_bias_gemm_validation(L):
    def call(A=addr(0), bi=addr(1), W=addr(2), bias=None, res=None, out=addr(4), M=64, N=64, K=64, act=0, dt=0):
        return L.fl_input_bias_gemm(A, bi, W, bias, res, out, M, N, K, act, dt, None)
    assert call(A=None) == INVALID and call(bi=None) == INVALID and call(W=None) == INVALID
    assert call(out=None) == INVALID and call(act=5) == INVALID and call(dt=3) == INVALID
    assert call(K=12) == ALIGN and call(bi=addr(1, 2)) == ALIGN
    assert call(out=addr(2, 16)) == INVALID                   # out overlaps W
    assert call(res=addr(4, 16)) == INVALID and "alias" in fl.last_error()
    assert call(res=addr(4)) in (OK, UNSUPPORTED, CUDA)        # exact alias allowed


def test_rms_norm_validation(L):
    def call(x=addr(0), g=addr(1), out=addr(2), M=4, K=64, eps=1e-6, dt=0):
        return L.fl_rms_norm(x, g, out, M, K, eps, dt, None)
    assert call(x=None) == INVALID and call(g=None) == INVALID and call(out=None) == INVALID
    assert call(M=0) == INVALID and call(K=0) == INVALID and call(K=20) == ALIGN
    assert call(eps=float("nan")) == INVALID and call(dt=5) == INVALID
    assert call(out=addr(0, 16)) == INVALID                    # partial overlap with x
    assert call(out=addr(1)) == INVALID                        # out overlaps gamma
    assert call(out=addr(0)) in (OK, UNSUPPORTED, CUDA)        # in place


def test_layer_create_validation(L):
    names = fl.DecoderLayer.NAMES

    def desc(**over):
        d = fl.LayerDesc(dtype=0, M=4, D=64, Dkv=32, F=128, eps=1e-6,
                         **{n: BASE + i * (1 << 32) for i, n in enumerate(names)})
        d.bias_o = None
        for k, v in over.items():
            setattr(d, k, v)
        return d

    h = ctypes.c_void_p(1234)
    assert L.fl_layer_create(None, ctypes.byref(h)) == INVALID and not h.value
    assert L.fl_layer_create(ctypes.byref(desc(dtype=3)), ctypes.byref(h)) == INVALID
    assert L.fl_layer_create(ctypes.byref(desc(M=0)), ctypes.byref(h)) == INVALID
    assert L.fl_layer_create(ctypes.byref(desc(Dkv=20)), ctypes.byref(h)) == ALIGN
    assert L.fl_layer_create(ctypes.byref(desc(Wo=None)), ctypes.byref(h)) == INVALID
    assert L.fl_layer_create(ctypes.byref(desc(q=BASE + 8)), ctypes.byref(h)) == ALIGN
    assert L.fl_layer_create(ctypes.byref(desc(eps=-1.0)), ctypes.byref(h)) == INVALID
    d = desc()
    d.h = d.x
    assert L.fl_layer_create(ctypes.byref(d), ctypes.byref(h)) == INVALID
    assert not h.value
    assert L.fl_layer_issue(None, 0, None) == INVALID
    L.fl_layer_destroy(None)  # no-op
    assert L.fl_graph_launch(None, None) == INVALID
    assert L.fl_capture_end(None, None) == INVALID
    L.fl_graph_destroy(None)  # no-op


def test_kernel_launch_counter_on_the_host(L):
    # no GPU work was issued through this process's rejected calls: the
    # counter only moves on successful launches
    n = ctypes.c_longlong(-1)
    assert L.fl_kernel_launches(ctypes.byref(n)) == OK and n.value >= 0
    before = n.value
    assert L.fl_gemm_epilogue(None, None, None, None, None, 0, 0, 0, 0, 0, None) != OK
    assert L.fl_kernel_launches(ctypes.byref(n)) == OK and n.value == before
    assert L.fl_kernel_launches(None) == INVALID
