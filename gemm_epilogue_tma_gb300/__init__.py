"""Python binding of libfusedlin, the fused transformer dense layer for GB300.

Argument marshalling only: every step of the computation runs in the CUDA
kernels of libfusedlin.so (built in-tree by gemm_epilogue_tma_gb300._build).
PyTorch supplies device memory and the current stream. If the library is
missing, every call raises; there is no fallback path.

Entry points mirror the C ABI declared in include/fusedlin.h:
    gemm_epilogue(A, W, bias, residual, out, pattern)   seven GEMM-first patterns
    norm_gemm(x, gamma, W, beta, bias, out, eps, norm, act)
    norm_gemm_multi(x, gamma, Ws, beta, biases, outs, acts, eps, norm)   one norm, several weights
    input_bias_gemm(A, bias_in, W, bias, residual, out, act)             (A + bias_in) W^T epilogue
    rms_norm(x, gamma, out, eps)                                          standalone RMSNorm
    swiglu_ffn(x, gamma, Wg, Wu, Wd, bias_down, out, eps, workspace)
"""
from __future__ import annotations

import ctypes
import os

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libfusedlin.so")

PATTERNS = (
    "gemm_bias_gelu", "gemm_bias_silu", "gemm_bias_relu", "gemm_bias", "gemm_bias_residual",
    "gemm_gelu", "gemm_silu", "layernorm_gemm", "rmsnorm_gemm",
)
NORMS = {"rms": 0, "layer": 1}
ACTS = {"none": 0, "gelu": 1, "silu": 2, "relu": 3}
DTYPE_CODES = {"f16": 0, "bf16": 1}
STATUS_NAMES = {0: "FL_OK", 1: "FL_ERR_INVALID_ARG", 2: "FL_ERR_UNSUPPORTED", 3: "FL_ERR_ALIGNMENT",
                4: "FL_ERR_WORKSPACE", 5: "FL_ERR_CUDA", 6: "FL_ERR_TIMEOUT"}
OPTIONS = {"tile_n": 0, "variant": 1, "timeout_ms": 2, "split_k": 3, "pdl": 4, "weight_preload": 5,
           "launch_cache": 6}

class LayerDesc(ctypes.Structure):
    """fl_layer_desc: sizes, dtype, eps and the device pointers of one decoder layer's dense part."""
    _fields_ = [("dtype", ctypes.c_int), ("M", ctypes.c_int), ("D", ctypes.c_int), ("Dkv", ctypes.c_int),
                ("F", ctypes.c_int), ("eps", ctypes.c_float)] + [
        (name, ctypes.c_void_p) for name in ("x", "gamma_attn", "Wq", "Wk", "Wv", "q", "k", "v", "attn", "Wo",
                                             "bias_o", "h", "gamma_ffn", "Wg", "Wu", "Wd", "out")]


# C ABI: name -> (restype, argtypes)
_vp, _i, _f, _sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
SIGNATURES = {
    "fl_gemm_epilogue": (_i, [_vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _vp]),
    "fl_norm_gemm": (_i, [_vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _i, _f, _i, _i, _i, _vp]),
    "fl_swiglu_ffn_workspace_size": (_sz, [_i, _i, _i]),
    "fl_swiglu_ffn": (_i, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _i, _f, _vp, _sz, _i, _vp]),
    "fl_swiglu_ffn_noalloc": (_i, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _i, _f, _i, _vp]),
    "fl_norm_gemm_multi": (_i, [_vp, _vp, _vp, _i, _vp, _vp, _vp, _vp, _vp, _i, _i, _f, _i, _i, _vp]),
    "fl_input_bias_gemm": (_i, [_vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _vp]),
    "fl_rms_norm": (_i, [_vp, _vp, _vp, _i, _i, _f, _i, _vp]),
    "fl_layer_create": (_i, [ctypes.POINTER(LayerDesc), ctypes.POINTER(_vp)]),
    "fl_layer_issue": (_i, [_vp, _i, _vp]),
    "fl_layer_destroy": (None, [_vp]),
    "fl_capture_begin": (_i, [_vp]),
    "fl_capture_end": (_i, [_vp, ctypes.POINTER(_vp)]),
    "fl_graph_launch": (_i, [_vp, _vp]),
    "fl_graph_destroy": (None, [_vp]),
    "fl_launch_cache_stats": (_i, [ctypes.POINTER(ctypes.c_longlong), ctypes.POINTER(ctypes.c_longlong)]),
    "fl_launch_cache_clear": (None, []),
    "fl_kernel_launches": (_i, [ctypes.POINTER(ctypes.c_longlong)]),
    "fl_last_error": (ctypes.c_char_p, []),
    "fl_device_status": (_i, [_vp]),
    "fl_set_option": (_i, [_i, _i]),
    "fl_debug_wait_timeout": (_i, [_i, _vp]),
    "fl_version": (ctypes.c_char_p, []),
}


class FusedLinError(RuntimeError):
    """A libfusedlin call returned a non-OK status."""

    def __init__(self, status: int, message: str):
        super().__init__(f"{STATUS_NAMES.get(status, status)}: {message}")
        self.status = status


_lib = None


def lib() -> ctypes.CDLL:
    """The loaded library (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError(f"{LIB_PATH} is missing: build it with "
                              "`python -m gemm_epilogue_tma_gb300._build` (needs nvcc)")
        handle = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(handle, name)
            fn.restype, fn.argtypes = res, args
        _lib = handle
    return _lib


def last_error() -> str:
    return lib().fl_last_error().decode()


def version() -> str:
    return lib().fl_version().decode()


def _check(status: int) -> None:
    if status != 0:
        raise FusedLinError(status, last_error())


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _dtype_code(t) -> int:
    import torch
    if t.dtype == torch.float16:
        return 0
    if t.dtype == torch.bfloat16:
        return 1
    raise TypeError(f"libfusedlin computes on fp16 or bf16 tensors, got {t.dtype}")


def _check_tensors(dt_ref, **tensors):
    for name, t in tensors.items():
        if t is None:
            continue
        if not t.is_cuda:
            raise ValueError(f"{name} must be a CUDA tensor")
        if not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous (row-major)")
        if t.dtype != dt_ref:
            raise TypeError(f"{name} has dtype {t.dtype}, expected {dt_ref}")


def gemm_epilogue(A, W, bias=None, residual=None, out=None, pattern="gemm_bias_gelu", stream=None):
    """out[M,N] = epilogue(A[M,K] W[N,K]^T) for a GEMM-first pattern name or enum value."""
    import torch
    p = PATTERNS.index(pattern) if isinstance(pattern, str) else int(pattern)
    M, K = A.shape
    N = W.shape[0]
    if W.shape[1] != K:
        raise ValueError(f"W has shape {tuple(W.shape)}, expected [N, {K}]")
    if out is None:
        out = torch.empty((M, N), dtype=A.dtype, device=A.device)
    _check_tensors(A.dtype, A=A, W=W, bias=bias, residual=residual, out=out)
    _check(lib().fl_gemm_epilogue(_ptr(A), _ptr(W), _ptr(bias), _ptr(residual), _ptr(out), M, N, K, p,
                                  _dtype_code(A), _stream(stream)))
    return out


def norm_gemm(x, gamma, W, beta=None, bias=None, out=None, eps=1e-6, norm="rms", act="none", stream=None):
    """out[M,N] = act(norm(x)[M,K] W[N,K]^T + bias); norm "rms" or "layer"."""
    import torch
    M, K = x.shape
    N = W.shape[0]
    if W.shape[1] != K:
        raise ValueError(f"W has shape {tuple(W.shape)}, expected [N, {K}]")
    if out is None:
        out = torch.empty((M, N), dtype=x.dtype, device=x.device)
    _check_tensors(x.dtype, x=x, gamma=gamma, W=W, beta=beta, bias=bias, out=out)
    _check(lib().fl_norm_gemm(_ptr(x), _ptr(gamma), _ptr(beta), _ptr(W), _ptr(bias), _ptr(out), M, N, K,
                              float(eps), NORMS[norm], ACTS[act], _dtype_code(x), _stream(stream)))
    return out


MAX_OUTPUTS = 4


def norm_gemm_multi(x, gamma, Ws, beta=None, biases=None, outs=None, acts=None, eps=1e-6, norm="rms", stream=None):
    """outs[i][M,N_i] = act_i(norm(x) Ws[i]^T + biases[i]) for every weight in one launch."""
    import torch
    n = len(Ws)
    if not 1 <= n <= MAX_OUTPUTS:
        raise ValueError(f"1..{MAX_OUTPUTS} weights, got {n}")
    M, K = x.shape
    for i, W in enumerate(Ws):
        if W.shape[1] != K:
            raise ValueError(f"Ws[{i}] has shape {tuple(W.shape)}, expected [N, {K}]")
    if outs is None:
        outs = [torch.empty((M, W.shape[0]), dtype=x.dtype, device=x.device) for W in Ws]
    biases = list(biases) if biases is not None else [None] * n
    acts = list(acts) if acts is not None else ["none"] * n
    if len(outs) != n or len(biases) != n or len(acts) != n:
        raise ValueError("Ws, outs, biases and acts must have the same length")
    _check_tensors(x.dtype, x=x, gamma=gamma, beta=beta,
                   **{f"W{i}": W for i, W in enumerate(Ws)}, **{f"out{i}": o for i, o in enumerate(outs)},
                   **{f"bias{i}": b for i, b in enumerate(biases)})
    arr = ctypes.c_void_p * n
    W_arr = arr(*[W.data_ptr() for W in Ws])
    b_arr = arr(*[(b.data_ptr() if b is not None else None) for b in biases])
    o_arr = arr(*[o.data_ptr() for o in outs])
    N_arr = (ctypes.c_int * n)(*[W.shape[0] for W in Ws])
    a_arr = (ctypes.c_int * n)(*[ACTS[a] for a in acts])
    _check(lib().fl_norm_gemm_multi(_ptr(x), _ptr(gamma), _ptr(beta), n, W_arr, b_arr, o_arr, N_arr, a_arr, M, K,
                                    float(eps), NORMS[norm], _dtype_code(x), _stream(stream)))
    return outs


def input_bias_gemm(A, bias_in, W, bias=None, residual=None, out=None, act="none", stream=None):
    """out[M,N] = act((A + bias_in) W^T + bias) (+ residual); bias_in runs along K."""
    import torch
    M, K = A.shape
    N = W.shape[0]
    if W.shape[1] != K:
        raise ValueError(f"W has shape {tuple(W.shape)}, expected [N, {K}]")
    if out is None:
        out = torch.empty((M, N), dtype=A.dtype, device=A.device)
    _check_tensors(A.dtype, A=A, bias_in=bias_in, W=W, bias=bias, residual=residual, out=out)
    _check(lib().fl_input_bias_gemm(_ptr(A), _ptr(bias_in), _ptr(W), _ptr(bias), _ptr(residual), _ptr(out), M, N,
                                    K, ACTS[act], _dtype_code(A), _stream(stream)))
    return out


def rms_norm(x, gamma, out=None, eps=1e-6, stream=None):
    """out[M,K] = x * gamma / sqrt(mean(x^2) + eps), rounded once (out may be x)."""
    import torch
    M, K = x.shape
    if out is None:
        out = torch.empty_like(x)
    _check_tensors(x.dtype, x=x, gamma=gamma, out=out)
    _check(lib().fl_rms_norm(_ptr(x), _ptr(gamma), _ptr(out), M, K, float(eps), _dtype_code(x), _stream(stream)))
    return out


class DecoderLayer:
    """The dense part of a decoder layer as a prepared call sequence (fl_layer_*).

    half 0: q, k, v = RMSNorm(x) [Wq; Wk; Wv]^T; the caller's attention then
    writes attn; half 1: h = attn Wo^T (+ bias_o) + x, out = SwiGLU_FFN(h) + h.
    Every tensor is fixed for the life of the layer: write new inputs into x
    and attn in place. Capture whole steps with Graph.capture().
    """

    NAMES = ("x", "gamma_attn", "Wq", "Wk", "Wv", "q", "k", "v", "attn", "Wo", "bias_o", "h", "gamma_ffn", "Wg",
             "Wu", "Wd", "out")

    def __init__(self, eps=1e-6, **tensors):
        x = tensors["x"]
        M, D = x.shape
        F = tensors["Wg"].shape[0]
        Dkv = tensors["Wk"].shape[0]
        _check_tensors(x.dtype, **tensors)
        self.tensors = tensors  # keep every buffer alive while the graphs exist
        desc = LayerDesc(dtype=_dtype_code(x), M=M, D=D, Dkv=Dkv, F=F, eps=float(eps),
                         **{n: (tensors[n].data_ptr() if tensors.get(n) is not None else None) for n in self.NAMES})
        h = ctypes.c_void_p()
        _check(lib().fl_layer_create(ctypes.byref(desc), ctypes.byref(h)))
        self._h = h

    def issue(self, half: int, stream=None) -> None:
        """Issue half 0 or 1 on the stream (capturable)."""
        _check(lib().fl_layer_issue(self._h, int(half), _stream(stream)))

    def close(self) -> None:
        if getattr(self, "_h", None):
            lib().fl_layer_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


class Graph:
    """A CUDA graph of library calls (fl_capture_begin / fl_capture_end / fl_graph_launch)."""

    def __init__(self, handle):
        self._h = handle

    @classmethod
    def capture(cls, fn, stream=None):
        """Run fn() (which issues library calls on `stream`) under capture; returns the graph.
        The stream must not be the legacy default stream (CUDA cannot capture it)."""
        s = _stream(stream)
        _check(lib().fl_capture_begin(s))
        try:
            fn()
        finally:
            h = ctypes.c_void_p()
            st = lib().fl_capture_end(s, ctypes.byref(h))
        _check(st)
        return cls(h)

    def launch(self, stream=None) -> None:
        _check(lib().fl_graph_launch(self._h, _stream(stream)))

    def close(self) -> None:
        if getattr(self, "_h", None):
            lib().fl_graph_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def swiglu_ffn_workspace_size(M: int, F: int, dtype) -> int:
    import torch
    code = {torch.float16: 0, torch.bfloat16: 1}.get(dtype, DTYPE_CODES.get(dtype))
    return int(lib().fl_swiglu_ffn_workspace_size(M, F, code))


def swiglu_ffn(x, gamma, Wg, Wu, Wd, bias_down=None, out=None, eps=1e-6, workspace=None, stream=None):
    """Llama-style SwiGLU FFN block: out = (silu(xh Wg^T) * (xh Wu^T)) Wd^T (+ bias_down) + x."""
    import torch
    M, D = x.shape
    F = Wg.shape[0]
    if out is None:
        out = torch.empty_like(x)
    need = swiglu_ffn_workspace_size(M, F, x.dtype)
    if workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=x.device)
    if not workspace.is_cuda or not workspace.is_contiguous():
        raise ValueError("workspace must be a contiguous CUDA tensor")
    _check_tensors(x.dtype, x=x, gamma=gamma, Wg=Wg, Wu=Wu, Wd=Wd, bias_down=bias_down, out=out)
    ws_bytes = workspace.numel() * workspace.element_size()
    _check(lib().fl_swiglu_ffn(_ptr(x), _ptr(gamma), _ptr(Wg), _ptr(Wu), _ptr(Wd), _ptr(bias_down), _ptr(out),
                               M, D, F, float(eps), _ptr(workspace), ws_bytes, _dtype_code(x), _stream(stream)))
    return out


def swiglu_ffn_noalloc(x, gamma, Wg, Wu, Wd, bias_down=None, out=None, eps=1e-6, stream=None):
    """swiglu_ffn for callers that may not allocate device memory: h lives in the
    library's fixed 8 MiB device array (M * F * 2 bytes at most). Calls whose
    kernels overlap on the GPU race on that array."""
    import torch
    M, D = x.shape
    F = Wg.shape[0]
    if out is None:
        out = torch.empty_like(x)
    _check_tensors(x.dtype, x=x, gamma=gamma, Wg=Wg, Wu=Wu, Wd=Wd, bias_down=bias_down, out=out)
    _check(lib().fl_swiglu_ffn_noalloc(_ptr(x), _ptr(gamma), _ptr(Wg), _ptr(Wu), _ptr(Wd), _ptr(bias_down),
                                       _ptr(out), M, D, F, float(eps), _dtype_code(x), _stream(stream)))
    return out


def launch_cache_stats():
    """(hits, misses) of the host-side launch cache since the library was loaded."""
    h, m = ctypes.c_longlong(), ctypes.c_longlong()
    _check(lib().fl_launch_cache_stats(ctypes.byref(h), ctypes.byref(m)))
    return h.value, m.value


def launch_cache_clear() -> None:
    lib().fl_launch_cache_clear()


def kernel_launches() -> int:
    """Kernels the library has launched (or recorded into a capture) since it was loaded."""
    n = ctypes.c_longlong()
    _check(lib().fl_kernel_launches(ctypes.byref(n)))
    return n.value


def device_status(stream=None) -> None:
    """Synchronise the stream and raise FusedLinError(FL_ERR_TIMEOUT) if a kernel's wait ran out."""
    _check(lib().fl_device_status(_stream(stream)))


def set_option(key: str, value: int) -> None:
    _check(lib().fl_set_option(OPTIONS[key], int(value)))


def debug_wait_timeout(limit_us: int, stream=None) -> None:
    """Launch the bounded-wait probe (a wait nothing completes); read the result with device_status()."""
    _check(lib().fl_debug_wait_timeout(int(limit_us), _stream(stream)))
