"""Python binding of libw4a16.so, the GB300 W4A16 group-quantised GEMM library.

Argument marshalling only: every step of the computation runs in the CUDA
kernels behind the C ABI (include/w4a16.h). PyTorch supplies device memory
and streams. There is no fallback: if the shared library is missing or
fails to load, importing this package raises.

Functions keep the C names:
    w4a16_gemm(x, qw, sc, y=None, group=32, algo="auto", overlap=False,
               stream=None, out_dtype="f32") -> y
    w4a16_quantize(w, group=32, stream=None) -> (qw, sc)
    w4a16_moe_sort(expert_ids, E, stream=None) -> (offsets, perm)
    w4a16_moe_workspace_size(T, topk, E, H, I) -> int
    w4a16_moe_workspace_layout(T, topk, E, H, I) -> {"perm", "h", "o"} byte offsets
    w4a16_moe_gemm(x, expert_ids, route_w, qw_gu, sc_gu, qw_dn, sc_dn,
                   workspace=None, y=None, group=32, stream=None) -> y
    w4a16_moe_route(x, router_w, topk, bias=None, route_scale=1.0, stream=None)
        -> (logits, expert_ids, route_w)
    w4a16_moe_block_workspace_size(T, topk, E, H, I, Is=0) -> int
    w4a16_moe_block(x, router_w, topk, qw_gu, sc_gu, qw_dn, sc_dn, shared=None,
                    bias=None, route_scale=1.0, group=32, workspace=None, y=None,
                    stream=None) -> (y, expert_ids, route_w)
    w4a16_status_string(code) -> str
    w4a16_last_device_status(stream=None) -> int
"""

from __future__ import annotations

import ctypes
import os

HERE = os.path.dirname(os.path.abspath(__file__))
# W4A16_LIBRARY selects another build of the library (the bounds-checking
# build, libw4a16_debug.so); by default the release build next to this file.
LIB_PATH = os.environ.get("W4A16_LIBRARY") or os.path.join(HERE, "libw4a16.so")

W4A16_OK = 0
W4A16_ERR_INVALID_ARG = 1
W4A16_ERR_UNSUPPORTED = 2
W4A16_ERR_ALIGNMENT = 3
W4A16_ERR_CUDA = 4
W4A16_ERR_TIMEOUT = 5
W4A16_ERR_BOUNDS = 6

ACT_F32 = 0
ACT_BF16 = 1

ALGOS = {"auto": 0, "simt": 1, "tc": 2, "stream": 3, "gemv": 4}
FLAG_OVERLAP = 1
FLAG_OUT_BF16 = 2

# name -> (restype, argtypes), mirroring include/w4a16.h
_VP, _I, _SZ = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
SIGNATURES = {
    "w4a16_gemm": (_I, [_VP, _I, _VP, _VP, _I, _I, _I, _I, _VP, _VP]),
    "w4a16_gemm_ex": (_I, [_VP, _I, _VP, _VP, _I, _I, _I, _I, _VP, _I, ctypes.c_uint, _VP]),
    "w4a16_gemm_launches": (_I, [_I, _I, _I, _I, _I, _I]),
    "w4a16_quantize": (_I, [_VP, _I, _I, _I, _VP, _VP, _VP]),
    "w4a16_moe_sort": (_I, [_VP, _I, _I, _VP, _VP, _VP]),
    "w4a16_moe_workspace_size": (_SZ, [_I, _I, _I, _I, _I]),
    "w4a16_moe_workspace_layout": (_I, [_I, _I, _I, _I, _I, ctypes.POINTER(_SZ),
                                        ctypes.POINTER(_SZ), ctypes.POINTER(_SZ)]),
    "w4a16_moe_gemm": (_I, [_VP, _I, _VP, _VP, _I, _I, _VP, _VP, _VP, _VP, _I, _I, _I, _I,
                            _VP, _SZ, _VP, _VP]),
    "w4a16_moe_gemm_noalloc": (_I, [_VP, _I, _VP, _VP, _I, _I, _VP, _VP, _VP, _VP, _I, _I, _I,
                                    _I, _VP, _VP]),
    "w4a16_moe_route": (_I, [_VP, _I, _I, _I, _VP, _VP, _I, _I, ctypes.c_float, _VP, _VP, _VP,
                             _VP]),
    "w4a16_moe_block_workspace_size": (_SZ, [_I, _I, _I, _I, _I, _I]),
    "w4a16_moe_block": (_I, [_VP, _I, _I, _VP, _VP, _I, _I, ctypes.c_float,
                             _VP, _VP, _VP, _VP, _I, _I,
                             _VP, _VP, _VP, _VP, _I,
                             _I, _VP, _SZ, _VP, _VP, _VP, _VP]),
    "w4a16_debug_fault_next_launch": (None, [_I]),
    "w4a16_status_string": (ctypes.c_char_p, [_I]),
    "w4a16_last_device_status": (_I, [_VP]),
}


class W4A16Error(RuntimeError):
    def __init__(self, fn: str, code: int):
        self.code = code
        super().__init__(f"{fn} failed: {status_string(code)} ({code})")


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(
            f"{LIB_PATH} is missing: build it with "
            "`python -c 'import __graft_entry__ as g; g.build()'` (nvcc, sm_103a)")
    lib = ctypes.CDLL(LIB_PATH)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    return lib


lib = _load()


def status_string(code: int) -> str:
    return lib.w4a16_status_string(int(code)).decode()


w4a16_status_string = status_string


def _check(fn: str, code: int):
    if code != W4A16_OK:
        raise W4A16Error(fn, code)


def _stream_handle(stream):
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr())


def _act_dtype(x):
    import torch
    if x.dtype == torch.float32:
        return ACT_F32
    if x.dtype == torch.bfloat16:
        return ACT_BF16
    raise TypeError("activations must be float32 or bfloat16")


def _need(t, dtype, name):
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def w4a16_gemm(x, qw, sc, y=None, group: int = 32, algo: str = "auto", overlap: bool = False,
               stream=None, out_dtype: str = "f32"):
    """y[M, N] = x[M, K] @ W_hat[N, K]^T via the C ABI.

    overlap=True sets W4A16_FLAG_OVERLAP: the weight stream may start while
    the previous kernel on the stream is still running (the caller promises
    that kernel does not write qw or sc). out_dtype="bf16" sets
    W4A16_FLAG_OUT_BF16: y is bf16, the fp32 result rounded to nearest even."""
    import torch
    xdt = _act_dtype(x)
    _need(x, x.dtype, "x")
    _need(qw, torch.int32, "qw")
    _need(sc, torch.float32, "sc")
    M, K = x.shape
    N = qw.shape[0]
    if out_dtype not in ("f32", "bf16"):
        raise ValueError("out_dtype must be 'f32' or 'bf16'")
    ydt = torch.bfloat16 if out_dtype == "bf16" else torch.float32
    if y is None:
        y = torch.empty((M, N), dtype=ydt, device=x.device)
    _need(y, ydt, "y")
    flags = (FLAG_OVERLAP if overlap else 0) | (FLAG_OUT_BF16 if out_dtype == "bf16" else 0)
    code = lib.w4a16_gemm_ex(_ptr(x), xdt, _ptr(qw), _ptr(sc), M, N, K, group, _ptr(y),
                             ALGOS[algo], flags, _stream_handle(stream))
    _check("w4a16_gemm", code)
    return y


def w4a16_gemm_launches(M: int, N: int, K: int, dtype: str = "f32", algo: str = "auto",
                        group: int = 32) -> int:
    """Kernel launches one w4a16_gemm call makes (negative status if rejected)."""
    return int(lib.w4a16_gemm_launches(M, N, K, group, ACT_BF16 if dtype == "bf16" else ACT_F32,
                                       ALGOS[algo]))


def w4a16_gemm_raw(x_ptr, xdt, qw_ptr, sc_ptr, M, N, K, group, y_ptr, algo=0, flags=0,
                   stream_ptr=0):
    """Pointer-level call (host code that manages its own buffers)."""
    return lib.w4a16_gemm_ex(ctypes.c_void_p(x_ptr), xdt, ctypes.c_void_p(qw_ptr),
                             ctypes.c_void_p(sc_ptr), M, N, K, group, ctypes.c_void_p(y_ptr),
                             algo, flags, ctypes.c_void_p(stream_ptr))


def w4a16_quantize(w, group: int = 32, qw=None, sc=None, stream=None):
    """Quantise fp32 w[N, K] on the device -> (qw int32 [N, K/8], sc fp32 [N, K/group])."""
    import torch
    _need(w, torch.float32, "w")
    N, K = w.shape
    if qw is None:
        qw = torch.empty((N, K // 8), dtype=torch.int32, device=w.device)
    if sc is None:
        sc = torch.empty((N, K // group), dtype=torch.float32, device=w.device)
    code = lib.w4a16_quantize(_ptr(w), N, K, group, _ptr(qw), _ptr(sc), _stream_handle(stream))
    _check("w4a16_quantize", code)
    return qw, sc


def w4a16_moe_sort(expert_ids, E: int, stream=None):
    """-> (offsets int32 [E+1], perm int32 [n_pairs])."""
    import torch
    _need(expert_ids, torch.int32, "expert_ids")
    n = expert_ids.numel()
    offsets = torch.empty(E + 1, dtype=torch.int32, device=expert_ids.device)
    perm = torch.empty(max(n, 1), dtype=torch.int32, device=expert_ids.device)
    code = lib.w4a16_moe_sort(_ptr(expert_ids), n, E, _ptr(offsets), _ptr(perm),
                              _stream_handle(stream))
    _check("w4a16_moe_sort", code)
    return offsets, perm[:n]


def w4a16_moe_workspace_size(T: int, topk: int, E: int, H: int, I: int) -> int:
    return int(lib.w4a16_moe_workspace_size(T, topk, E, H, I))


def w4a16_moe_workspace_layout(T: int, topk: int, E: int, H: int, I: int) -> dict:
    """Byte offsets of perm, h and o inside the MoE workspace (see the header)."""
    a, b, c = ctypes.c_size_t(), ctypes.c_size_t(), ctypes.c_size_t()
    code = lib.w4a16_moe_workspace_layout(T, topk, E, H, I, ctypes.byref(a), ctypes.byref(b),
                                          ctypes.byref(c))
    _check("w4a16_moe_workspace_layout", code)
    return {"perm": a.value, "h": b.value, "o": c.value}


def _moe_args(x, expert_ids, route_w, qw_gu, sc_gu, qw_dn, sc_dn, y):
    """Checks shared by the MoE layer wrappers -> (xdt, T, H, topk, E, I, y)."""
    import torch
    xdt = _act_dtype(x)
    _need(x, x.dtype, "x")
    _need(expert_ids, torch.int32, "expert_ids")
    _need(route_w, torch.float32, "route_w")
    for t, n, d in ((qw_gu, "qw_gu", torch.int32), (sc_gu, "sc_gu", torch.float32),
                    (qw_dn, "qw_dn", torch.int32), (sc_dn, "sc_dn", torch.float32)):
        _need(t, d, n)
    T, H = x.shape
    topk = expert_ids.shape[1]
    E = qw_gu.shape[0]
    I = qw_gu.shape[1] // 2
    if y is None:
        y = torch.empty((T, H), dtype=torch.float32, device=x.device)
    _need(y, torch.float32, "y")
    if tuple(y.shape) != (T, H):
        raise ValueError(f"y must have shape {(T, H)}, got {tuple(y.shape)}")
    return xdt, T, H, topk, E, I, y


def w4a16_moe_gemm(x, expert_ids, route_w, qw_gu, sc_gu, qw_dn, sc_dn, workspace=None,
                   y=None, group: int = 32, stream=None):
    """Grouped MoE layer on INT4 experts -> y fp32 [T, H]."""
    import torch
    xdt, T, H, topk, E, I, y = _moe_args(x, expert_ids, route_w, qw_gu, sc_gu, qw_dn, sc_dn, y)
    ws = w4a16_moe_workspace_size(T, topk, E, H, I)
    if workspace is None:
        workspace = torch.empty(ws, dtype=torch.uint8, device=x.device)
    code = lib.w4a16_moe_gemm(_ptr(x), xdt, _ptr(expert_ids), _ptr(route_w), T, topk,
                              _ptr(qw_gu), _ptr(sc_gu), _ptr(qw_dn), _ptr(sc_dn), E, H, I, group,
                              _ptr(workspace), workspace.numel() * workspace.element_size(),
                              _ptr(y), _stream_handle(stream))
    _check("w4a16_moe_gemm", code)
    return y


def w4a16_moe_gemm_noalloc(x, expert_ids, route_w, qw_gu, sc_gu, qw_dn, sc_dn, y=None,
                           group: int = 32, stream=None):
    """w4a16_moe_gemm without a workspace: the library's fixed 40 MiB device
    array holds the intermediates (for callers that cannot allocate). The
    array used is the current device's, so every tensor must live there."""
    import torch
    xdt, T, H, topk, E, I, y = _moe_args(x, expert_ids, route_w, qw_gu, sc_gu, qw_dn, sc_dn, y)
    cur = torch.cuda.current_device()
    for t, n in ((x, "x"), (expert_ids, "expert_ids"), (route_w, "route_w"), (qw_gu, "qw_gu"),
                 (sc_gu, "sc_gu"), (qw_dn, "qw_dn"), (sc_dn, "sc_dn"), (y, "y")):
        if t.device.index != cur:
            raise ValueError(f"{n} is on {t.device}, not on the current device cuda:{cur}")
    code = lib.w4a16_moe_gemm_noalloc(_ptr(x), xdt, _ptr(expert_ids), _ptr(route_w), T, topk,
                                      _ptr(qw_gu), _ptr(sc_gu), _ptr(qw_dn), _ptr(sc_dn), E, H, I,
                                      group, _ptr(y), _stream_handle(stream))
    _check("w4a16_moe_gemm_noalloc", code)
    return y


def w4a16_debug_fault_next_launch(enable: bool = True) -> None:
    """Testing aid: the next launch of a CUDA-core GEMM kernel (decode GEMV or
    streaming) skips its weight copies, times out after about a second and
    records W4A16_ERR_TIMEOUT."""
    lib.w4a16_debug_fault_next_launch(1 if enable else 0)


def w4a16_last_device_status(stream=None) -> int:
    return int(lib.w4a16_last_device_status(_stream_handle(stream)))


def w4a16_moe_route(x, router_w, topk: int, bias=None, route_scale: float = 1.0, stream=None):
    """MoE router -> (logits fp32 [T, E], expert_ids int32 [T, topk], route_w fp32 [T, topk])."""
    import torch
    xdt = _act_dtype(x)
    _need(x, x.dtype, "x")
    _need(router_w, torch.float32, "router_w")
    if bias is not None:
        _need(bias, torch.float32, "bias")
    T, H = x.shape
    E = router_w.shape[0]
    logits = torch.empty((T, E), dtype=torch.float32, device=x.device)
    ids = torch.empty((T, topk), dtype=torch.int32, device=x.device)
    rw = torch.empty((T, topk), dtype=torch.float32, device=x.device)
    code = lib.w4a16_moe_route(_ptr(x), xdt, T, H, _ptr(router_w),
                               _ptr(bias) if bias is not None else None, E, topk,
                               float(route_scale), _ptr(logits), _ptr(ids), _ptr(rw),
                               _stream_handle(stream))
    _check("w4a16_moe_route", code)
    return logits, ids, rw


def w4a16_moe_block_workspace_size(T: int, topk: int, E: int, H: int, I: int, Is: int = 0) -> int:
    return int(lib.w4a16_moe_block_workspace_size(T, topk, E, H, I, Is))


def w4a16_moe_block(x, router_w, topk: int, qw_gu, sc_gu, qw_dn, sc_dn, shared=None, bias=None,
                    route_scale: float = 1.0, group: int = 32, workspace=None, y=None,
                    stream=None):
    """Whole MoE block: router, routed experts and the shared expert.

    ``shared`` is (qw_sgu [2Is, H/8], sc_sgu, qw_sdn [H, Is/8], sc_sdn) or None.
    Returns (y fp32 [T, H], expert_ids int32 [T, topk], route_w fp32 [T, topk])."""
    import torch
    xdt = _act_dtype(x)
    _need(x, x.dtype, "x")
    _need(router_w, torch.float32, "router_w")
    if bias is not None:
        _need(bias, torch.float32, "bias")
    for t, n, d in ((qw_gu, "qw_gu", torch.int32), (sc_gu, "sc_gu", torch.float32),
                    (qw_dn, "qw_dn", torch.int32), (sc_dn, "sc_dn", torch.float32)):
        _need(t, d, n)
    T, H = x.shape
    E = qw_gu.shape[0]
    I = qw_gu.shape[1] // 2
    if shared is not None:
        for t, n, d in zip(shared, ("qw_sgu", "sc_sgu", "qw_sdn", "sc_sdn"),
                           (torch.int32, torch.float32, torch.int32, torch.float32)):
            _need(t, d, n)
        Is = shared[0].shape[0] // 2
        sp = [_ptr(t) for t in shared]
    else:
        Is = 0
        sp = [None] * 4
    ws = w4a16_moe_block_workspace_size(T, topk, E, H, I, Is)
    if workspace is None:
        workspace = torch.empty(max(ws, 1), dtype=torch.uint8, device=x.device)
    if y is None:
        y = torch.empty((T, H), dtype=torch.float32, device=x.device)
    ids = torch.empty((T, topk), dtype=torch.int32, device=x.device)
    rw = torch.empty((T, topk), dtype=torch.float32, device=x.device)
    code = lib.w4a16_moe_block(_ptr(x), xdt, T, _ptr(router_w),
                               _ptr(bias) if bias is not None else None, E, topk,
                               float(route_scale), _ptr(qw_gu), _ptr(sc_gu), _ptr(qw_dn),
                               _ptr(sc_dn), H, I, sp[0], sp[1], sp[2], sp[3], Is, group,
                               _ptr(workspace), workspace.numel() * workspace.element_size(),
                               _ptr(ids), _ptr(rw), _ptr(y), _stream_handle(stream))
    _check("w4a16_moe_block", code)
    return y, ids, rw
