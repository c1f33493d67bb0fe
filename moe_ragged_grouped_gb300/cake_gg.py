"""Thin Python binding of the C ABI in include/cake_gg.h (ctypes; marshalling only).

Every function here converts arguments (torch tensors -> device pointers, the
current torch CUDA stream -> cudaStream_t) and calls the library of the same
name; all computation runs in the library's CUDA kernels.  There is no CPU or
eager fallback: if ``libcake_gg.so`` is missing, every call raises.

PyTorch is used only for device memory and streams.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libcake_gg.so")

CAKE_GG_OK = 0
CAKE_GG_ERR_INVALID_ARG = 1
CAKE_GG_ERR_ALIGNMENT = 2
CAKE_GG_ERR_OVERFLOW = 3
CAKE_GG_ERR_UNSUPPORTED = 4
CAKE_GG_ERR_WORKSPACE = 5
CAKE_GG_ERR_CUDA = 6
CAKE_GG_ERR_BAD_OFFSETS = 7
CAKE_GG_ERR_TIMEOUT = 8
CAKE_GG_ERR_SCRATCH_LIMIT = 9
CAKE_GG_NOALLOC_SCRATCH_BYTES = 32 << 20

CAKE_GG_FWD, CAKE_GG_DGRAD, CAKE_GG_WGRAD = 0, 1, 2
CAKE_GG_BF16, CAKE_GG_FP32 = 0, 1
CAKE_GG_DEBUG_DROP_FIRST_LOAD = 1

PASSES = {"fwd": CAKE_GG_FWD, "dgrad": CAKE_GG_DGRAD, "wgrad": CAKE_GG_WGRAD}
DTYPES = {"bf16": CAKE_GG_BF16, "fp32": CAKE_GG_FP32}

EXPORTED = ["cake_gg_plan", "cake_gg_fwd", "cake_gg_dgrad", "cake_gg_wgrad",
            "cake_gg_check_status", "cake_gg_strerror", "cake_gg_tile_walk", "cake_gg_corun_spinner",
            "cake_gg_router_plan", "cake_gg_router_fp32"]


class CakeGGPlan(ctypes.Structure):
    """Mirror of cake_gg_plan_t (same field order, same C layout)."""
    _fields_ = [
        ("abi_version", ctypes.c_int32),
        ("pass_", ctypes.c_int32),
        ("E", ctypes.c_int32),
        ("N", ctypes.c_int32),
        ("K", ctypes.c_int32),
        ("out_dtype", ctypes.c_int32),
        ("M_max", ctypes.c_int64),
        ("deterministic", ctypes.c_int32),
        ("max_sms", ctypes.c_int32),
        ("tile_m", ctypes.c_int32),
        ("tile_n", ctypes.c_int32),
        ("tile_k", ctypes.c_int32),
        ("stages", ctypes.c_int32),
        ("pair", ctypes.c_int32),
        ("swap_ab", ctypes.c_int32),
        ("split_chunk", ctypes.c_int32),
        ("debug_flags", ctypes.c_int32),
        ("timeout_ns", ctypes.c_uint64),
        ("workspace_bytes", ctypes.c_uint64),
        ("staging_bufs", ctypes.c_int32),
        ("cluster_splits", ctypes.c_int32),
        ("tail_units", ctypes.c_int32),
        ("tail_splits", ctypes.c_int32),
        ("streamk_kblocks", ctypes.c_int32),
        ("epi_groups", ctypes.c_int32),
        ("tail_nsplit", ctypes.c_int32),
        ("reserved", ctypes.c_int32 * 1),
    ]

    def as_dict(self):
        return {f[0]: getattr(self, f[0]) for f in self._fields_ if f[0] != "reserved"}


class CakeGGRouterPlan(ctypes.Structure):
    """Mirror of cake_gg_router_plan_t (same field order, same C layout)."""
    _fields_ = [
        ("abi_version", ctypes.c_int32),
        ("R", ctypes.c_int32),
        ("T", ctypes.c_int64),
        ("K", ctypes.c_int32),
        ("reserved", ctypes.c_int32),
        ("workspace_bytes", ctypes.c_uint64),
        ("gemm", CakeGGPlan),
    ]


class CakeGGError(RuntimeError):
    def __init__(self, code, where):
        super().__init__(f"{where}: {cake_gg_strerror(code)} (status {code})")
        self.code = code


_lib = None


def load_library(path: str = LIB_PATH):
    """Load libcake_gg.so; raise if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(
            f"{path} is missing: build it with moe_ragged_grouped_gb300.build.build() "
            "(there is no fallback implementation)")
    lib = ctypes.CDLL(path)
    vp, i32, i64, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t
    plan_p = ctypes.POINTER(CakeGGPlan)
    lib.cake_gg_plan.argtypes = [plan_p, ctypes.c_int, i32, i64, i32, i32, ctypes.c_int, ctypes.c_int, i32]
    lib.cake_gg_plan.restype = ctypes.c_int
    for name in ("cake_gg_fwd", "cake_gg_dgrad", "cake_gg_wgrad"):
        f = getattr(lib, name)
        f.argtypes = [plan_p, vp, vp, vp, vp, ctypes.c_int, ctypes.c_int, vp, sz, vp]
        f.restype = ctypes.c_int
    lib.cake_gg_check_status.argtypes = [vp, vp]
    lib.cake_gg_corun_spinner.argtypes = [i32, ctypes.c_uint64, vp]
    lib.cake_gg_corun_spinner.restype = ctypes.c_int
    lib.cake_gg_check_status.restype = ctypes.c_int
    lib.cake_gg_strerror.argtypes = [ctypes.c_int]
    lib.cake_gg_strerror.restype = ctypes.c_char_p
    lib.cake_gg_tile_walk.argtypes = [plan_p, ctypes.POINTER(ctypes.c_int32), i64,
                                      ctypes.POINTER(ctypes.c_int32), ctypes.POINTER(ctypes.c_int64)]
    lib.cake_gg_tile_walk.restype = ctypes.c_int
    lib.cake_gg_wgrad_noalloc.argtypes = [plan_p, vp, vp, vp, vp, ctypes.c_int, ctypes.c_int, vp]
    lib.cake_gg_wgrad_noalloc.restype = ctypes.c_int
    rplan_p = ctypes.POINTER(CakeGGRouterPlan)
    lib.cake_gg_router_plan.argtypes = [rplan_p, i64, i32, i32, i32]
    lib.cake_gg_router_plan.restype = ctypes.c_int
    lib.cake_gg_router_fp32.argtypes = [rplan_p, vp, vp, vp, vp, sz, vp]
    lib.cake_gg_router_fp32.restype = ctypes.c_int
    _lib = lib
    return lib


def _ptr(x):
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return x.data_ptr()


def _stream(stream, *tensors):
    if stream is not None:
        return stream if isinstance(stream, int) else stream.cuda_stream
    for t in tensors:
        if t is not None and not isinstance(t, int) and getattr(t, "is_cuda", False):
            import torch
            return torch.cuda.current_stream(t.device).cuda_stream
    return 0


def _dtype_code(d):
    return DTYPES[d] if isinstance(d, str) else int(d)


def _pass_code(p):
    return PASSES[p] if isinstance(p, str) else int(p)


# ---------------------------------------------------------------- C ABI, same names


def cake_gg_strerror(code: int) -> str:
    return load_library().cake_gg_strerror(int(code)).decode()


def cake_gg_plan(pass_, E, M_max, N, K, out_dtype, deterministic, max_sms=0) -> CakeGGPlan:
    """cake_gg_plan(): returns the filled plan; raises CakeGGError on a non-zero status."""
    plan = CakeGGPlan()
    rc = load_library().cake_gg_plan(ctypes.byref(plan), _pass_code(pass_), int(E), int(M_max), int(N),
                                     int(K), _dtype_code(out_dtype), int(bool(deterministic)), int(max_sms))
    if rc != CAKE_GG_OK:
        raise CakeGGError(rc, "cake_gg_plan")
    return plan


def _call(name, plan, a, b, out, offsets, out_dtype, deterministic, workspace, workspace_bytes, stream):
    lib = load_library()
    if workspace_bytes is None:
        workspace_bytes = 0 if workspace is None else (
            workspace.numel() * workspace.element_size() if not isinstance(workspace, int) else plan.workspace_bytes)
    s = _stream(stream, a, b, out)
    return getattr(lib, name)(ctypes.byref(plan), _ptr(a), _ptr(b), _ptr(out), _ptr(offsets),
                              _dtype_code(out_dtype), int(bool(deterministic)), _ptr(workspace),
                              int(workspace_bytes), s)


def cake_gg_fwd(plan, X, W, Y, offsets, out_dtype, deterministic, workspace, workspace_bytes=None,
                stream=None) -> int:
    """cake_gg_fwd(): Y = X W_e^T per expert; returns the status code."""
    return _call("cake_gg_fwd", plan, X, W, Y, offsets, out_dtype, deterministic, workspace,
                 workspace_bytes, stream)


def cake_gg_dgrad(plan, G, W, dX, offsets, out_dtype, deterministic, workspace, workspace_bytes=None,
                  stream=None) -> int:
    """cake_gg_dgrad(): dX = G W_e per expert; returns the status code."""
    return _call("cake_gg_dgrad", plan, G, W, dX, offsets, out_dtype, deterministic, workspace,
                 workspace_bytes, stream)


def cake_gg_wgrad(plan, G, X, dW, offsets, out_dtype, deterministic, workspace, workspace_bytes=None,
                  stream=None) -> int:
    """cake_gg_wgrad(): dW_e = G_e^T X_e per expert; returns the status code."""
    return _call("cake_gg_wgrad", plan, G, X, dW, offsets, out_dtype, deterministic, workspace,
                 workspace_bytes, stream)


def cake_gg_wgrad_noalloc(plan, G, X, dW, offsets, out_dtype, deterministic, stream=None) -> int:
    """cake_gg_wgrad_noalloc(): the weight gradient using the library's fixed scratch.

    For callers that cannot allocate device memory (no workspace argument, no
    allocation inside the call).  Returns the status code;
    CAKE_GG_ERR_SCRATCH_LIMIT when plan.workspace_bytes exceeds
    CAKE_GG_NOALLOC_SCRATCH_BYTES.
    """
    s = _stream(stream, G, X, dW)
    return load_library().cake_gg_wgrad_noalloc(ctypes.byref(plan), _ptr(G), _ptr(X), _ptr(dW), _ptr(offsets),
                                                _dtype_code(out_dtype), int(bool(deterministic)), s)


def cake_gg_check_status(workspace, stream=None) -> int:
    """cake_gg_check_status(): synchronises the stream and returns the device status word."""
    return load_library().cake_gg_check_status(_ptr(workspace), _stream(stream, workspace))


def cake_gg_corun_spinner(ctas, ns, stream) -> int:
    """cake_gg_corun_spinner(): hold `ctas` SMs for `ns` nanoseconds on `stream` (a cudaStream_t value)."""
    return load_library().cake_gg_corun_spinner(int(ctas), int(ns), ctypes.c_void_p(int(stream)))


def cake_gg_tile_walk(plan, offsets) -> np.ndarray:
    """cake_gg_tile_walk(): the kernel's tile list for host offsets, as an int32 [count, 10] array."""
    lib = load_library()
    off = np.ascontiguousarray(offsets, dtype=np.int32)
    count = ctypes.c_int64(0)
    rc = lib.cake_gg_tile_walk(ctypes.byref(plan), off.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)), 0,
                               None, ctypes.byref(count))
    if rc != CAKE_GG_OK:
        raise CakeGGError(rc, "cake_gg_tile_walk")
    out = np.zeros((count.value, 10), dtype=np.int32)
    rc = lib.cake_gg_tile_walk(ctypes.byref(plan), off.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)),
                               count.value, out.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)),
                               ctypes.byref(count))
    if rc != CAKE_GG_OK:
        raise CakeGGError(rc, "cake_gg_tile_walk")
    return out


def cake_gg_router_plan(T, R, K, max_sms=0) -> CakeGGRouterPlan:
    """cake_gg_router_plan(): plan of the FP32 router GEMM (BF16x3 emulation); raises on error."""
    rp = CakeGGRouterPlan()
    rc = load_library().cake_gg_router_plan(ctypes.byref(rp), int(T), int(R), int(K), int(max_sms))
    if rc != CAKE_GG_OK:
        raise CakeGGError(rc, "cake_gg_router_plan")
    return rp


def cake_gg_router_fp32(rp, X, W, Y, workspace, workspace_bytes=None, stream=None) -> int:
    """cake_gg_router_fp32(): Y = X W^T by BF16x3 emulation on float32 torch tensors; returns the status."""
    s = _stream(stream, X, W, Y)
    nb = int(workspace.numel() * workspace.element_size()) if workspace_bytes is None else int(workspace_bytes)
    return load_library().cake_gg_router_fp32(ctypes.byref(rp), _ptr(X), _ptr(W), _ptr(Y), _ptr(workspace), nb, s)


# ---------------------------------------------------------------- tensor-level helpers


def _torch_out_dtype(out_dtype):
    import torch
    return torch.float32 if _dtype_code(out_dtype) == CAKE_GG_FP32 else torch.bfloat16


def make_workspace(plan, device):
    """A zero-filled workspace of plan.workspace_bytes (the library expects zeros before first use)."""
    import torch
    n = max(int(plan.workspace_bytes), 256)
    return torch.zeros(n, dtype=torch.uint8, device=device)


def grouped_gemm(pass_, a, b, offsets, out_dtype="bf16", deterministic=True, max_sms=0, out=None,
                 plan=None, workspace=None, stream=None, check=True):
    """Run one pass on torch CUDA tensors, allocating the output and workspace through torch.

    fwd:   a = X [M, K], b = W [E, N, K] -> Y [M, N]
    dgrad: a = G [M, N], b = W [E, N, K] -> dX [M, K]
    wgrad: a = G [M, N], b = X [M, K], E from offsets -> dW [E, N, K]
    Rows >= offsets[E] of Y / dX are left as allocated (uninitialised).
    """
    import torch
    p = _pass_code(pass_)
    E = int(offsets.numel()) - 1
    M = int(a.shape[0])
    if p == CAKE_GG_FWD:
        N, K = int(b.shape[1]), int(b.shape[2])
        shape = (M, N)
    elif p == CAKE_GG_DGRAD:
        N, K = int(b.shape[1]), int(b.shape[2])
        shape = (M, K)
    else:
        N, K = int(a.shape[1]), int(b.shape[1])
        shape = (E, N, K)
    if plan is None:
        plan = cake_gg_plan(p, E, M, N, K, out_dtype, deterministic, max_sms)
    if out is None:
        out = torch.empty(shape, dtype=_torch_out_dtype(out_dtype), device=a.device)
    if workspace is None:
        workspace = make_workspace(plan, a.device)
    fn = {CAKE_GG_FWD: cake_gg_fwd, CAKE_GG_DGRAD: cake_gg_dgrad, CAKE_GG_WGRAD: cake_gg_wgrad}[p]
    rc = fn(plan, a, b, out, offsets, out_dtype, deterministic, workspace, stream=stream)
    if rc != CAKE_GG_OK:
        raise CakeGGError(rc, f"cake_gg pass {pass_}")
    if check:
        st = cake_gg_check_status(workspace, stream)
        if st != CAKE_GG_OK:
            raise CakeGGError(st, f"cake_gg pass {pass_} (device status)")
    return out


def router_gemm(X, W, max_sms=0, out=None, plan=None, workspace=None, stream=None, check=True):
    """FP32 router logits Y [T, R] = X [T, K] W [R, K]^T by BF16x3 emulation (float32 torch tensors).

    Allocates the output and the workspace through torch when not given.
    """
    import torch
    T, K = int(X.shape[0]), int(X.shape[1])
    R = int(W.shape[0])
    if plan is None:
        plan = cake_gg_router_plan(T, R, K, max_sms)
    if out is None:
        out = torch.empty((T, R), dtype=torch.float32, device=X.device)
    if workspace is None:
        workspace = torch.zeros(max(int(plan.workspace_bytes), 256), dtype=torch.uint8, device=X.device)
    rc = cake_gg_router_fp32(plan, X, W, out, workspace, stream=stream)
    if rc != CAKE_GG_OK:
        raise CakeGGError(rc, "cake_gg_router_fp32")
    if check:
        st = cake_gg_check_status(workspace, stream)
        if st != CAKE_GG_OK:
            raise CakeGGError(st, "cake_gg_router_fp32 (device status)")
    return out
