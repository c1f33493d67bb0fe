"""FP64 CPU oracle for the ragged BF16 grouped GEMM -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline /
reference legs may import this package.  The library under
``moe_ragged_grouped_gb300`` never imports it, and it imports nothing from the
library: the two share no code.

The arithmetic lives in ``cake_oracle.c`` (plain C, FP64, sequential sums in
index order); this module only compiles it with gcc and marshals numpy arrays.
What it computes follows flashinfer PR #8258 (opening summary: forward
Y = X W^T, data gradient dX = G W, weight gradient dW = G^T X over ragged
expert row groups) and PR #8363 ("Definitions": [T, d_in] activations,
[T, d_out] output gradients, [d_out, d_in] weight gradient).

BF16 tensors are passed as ``numpy.uint16`` arrays of raw bit patterns.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import tempfile

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "cake_oracle.c")
_LIB_PATH = os.path.join(_HERE, "libcake_oracle.so")
_lib = None

_U16P = ctypes.POINTER(ctypes.c_uint16)
_I32P = ctypes.POINTER(ctypes.c_int32)
_I64P = ctypes.POINTER(ctypes.c_int64)
_F64P = ctypes.POINTER(ctypes.c_double)
_F32P = ctypes.POINTER(ctypes.c_float)


def compile_oracle(out_path: str = _LIB_PATH, mutant: int = 0) -> str:
    """Compile cake_oracle.c into a shared library (gcc, OpenMP, no FMA contraction).

    ``mutant`` > 0 plants the numbered deliberate mistake (used only by the test
    that shows the pins catch such mistakes).
    """
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp",
           "-ffp-contract=off", "-fno-fast-math", f"-DORACLE_MUTANT={int(mutant)}",
           _SRC, "-o", out_path]
    subprocess.run(cmd, check=True)
    return out_path


def _bind(lib):
    ent = [_U16P, _U16P, _I32P, ctypes.c_int32, ctypes.c_int64, ctypes.c_int32, ctypes.c_int32]
    for name in ("oracle_fwd", "oracle_dgrad", "oracle_wgrad"):
        f = getattr(lib, name)
        f.argtypes = ent + [_F64P]
        f.restype = ctypes.c_int
    for name in ("oracle_fwd_at", "oracle_dgrad_at"):
        f = getattr(lib, name)
        f.argtypes = ent + [_I64P, _I64P, ctypes.c_int64, _F64P]
        f.restype = ctypes.c_int
    lib.oracle_wgrad_at.argtypes = ent + [_I64P, _I64P, _I64P, ctypes.c_int64, _F64P]
    lib.oracle_wgrad_at.restype = ctypes.c_int
    lib.oracle_num_threads.argtypes = []
    lib.oracle_num_threads.restype = ctypes.c_int
    rt = [_F32P, _F32P, ctypes.c_int64, ctypes.c_int32, ctypes.c_int32]
    for name in ("oracle_router_bf16x3", "oracle_router_exact"):
        f = getattr(lib, name)
        f.argtypes = rt + [_F64P]
        f.restype = ctypes.c_int
    lib.oracle_router_bf16x3_at.argtypes = rt + [_I64P, _I64P, ctypes.c_int64, _F64P]
    lib.oracle_router_bf16x3_at.restype = ctypes.c_int
    lib.oracle_round_bf16.argtypes = [ctypes.c_float]
    lib.oracle_round_bf16.restype = ctypes.c_float
    return lib


def load(mutant: int = 0):
    """Return the compiled oracle library, building it when missing or stale."""
    global _lib
    if mutant:
        tmp = tempfile.mkdtemp(prefix="cake_oracle_mutant_")
        return _bind(ctypes.CDLL(compile_oracle(os.path.join(tmp, "lib.so"), mutant)))
    if _lib is None:
        if (not os.path.exists(_LIB_PATH)
                or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC)):
            compile_oracle()
        _lib = _bind(ctypes.CDLL(_LIB_PATH))
    return _lib


def _u16(a):
    a = np.ascontiguousarray(a)
    if a.dtype != np.uint16:
        raise TypeError("BF16 operands are passed as uint16 bit patterns")
    return a, a.ctypes.data_as(_U16P)


def _off(off):
    o = np.ascontiguousarray(off, dtype=np.int32)
    return o, o.ctypes.data_as(_I32P)


def _check(rc, name):
    if rc != 0:
        raise ValueError(f"{name}: invalid arguments (offsets or sizes)")


def fwd(X, W, off, lib=None):
    """Y [off[E], N] in FP64 from X [M, K], W [E, N, K] (uint16 BF16 bits)."""
    lib = lib or load()
    X, px = _u16(X); W, pw = _u16(W); off, po = _off(off)
    E, N, K = W.shape
    Y = np.zeros((int(off[-1]), N), dtype=np.float64)
    _check(lib.oracle_fwd(px, pw, po, E, X.shape[0], N, K, Y.ctypes.data_as(_F64P)), "fwd")
    return Y


def dgrad(G, W, off, lib=None):
    """dX [off[E], K] in FP64 from G [M, N], W [E, N, K]."""
    lib = lib or load()
    G, pg = _u16(G); W, pw = _u16(W); off, po = _off(off)
    E, N, K = W.shape
    dX = np.zeros((int(off[-1]), K), dtype=np.float64)
    _check(lib.oracle_dgrad(pg, pw, po, E, G.shape[0], N, K, dX.ctypes.data_as(_F64P)), "dgrad")
    return dX


def wgrad(G, X, off, E, lib=None):
    """dW [E, N, K] in FP64 from G [M, N], X [M, K]."""
    lib = lib or load()
    G, pg = _u16(G); X, px = _u16(X); off, po = _off(off)
    N, K = G.shape[1], X.shape[1]
    dW = np.zeros((E, N, K), dtype=np.float64)
    _check(lib.oracle_wgrad(pg, px, po, E, G.shape[0], N, K, dW.ctypes.data_as(_F64P)), "wgrad")
    return dW


def _idx(a):
    a = np.ascontiguousarray(a, dtype=np.int64)
    return a, a.ctypes.data_as(_I64P)


def fwd_at(X, W, off, rows, cols, lib=None):
    """Y[rows[i], cols[i]] for each i, in FP64."""
    lib = lib or load()
    X, px = _u16(X); W, pw = _u16(W); off, po = _off(off)
    E, N, K = W.shape
    rows, pr = _idx(rows); cols, pc = _idx(cols)
    out = np.zeros(rows.shape[0], dtype=np.float64)
    _check(lib.oracle_fwd_at(px, pw, po, E, X.shape[0], N, K, pr, pc, rows.shape[0],
                             out.ctypes.data_as(_F64P)), "fwd_at")
    return out


def dgrad_at(G, W, off, rows, cols, lib=None):
    """dX[rows[i], cols[i]] for each i, in FP64."""
    lib = lib or load()
    G, pg = _u16(G); W, pw = _u16(W); off, po = _off(off)
    E, N, K = W.shape
    rows, pr = _idx(rows); cols, pc = _idx(cols)
    out = np.zeros(rows.shape[0], dtype=np.float64)
    _check(lib.oracle_dgrad_at(pg, pw, po, E, G.shape[0], N, K, pr, pc, rows.shape[0],
                               out.ctypes.data_as(_F64P)), "dgrad_at")
    return out


def wgrad_at(G, X, off, E, es, ns, ks, lib=None):
    """dW[es[i], ns[i], ks[i]] for each i, in FP64."""
    lib = lib or load()
    G, pg = _u16(G); X, px = _u16(X); off, po = _off(off)
    N, K = G.shape[1], X.shape[1]
    es, pe = _idx(es); ns, pn = _idx(ns); ks, pk = _idx(ks)
    out = np.zeros(es.shape[0], dtype=np.float64)
    _check(lib.oracle_wgrad_at(pg, px, po, E, G.shape[0], N, K, pe, pn, pk, es.shape[0],
                               out.ctypes.data_as(_F64P)), "wgrad_at")
    return out


# ---- FP32 router GEMM (BF16x3 emulation; flashinfer PR #8438, "Summary") ----

def _f32(a):
    a = np.ascontiguousarray(a)
    if a.dtype != np.float32:
        raise TypeError("router operands are float32")
    return a, a.ctypes.data_as(_F32P)


def router_bf16x3(X, W, lib=None):
    """Y [T, R] in FP64: sum over k of x_hi w_hi + x_hi w_lo + x_lo w_hi (X [T, K], W [R, K] float32)."""
    lib = lib or load()
    X, px = _f32(X); W, pw = _f32(W)
    (T, K), R = X.shape, W.shape[0]
    Y = np.zeros((T, R), dtype=np.float64)
    _check(lib.oracle_router_bf16x3(px, pw, T, R, K, Y.ctypes.data_as(_F64P)), "router_bf16x3")
    return Y


def router_exact(X, W, lib=None):
    """Y [T, R] in FP64 by the definition sum over k of x w."""
    lib = lib or load()
    X, px = _f32(X); W, pw = _f32(W)
    (T, K), R = X.shape, W.shape[0]
    Y = np.zeros((T, R), dtype=np.float64)
    _check(lib.oracle_router_exact(px, pw, T, R, K, Y.ctypes.data_as(_F64P)), "router_exact")
    return Y


def router_bf16x3_at(X, W, ts, rs, lib=None):
    """Y[ts[i], rs[i]] by the BF16x3 emulation, in FP64."""
    lib = lib or load()
    X, px = _f32(X); W, pw = _f32(W)
    (T, K), R = X.shape, W.shape[0]
    ts, pt = _idx(ts); rs, pr = _idx(rs)
    out = np.zeros(ts.shape[0], dtype=np.float64)
    _check(lib.oracle_router_bf16x3_at(px, pw, T, R, K, pt, pr, ts.shape[0], out.ctypes.data_as(_F64P)),
           "router_bf16x3_at")
    return out


def round_bf16(v, lib=None) -> float:
    """The oracle's round-to-nearest-even BF16 of one float32 value (widened back to float)."""
    return float((lib or load()).oracle_round_bf16(float(v)))


def router_tolerance(abs_dot, L):
    """Per-element bound for a GPU BF16x3 router logit against the emulation (router_bf16x3).

    The GPU sums the same L = 3K exact BF16 products in FP32 (tensor-core
    accumulation, order hardware-defined): |gpu - emu| <= 2^-22 * L * sum_k
    |x_k w_k|, the sequential FP32 bound L * 2^-24 * sum|terms| with a factor 4
    of margin for the accumulator's alignment.  ``abs_dot`` is sum_k |x_k| |w_k|.
    """
    return 2.0 ** -22 * float(L) * np.asarray(abs_dot, dtype=np.float64)


def router_emulation_bound(abs_dot):
    """|emulation - definition| <= 3 * 2^-16 * sum_k |x_k| |w_k| (the dropped x_lo w_lo and split residues)."""
    return 3.0 * 2.0 ** -16 * np.asarray(abs_dot, dtype=np.float64)


def num_threads(lib=None) -> int:
    return int((lib or load()).oracle_num_threads())


def bf16_bits_to_f64(a) -> np.ndarray:
    """Exact widening of BF16 bit patterns (uint16) to float64, for tests."""
    a = np.ascontiguousarray(a, dtype=np.uint16)
    return (a.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def tolerance(ref, L, max_a, max_b):
    """Per-element parity bound |gpu - ref| <= 2^-8 |ref| + 2^-18 * L * max|a| * max|b|.

    L is the pass's reduction length (K for forward, N for the data gradient,
    the expert's row count for the weight gradient); max|a|, max|b| are the
    maxima over the pass's two input operands.
    """
    return 2.0 ** -8 * np.abs(ref) + 2.0 ** -18 * np.asarray(L, dtype=np.float64) * max_a * max_b
