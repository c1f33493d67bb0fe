"""Shared helpers of the GPU parity tests: run a pass through the C ABI on
seeded inputs and compare it with the FP64 oracle under the parity bound

    |gpu - ref| <= 2^-8 |ref| + 2^-18 * L * max|a| * max|b|

with L the element's reduction length (K forward, N data gradient, the
expert's row count weight gradient) and max|a|, max|b| the maxima of the
pass's two input operands.
"""
from __future__ import annotations

import numpy as np

import oracle
from moe_ragged_grouped_gb300 import cake_gg as gg
from moe_ragged_grouped_gb300 import workloads as wl

SENTINEL_BF16 = 0x7FC1          # a NaN bit pattern
SENTINEL_F32 = 0x7FC00001


def to_dev(bits, device="cuda"):
    return wl.to_torch_bf16(bits, device)


def out_to_f64(t):
    import torch
    if t.dtype == torch.bfloat16:
        return oracle.bf16_bits_to_f64(wl.torch_bf16_to_bits(t))
    return t.detach().to("cpu").double().numpy()


def guarded_empty(shape, out_dtype, device="cuda", guard=4096):
    """An output view with sentinel-filled guard bands before and after it."""
    import torch
    n = int(np.prod(shape))
    if out_dtype == "fp32":
        buf = torch.empty(n + 2 * guard, dtype=torch.int32, device=device).fill_(SENTINEL_F32)
        view = buf[guard:guard + n].view(torch.float32).view(shape)
    else:
        buf = torch.empty(n + 2 * guard, dtype=torch.int16, device=device).fill_(SENTINEL_BF16)
        view = buf[guard:guard + n].view(torch.bfloat16).view(shape)
    return buf, view, guard


def guards_intact(buf, guard, n, out_dtype):
    b = buf.to("cpu").numpy()
    s = SENTINEL_F32 if out_dtype == "fp32" else np.int16(SENTINEL_BF16)
    return bool((b[:guard] == s).all() and (b[guard + n:] == s).all())


def run(pass_, X, W, G, off, out_dtype, det, max_sms=0, out=None, plan=None, workspace=None):
    """Run one pass through the C ABI (device tensors in, device tensor out)."""
    import torch
    offs = torch.from_numpy(np.ascontiguousarray(off, np.int32)).to(X.device)
    if pass_ == "fwd":
        a, b = X, W
    elif pass_ == "dgrad":
        a, b = G, W
    else:
        a, b = G, X
    return gg.grouped_gemm(pass_, a, b, offs, out_dtype=out_dtype, deterministic=det, max_sms=max_sms,
                           out=out, plan=plan, workspace=workspace)


def reference(pass_, Xb, Wb, Gb, off):
    """FP64 oracle output (numpy) from uint16 BF16 bits."""
    E = Wb.shape[0]
    if pass_ == "fwd":
        return oracle.fwd(Xb, Wb, off)
    if pass_ == "dgrad":
        return oracle.dgrad(Gb, Wb, off)
    return oracle.wgrad(Gb, Xb, off, E)


def reduction_lengths(pass_, off, N, K, shape):
    if pass_ == "fwd":
        return np.full(shape, K, np.float64)
    if pass_ == "dgrad":
        return np.full(shape, N, np.float64)
    sizes = np.diff(off).astype(np.float64)
    return np.broadcast_to(sizes[:, None, None], shape)


def operand_maxima(pass_, Xb, Wb, Gb, off):
    M = int(off[-1])
    mx = lambda a: float(np.abs(oracle.bf16_bits_to_f64(a)).max()) if a.size else 0.0
    if pass_ == "fwd":
        return mx(Xb[:M]), mx(Wb)
    if pass_ == "dgrad":
        return mx(Gb[:M]), mx(Wb)
    return mx(Gb[:M]), mx(Xb[:M])


def assert_parity(pass_, got, ref, Xb, Wb, Gb, off, what=""):
    N, K = Wb.shape[1], Wb.shape[2]
    L = reduction_lengths(pass_, off, N, K, ref.shape)
    ma, mb = operand_maxima(pass_, Xb, Wb, Gb, off)
    tol = oracle.tolerance(ref, L, ma, mb)
    err = np.abs(got - ref)
    bad = ~(err <= tol)
    if bad.any():
        idx = np.argwhere(bad)[:5]
        raise AssertionError(
            f"{what}: {int(bad.sum())} of {bad.size} elements outside the parity bound; "
            f"first {idx.tolist()}: got {[float(got[tuple(i)]) for i in idx]} "
            f"ref {[float(ref[tuple(i)]) for i in idx]}")
    return float((err / np.maximum(tol, 1e-300)).max()) if err.size else 0.0
