"""A ragged grouped linear layer for torch autograd, on the C-ABI kernels.

    Y = grouped_linear(X, W, offsets)          # Y[r] = X[r] @ W[e]^T for rows r of expert e

Forward runs the grouped GEMM's forward pass; backward runs its data gradient
(dX = G W_e) and weight gradient (dW_e = G_e^T X_e), the three passes of the
MoE expert layer (flashinfer PR #8258, opening summary).  Under
``torch.utils.checkpoint`` the forward runs again before the backward: the
pages' "ckpt" operation (forward + backward with the forward recomputed).

    Y = checkpointed_grouped_linear(X, W, offsets, early_stop=True)

is the pages' pair of checkpointed operations (PR #8258, "Operations and
shapes": one grouped GEMM in a non-reentrant checkpoint, early stop off =
"ckpt", on = "ckpt ES").  The backward needs only the layer's inputs, which
the recompute saves again before anything else; with early stop on, the
checkpoint stops the recompute as soon as those are saved, so the recomputed
forward's output is never read and its GEMM is not launched (the pages credit
their earlier PR #8114 with skipping that recompute).  With early stop off
the recompute runs the forward GEMM, as stock checkpointing does.

This module only marshals arguments: every pass runs in libcake_gg.so.  Plans
and workspaces are cached per (pass, shape, dtype, mode, device, stream) and
reused across calls, as the workspace contract allows (zero-filled once,
ready again after every call, calls on one workspace ordered on one stream).
Rows at or past offsets[E] of Y and dX are left unwritten (uninitialised).
"""
from __future__ import annotations

import contextlib
import threading

from . import cake_gg as gg

_cache: dict = {}
# set while a checkpointed_grouped_linear with early stop recomputes its forward
_recompute = threading.local()


def _plan_ws(pass_, E, M, N, K, out_dtype, det, device, stream):
    key = (pass_, E, M, N, K, out_dtype, bool(det), str(device), int(stream))
    hit = _cache.get(key)
    if hit is None:
        plan = gg.cake_gg_plan(pass_, E, M, N, K, out_dtype, det)
        hit = (plan, gg.make_workspace(plan, device))
        _cache[key] = hit
    return hit


def _run(pass_, a, b, offsets, out_shape, out_dtype, det, E, M, N, K):
    import torch
    stream = torch.cuda.current_stream(a.device).cuda_stream
    plan, ws = _plan_ws(pass_, E, M, N, K, out_dtype, det, a.device, stream)
    out = torch.empty(out_shape, dtype=torch.float32 if out_dtype == "fp32" else torch.bfloat16, device=a.device)
    fn = {"fwd": gg.cake_gg_fwd, "dgrad": gg.cake_gg_dgrad, "wgrad": gg.cake_gg_wgrad}[pass_]
    rc = fn(plan, a, b, out, offsets, out_dtype, det, ws, stream=stream)
    if rc != gg.CAKE_GG_OK:
        raise gg.CakeGGError(rc, f"grouped_linear {pass_}")
    return out


def _make_function():
    import torch

    class GroupedLinear(torch.autograd.Function):
        """Y = X W_e^T per expert group; BF16 in and out, FP32 accumulation."""

        @staticmethod
        def forward(ctx, X, W, offsets, deterministic, wgrad_dtype):
            if X.dtype != torch.bfloat16 or W.dtype != torch.bfloat16:
                raise TypeError("grouped_linear takes BF16 X and W")
            if offsets.dtype != torch.int32:
                raise TypeError("offsets must be int32 [E+1]")
            X, W = X.contiguous(), W.contiguous()
            E, N, K = int(W.shape[0]), int(W.shape[1]), int(W.shape[2])
            M = int(X.shape[0])
            if int(offsets.numel()) != E + 1 or int(X.shape[1]) != K:
                raise ValueError("shapes: X [M, K], W [E, N, K], offsets [E+1]")
            ctx.save_for_backward(X, W, offsets)
            ctx.det, ctx.wgrad_dtype = bool(deterministic), wgrad_dtype
            if getattr(_recompute, "skip_forward", False):
                # an early-stopped recompute: only the saved inputs are kept, the
                # output is discarded unread, so the GEMM is not launched
                return torch.empty((M, N), dtype=torch.bfloat16, device=X.device)
            return _run("fwd", X, W, offsets, (M, N), "bf16", ctx.det, E, M, N, K)

        @staticmethod
        def backward(ctx, G):
            X, W, offsets = ctx.saved_tensors
            G = G.contiguous()
            if G.dtype != torch.bfloat16:
                G = G.to(torch.bfloat16)
            E, N, K = int(W.shape[0]), int(W.shape[1]), int(W.shape[2])
            M = int(X.shape[0])
            dX = dW = None
            if ctx.needs_input_grad[0]:
                dX = _run("dgrad", G, W, offsets, (M, K), "bf16", ctx.det, E, M, N, K)
            if ctx.needs_input_grad[1]:
                dW = _run("wgrad", G, X, offsets, (E, N, K), ctx.wgrad_dtype, ctx.det, E, M, N, K)
                if dW.dtype != W.dtype:
                    dW = dW.to(W.dtype)
            return dX, dW, None, None, None

    return GroupedLinear


_fn = None


def grouped_linear(X, W, offsets, deterministic=True, wgrad_dtype="bf16"):
    """Y [M, N] = X [M, K] @ W[e]^T for the rows [offsets[e], offsets[e+1]) of each expert e.

    Differentiable in X and W.  ``wgrad_dtype`` = "fp32" accumulates the weight
    gradient's output in FP32 before it is cast to W's dtype for autograd.
    """
    global _fn
    if _fn is None:
        _fn = _make_function()
    return _fn.apply(X, W, offsets, deterministic, wgrad_dtype)


@contextlib.contextmanager
def _recompute_without_forward():
    prev = getattr(_recompute, "skip_forward", False)
    _recompute.skip_forward = True
    try:
        yield
    finally:
        _recompute.skip_forward = prev


def checkpointed_grouped_linear(X, W, offsets, early_stop=True, deterministic=True, wgrad_dtype="bf16"):
    """grouped_linear inside a non-reentrant ``torch.utils.checkpoint``.

    ``early_stop`` False: the pages' "ckpt" -- forward, then in the backward the
    forward recomputed, the data gradient and the weight gradient (2 x fwd + bwd).
    ``early_stop`` True: "ckpt ES" -- the checkpoint stops its recompute once the
    layer's inputs are saved again, which happens before the forward GEMM would
    run, so the backward launches only the data and weight gradients.  Results
    are bitwise those of the plain grouped_linear in deterministic mode.
    """
    import torch
    from torch.utils.checkpoint import checkpoint, set_checkpoint_early_stop

    def contexts():
        return contextlib.nullcontext(), (_recompute_without_forward() if early_stop
                                          else contextlib.nullcontext())

    with set_checkpoint_early_stop(bool(early_stop)):
        return checkpoint(grouped_linear, X, W, offsets, deterministic, wgrad_dtype,
                          use_reentrant=False, context_fn=contexts)
