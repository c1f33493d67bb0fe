"""The autograd layer over the C-ABI kernels: gradients against the FP64 oracle, and the
checkpointed step -- "ckpt" (forward recomputed before the backward) and "ckpt ES" (early
stop: the recompute launches no GEMM), the pages' checkpointed operations (PR #8258,
"Operations and shapes")."""
import numpy as np
import pytest

import oracle
from moe_ragged_grouped_gb300 import workloads as wl


def test_rejects_wrong_dtypes_before_any_device_work():
    import torch
    from moe_ragged_grouped_gb300.autograd import grouped_linear
    X = torch.zeros(4, 8)
    W = torch.zeros(1, 8, 8)
    with pytest.raises(TypeError):
        grouped_linear(X, W, torch.tensor([0, 4], dtype=torch.int32))
    with pytest.raises(TypeError):
        grouped_linear(X.bfloat16(), W.bfloat16(), torch.tensor([0, 4], dtype=torch.int64))


def _setup(sizes, N, K, seed):
    """Device tensors and their host BF16 bits (the oracle's inputs)."""
    import torch
    from moe_ragged_grouped_gb300 import build as gg_build
    from moe_ragged_grouped_gb300 import cake_gg as gg
    gg_build.build()
    gg.load_library()
    rng = np.random.default_rng(seed)
    E, M = len(sizes), sum(sizes)
    bits = (wl.randn_bf16((M, K), 1.0, rng), wl.randn_bf16((E, N, K), K ** -0.5, rng),
            wl.randn_bf16((M, N), 1.0, rng))   # X, W, upstream gradient R
    X, W, R = (wl.to_torch_bf16(b, "cuda") for b in bits)
    off = torch.from_numpy(wl.offsets_from_sizes(sizes)).cuda()
    return X, W, R, off, bits


def _bits(t):
    import torch
    return wl.torch_bf16_to_bits(t.detach().to(torch.bfloat16))


def _assert_oracle_parity(Y, dX, dW, bits, off):
    """Y, dX, dW against the FP64 oracle on the same BF16 bits, under the parity bound
    |gpu - ref| <= 2^-8 |ref| + 2^-18 L max|a| max|b| with the operands' true maxima."""
    Xb, Wb, Rb = bits
    o = off.cpu().numpy()
    M = int(o[-1])
    f = lambda a: float(np.abs(oracle.bf16_bits_to_f64(a)).max()) if a.size else 0.0
    N, K = Wb.shape[1], Wb.shape[2]
    L_w = np.broadcast_to(np.diff(o).astype(np.float64)[:, None, None], Wb.shape)
    cases = (("Y", Y[:M], oracle.fwd(Xb, Wb, o), K, f(Xb[:M]), f(Wb)),
             ("dX", dX[:M], oracle.dgrad(Rb, Wb, o), N, f(Rb[:M]), f(Wb)),
             ("dW", dW, oracle.wgrad(Rb, Xb, o, Wb.shape[0]), L_w, f(Rb[:M]), f(Xb[:M])))
    for name, got_t, ref, L, ma, mb in cases:
        got = oracle.bf16_bits_to_f64(_bits(got_t)).reshape(ref.shape)
        tol = oracle.tolerance(ref, L, ma, mb)
        bad = ~(np.abs(got - ref) <= tol)
        assert not bad.any(), f"{name}: {int(bad.sum())} of {bad.size} elements outside the parity bound"


@pytest.mark.gpu
@pytest.mark.parametrize("wgrad_dtype", ["bf16", "fp32"])
def test_gradients_match_the_oracle(wgrad_dtype):
    """Y, dX and dW of one forward + backward against the FP64 oracle (an empty expert gets an
    exact zero dW: its bound is 0); with wgrad_dtype = fp32 the weight gradient is accumulated
    into FP32 output and then rounded once more to W's BF16 for autograd."""
    from moe_ragged_grouped_gb300.autograd import grouped_linear
    sizes, N, K = [0, 700, 1300, 33], 384, 512
    X, W, R, off, bits = _setup(sizes, N, K, seed=31)
    Xg, Wg = X.clone().requires_grad_(), W.clone().requires_grad_()
    Y = grouped_linear(Xg, Wg, off, wgrad_dtype=wgrad_dtype)
    Y.backward(R)
    _assert_oracle_parity(Y, Xg.grad, Wg.grad, bits, off)


def _cpu_stand_in(calls):
    """A CPU stand-in for the C-ABI launch (host logic only): records the pass and computes it
    with torch on the CPU, so the checkpoint's launch sequence can be observed without a GPU."""
    import torch

    def run(pass_, a, b, offsets, out_shape, out_dtype, det, E, M, N, K):
        calls.append(pass_)
        o = offsets.tolist()
        out = torch.zeros(out_shape, dtype=torch.float64)
        for e in range(E):
            r0, r1 = o[e], o[e + 1]
            if pass_ == "fwd":
                out[r0:r1] = a[r0:r1].double() @ b[e].double().T
            elif pass_ == "dgrad":
                out[r0:r1] = a[r0:r1].double() @ b[e].double()
            else:
                out[e] = a[r0:r1].double().T @ b[r0:r1].double()
        return out.to(torch.bfloat16)
    return run


def test_checkpoint_early_stop_skips_the_recomputed_forward(monkeypatch):
    """Launch sequence of one forward + backward: plain = fwd, dgrad, wgrad; "ckpt" (early stop
    off) = fwd, fwd again, dgrad, wgrad; "ckpt ES" = fwd, dgrad, wgrad.  Results equal the plain
    step's bitwise in both checkpointed modes (the skipped recompute's output is never read)."""
    import torch
    from moe_ragged_grouped_gb300 import autograd as ag
    calls = []
    monkeypatch.setattr(ag, "_run", _cpu_stand_in(calls))
    g = torch.Generator().manual_seed(5)
    X = torch.randn(37, 16, generator=g).bfloat16()
    W = torch.randn(3, 24, 16, generator=g).bfloat16()
    off = torch.tensor([0, 20, 20, 37], dtype=torch.int32)
    R = torch.randn(37, 24, generator=g).bfloat16()
    seen, res = {}, {}
    for mode in ("plain", "ckpt", "ckpt ES"):
        calls.clear()
        Xg, Wg = X.clone().requires_grad_(), W.clone().requires_grad_()
        if mode == "plain":
            Y = ag.grouped_linear(Xg, Wg, off)
        else:
            Y = ag.checkpointed_grouped_linear(Xg, Wg, off, early_stop=(mode == "ckpt ES"))
        Y.backward(R)
        seen[mode] = list(calls)
        res[mode] = (Y.detach(), Xg.grad, Wg.grad)
    assert seen == {"plain": ["fwd", "dgrad", "wgrad"], "ckpt": ["fwd", "fwd", "dgrad", "wgrad"],
                    "ckpt ES": ["fwd", "dgrad", "wgrad"]}
    for mode in ("ckpt", "ckpt ES"):
        for a, b in zip(res["plain"], res[mode]):
            assert torch.equal(a, b), mode


@pytest.mark.gpu
def test_checkpointed_steps_equal_plain_step_bitwise():
    """The plain step, torch's own checkpoint around grouped_linear, and the "ckpt" / "ckpt ES"
    entry point give the same bits; the plain step's gradients are also checked against the
    oracle."""
    import torch
    from torch.utils.checkpoint import checkpoint
    from moe_ragged_grouped_gb300.autograd import checkpointed_grouped_linear, grouped_linear
    X, W, R, off, bits = _setup([5000, 1900, 0, 1200], 512, 768, seed=32)
    grads = []
    for mode in ("plain", "torch", "torch", "ckpt", "ckpt ES", "ckpt ES"):
        Xg, Wg = X.clone().requires_grad_(), W.clone().requires_grad_()
        if mode == "torch":
            Y = checkpoint(grouped_linear, Xg, Wg, off, use_reentrant=False)
        elif mode == "plain":
            Y = grouped_linear(Xg, Wg, off)
        else:
            Y = checkpointed_grouped_linear(Xg, Wg, off, early_stop=(mode == "ckpt ES"))
        (Y.float() * R.float()).sum().backward()
        grads.append((Y.detach().clone(), Xg.grad.clone(), Wg.grad.clone()))
    _assert_oracle_parity(*grads[0], bits, off)
    for i in range(1, len(grads)):
        for a, b in zip(grads[0], grads[i]):
            assert torch.equal(a.view(torch.int16), b.view(torch.int16)), i
