"""The autograd layer over the C-ABI kernels: gradients, and the checkpointed step
(forward recomputed before the backward: the pages' "ckpt" operation)."""
import numpy as np
import pytest

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
    import torch
    from moe_ragged_grouped_gb300 import build as gg_build
    from moe_ragged_grouped_gb300 import cake_gg as gg
    gg_build.build()
    gg.load_library()
    rng = np.random.default_rng(seed)
    E, M = len(sizes), sum(sizes)
    X = wl.to_torch_bf16(wl.randn_bf16((M, K), 1.0, rng), "cuda")
    W = wl.to_torch_bf16(wl.randn_bf16((E, N, K), K ** -0.5, rng), "cuda")
    R = wl.to_torch_bf16(wl.randn_bf16((M, N), 1.0, rng), "cuda")   # upstream gradient
    off = torch.from_numpy(wl.offsets_from_sizes(sizes)).cuda()
    return X, W, R, off


@pytest.mark.gpu
@pytest.mark.parametrize("wgrad_dtype", ["bf16", "fp32"])
def test_gradients_match_fp32_reference(wgrad_dtype):
    import torch
    from moe_ragged_grouped_gb300.autograd import grouped_linear
    sizes, N, K = [0, 700, 1300, 33], 384, 512
    X, W, R, off = _setup(sizes, N, K, seed=31)
    Xg, Wg = X.clone().requires_grad_(), W.clone().requires_grad_()
    Y = grouped_linear(Xg, Wg, off, wgrad_dtype=wgrad_dtype)
    Y.backward(R)
    o = off.cpu().numpy()
    for e in range(len(sizes)):
        r0, r1 = int(o[e]), int(o[e + 1])
        if r1 == r0:
            assert bool((Wg.grad[e] == 0).all())  # empty expert: exact zero weight gradient
            continue
        x, w, g = X[r0:r1].float(), W[e].float(), R[r0:r1].float()
        for got, ref, L, ma, mb in ((Y[r0:r1], x @ w.T, K, x, w), (Xg.grad[r0:r1], g @ w, N, g, w),
                                    (Wg.grad[e], g.T @ x, max(r1 - r0, 1), g, x)):
            tol = 2.0 ** -8 * ref.abs() + 2.0 ** -18 * L * ma.abs().max().clamp(min=1) * mb.abs().max().clamp(min=1)
            assert bool(((got.float() - ref).abs() <= tol + 1e-30).all()), f"expert {e}"


@pytest.mark.gpu
def test_checkpointed_step_equals_plain_step_bitwise():
    import torch
    from torch.utils.checkpoint import checkpoint
    from moe_ragged_grouped_gb300.autograd import grouped_linear
    X, W, R, off = _setup([5000, 1900, 0, 1200], 512, 768, seed=32)
    grads = []
    for use_ckpt in (False, True, True):
        Xg, Wg = X.clone().requires_grad_(), W.clone().requires_grad_()
        if use_ckpt:
            Y = checkpoint(grouped_linear, Xg, Wg, off, use_reentrant=False)
        else:
            Y = grouped_linear(Xg, Wg, off)
        (Y.float() * R.float()).sum().backward()
        grads.append((Y.detach().clone(), Xg.grad.clone(), Wg.grad.clone()))
    for i in (1, 2):
        for a, b in zip(grads[0], grads[i]):
            assert torch.equal(a.view(torch.int16), b.view(torch.int16))
