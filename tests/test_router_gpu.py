"""GPU parity of the FP32 router GEMM (BF16x3 emulation) against the FP64 oracle.

The dense projection family's router GEMM (flashinfer PR #8438, "Summary": a
router GEMM over 256 experts in FP32, emulated with three BF16 products):
logits Y = X W^T from
FP32 X [T, K] and W [R, K].  Every call goes through the C ABI
(cake_gg_router_plan / cake_gg_router_fp32).  The GPU result is compared with
the oracle's emulation (same split, exact products, FP64 sum) under the FP32
accumulation bound, and with the definition X W^T under that bound plus the
emulation's own 3 * 2^-16 sum|x w|.
"""
import numpy as np
import pytest

import oracle
from moe_ragged_grouped_gb300 import cake_gg as gg
from moe_ragged_grouped_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


def _run(X, W, extra_rows=0, max_sms=0):
    import torch
    T, R = X.shape[0], W.shape[0]
    Xd = torch.from_numpy(X).cuda()
    Wd = torch.from_numpy(W).cuda()
    Ybuf = torch.full((T + extra_rows, R), float("nan"), dtype=torch.float32, device="cuda")
    Y = gg.router_gemm(Xd, Wd, max_sms=max_sms, out=Ybuf[:T])
    torch.cuda.synchronize()
    full = Ybuf.cpu().numpy()
    if extra_rows:
        assert np.all(np.isnan(full[T:])), "rows past T were written"
    return full[:T].astype(np.float64)


def _check(gpu, X, W, lib):
    emu = oracle.router_bf16x3(X, W, lib)
    ref = oracle.router_exact(X, W, lib)
    abs_dot = np.abs(X).astype(np.float64) @ np.abs(W).astype(np.float64).T
    tol = oracle.router_tolerance(abs_dot, 3 * X.shape[1])
    err_emu = np.abs(gpu - emu)
    assert np.all(err_emu <= tol), f"max err vs emulation {np.max(err_emu / np.maximum(tol, 1e-300)):.3f} x tol"
    err_ref = np.abs(gpu - ref)
    assert np.all(err_ref <= tol + oracle.router_emulation_bound(abs_dot))
    return float(np.max(err_ref / np.maximum(abs_dot, 1e-300)))


@pytest.mark.parametrize("T,K,R", [(300, 200, 256), (129, 64, 8), (1000, 1096, 256), (257, 8, 16)])
def test_router_matches_oracle(T, K, R, oracle_lib):
    X, W = wl.router_inputs(T, K, R, seed=T + K)
    rel = _check(_run(X, W, extra_rows=3), X, W, oracle_lib)
    assert rel < 2.0 ** -14   # far more accurate than one BF16 product (2^-8)


def test_router_beats_plain_bf16(oracle_lib):
    """The emulation is well inside the error of rounding X and W to BF16 once (what it replaces)."""
    X, W = wl.router_inputs(256, 512, 64, seed=5)
    gpu = _run(X, W)
    ref = oracle.router_exact(X, W, oracle_lib)
    Xb = np.vectorize(lambda v: oracle.round_bf16(v, oracle_lib))(X).astype(np.float64)
    Wb = np.vectorize(lambda v: oracle.round_bf16(v, oracle_lib))(W).astype(np.float64)
    plain = Xb @ Wb.T
    assert np.max(np.abs(gpu - ref)) * 64 < np.max(np.abs(plain - ref))


def test_router_exact_for_small_integers(oracle_lib):
    """BF16-representable inputs with small integer values: every partial sum is exact in FP32,
    so the GPU equals the definition bitwise."""
    rng = np.random.default_rng(7)
    X = rng.integers(-8, 9, (300, 128)).astype(np.float32)
    W = rng.integers(-8, 9, (32, 128)).astype(np.float32)
    gpu = _run(X, W)
    np.testing.assert_array_equal(gpu, oracle.router_exact(X, W, oracle_lib))


def test_router_no_tokens():
    import torch
    W = torch.randn(256, 64, device="cuda")
    X = torch.empty(0, 64, device="cuda")
    Y = gg.router_gemm(X, W)
    assert Y.shape == (0, 256)


def test_router_deterministic_and_sm_cap_invariant():
    import torch
    X, W = wl.router_inputs(1000, 512, 256, seed=9)
    a = _run(X, W)
    b = _run(X, W)
    c = _run(X, W, max_sms=10)
    assert np.array_equal(a.view(np.int64), b.view(np.int64))
    assert np.array_equal(a.view(np.int64), c.view(np.int64))


def test_router_full_size_sampled(oracle_lib):
    """T = 16384, K = 4096, R = 256 (the benchmark's router workload) on sampled logits."""
    import torch
    T, K, R = wl.ROUTER_T, wl.ROUTER_K, wl.ROUTER_R
    Xd, Wd = wl.router_inputs_torch(T, K, R, seed=0)
    Y = gg.router_gemm(Xd, Wd)
    torch.cuda.synchronize()
    X, W = Xd.cpu().numpy(), Wd.cpu().numpy()
    rng = np.random.default_rng(1)
    ts = np.concatenate([rng.integers(0, T, 2000), [0, T - 1, 127, 128, 255, 256]])
    rs = np.concatenate([rng.integers(0, R, 2000), [0, R - 1, 0, R - 1, 128, 127]])
    emu = oracle.router_bf16x3_at(X, W, ts, rs, oracle_lib)
    abs_dot = np.einsum("ik,ik->i", np.abs(X[ts]).astype(np.float64), np.abs(W[rs]).astype(np.float64))
    gpu = Y.cpu().numpy()[ts, rs].astype(np.float64)
    assert np.all(np.abs(gpu - emu) <= oracle.router_tolerance(abs_dot, 3 * K))


def test_router_full_size_every_logit_and_bitwise(oracle_lib):
    """T = 16384, K = 4096, R = 256, every logit: within the emulation's bound of the
    definition X W^T (summed in FP64), and bitwise equal across repeated calls and an SM
    cap (a k-block whose split A tile were read before it was written, or overwritten
    while read, would break both)."""
    import torch
    T, K, R = wl.ROUTER_T, wl.ROUTER_K, wl.ROUTER_R
    Xd, Wd = wl.router_inputs_torch(T, K, R, seed=3)
    runs = []
    for cap in (0, 0, 0, 64):
        runs.append(gg.router_gemm(Xd, Wd, max_sms=cap).cpu().numpy())
    for r in runs[1:]:
        assert np.array_equal(runs[0].view(np.int32), r.view(np.int32))
    X, W = Xd.cpu().numpy().astype(np.float64), Wd.cpu().numpy().astype(np.float64)
    ref = X @ W.T
    abs_dot = np.abs(X) @ np.abs(W).T
    tol = oracle.router_tolerance(abs_dot, 3 * K) + oracle.router_emulation_bound(abs_dot)
    assert np.all(np.abs(runs[0].astype(np.float64) - ref) <= tol)
