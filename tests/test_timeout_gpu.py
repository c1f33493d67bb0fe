"""Bounded waits: a stage that never fills makes the kernel report a timeout.

With the test-only plan flag CAKE_GG_DEBUG_DROP_FIRST_LOAD, CTA 0 arms its
first pipeline stage (expects the bytes) but issues no copy into it.  Every
wait in the kernel is bounded by plan.timeout_ns, so the consumer gives up,
the status word reads CAKE_GG_ERR_TIMEOUT, the CTAs drain what they issued,
free their tensor memory and return: no trap, no hang.  The context stays
usable: the next regular call on the same tensors is correct.
"""
import numpy as np
import pytest

import oracle
from moe_ragged_grouped_gb300 import build as gg_build
from moe_ragged_grouped_gb300 import cake_gg as gg
from moe_ragged_grouped_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def lib():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    gg_build.build()
    return gg.load_library()


@pytest.mark.parametrize("pair_env", [None, "0"])
@pytest.mark.parametrize("pass_", ["fwd", "wgrad"])
def test_dropped_copy_times_out_and_context_survives(pass_, pair_env, monkeypatch):
    import torch
    if pair_env is not None:
        monkeypatch.setenv("CAKE_GG_PAIR", pair_env)
    wk = wl.tiny()
    Xb, Wb, Gb = wk.make_numpy(seed=0)
    off = wk.offsets
    X, W, G = (wl.to_torch_bf16(a, "cuda") for a in (Xb, Wb, Gb))
    offs = torch.from_numpy(off).cuda()
    a, b = (X, W) if pass_ == "fwd" else (G, X)
    plan = gg.cake_gg_plan(pass_, wk.E, wk.M, wk.N, wk.K, "fp32", 1)
    plan.debug_flags = gg.CAKE_GG_DEBUG_DROP_FIRST_LOAD
    plan.timeout_ns = 100_000_000  # 0.1 s
    ws = gg.make_workspace(plan, "cuda")
    shape = (wk.M, wk.N) if pass_ == "fwd" else (wk.E, wk.N, wk.K)
    out = torch.zeros(shape, dtype=torch.float32, device="cuda")
    fn = gg.cake_gg_fwd if pass_ == "fwd" else gg.cake_gg_wgrad
    assert fn(plan, a, b, out, offs, "fp32", 1, ws) == gg.CAKE_GG_OK
    assert gg.cake_gg_check_status(ws) == gg.CAKE_GG_ERR_TIMEOUT
    # the same context, a regular plan: correct results
    good = gg.grouped_gemm(pass_, a, b, offs, out_dtype="fp32", deterministic=1)
    torch.cuda.synchronize()
    ref = oracle.fwd(Xb, Wb, off) if pass_ == "fwd" else oracle.wgrad(Gb, Xb, off, wk.E)
    got = good.double().cpu().numpy()
    L = wk.K if pass_ == "fwd" else 128
    f = lambda t: float(np.abs(oracle.bf16_bits_to_f64(t)).max())
    ma, mb = (f(Xb), f(Wb)) if pass_ == "fwd" else (f(Gb), f(Xb))
    assert (np.abs(got - ref) <= oracle.tolerance(ref, L, ma, mb)).all()


def test_dropped_copy_in_a_cluster_split_times_out_and_context_survives():
    """A thin weight gradient (d_out = 48, K = 1024, 4096 rows) runs each output tile as a
    cluster of eight splits that push their FP32 partial slices into each other's shared memory.
    Rank 0 of the first cluster loses its first copy: its MMA and epilogue give up, it lets the
    slices its peers pushed to it land before retiring, and its peers -- which never receive rank
    0's parts -- give up on their own bounded waits.  The call reports CAKE_GG_ERR_TIMEOUT and
    the next regular call on the same tensors is correct."""
    import torch
    E, M, N, K = 1, 4096, 48, 1024
    rng = np.random.default_rng(41)
    Xb = wl.randn_bf16((M, K), 1.0, rng)
    Gb = wl.randn_bf16((M, N), 1.0, rng)
    off = wl.offsets_from_sizes([M])
    X, G = wl.to_torch_bf16(Xb, "cuda"), wl.to_torch_bf16(Gb, "cuda")
    offs = torch.from_numpy(off).cuda()
    plan = gg.cake_gg_plan("wgrad", E, M, N, K, "fp32", 1)
    assert plan.cluster_splits == 8 and plan.swap_ab == 1
    plan.debug_flags = gg.CAKE_GG_DEBUG_DROP_FIRST_LOAD
    plan.timeout_ns = 100_000_000  # 0.1 s
    ws = gg.make_workspace(plan, "cuda")
    out = torch.zeros((E, N, K), dtype=torch.float32, device="cuda")
    assert gg.cake_gg_wgrad(plan, G, X, out, offs, "fp32", 1, ws) == gg.CAKE_GG_OK
    assert gg.cake_gg_check_status(ws) == gg.CAKE_GG_ERR_TIMEOUT
    good = gg.grouped_gemm("wgrad", G, X, offs, out_dtype="fp32", deterministic=1)
    torch.cuda.synchronize()
    ref = oracle.wgrad(Gb, Xb, off, E)
    f = lambda t: float(np.abs(oracle.bf16_bits_to_f64(t)).max())
    assert (np.abs(good.double().cpu().numpy() - ref) <= oracle.tolerance(ref, M, f(Gb), f(Xb))).all()


@pytest.mark.parametrize("csplit,wide", [("2", False), ("3", True)])
def test_dropped_copy_in_a_pair_cluster_split_times_out_and_context_survives(csplit, wide, monkeypatch):
    """A weight gradient of 256-row pair tiles whose splits run as one cluster of pairs and
    reduce into each other's operand rings (256 x 512 tiles: in rounds over column windows).
    The even CTA of the first cluster's first pair loses its first copy: that pair's MMA never
    completes, the other pairs wait in vain for the first pair's ring to be offered, and every
    role gives up on its bounded wait.  The call reports CAKE_GG_ERR_TIMEOUT and the next
    regular call is correct."""
    import torch
    monkeypatch.setenv("CAKE_GG_CSPLIT", csplit)
    if wide:
        monkeypatch.setenv("CAKE_GG_WIDE", "2")
    E, M, N, K = (1, 8300, 256, 1152) if wide else (1, 3000, 512, 512)
    rng = np.random.default_rng(42)
    Xb = wl.randn_bf16((M, K), 1.0, rng)
    Gb = wl.randn_bf16((M, N), 1.0, rng)
    off = wl.offsets_from_sizes([M])
    X, G = wl.to_torch_bf16(Xb, "cuda"), wl.to_torch_bf16(Gb, "cuda")
    offs = torch.from_numpy(off).cuda()
    plan = gg.cake_gg_plan("wgrad", E, M, N, K, "fp32", 1)
    assert plan.cluster_splits == int(csplit) and plan.pair == 2 and plan.tile_n == (512 if wide else 256)
    plan.debug_flags = gg.CAKE_GG_DEBUG_DROP_FIRST_LOAD
    plan.timeout_ns = 100_000_000  # 0.1 s
    ws = gg.make_workspace(plan, "cuda")
    out = torch.zeros((E, N, K), dtype=torch.float32, device="cuda")
    assert gg.cake_gg_wgrad(plan, G, X, out, offs, "fp32", 1, ws) == gg.CAKE_GG_OK
    assert gg.cake_gg_check_status(ws) == gg.CAKE_GG_ERR_TIMEOUT
    good = gg.grouped_gemm("wgrad", G, X, offs, out_dtype="fp32", deterministic=1)
    torch.cuda.synchronize()
    ref = oracle.wgrad(Gb, Xb, off, E)
    f = lambda t: float(np.abs(oracle.bf16_bits_to_f64(t)).max())
    assert (np.abs(good.double().cpu().numpy() - ref) <= oracle.tolerance(ref, M, f(Gb), f(Xb))).all()
