"""The no-allocation weight-gradient entry point against the regular one.

cake_gg_wgrad_noalloc serves callers that cannot allocate device memory (for
example a custom-operator interface that passes only input / output pointers
and a stream, or a training loop that must not allocate once it runs).  It
uses a fixed scratch array inside the library instead of a caller workspace.
Here its output, on two calls in a row, must match cake_gg_wgrad's output on
the same inputs within the parity bound the other tests use (and bitwise in
deterministic mode, where both follow the same fixed summation order), and
the FP64 oracle's within that bound.

This file is collected last so that a run stopping at the first failure has
already run every other test.
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


def _inputs(sizes, N, K, seed):
    rng = np.random.default_rng(seed)
    E, M = len(sizes), sum(sizes) + 3
    Xb = wl.randn_bf16((M, K), 1.0, rng)
    Gb = wl.randn_bf16((M, N), 1.0, rng)
    return Xb, Gb, wl.offsets_from_sizes(sizes)


def _f64(t):
    import torch
    if t.dtype == torch.bfloat16:
        return oracle.bf16_bits_to_f64(wl.torch_bf16_to_bits(t))
    return t.double().cpu().numpy()


@pytest.mark.parametrize("sizes,N,K,env", [
    ([3000], 48, 512, None),                 # thin: operands swapped, split reduction
    ([0, 700, 1500, 33], 128, 256, "3"),     # ragged, empty expert, forced split
    ([400, 900], 192, 320, None),            # no split
])
@pytest.mark.parametrize("out_dtype", ["fp32", "bf16"])
@pytest.mark.parametrize("det", [1, 0])
def test_noalloc_matches_workspace_entry_point(sizes, N, K, env, out_dtype, det, monkeypatch):
    import torch
    if env:
        monkeypatch.setenv("CAKE_GG_SPLIT_CHUNK", env)
    Xb, Gb, off = _inputs(sizes, N, K, seed=21)
    E, M = len(sizes), Xb.shape[0]
    X, G = wl.to_torch_bf16(Xb, "cuda"), wl.to_torch_bf16(Gb, "cuda")
    offs = torch.from_numpy(off).cuda()
    plan = gg.cake_gg_plan("wgrad", E, M, N, K, out_dtype, det)
    assert plan.workspace_bytes <= gg.CAKE_GG_NOALLOC_SCRATCH_BYTES
    ref = gg.grouped_gemm("wgrad", G, X, offs, out_dtype=out_dtype, deterministic=det, plan=plan)
    ref64 = _f64(ref)
    # parity bound of the other tests, with the regular entry point's result as reference
    L = np.broadcast_to(np.diff(off).astype(np.float64)[:, None, None], ref64.shape)
    ma = float(np.abs(oracle.bf16_bits_to_f64(Gb[:off[-1]])).max())
    mb = float(np.abs(oracle.bf16_bits_to_f64(Xb[:off[-1]])).max())
    tol = oracle.tolerance(ref64, L, ma, mb)
    tdt = torch.float32 if out_dtype == "fp32" else torch.bfloat16
    oracle64 = oracle.wgrad(Gb, Xb, off, E)
    tol_oracle = oracle.tolerance(oracle64, L, ma, mb)
    for call in range(2):
        dW = torch.full((E, N, K), float("nan"), dtype=tdt, device="cuda")
        rc = gg.cake_gg_wgrad_noalloc(plan, G, X, dW, offs, out_dtype, det)
        assert rc == gg.CAKE_GG_OK, gg.cake_gg_strerror(rc)
        torch.cuda.synchronize()
        got = _f64(dW)
        assert (np.abs(got - ref64) <= tol).all(), f"call {call}: outside the parity bound"
        assert (np.abs(got - oracle64) <= tol_oracle).all(), f"call {call}: outside the oracle's parity bound"
        if det:
            assert torch.equal(dW.view(torch.int16 if out_dtype == "bf16" else torch.int32),
                               ref.view(torch.int16 if out_dtype == "bf16" else torch.int32)), f"call {call}"


@pytest.mark.parametrize("out_dtype,det", [("bf16", 1), ("fp32", 0)])
def test_noalloc_with_a_split_tail_matches_bitwise(out_dtype, det):
    """A plan whose last partial wave runs as split pieces (16 MB of partial slots inside the
    fixed scratch): two calls in a row give the workspace entry point's bits (tail pieces are
    summed in piece order in both modes)."""
    import torch
    sizes, N, K = [8300, 8200, 8192, 8100], 3072, 4096
    Xb, Gb, off = _inputs(sizes, N, K, seed=23)
    E, M = len(sizes), Xb.shape[0]
    X, G = wl.to_torch_bf16(Xb, "cuda"), wl.to_torch_bf16(Gb, "cuda")
    offs = torch.from_numpy(off).cuda()
    plan = gg.cake_gg_plan("wgrad", E, M, N, K, out_dtype, det)
    assert plan.tail_splits == 8 and plan.workspace_bytes <= gg.CAKE_GG_NOALLOC_SCRATCH_BYTES
    ref = gg.grouped_gemm("wgrad", G, X, offs, out_dtype=out_dtype, deterministic=det, plan=plan)
    iv = torch.int16 if out_dtype == "bf16" else torch.int32
    # sampled outputs against the oracle: one element per 128 x 64 block of every expert's dW
    rng = np.random.default_rng(24)
    es, ns, ks = [], [], []
    for e in range(E):
        for n0 in range(0, N, 128):
            for k0 in range(0, K, 64):
                es.append(e)
                ns.append(n0 + int(rng.integers(0, min(128, N - n0))))
                ks.append(k0 + int(rng.integers(0, min(64, K - k0))))
    es, ns, ks = (np.array(v, np.int64) for v in (es, ns, ks))
    ref_s = oracle.wgrad_at(Gb, Xb, off, E, es, ns, ks)
    L = np.diff(off).astype(np.float64)[es]
    ma = float(np.abs(oracle.bf16_bits_to_f64(Gb[:off[-1]])).max())
    mb = float(np.abs(oracle.bf16_bits_to_f64(Xb[:off[-1]])).max())
    tol = oracle.tolerance(ref_s, L, ma, mb)
    idx = torch.from_numpy(es * N * K + ns * K + ks).cuda()
    for call in range(2):
        dW = torch.full_like(ref, float("nan"))
        rc = gg.cake_gg_wgrad_noalloc(plan, G, X, dW, offs, out_dtype, det)
        assert rc == gg.CAKE_GG_OK, gg.cake_gg_strerror(rc)
        torch.cuda.synchronize()
        assert torch.equal(dW.view(iv), ref.view(iv)), f"call {call}"
        got = _f64(dW.view(-1)[idx])
        assert (np.abs(got - ref_s) <= tol).all(), f"call {call}: sampled outputs outside the oracle's bound"


def test_noalloc_rejects_problems_beyond_its_scratch():
    import torch
    # T = 2^20 rows of a thin projection needs far more partial-tile scratch than the fixed maximum
    os_env = {"CAKE_GG_SPLIT_CHUNK": "1"}
    import os
    old = {k: os.environ.get(k) for k in os_env}
    os.environ.update(os_env)
    try:
        plan = gg.cake_gg_plan("wgrad", 1, 1 << 20, 48, 4096, "fp32", 1)
    finally:
        for k, v in old.items():
            if v is None:
                del os.environ[k]
            else:
                os.environ[k] = v
    assert plan.workspace_bytes > gg.CAKE_GG_NOALLOC_SCRATCH_BYTES
    X = torch.empty((16, 4096), dtype=torch.bfloat16, device="cuda")
    rc = gg.cake_gg_wgrad_noalloc(plan, X, X, X, torch.zeros(2, dtype=torch.int32, device="cuda"), "fp32", 1)
    assert rc == gg.CAKE_GG_ERR_SCRATCH_LIMIT
    assert "scratch" in gg.cake_gg_strerror(rc)
