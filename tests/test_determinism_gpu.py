"""Deterministic mode: bitwise reproducible across runs and across SM caps.

flashinfer PR #8258 (opening summary) calls the deterministic variant
"bitwise reproducible from run to run"; here the bar is also bitwise equality
between launches capped at 100 and 148 SMs, because tile shapes, split
factors and every element's summation order are fixed by the plan, never by
the number of CTAs.
"""
import numpy as np
import pytest

from moe_ragged_grouped_gb300 import build as gg_build
from moe_ragged_grouped_gb300 import cake_gg as gg
from moe_ragged_grouped_gb300 import workloads as wl

from gg_testutil import run, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def lib():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    gg_build.build()
    return gg.load_library()


def inputs(sizes, N, K, seed):
    rng = np.random.default_rng(seed)
    E, M = len(sizes), sum(sizes)
    return (to_dev(wl.randn_bf16((M, K), 1.0, rng)), to_dev(wl.randn_bf16((E, N, K), K ** -0.5, rng)),
            to_dev(wl.randn_bf16((M, N), 1.0, rng)), wl.offsets_from_sizes(sizes))


@pytest.mark.parametrize("pass_,sizes,N,K,env", [
    ("fwd", [0, 777, 2048, 301], 384, 512, None),
    ("dgrad", [0, 777, 2048, 301], 384, 512, None),
    ("wgrad", [0, 777, 2048, 301], 384, 512, None),
    ("wgrad", [0, 5000, 1900, 33], 128, 256, "3"),     # split reduction
    ("wgrad", [8192], 48, 1024, None),                  # thin, swapped, split
])
def test_bitwise_across_runs_and_sm_caps(pass_, sizes, N, K, env, monkeypatch):
    import torch
    if env:
        monkeypatch.setenv("CAKE_GG_SPLIT_CHUNK", env)
    X, W, G, off = inputs(sizes, N, K, seed=11)
    ref = run(pass_, X, W, G, off, "fp32", 1)
    for i in range(20):
        again = run(pass_, X, W, G, off, "fp32", 1)
        assert torch.equal(again.view(torch.int32), ref.view(torch.int32)), f"run {i} differs"
    for cap in (100, 148, 7, 1):
        capped = run(pass_, X, W, G, off, "fp32", 1, max_sms=cap)
        assert torch.equal(capped.view(torch.int32), ref.view(torch.int32)), f"max_sms={cap} differs"


@pytest.mark.parametrize("pass_", ["fwd", "dgrad", "wgrad"])
def test_many_experts_bitwise_across_sm_caps(pass_):
    """E = 300 (tables built block-wide, heaviest first): bitwise equal across runs and SM
    caps."""
    import torch
    rng = np.random.default_rng(31)
    sizes = [int(v) for v in rng.multinomial(12000, rng.dirichlet(np.full(300, 0.5)))]
    X, W, G, off = inputs(sizes, 128, 256, seed=31)
    ref = run(pass_, X, W, G, off, "fp32", 1)
    for cap in (0, 100, 148, 7):
        again = run(pass_, X, W, G, off, "fp32", 1, max_sms=cap)
        assert torch.equal(again.view(torch.int32), ref.view(torch.int32)), f"max_sms={cap} differs"


def test_forward_rows_independent_of_other_experts():
    """A forward output row depends only on its own row and its expert's weights."""
    import torch
    X, W, G, off = inputs([300, 500, 200], 256, 256, seed=12)
    Y = run("fwd", X, W, G, off, "fp32", 1)
    # move the boundary between experts 0 and 1 past row 300: rows of expert 2 are unchanged
    off2 = np.array([0, 100, 800, 1000], np.int32)
    Y2 = run("fwd", X, W, G, off2, "fp32", 1)
    assert torch.equal(Y[800:1000].view(torch.int32), Y2[800:1000].view(torch.int32))
    assert torch.equal(Y[0:100].view(torch.int32), Y2[0:100].view(torch.int32))


@pytest.mark.parametrize("pass_", ["fwd", "dgrad", "wgrad"])
@pytest.mark.parametrize("tile_n", ["64", "128"])
def test_results_do_not_depend_on_tile_width(pass_, tile_n, monkeypatch):
    """Each output element's K-order is fixed by the k-steps, not by the MMA's N: an N-tile of
    64 or 128 columns gives the same bits as the planned 256 (flashinfer PR #8363 reports the same
    for its 192- vs 256-wide programs)."""
    import torch
    X, W, G, off = inputs([0, 777, 2048, 301], 512, 768, seed=21)
    ref = run(pass_, X, W, G, off, "fp32", 1)
    monkeypatch.setenv("CAKE_GG_TILE_N", tile_n)
    other = run(pass_, X, W, G, off, "fp32", 1)
    M = int(off[-1])
    if pass_ != "wgrad":
        ref, other = ref[:M], other[:M]
    assert torch.equal(ref.view(torch.int32), other.view(torch.int32))
