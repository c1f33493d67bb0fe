"""GPU parity: the CUDA path (through the C ABI) against the FP64 oracle.

Element-by-element comparisons on seeded inputs sized so the oracle finishes
in seconds while still spanning several tiles and ragged tails; exact
(bitwise) comparisons where the inputs make every FP32 sum exact; guard bands
around every output; rows beyond the last offset untouched.
"""
import os

import numpy as np
import pytest

import oracle
from moe_ragged_grouped_gb300 import build as gg_build
from moe_ragged_grouped_gb300 import cake_gg as gg
from moe_ragged_grouped_gb300 import workloads as wl

from gg_testutil import (assert_parity, guarded_empty, guards_intact, out_to_f64, reference, run,
                         to_dev)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def lib():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    gg_build.build()
    return gg.load_library()


def make_inputs(sizes, N, K, seed, extra_rows=0, nan_tail=True):
    rng = np.random.default_rng(seed)
    E, M = len(sizes), sum(sizes) + extra_rows
    Xb = wl.randn_bf16((M, K), 1.0, rng)
    Wb = wl.randn_bf16((E, N, K), 1.0 / np.sqrt(K), rng)
    Gb = wl.randn_bf16((M, N), 1.0, rng)
    if nan_tail and extra_rows:
        Xb[sum(sizes):] = 0x7FC0
        Gb[sum(sizes):] = 0x7FC0
    return Xb, Wb, Gb, wl.offsets_from_sizes(sizes)


def out_shape(pass_, M, E, N, K):
    return {"fwd": (M, N), "dgrad": (M, K), "wgrad": (E, N, K)}[pass_]


def check_case(pass_, sizes, N, K, out_dtype, det, seed=0, extra_rows=0, max_sms=0):
    Xb, Wb, Gb, off = make_inputs(sizes, N, K, seed, extra_rows)
    X, W, G = to_dev(Xb), to_dev(Wb), to_dev(Gb)
    E, M = len(sizes), Xb.shape[0]
    shape = out_shape(pass_, M, E, N, K)
    buf, view, guard = guarded_empty(shape, out_dtype)
    run(pass_, X, W, G, off, out_dtype, det, max_sms=max_sms, out=view)
    import torch
    torch.cuda.synchronize()
    assert guards_intact(buf, guard, int(np.prod(shape)), out_dtype), "guard band overwritten"
    got = out_to_f64(view)
    ref = reference(pass_, Xb, Wb, Gb, off)
    if pass_ != "wgrad":
        tail = got[off[-1]:]
        assert np.isnan(tail).all(), "rows beyond offsets[E] were written"
        got = got[:off[-1]]
    return assert_parity(pass_, got, ref, Xb, Wb, Gb, off, f"{pass_} {out_dtype} det={det} sizes={sizes}")


PASSES = ["fwd", "dgrad", "wgrad"]


def many_expert_sizes(E, M, seed, alpha):
    """Ragged sizes of E experts summing to M (Dirichlet shares, so some are empty)."""
    rng = np.random.default_rng(seed)
    sizes = [int(v) for v in rng.multinomial(M, rng.dirichlet(np.full(E, alpha)))]
    sizes[0] = sizes[E // 2] = sizes[-1] = 0
    return sizes


@pytest.mark.parametrize("pass_", PASSES)
@pytest.mark.parametrize("det", [1, 0])
def test_many_experts_block_built_tables(pass_, det):
    """E = 200 > 32: the walk tables (offsets, heaviest-first order, prefixes) are built by the
    whole CTA rather than one warp; skewed sizes with empty experts, first and last included."""
    sizes = many_expert_sizes(200, 9000, 29, 0.7)
    check_case(pass_, sizes, 128, 192, "fp32", det, seed=29, extra_rows=5)


@pytest.mark.parametrize("pass_", PASSES)
def test_maximum_expert_count(pass_):
    """E = 1024, the most the on-chip tables hold: mostly tiny experts, two long ones, empty
    ones anywhere."""
    rng = np.random.default_rng(30)
    sizes = [int(v) for v in rng.integers(0, 12, 1024)]
    sizes[0] = sizes[-1] = sizes[511] = 0
    sizes[100], sizes[900] = 700, 1300
    check_case(pass_, sizes, 64, 128, "bf16", 1, seed=30, extra_rows=3)


@pytest.mark.parametrize("pass_", PASSES)
@pytest.mark.parametrize("N,K", [(8, 8), (8, 136), (136, 8), (24, 40)])
@pytest.mark.parametrize("out_dtype", ["bf16", "fp32"])
def test_smallest_widths(pass_, N, K, out_dtype):
    """N and K down to 8, the smallest the interface takes: every tile and copy box reaches
    past the tensor's edge (zero fill on loads, clipped or masked stores)."""
    check_case(pass_, [0, 130, 1, 257], N, K, out_dtype, 1, seed=32, extra_rows=3)


@pytest.mark.parametrize("pass_", PASSES)
@pytest.mark.parametrize("out_dtype", ["bf16", "fp32"])
@pytest.mark.parametrize("det", [1, 0])
def test_tiny_config(pass_, out_dtype, det):
    """E=4 experts x 128 rows, K=256, N=128 (X~N(0,1), W~N(0,1/K), G~N(0,1), seed 0)."""
    check_case(pass_, [128] * 4, 128, 256, out_dtype, det, seed=0)


@pytest.mark.parametrize("pass_", PASSES)
@pytest.mark.parametrize("out_dtype", ["bf16", "fp32"])
def test_ragged_groups_with_empty_experts(pass_, out_dtype):
    check_case(pass_, [0, 1, 129, 300, 0, 77], 192, 320, out_dtype, 1, seed=1, extra_rows=9)


@pytest.mark.parametrize("pass_", PASSES)
def test_wide_tiles_several_ktiles(pass_):
    check_case(pass_, [257, 511, 6], 512, 576, "fp32", 1, seed=2, extra_rows=3)


@pytest.mark.parametrize("det", [1, 0])
@pytest.mark.parametrize("out_dtype", ["bf16", "fp32"])
def test_thin_weight_gradient_swapped_split(det, out_dtype):
    """Dense projection shape family: E=1, d_out=48 (MMA rows over d_in, split reduction)."""
    check_case("wgrad", [3000], 48, 512, out_dtype, det, seed=3, extra_rows=5)


@pytest.mark.parametrize("det", [1, 0])
@pytest.mark.parametrize("sizes", [[1500, 517, 0, 64], [4000]])
def test_split_reduction_forced(det, sizes, monkeypatch):
    monkeypatch.setenv("CAKE_GG_SPLIT_CHUNK", "3")
    check_case("wgrad", sizes, 128, 256, "fp32", det, seed=4, extra_rows=7)


@pytest.mark.parametrize("pass_", PASSES)
@pytest.mark.parametrize("det", [1, 0])
def test_exact_integer_inputs_are_bitwise(pass_, det, monkeypatch):
    """Inputs in {-2..2}: every FP32 sum is exact in any order, so GPU == oracle bitwise."""
    if pass_ == "wgrad":
        monkeypatch.setenv("CAKE_GG_SPLIT_CHUNK", "2")
    rng = np.random.default_rng(5)
    sizes = [700, 0, 333, 64]
    E, N, K = len(sizes), 128, 192
    M = sum(sizes)
    Xb = wl.small_int_bf16((M, K), rng)
    Wb = wl.small_int_bf16((E, N, K), rng)
    Gb = wl.small_int_bf16((M, N), rng)
    off = wl.offsets_from_sizes(sizes)
    got = out_to_f64(run(pass_, to_dev(Xb), to_dev(Wb), to_dev(Gb), off, "fp32", det))
    ref = reference(pass_, Xb, Wb, Gb, off)
    if pass_ != "wgrad":
        got = got[:off[-1]]
    np.testing.assert_array_equal(got, ref)


def test_one_hot_forward_selects_weight_columns():
    rng = np.random.default_rng(6)
    sizes = [130, 70]
    E, N, K = 2, 128, 256
    M = sum(sizes)
    Wb = wl.randn_bf16((E, N, K), 1.0, rng)
    Xb = np.zeros((M, K), np.uint16)
    ks = rng.integers(0, K, M)
    Xb[np.arange(M), ks] = 0x3F80
    off = wl.offsets_from_sizes(sizes)
    got = wl.torch_bf16_to_bits(run("fwd", to_dev(Xb), to_dev(Wb), to_dev(np.zeros((M, N), np.uint16)),
                                    off, "bf16", 1))
    for r in range(M):
        e = 0 if r < off[1] else 1
        np.testing.assert_array_equal(got[r], Wb[e][:, ks[r]])


def test_all_zero_and_empty_weight_gradient():
    sizes = [0, 200, 0]
    Xb, Wb, Gb, off = make_inputs(sizes, 64, 128, seed=7)
    got = out_to_f64(run("wgrad", to_dev(Xb), to_dev(Wb), to_dev(Gb), off, "fp32", 1))
    assert not got[0].any() and not got[2].any() and got[1].any()
    z = np.zeros_like(Xb)
    got = out_to_f64(run("fwd", to_dev(z), to_dev(Wb), to_dev(Gb), off, "fp32", 1))
    assert not got[:off[-1]].any()


def test_no_rows_at_all():
    import torch
    Wb = wl.randn_bf16((3, 64, 64), 1.0, np.random.default_rng(0))
    X = torch.zeros((0, 64), dtype=torch.bfloat16, device="cuda")
    G = torch.zeros((0, 64), dtype=torch.bfloat16, device="cuda")
    off = np.zeros(4, np.int32)
    dW = torch.full((3, 64, 64), 7.0, device="cuda")
    run("wgrad", X, to_dev(Wb), G, off, "fp32", 1, out=dW)
    assert not dW.any()


def test_device_detects_bad_offsets_and_recovers():
    import torch
    Xb, Wb, Gb, off = make_inputs([100, 100], 64, 64, seed=8)
    X, W, G = to_dev(Xb), to_dev(Wb), to_dev(Gb)
    bad = torch.tensor([0, 150, 120], dtype=torch.int32, device="cuda")   # decreasing
    with pytest.raises(gg.CakeGGError) as ei:
        gg.grouped_gemm("fwd", X, W, bad, out_dtype="bf16")
    assert ei.value.code == gg.CAKE_GG_ERR_BAD_OFFSETS
    too_big = torch.tensor([0, 150, 201], dtype=torch.int32, device="cuda")  # > M_max
    with pytest.raises(gg.CakeGGError) as ei:
        gg.grouped_gemm("wgrad", G, X, too_big, out_dtype="fp32")
    assert ei.value.code == gg.CAKE_GG_ERR_BAD_OFFSETS
    # the context is still usable
    check_case("fwd", [100, 100], 64, 64, "bf16", 1, seed=8)


def test_dgrad_equals_forward_with_transposed_weights():
    """GPU vs GPU: dX = G W equals the forward pass with W'_e = W_e^T stored [E, K, N]."""
    import torch
    Xb, Wb, Gb, off = make_inputs([300, 0, 200, 77], 192, 256, seed=13)
    G, W = to_dev(Gb), to_dev(Wb)
    Wt = W.transpose(1, 2).contiguous()
    offs = torch.from_numpy(off).cuda()
    dX = gg.grouped_gemm("dgrad", G, W, offs, out_dtype="fp32")
    Yt = gg.grouped_gemm("fwd", G, Wt, offs, out_dtype="fp32")
    M = int(off[-1])
    a, b = dX[:M].double().cpu().numpy(), Yt[:M].double().cpu().numpy()
    ma = float(np.abs(oracle.bf16_bits_to_f64(Gb[:M])).max())
    mb = float(np.abs(oracle.bf16_bits_to_f64(Wb)).max())
    assert (np.abs(a - b) <= oracle.tolerance(b, 192, ma, mb)).all()


@pytest.mark.parametrize("pass_", PASSES)
def test_single_and_paired_ctas_agree_bitwise(pass_, monkeypatch):
    """Pairing CTAs changes only how the B tile reaches shared memory, never a result bit."""
    import torch
    Xb, Wb, Gb, off = make_inputs([0, 513, 1000, 130], 384, 512, seed=14)
    X, W, G = to_dev(Xb), to_dev(Wb), to_dev(Gb)
    paired = run(pass_, X, W, G, off, "fp32", 1)
    monkeypatch.setenv("CAKE_GG_PAIR", "0")
    single = run(pass_, X, W, G, off, "fp32", 1)
    M = int(off[-1])
    if pass_ != "wgrad":
        paired, single = paired[:M], single[:M]
    assert torch.equal(paired.view(torch.int32), single.view(torch.int32))


@pytest.mark.parametrize("pass_", PASSES)
@pytest.mark.parametrize("tile_k", ["128", "256"])
def test_deeper_stages(pass_, tile_k, monkeypatch):
    """Stages holding two or four 64-deep k-chunks (single CTAs), on ragged groups with a NaN tail."""
    monkeypatch.setenv("CAKE_GG_PAIR", "0")
    monkeypatch.setenv("CAKE_GG_TILE_K", tile_k)
    check_case(pass_, [0, 1, 129, 300, 0, 77], 192, 320, "fp32", 1, seed=15, extra_rows=9)
    if pass_ == "wgrad":
        monkeypatch.setenv("CAKE_GG_SPLIT_CHUNK", "2")
        check_case(pass_, [2000, 0, 517], 128, 256, "fp32", 1, seed=16, extra_rows=5)


@pytest.mark.parametrize("out_dtype", ["bf16", "fp32"])
def test_thin_forward(out_dtype):
    """Dense projection forward with d_out = 48: deeper stages, one 64-wide column tile."""
    check_case("fwd", [1000], 48, 512, out_dtype, 1, seed=17, extra_rows=3)


@pytest.mark.parametrize("csplit", ["2", "5", "8"])
@pytest.mark.parametrize("det,out_dtype", [(1, "fp32"), (0, "bf16")])
def test_cluster_split_weight_gradient(csplit, det, out_dtype, monkeypatch):
    """Thin weight gradient whose splits run as one cluster and reduce through distributed
    shared memory: experts empty, shorter than one stage, and long."""
    monkeypatch.setenv("CAKE_GG_CSPLIT", csplit)
    check_case("wgrad", [0, 100, 3000, 65, 1], 48, 512, out_dtype, det, seed=18, extra_rows=6)


@pytest.mark.parametrize("csplit,det,out_dtype", [("2", 1, "fp32"), ("3", 1, "fp32"), ("4", 0, "fp32"),
                                                  ("2", 0, "bf16"), ("4", 1, "bf16")])
@pytest.mark.parametrize("max_sms", [0, 8])
def test_pair_cluster_split_weight_gradient(csplit, det, out_dtype, max_sms, monkeypatch):
    """Weight gradient of 256-row pair tiles whose splits run as one cluster of pairs and reduce
    into their operand rings: experts empty, shorter than one stage and long; a partial last
    column tile (320 = 256 + 64); on 8 SMs one or two clusters take every tile in turn (each
    tile's copies wait until the previous tile's slice is summed)."""
    monkeypatch.setenv("CAKE_GG_CSPLIT", csplit)
    plan = gg.cake_gg_plan("wgrad", 5, 3200, 512, 320, out_dtype, det)
    assert plan.pair == 2 and plan.cluster_splits == int(csplit)
    check_case("wgrad", [0, 100, 3000, 65, 1], 512, 320, out_dtype, det, seed=29, extra_rows=6, max_sms=max_sms)


@pytest.mark.parametrize("out_dtype", ["fp32", "bf16"])
def test_pair_cluster_split_bitwise_equal_to_workspace_slots(out_dtype, monkeypatch):
    """Two splits summed on chip give the bits of the same two splits summed from workspace slots
    (p0 + p1, one rounding): the reduction's place never changes a result."""
    import torch
    Xb, Wb, Gb, off = make_inputs([3000], 512, 512, seed=30, extra_rows=2)
    X, W, G = to_dev(Xb), to_dev(Wb), to_dev(Gb)
    monkeypatch.setenv("CAKE_GG_CSPLIT", "2")
    on_chip = run("wgrad", X, W, G, off, out_dtype, 1)
    monkeypatch.setenv("CAKE_GG_CSPLIT", "0")
    monkeypatch.setenv("CAKE_GG_SPLIT_CHUNK", str(-(-(-(-3000 // 128)) // 2)))
    slots = run("wgrad", X, W, G, off, out_dtype, 1)
    i = torch.int32 if out_dtype == "fp32" else torch.int16
    assert torch.equal(on_chip.view(i), slots.view(i))


@pytest.mark.parametrize("pass_", ["fwd", "dgrad"])
@pytest.mark.parametrize("red", [192, 48])
@pytest.mark.parametrize("out_dtype", ["bf16", "fp32"])
@pytest.mark.parametrize("max_sms", [2, 6, 0])
def test_two_epilogue_groups(pass_, red, out_dtype, max_sms, monkeypatch):
    """A short reduction (192: three 64-deep k-blocks, 2-SM pairs; 48: one partial k-block,
    single CTAs) gives the forward / data gradient a second epilogue warpgroup that takes every
    other tile: ragged groups with a NaN tail, a partial last column tile (640 = 2 x 256 + 128),
    and one or three pairs running every tile in turn (both groups' accumulator and staging
    phases carried across tiles)."""
    N, K = (640, red) if pass_ == "fwd" else (red, 640)
    plan = gg.cake_gg_plan(pass_, 4, 3200, N, K, out_dtype, 1)
    assert plan.epi_groups == 2 and plan.pair == (2 if red > 64 else 1)
    check_case(pass_, [0, 777, 2048, 301], N, K, out_dtype, 1, seed=31, extra_rows=5, max_sms=max_sms)


@pytest.mark.parametrize("pass_", ["fwd", "dgrad"])
def test_two_epilogue_groups_bitwise_equal_to_one(pass_, monkeypatch):
    """Which warpgroup stores a tile never changes its bits."""
    import torch
    N, K = (640, 192) if pass_ == "fwd" else (192, 640)
    Xb, Wb, Gb, off = make_inputs([0, 777, 2048, 301], N, K, seed=32, extra_rows=3)
    X, W, G = to_dev(Xb), to_dev(Wb), to_dev(Gb)
    two = run(pass_, X, W, G, off, "bf16", 1)
    monkeypatch.setenv("CAKE_GG_EPI_GROUPS", "1")
    one = run(pass_, X, W, G, off, "bf16", 1)
    M = int(off[-1])
    assert torch.equal(two[:M].view(torch.int16), one[:M].view(torch.int16))


@pytest.mark.parametrize("csplit,out_dtype", [("2", "fp32"), ("3", "fp32"), ("4", "fp32"), ("3", "bf16")])
@pytest.mark.parametrize("max_sms", [0, 12])
def test_wide_pair_cluster_split_in_rounds(csplit, out_dtype, max_sms, monkeypatch):
    """256 x 512 pair tiles split by clusters of S pairs: each owner's slice is wider than the
    ring holds at once, so the reduction runs in rounds over column windows of it (the receive
    buffer and the staged output one window's); ragged experts, a partial last column tile
    (1152 = 2 x 512 + 128), and on 12 SMs one or two clusters taking every tile in turn."""
    monkeypatch.setenv("CAKE_GG_WIDE", "2")
    monkeypatch.setenv("CAKE_GG_CSPLIT", csplit)
    plan = gg.cake_gg_plan("wgrad", 2, 16604, 256, 1152, out_dtype, 1)
    assert plan.tile_n == 512 and plan.pair == 2 and plan.cluster_splits == int(csplit)
    check_case("wgrad", [9000, 7600], 256, 1152, out_dtype, 1, seed=36, extra_rows=4, max_sms=max_sms)


def test_wide_pair_cluster_split_bitwise_equal_to_workspace_slots(monkeypatch):
    """Three splits of 256 x 512 tiles summed on chip in two rounds give the bits of the same
    three splits summed from workspace slots."""
    import torch
    monkeypatch.setenv("CAKE_GG_WIDE", "2")
    Xb, Wb, Gb, off = make_inputs([16600], 256, 1152, seed=37, extra_rows=4)
    X, W, G = to_dev(Xb), to_dev(Wb), to_dev(Gb)
    monkeypatch.setenv("CAKE_GG_CSPLIT", "3")
    on_chip = run("wgrad", X, W, G, off, "fp32", 1)
    monkeypatch.setenv("CAKE_GG_CSPLIT", "0")
    monkeypatch.setenv("CAKE_GG_SPLIT_CHUNK", str(-(-(-(-16600 // 64)) // 3)))
    slots = run("wgrad", X, W, G, off, "fp32", 1)
    assert torch.equal(on_chip.view(torch.int32), slots.view(torch.int32))


@pytest.mark.parametrize("nq,det,out_dtype", [("4", 1, "fp32"), ("4", 0, "bf16"), ("2", 1, "bf16")])
@pytest.mark.parametrize("max_sms", [0, 8])
def test_nsplit_tail_weight_gradient(nq, det, out_dtype, max_sms, monkeypatch):
    """256 x 512 weight-gradient tiles whose last units run as 2 or 4 column pieces, each over
    all of its expert's k-blocks: ragged experts (one of 7600 rows: a partial last stage), a
    partial last column tile (1152 = 2 x 512 + 128: pieces past K store nothing), every unit a
    tail unit; on 8 SMs four pairs take every piece in turn."""
    monkeypatch.setenv("CAKE_GG_WIDE", "2")
    monkeypatch.setenv("CAKE_GG_SPLIT_CHUNK", "0")
    monkeypatch.setenv("CAKE_GG_NTAIL", nq)
    plan = gg.cake_gg_plan("wgrad", 2, 16604, 256, 1152, out_dtype, det)
    assert plan.tile_n == 512 and plan.tail_nsplit == int(nq) and plan.tail_units == 6
    check_case("wgrad", [9000, 7600], 256, 1152, out_dtype, det, seed=33, extra_rows=4, max_sms=max_sms)


def test_nsplit_tail_bitwise_equal_to_whole_units(monkeypatch):
    """N-split tail pieces sum the same k-blocks in the same order as the whole unit: the bits of
    the plan without a tail split."""
    import torch
    monkeypatch.setenv("CAKE_GG_WIDE", "2")
    monkeypatch.setenv("CAKE_GG_SPLIT_CHUNK", "0")
    Xb, Wb, Gb, off = make_inputs([9000, 7600], 256, 1152, seed=34, extra_rows=4)
    X, W, G = to_dev(Xb), to_dev(Wb), to_dev(Gb)
    monkeypatch.setenv("CAKE_GG_NTAIL", "4")
    pieces = run("wgrad", X, W, G, off, "fp32", 1)
    monkeypatch.setenv("CAKE_GG_TAIL", "0")
    whole = run("wgrad", X, W, G, off, "fp32", 1)
    assert torch.equal(pieces.view(torch.int32), whole.view(torch.int32))


@pytest.mark.parametrize("det", [1, 0])
def test_thin_weight_gradient_through_workspace_slots(det, monkeypatch):
    """The same thin shape with the cluster reduction disabled: partials through the workspace."""
    monkeypatch.setenv("CAKE_GG_CSPLIT", "0")
    check_case("wgrad", [3000], 48, 512, "fp32", det, seed=3, extra_rows=5)


@pytest.mark.parametrize("pass_", ["fwd", "dgrad"])
@pytest.mark.parametrize("out_dtype", ["bf16", "fp32"])
@pytest.mark.parametrize("max_sms", [2, 0])
def test_double_staging_partial_last_tile(pass_, out_dtype, max_sms, monkeypatch):
    """Two alternating staging buffers per epilogue warp, an output width that leaves the last
    column tile partial (384 = 256 + 128), and one CTA pair running every tile in turn: each
    staging write must be followed by its own committed store."""
    monkeypatch.setenv("CAKE_GG_STAGING_BUFS", "2")
    N, K = (384, 512) if pass_ == "fwd" else (512, 384)
    check_case(pass_, [0, 777, 2048, 301], N, K, out_dtype, 1, seed=19, extra_rows=4, max_sms=max_sms)


@pytest.mark.parametrize("pass_", ["fwd", "dgrad"])
@pytest.mark.parametrize("width", [320, 448])
@pytest.mark.parametrize("max_sms", [2, 0])
def test_double_staging_odd_slab_count(pass_, width, max_sms, monkeypatch):
    """BF16 output 320 = 256 + 64 or 448 = 256 + 192 wide: the last column tile stores an odd
    number of 64-column slabs (1 or 3), so a warp's next tile starts on the buffer its previous
    tile's last store may still be reading unless the buffers alternate across tiles."""
    monkeypatch.setenv("CAKE_GG_STAGING_BUFS", "2")
    N, K = (width, 256) if pass_ == "fwd" else (256, width)
    check_case(pass_, [0, 777, 2048, 301, 1500], N, K, "bf16", 1, seed=28, extra_rows=4, max_sms=max_sms)


@pytest.mark.parametrize("pass_", PASSES)
@pytest.mark.parametrize("tile_k", ["64", "128"])
def test_pairs_at_both_stage_depths_and_few_ctas(pass_, tile_k, monkeypatch):
    """2-SM pairs with 64- and 128-deep stages, on a grid of one and three pairs (many tiles per
    CTA, ring and accumulator phases carried across tiles), ragged groups with a NaN tail."""
    monkeypatch.setenv("CAKE_GG_TILE_K", tile_k)
    for cap in (2, 6):
        check_case(pass_, [0, 777, 2048, 301], 384, 512, "fp32", 1, seed=20, extra_rows=5, max_sms=cap)


@pytest.mark.parametrize("sizes,N,K", [([0, 5000, 1900, 33, 0, 777], 384, 512), ([3000, 200, 17], 256, 128)])
@pytest.mark.parametrize("max_sms", [0, 6])
def test_dynamic_and_static_unit_order_agree_bitwise(sizes, N, K, max_sms, monkeypatch):
    """Weight-gradient units taken from a global counter (heaviest first) give the same bits as the
    static stride: a tile's arithmetic never depends on the CTA that computes it."""
    import torch
    Xb, Wb, Gb, off = make_inputs(sizes, N, K, seed=21, extra_rows=3)
    X, W, G = to_dev(Xb), to_dev(Wb), to_dev(Gb)
    dyn = run("wgrad", X, W, G, off, "fp32", 1, max_sms=max_sms)
    monkeypatch.setenv("CAKE_GG_DYN", "0")
    stat = run("wgrad", X, W, G, off, "fp32", 1, max_sms=max_sms)
    assert torch.equal(dyn.view(torch.int32), stat.view(torch.int32))


def test_scheduler_words_return_to_zero():
    """The status word, the unit counter and the retired-CTA counter in the workspace header are
    zero after every call, so the workspace needs no clearing between calls; the ticket tag
    (header word 32, byte 128) advances by one per call."""
    import torch
    Xb, Wb, Gb, off = make_inputs([700, 0, 1300], 256, 512, seed=22)
    X, W, G = to_dev(Xb), to_dev(Wb), to_dev(Gb)
    E, M = 3, Xb.shape[0]
    plans = [gg.cake_gg_plan("wgrad", E, M, 256, 512, od, 1, cap) for od in ("bf16", "fp32") for cap in (0, 4)]
    ws = torch.zeros(max(int(pl.workspace_bytes) for pl in plans), dtype=torch.uint8, device="cuda")
    offs = torch.from_numpy(off).cuda()
    for i, cap in enumerate((0, 4, 0)):
        plan = gg.cake_gg_plan("wgrad", E, M, 256, 512, "bf16", 1, cap)
        gg.grouped_gemm("wgrad", G, X, offs, out_dtype="bf16", plan=plan, workspace=ws)
        torch.cuda.synchronize()
        head = ws[:256].view(torch.int32).cpu().numpy().copy()
        assert head[32] == i + 1, head[32]
        head[32] = 0
        assert (head == 0).all(), head.nonzero()
    ref = reference("wgrad", Xb, Wb, Gb, off)
    out = gg.grouped_gemm("wgrad", G, X, offs, out_dtype="fp32", plan=gg.cake_gg_plan("wgrad", E, M, 256, 512, "fp32", 1),
                          workspace=ws)
    assert_parity("wgrad", out_to_f64(out), ref, Xb, Wb, Gb, off, "after reuse")


@pytest.mark.parametrize("det,out_dtype", [(1, "fp32"), (0, "bf16"), (1, "bf16")])
def test_wide_weight_gradient_tiles(det, out_dtype, monkeypatch):
    """256 x 512 pair tiles (two N = 256 MMAs per k-step into one 512-column accumulator):
    an empty expert, a last column tile of 64 (K = 1088), a last pair whose odd CTA lies past
    N = 384, NaN rows past the last offset.  (The plan takes these tiles for shapes this small
    only when forced: 18 units fill less than half a wave.)"""
    import torch
    from moe_ragged_grouped_gb300 import cake_gg as gg_
    monkeypatch.setenv("CAKE_GG_WIDE", "2")
    plan = gg_.cake_gg_plan("wgrad", 3, 25004, 384, 1088, out_dtype, det)
    assert plan.tile_n == 512 and plan.pair == 2
    check_case("wgrad", [12000, 0, 13000], 384, 1088, out_dtype, det, seed=24, extra_rows=4)


def test_wide_tiles_bitwise_equal_to_256_wide(monkeypatch):
    """Unsplit plans (a split's boundaries depend on the stage depth): every output element sees
    the same sequence of K = 16 MMA steps in both tile widths."""
    import torch
    monkeypatch.setenv("CAKE_GG_SPLIT_CHUNK", "0")
    monkeypatch.setenv("CAKE_GG_WIDE", "2")
    Xb, Wb, Gb, off = make_inputs([12000, 0, 13000], 384, 1088, seed=25)
    X, W, G = to_dev(Xb), to_dev(Wb), to_dev(Gb)
    assert gg.cake_gg_plan("wgrad", 3, 25004, 384, 1088, "fp32", 1).tile_n == 512
    wide = run("wgrad", X, W, G, off, "fp32", 1)
    monkeypatch.setenv("CAKE_GG_WIDE", "0")
    narrow = run("wgrad", X, W, G, off, "fp32", 1)
    assert torch.equal(wide.view(torch.int32), narrow.view(torch.int32))


@pytest.mark.parametrize("pass_", ["fwd", "dgrad"])
@pytest.mark.parametrize("det,out_dtype", [(1, "bf16"), (0, "fp32")])
def test_wide_forward_and_data_gradient_tiles(pass_, det, out_dtype, monkeypatch):
    """256 x 512 pair tiles for the forward (K-major W: two 128-row boxes per CTA) and the data
    gradient (MN-major W: two stacked boxes per CTA): ragged experts, an empty one, a partial
    last row tile, NaN rows past the last offset."""
    monkeypatch.setenv("CAKE_GG_WIDE_FD", "1")
    plan = gg.cake_gg_plan(pass_, 4, 2037, 1024, 1536, out_dtype, det)
    assert plan.tile_n == 512 and plan.pair == 2 and plan.tile_k == 64
    check_case(pass_, [700, 0, 1300, 33], 1024, 1536, out_dtype, det, seed=26, extra_rows=4)


@pytest.mark.parametrize("pass_", ["fwd", "dgrad"])
def test_wide_forward_and_data_gradient_bitwise_equal_to_256_wide(pass_, monkeypatch):
    """Each output element sees the same sequence of K = 16 MMA steps in both tile widths."""
    import torch
    Xb, Wb, Gb, off = make_inputs([1500, 0, 2100], 1024, 1536, seed=27)
    X, W, G = to_dev(Xb), to_dev(Wb), to_dev(Gb)
    monkeypatch.setenv("CAKE_GG_WIDE_FD", "1")
    wide = run(pass_, X, W, G, off, "fp32", 1)
    monkeypatch.setenv("CAKE_GG_WIDE_FD", "0")
    narrow = run(pass_, X, W, G, off, "fp32", 1)
    assert torch.equal(wide.view(torch.int32), narrow.view(torch.int32))


@pytest.mark.parametrize("pass_", PASSES)
def test_results_unchanged_next_to_a_spinner(pass_):
    """A bounded spinner on another stream holds 32 SMs for 5 ms: CTAs that start late find the
    unit counter drained or take what is left.  Each result next to the spinner is within the
    parity bound of the FP64 oracle and bitwise equal to the result without it."""
    import torch
    Xb, Wb, Gb, off = make_inputs([3000, 0, 5000, 1200], 512, 768, seed=26)
    X, W, G = to_dev(Xb), to_dev(Wb), to_dev(Gb)
    ref = run(pass_, X, W, G, off, "fp32", 1)
    ref64 = reference(pass_, Xb, Wb, Gb, off)
    side = torch.cuda.Stream()
    M = int(off[-1])
    for i in range(2):
        assert gg.cake_gg_corun_spinner(32, 5_000_000, side.cuda_stream) == gg.CAKE_GG_OK
        out = run(pass_, X, W, G, off, "fp32", 1)
        torch.cuda.synchronize()
        a, b = (ref, out) if pass_ == "wgrad" else (ref[:M], out[:M])
        assert_parity(pass_, out_to_f64(b), ref64, Xb, Wb, Gb, off, f"{pass_} next to a spinner, run {i}")
        assert torch.equal(a.view(torch.int32), b.view(torch.int32))


def test_spinner_rejects_bad_arguments():
    assert gg.cake_gg_corun_spinner(0, 1000, 0) == gg.CAKE_GG_ERR_INVALID_ARG
    assert gg.cake_gg_corun_spinner(8, 20_000_000_000, 0) == gg.CAKE_GG_ERR_INVALID_ARG


@pytest.mark.parametrize("det,env", [(1, {"CAKE_GG_SPLIT_CHUNK": "8"}), (0, {"CAKE_GG_SPLIT_CHUNK": "8"}),
                                     (1, {"CAKE_GG_TAIL": "1"})])
def test_ticketed_weight_gradient_replayed_from_a_cuda_graph(det, env, monkeypatch):
    """Split tiles finish through tickets tagged with a per-call number that the workspace keeps
    and each call advances on the device, so a call captured once in a CUDA graph and replayed
    gets a fresh number every replay: each of three replays is within the oracle's bound (and,
    deterministic, bitwise the eager call's result)."""
    import torch
    for k, v in env.items():
        monkeypatch.setenv(k, v)
    if "CAKE_GG_TAIL" in env:
        sizes, N, K = [8300, 8200, 8192, 8100], 3072, 4096   # a split tail: 4 units x 8 pieces
    else:
        sizes, N, K = [3000, 0, 5000, 1200], 512, 768
    Xb, Wb, Gb, off = make_inputs(sizes, N, K, seed=28)
    X, G = to_dev(Xb), to_dev(Gb)
    E, M = len(sizes), Xb.shape[0]
    plan = gg.cake_gg_plan("wgrad", E, M, N, K, "fp32", det)
    assert plan.split_chunk == 8 or plan.tail_splits > 1
    ws = gg.make_workspace(plan, "cuda")
    offs = torch.from_numpy(off).cuda()
    out = torch.empty((E, N, K), dtype=torch.float32, device="cuda")
    stream = torch.cuda.Stream()
    with torch.cuda.stream(stream):
        assert gg.cake_gg_wgrad(plan, G, X, out, offs, "fp32", det, ws, stream=stream.cuda_stream) == gg.CAKE_GG_OK
    torch.cuda.synchronize()
    eager = out.clone()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        rc = gg.cake_gg_wgrad(plan, G, X, out, offs, "fp32", det, ws, stream=stream.cuda_stream)
    assert rc == gg.CAKE_GG_OK
    if K > 1024:
        # sampled: one element per 128 x 64 block of every expert's dW
        rng = np.random.default_rng(3)
        es = np.repeat(np.arange(E), (N // 128) * (K // 64))
        nb = np.tile(np.repeat(np.arange(0, N, 128), K // 64), E)
        kb = np.tile(np.tile(np.arange(0, K, 64), N // 128), E)
        ns, ks = nb + rng.integers(0, 128, nb.size), kb + rng.integers(0, 64, kb.size)
        ref = oracle.wgrad_at(Gb, Xb, off, E, es, ns, ks)
        idx = torch.from_numpy(es * N * K + ns * K + ks).cuda()
        ma = float(np.abs(oracle.bf16_bits_to_f64(Gb[:off[-1]])).max())
        mb = float(np.abs(oracle.bf16_bits_to_f64(Xb[:off[-1]])).max())
        tol = oracle.tolerance(ref, np.diff(off).astype(np.float64)[es], ma, mb)
    else:
        ref = oracle.wgrad(Gb, Xb, off, E)
    for i in range(3):
        out.fill_(float("nan"))
        graph.replay()
        torch.cuda.synchronize()
        if K > 1024:
            got = out.view(-1)[idx].double().cpu().numpy()
            assert (np.abs(got - ref) <= tol).all(), f"replay {i}"
        else:
            assert_parity("wgrad", out_to_f64(out), ref, Xb, Wb, Gb, off, f"replay {i}")
        if det:
            assert torch.equal(out.view(torch.int32), eager.view(torch.int32)), f"replay {i}"
    assert gg.cake_gg_check_status(ws, stream.cuda_stream) == gg.CAKE_GG_OK


@pytest.mark.parametrize("sizes,N,K", [([3000], 384, 1024), ([1000], 512, 2048), ([5000], 256, 768)])
@pytest.mark.parametrize("det,out_dtype", [(1, "fp32"), (0, "bf16"), (1, "bf16")])
def test_streamk_weight_gradient(sizes, N, K, det, out_dtype, monkeypatch):
    """Stream-K walk forced on small one-expert shapes (segments of a few k-blocks cross several
    tile boundaries; a ragged last k-block; NaN rows past the expert): every element against the
    oracle, guard bands intact."""
    monkeypatch.setenv("CAKE_GG_STREAMK", "2")
    plan = gg.cake_gg_plan("wgrad", 1, sum(sizes) + 3, N, K, out_dtype, det)
    assert plan.streamk_kblocks > 0
    check_case("wgrad", sizes, N, K, out_dtype, det, seed=29, extra_rows=3)


def test_streamk_bitwise_across_sm_caps_and_equal_pieces(monkeypatch):
    """The stream-K pieces are a function of the plan and the offsets alone: SM caps 7, 100, 148
    and the full device give the same bits; exact-integer inputs give the oracle's bits."""
    import torch
    monkeypatch.setenv("CAKE_GG_STREAMK", "2")
    Xb, Wb, Gb, off = make_inputs([3000], 384, 1024, seed=30, extra_rows=3)
    X, W, G = to_dev(Xb), to_dev(Wb), to_dev(Gb)
    ref = run("wgrad", X, W, G, off, "fp32", 1)
    for cap in (7, 100, 148, 0):
        out = run("wgrad", X, W, G, off, "fp32", 1, max_sms=cap)
        assert torch.equal(out.view(torch.int32), ref.view(torch.int32)), f"max_sms={cap}"
    # small integers: every FP32 sum is exact, so the pieces' sum is the oracle's value exactly
    rng = np.random.default_rng(31)
    Xi = wl.f32_to_bf16_bits(rng.integers(-2, 3, Xb.shape).astype(np.float32))
    Gi = wl.f32_to_bf16_bits(rng.integers(-2, 3, Gb.shape).astype(np.float32))
    for det in (1, 0):
        out = run("wgrad", to_dev(Xi), W, to_dev(Gi), off, "fp32", det)
        assert np.array_equal(out.double().cpu().numpy(), oracle.wgrad(Gi, Xi, off, 1))


def test_streamk_with_no_rows_writes_zeros(monkeypatch):
    import torch
    monkeypatch.setenv("CAKE_GG_STREAMK", "2")
    Xb, Wb, Gb, _ = make_inputs([2000], 512, 1024, seed=32)
    X, G = to_dev(Xb), to_dev(Gb)
    plan = gg.cake_gg_plan("wgrad", 1, 2000, 512, 1024, "fp32", 1)
    assert plan.streamk_kblocks > 0
    offs = torch.zeros(2, dtype=torch.int32, device="cuda")
    out = torch.full((1, 512, 1024), float("nan"), device="cuda")
    gg.grouped_gemm("wgrad", G, X, offs, out_dtype="fp32", plan=plan, out=out)
    torch.cuda.synchronize()
    assert bool((out == 0).all())
