"""Host-side checks of the C ABI (no GPU needed, no compute calls).

* the library loads and exports every entry point include/cake_gg.h declares;
* cake_gg_plan validates its arguments and never depends on max_sms;
* the kernel's tile walk (host replica, same code as the device) covers every
  output element exactly once, partitions each expert's reduction into
  contiguous splits, and walks the weight gradient heaviest-first.
"""
import ctypes
import os
import re

import numpy as np
import pytest

from moe_ragged_grouped_gb300 import build as gg_build
from moe_ragged_grouped_gb300 import cake_gg as gg
from moe_ragged_grouped_gb300 import workloads as wl

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module", autouse=True)
def built_library():
    gg_build.build()
    gg.load_library()


def declared_entry_points():
    names = []
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            text = open(os.path.join(ROOT, "include", fn)).read()
            names += re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(cake_gg_\w+)\s*\(", text, re.M)
    return sorted(set(names))


def test_library_exports_every_declared_symbol():
    names = declared_entry_points()
    assert "cake_gg_plan" in names and "cake_gg_wgrad" in names
    lib = ctypes.CDLL(gg.LIB_PATH)
    for n in names:
        assert hasattr(lib, n), f"{n} declared in include/ but not exported"
    assert set(gg.EXPORTED) <= set(names)


def test_plan_struct_layout_matches_header():
    # 6 int32, int64, 10 int32, 2 uint64, staging_bufs + 7 int32 reserved
    assert ctypes.sizeof(gg.CakeGGPlan) == 120
    assert gg.CakeGGPlan.M_max.offset == 24
    assert gg.CakeGGPlan.timeout_ns.offset == 72
    assert gg.CakeGGPlan.workspace_bytes.offset == 80


def test_strerror_never_null():
    for code in range(-1, 12):
        assert isinstance(gg.cake_gg_strerror(code), str)
    assert "workspace" in gg.cake_gg_strerror(gg.CAKE_GG_ERR_WORKSPACE)


@pytest.mark.parametrize("args,code", [
    (("fwd", 0, 128, 64, 64, "bf16", 1), gg.CAKE_GG_ERR_INVALID_ARG),        # E = 0
    (("fwd", 1025, 128, 64, 64, "bf16", 1), gg.CAKE_GG_ERR_INVALID_ARG),     # E too large
    (("fwd", 2, 128, 60, 64, "bf16", 1), gg.CAKE_GG_ERR_ALIGNMENT),          # N % 8
    (("dgrad", 2, 128, 64, 12, "bf16", 1), gg.CAKE_GG_ERR_ALIGNMENT),        # K % 8
    (("wgrad", 2, -1, 64, 64, "fp32", 1), gg.CAKE_GG_ERR_INVALID_ARG),       # M < 0
    (("wgrad", 2, 2 ** 31, 64, 64, "fp32", 1), gg.CAKE_GG_ERR_INVALID_ARG),  # M too large
    ((5, 2, 128, 64, 64, "bf16", 1), gg.CAKE_GG_ERR_INVALID_ARG),            # bad pass
    (("fwd", 2, 128, 64, 64, 7, 1), gg.CAKE_GG_ERR_UNSUPPORTED),             # bad dtype
    (("wgrad", 1024, 2 ** 31 - 1, 2 ** 30, 2 ** 30, "fp32", 1), gg.CAKE_GG_ERR_OVERFLOW),
])
def test_plan_rejects_bad_arguments(args, code):
    with pytest.raises(gg.CakeGGError) as ei:
        gg.cake_gg_plan(*args)
    assert ei.value.code == code


def test_plan_rejects_negative_max_sms():
    with pytest.raises(gg.CakeGGError):
        gg.cake_gg_plan("fwd", 1, 128, 64, 64, "bf16", 1, -3)


@pytest.mark.parametrize("pass_", ["fwd", "dgrad", "wgrad"])
@pytest.mark.parametrize("shape", [(8, 131072, 3072, 4096), (1, 16384, 48, 4096), (4, 512, 128, 256),
                                   (32, 131072, 4096, 1536), (1, 16384, 512, 5120)])
def test_plan_choices_do_not_depend_on_max_sms(pass_, shape):
    E, M, N, K = shape
    plans = [gg.cake_gg_plan(pass_, E, M, N, K, "fp32", 1, s).as_dict() for s in (0, 100, 148, 152)]
    for p in plans[1:]:
        for key in ("tile_m", "tile_n", "tile_k", "stages", "swap_ab", "split_chunk", "workspace_bytes"):
            assert p[key] == plans[0][key]
    assert plans[0]["tile_n"] % 64 == 0 and (64 <= plans[0]["tile_n"] <= 256 or plans[0]["tile_n"] == 512)


def test_thin_weight_gradient_swaps_and_splits():
    p = gg.cake_gg_plan("wgrad", 1, 16384, 48, 4096, "fp32", 1)
    assert p.swap_ab == 1 and p.tile_n == 64 and (p.split_chunk > 0 or p.cluster_splits > 1)
    q = gg.cake_gg_plan("wgrad", 8, 131072, 3072, 4096, "bf16", 1)
    assert q.swap_ab == 0 and q.split_chunk == 0
    # long units: 256 x 512 pair tiles, 768 units = 10 waves of 76 pairs + 8; those 8 run as 4
    # pieces each through FP32 partial slots (8 units x 2 CTAs x 4 pieces x 128 x 512 floats)
    assert q.tile_n == 512 and q.tile_k == 64
    assert (q.tail_units, q.tail_splits) == (8, 4)
    assert q.workspace_bytes >= 256 + 8 * 2 * 4 * 128 * 512 * 4


def _check_walk_coverage(pass_, sizes, N, K, det=1, env=None):
    if env:
        os.environ.update(env)
    try:
        off = wl.offsets_from_sizes(sizes)
        E, M = len(sizes), int(off[-1]) + 5
        plan = gg.cake_gg_plan(pass_, E, M, N, K, "fp32", det)
    finally:
        for k in (env or {}):
            del os.environ[k]
    tiles = gg.cake_gg_tile_walk(plan, off)
    bm, bn = plan.tile_m, plan.tile_n
    if pass_ in ("fwd", "dgrad"):
        nout = N if pass_ == "fwd" else K
        cover = np.zeros((M, nout), np.int32)
        for e, mt, nt, s, S, kb0, kb1, _ in tiles[:, :8]:
            assert S == 1 and s == 0 and kb0 == 0
            r0 = off[e] + mt * bm
            assert r0 < off[e + 1]
            cover[r0:min(r0 + bm, off[e + 1]), nt * bn:min((nt + 1) * bn, nout)] += 1
        assert (cover[:off[-1]] == 1).all() and (cover[off[-1]:] == 0).all()
    else:
        mdim, ndim = (K, N) if plan.swap_ab else (N, K)
        # weight-gradient tiles are aligned bm x bn blocks of each expert's output: coverage
        # exactly once <=> every (expert, m-tile, n-tile) block appears as one split group
        n_mt, n_nt = -(-mdim // bm), -(-ndim // bn)
        cover = np.zeros((len(sizes), n_mt, n_nt), np.int32)
        # N-split tail pieces: column ranges of one tile that partition it, each over
        # all of its k-blocks; every other unit covers the whole tile
        pieces = {}
        for e, mt, nt, s, S, kb0, kb1, ticket, c0, cw in tiles:
            pieces.setdefault((e, mt, nt), []).append((c0, cw))
        for key, cols in pieces.items():
            cols = sorted(set(cols))
            assert cols[0][0] == 0 and sum(w for _, w in cols) == bn
            assert all(a[0] + a[1] == b[0] for a, b in zip(cols, cols[1:]))
        splits = {}
        for e, mt, nt, s, S, kb0, kb1, ticket, c0, cw in tiles:
            if cw < bn:
                assert S == 1 and s == 0 and kb0 == 0
                if c0 > 0:
                    continue   # (counted once, with its first piece)
            splits.setdefault((e, mt, nt), []).append((s, S, kb0, kb1, ticket))
        for (e, mt, nt), lst in splits.items():
            lst.sort()
            S = lst[0][1]
            assert [x[0] for x in lst] == list(range(S))
            nkb = -(-(off[e + 1] - off[e]) // plan.tile_k)
            # contiguous partition of [0, nkb)
            assert lst[0][2] == 0 and lst[-1][3] == nkb
            for a, b in zip(lst, lst[1:]):
                # cluster splits and split tails give every tile a fixed piece count;
                # trailing pieces of a short expert may be empty
                assert a[3] == b[2] and (b[2] < b[3] or plan.cluster_splits > 0 or plan.tail_splits > 0)
            assert len({x[4] for x in lst}) == 1
            assert 0 <= mt < n_mt and 0 <= nt < n_nt
            cover[e, mt, nt] += 1
        assert (cover == 1).all()
        # heaviest-first over experts (k-blocks per split, ties by expert index)
        costs = []
        for e, mt, nt, s, S, kb0, kb1, _ in tiles[:, :8]:
            if not costs or costs[-1][0] != e:
                costs.append((e, -(-(-(-(off[e + 1] - off[e]) // plan.tile_k)) // S)))
        seq = [c for _, c in costs]
        assert seq == sorted(seq, reverse=True)
    return plan, tiles


@pytest.mark.parametrize("pass_", ["fwd", "dgrad", "wgrad"])
@pytest.mark.parametrize("sizes", [[128] * 4, [0, 1, 129, 300, 0], [5000], [0, 21381 // 16, 34780 // 16, 79903 // 16],
                                   [17, 0, 0, 64, 63, 65, 1]])
def test_tile_walk_covers_each_output_once(pass_, sizes):
    _check_walk_coverage(pass_, sizes, N=192, K=320)


def test_tile_walk_split_partitions():
    plan, tiles = _check_walk_coverage("wgrad", [0, 3000, 700, 64], N=128, K=256,
                                       env={"CAKE_GG_SPLIT_CHUNK": "4"})
    assert plan.split_chunk == 4
    assert max(t[4] for t in tiles) == -(-(-(-3000 // plan.tile_k)) // 4)


def test_tile_walk_thin_swap():
    plan, tiles = _check_walk_coverage("wgrad", [16384], N=48, K=4096)
    assert plan.swap_ab == 1 and plan.cluster_splits >= 2 and plan.workspace_bytes == 256
    assert len({(t[1], t[2]) for t in tiles}) == 32
    assert len(tiles) == 32 * plan.cluster_splits


def test_tile_walk_pair_cluster_split():
    """4096 -> 512 weight gradient at T = 16384: 32 pair tiles of 256 x 256, each split in two
    by a cluster of two pairs (4 CTAs) that reduces on chip -- every (m-tile, n-tile) once, the
    two splits contiguous halves of the 128 k-blocks, no workspace partials."""
    plan, tiles = _check_walk_coverage("wgrad", [16384], N=512, K=4096)
    assert plan.pair == 2 and plan.cluster_splits == 2 and plan.split_chunk == 0 and plan.swap_ab == 0
    assert plan.workspace_bytes == 256
    assert len(tiles) == 4 * 16 * 2
    assert {(t[5], t[6]) for t in tiles} == {(0, 64), (64, 128)}


def test_tile_walk_pair_cluster_split_with_small_and_empty_experts():
    plan, _ = _check_walk_coverage("wgrad", [0, 100, 3000, 65, 1], N=512, K=512, env={"CAKE_GG_CSPLIT": "3"})
    assert plan.pair == 2 and plan.cluster_splits == 3


def test_few_tile_weight_gradient_width_choice():
    """Few-tile dense weight gradients (T = 16384): 5120 -> 512 takes 256 x 512 tiles split in
    three (20 x 3 units in one wave instead of 40 x 3 in two), reduced on chip by clusters of
    three pairs; 4096 -> 512 keeps 256-wide tiles reduced on chip; 4096 -> 1024 and 5120 -> 1024
    keep 256-wide tiles (unsplit / split tail)."""
    p = gg.cake_gg_plan("wgrad", 1, 16384, 512, 5120, "fp32", 1)
    assert (p.tile_n, p.tile_k, p.cluster_splits, p.split_chunk, p.workspace_bytes) == (512, 64, 3, 0, 256)
    p = gg.cake_gg_plan("wgrad", 1, 16384, 512, 4096, "fp32", 1)
    assert p.tile_n == 256 and p.cluster_splits == 2
    p = gg.cake_gg_plan("wgrad", 1, 16384, 1024, 4096, "fp32", 1)
    assert p.tile_n == 256 and p.split_chunk == 0
    p = gg.cake_gg_plan("wgrad", 1, 16384, 1024, 5120, "fp32", 1)
    assert p.tile_n == 256 and (p.tail_units, p.tail_splits) == (4, 8)


def test_pair_cluster_split_needs_every_cluster_resident():
    # 5120 -> 512 with 256-wide tiles: 40 pair tiles split in three, more clusters of three
    # pairs than fit at once (23) -> global split slots
    os.environ["CAKE_GG_WIDE"] = "0"
    try:
        plan = gg.cake_gg_plan("wgrad", 1, 16384, 512, 5120, "fp32", 1)
    finally:
        del os.environ["CAKE_GG_WIDE"]
    assert plan.tile_n == 256 and plan.cluster_splits == 0 and plan.split_chunk > 0


def test_tile_walk_nsplit_tail_two_experts():
    """Two experts of 16384 rows, 3072 x 4096: 192 units of 256 x 512, a last wave of 40 of
    the 76 pairs -- too full for the K-split tail -- runs by the N-split rule as 4 column pieces
    of 128 per unit (160 pieces), each over all of its expert's k-blocks.  (The rule is off
    unless asked for: measured slower.)"""
    assert gg.cake_gg_plan("wgrad", 2, 32768, 3072, 4096, "bf16", 1).tail_nsplit == 0
    plan, tiles = _check_walk_coverage("wgrad", [16384, 16384], N=3072, K=4096, env={"CAKE_GG_NTAIL": "1"})
    assert plan.tile_n == 512 and plan.pair == 2
    assert (plan.tail_units, plan.tail_nsplit, plan.tail_splits) == (40, 4, 0)
    assert plan.workspace_bytes == 256
    pieces = tiles[tiles[:, 9] < 512]
    assert len(pieces) == 40 * 4 * 2 and set(pieces[:, 9]) == {128}
    assert (pieces[:, 5] == 0).all() and (pieces[:, 6] == 16384 // plan.tile_k).all()


def test_tile_walk_nsplit_tail_forced_ragged():
    os.environ["CAKE_GG_WIDE"] = "2"
    try:
        plan, tiles = _check_walk_coverage("wgrad", [9000, 0, 16000], N=256, K=1152,
                                           env={"CAKE_GG_NTAIL": "4", "CAKE_GG_SPLIT_CHUNK": "0"})
    finally:
        del os.environ["CAKE_GG_WIDE"]
    assert plan.tile_n == 512 and plan.tail_nsplit == 4 and plan.tail_units == 9


def test_tile_walk_cluster_split_with_small_and_empty_experts():
    _check_walk_coverage("wgrad", [0, 100, 3000, 65, 1], N=48, K=512, env={"CAKE_GG_CSPLIT": "4"})


def test_tile_walk_rejects_bad_offsets():
    plan = gg.cake_gg_plan("fwd", 2, 100, 64, 64, "bf16", 1)
    for bad in ([1, 5, 9], [0, 9, 5], [0, 5, 101]):
        with pytest.raises(gg.CakeGGError) as ei:
            gg.cake_gg_tile_walk(plan, np.array(bad, np.int32))
        assert ei.value.code == gg.CAKE_GG_ERR_BAD_OFFSETS


def test_compute_calls_reject_bad_arguments_before_any_cuda_call():
    """Host validation runs before the library touches CUDA (works without a GPU)."""
    plan = gg.cake_gg_plan("fwd", 2, 256, 64, 64, "bf16", 1)
    good = 1 << 20
    # null pointer
    assert gg.cake_gg_fwd(plan, 0, good, good, good, "bf16", 1, good, 4096, 0) == gg.CAKE_GG_ERR_INVALID_ARG
    # misaligned pointer
    assert gg.cake_gg_fwd(plan, good + 2, good, good, good, "bf16", 1, good, 4096, 0) == gg.CAKE_GG_ERR_ALIGNMENT
    # plan / call mismatch: dtype, determinism, pass
    assert gg.cake_gg_fwd(plan, good, good, good, good, "fp32", 1, good, 4096, 0) == gg.CAKE_GG_ERR_INVALID_ARG
    assert gg.cake_gg_fwd(plan, good, good, good, good, "bf16", 0, good, 4096, 0) == gg.CAKE_GG_ERR_INVALID_ARG
    assert gg.cake_gg_dgrad(plan, good, good, good, good, "bf16", 1, good, 4096, 0) == gg.CAKE_GG_ERR_INVALID_ARG
    # workspace too small
    assert gg.cake_gg_fwd(plan, good, good, good, good, "bf16", 1, good, 16, 0) == gg.CAKE_GG_ERR_WORKSPACE
    wplan = gg.cake_gg_plan("wgrad", 1, 16384, 48, 4096, "fp32", 1)
    assert gg.cake_gg_wgrad(wplan, good, good, good, good, "fp32", 1, good,
                            wplan.workspace_bytes - 1, 0) == gg.CAKE_GG_ERR_WORKSPACE


def test_tile_walk_split_tail():
    """The last partial wave of weight-gradient units runs as pieces: every output element is still
    covered once, each tail tile's pieces partition its expert's k-blocks, the rest stay whole."""
    plan, tiles = _check_walk_coverage("wgrad", [16384] * 8, N=3072, K=4096)
    assert plan.tile_n == 512 and plan.tail_units == 8 and plan.tail_splits == 4
    pieces = [t for t in tiles if t[4] > 1]
    assert len(pieces) == plan.tail_units * plan.pair * plan.tail_splits
    assert len(tiles) - len(pieces) == (8 * 12 * 8 - plan.tail_units) * plan.pair
    # nearly balanced experts: the pieces belong to the lightest expert, walked last
    plan, tiles = _check_walk_coverage("wgrad", [8300, 8200, 8192, 8100], N=3072, K=4096)
    assert (plan.tile_n, plan.tail_units, plan.tail_splits) == (512, 4, 8)
    assert {t[0] for t in tiles if t[4] > 1} == {3}
    # skewed experts (lightest below 80% of the heaviest): the plan reserves a tail, the walk
    # keeps every unit whole (its last units are short already)
    plan, tiles = _check_walk_coverage("wgrad", [59491, 25895, 15919, 11271], N=6144, K=2048)
    assert plan.tail_splits > 1
    assert not [t for t in tiles if t[4] > 1]


@pytest.mark.parametrize("sizes,N,K,force", [([16384], 512, 4096, False), ([16384], 1024, 5120, False),
                                             ([16300], 512, 4096, False), ([1000], 512, 1024, True),
                                             ([300], 384, 2048, True)])
def test_tile_walk_streamk(sizes, N, K, force):
    """Stream-K walk of a one-expert weight gradient: every output tile is covered once by pieces
    that partition its k-blocks in order; every virtual pair does at most L k-blocks; the m-units
    of a segment get the same (n-tile, k-range) pieces (they read the same operand rows)."""
    env = {"CAKE_GG_STREAMK": "2" if force else "1"}
    plan, tiles = _check_walk_coverage("wgrad", sizes, N=N, K=K, env=env)
    L = plan.streamk_kblocks
    assert L > 0 and plan.split_chunk == 0 and plan.tail_splits == 0
    KB = -(-sizes[0] // plan.tile_k)
    n_tiles = -(-K // plan.tile_n)
    m_units = -(-(-(-N // 128)) // 2)
    # each m-unit's pieces (its even CTA's tiles) as linear k-block ranges of [0, n_tiles * KB)
    per_v = {}
    for e, mt, nt, s, S, kb0, kb1, _ in tiles[:, :8]:
        if mt % 2 == 0:
            per_v.setdefault(mt // 2, []).append((nt * KB + kb0, nt * KB + kb1))
    assert len(per_v) == m_units
    # the linear k-block ranges of each m-unit tile the work [0, n_tiles * KB) and cut it every L
    for mu, ranges in per_v.items():
        ranges.sort()
        assert ranges[0][0] == 0 and ranges[-1][1] == n_tiles * KB
        for (a0, a1), (b0, b1) in zip(ranges, ranges[1:]):
            assert a1 == b0
        cuts = sorted({r[0] for r in ranges} | {n_tiles * KB})
        for c in cuts:
            assert c % L == 0 or c % KB == 0
        # a segment's pieces sum to L k-blocks (the last one to the remainder)
        seg = {}
        for a0, a1 in ranges:
            seg[a0 // L] = seg.get(a0 // L, 0) + (a1 - a0)
        assert max(seg.values()) <= L
    assert len({tuple(sorted(r)) for r in per_v.values()}) == 1   # the m-units run the same pieces


def test_tile_walk_streamk_empty_expert_writes_zero_tiles():
    """No rows at run time (the plan was made for more): every tile is one piece of one k-block
    whose rows all lie past the expert's end (zeroed), so dW is written as exact zeros."""
    os.environ["CAKE_GG_STREAMK"] = "2"
    try:
        plan = gg.cake_gg_plan("wgrad", 1, 4096, 512, 1024, "fp32", 1)
    finally:
        del os.environ["CAKE_GG_STREAMK"]
    assert plan.streamk_kblocks > 0
    tiles = gg.cake_gg_tile_walk(plan, np.array([0, 0], np.int32))
    assert {(t[1], t[2]) for t in tiles} == {(m, n) for m in range(4) for n in range(1024 // plan.tile_n)}
    assert all(t[5] == 0 and t[6] == 1 for t in tiles)


@pytest.mark.parametrize("E,M,N,K,od,field,det_value", [
    (1, 16384, 512, 4096, "fp32", "cluster_splits", 2),   # split (on chip, two-pair clusters) dropped
    (1, 16384, 1024, 5120, "fp32", "tail_splits", 8),     # split tail dropped
    (1, 16384, 4096, 4096, "fp32", "tile_n", 512),        # 256 x 512 tiles dropped
    (8, 131072, 4096, 6144, "bf16", "tail_splits", 2),    # split tail dropped
    (1, 16384, 48, 4096, "fp32", "cluster_splits", 4),    # on-chip reduction dropped (workspace slots)
    (1, 16384, 512, 5120, "fp32", "cluster_splits", 3),
])
def test_nondeterministic_planner_drops_rules_that_failed_the_decision_protocol(E, M, N, K, od, field, det_value):
    """At points where a plan rule failed the pages' decision protocol (measured with bench.py
    --decide), the non-deterministic planner runs the baseline plan; the deterministic planner keeps
    the rule; CAKE_GG_DECIDED=0 restores the rule for non-deterministic plans."""
    det = gg.cake_gg_plan("wgrad", E, M, N, K, od, 1).as_dict()
    nd = gg.cake_gg_plan("wgrad", E, M, N, K, od, 0).as_dict()
    assert det[field] == det_value
    assert nd[field] != det_value
    os.environ["CAKE_GG_DECIDED"] = "0"
    try:
        nd_rule = gg.cake_gg_plan("wgrad", E, M, N, K, od, 0).as_dict()
    finally:
        del os.environ["CAKE_GG_DECIDED"]
    choices = ("tile_n", "tile_k", "stages", "pair", "swap_ab", "split_chunk", "cluster_splits", "tail_units",
               "tail_splits", "staging_bufs", "streamk_kblocks")
    assert {k: nd_rule[k] for k in choices} == {k: det[k] for k in choices}


def _slack_rule_reference(sizes, plan):
    """Independent restatement of the slack-placement rule (PR #8258, opening summary, 2nd
    paragraph): walk the experts heaviest first (ties by index); every unit of an expert lasts its
    k-blocks; the walk's units go, in order, to whichever of the 76 pairs becomes free first (a heap
    of pair loads); each of the last tail_units units must fit on the least-loaded pair within the
    largest load plus one tail share (k-blocks / tail_splits) plus the split's own cost.  True: the
    tail runs whole."""
    import heapq
    bk = plan.tile_k
    m_units = -(-(-(-plan.N // 128)) // 2)
    n_tiles = -(-plan.K // plan.tile_n)
    kb = [-(-s_ // bk) for s_ in sizes]
    order = sorted(range(len(sizes)), key=lambda e: (-kb[e], e))
    walk = [kb[e] for e in order for _ in range(m_units * n_tiles)]
    T = plan.tail_units
    loads = [0] * 76
    heapq.heapify(loads)
    for c in walk[:len(walk) - T]:
        heapq.heappush(loads, heapq.heappop(loads) + c)
    # what a split costs on top of its pieces, in k-blocks: partial tile write + read (x2) and the
    # finish, as the planner's split model charges it
    ovh = -(-(4096 * plan.tile_n * 64) // ((16384 + 128 * plan.tile_n) * bk)) + -(-(4 * 64) // bk)
    for c in walk[len(walk) - T:]:
        lo = heapq.heappop(loads)
        if (lo + c - max(loads + [lo]) - ovh) * plan.tail_splits > c:
            return False
        heapq.heappush(loads, lo + c)
    return True


@pytest.mark.parametrize("seed", range(12))
def test_split_tail_slack_placement_matches_a_heap_schedule(seed):
    """The walk's decision (tail pieces present or not) equals the reference rule above on ragged
    experts around the planned size (the plan assumes balanced experts: 4 x 8192 rows)."""
    rng = np.random.default_rng(seed)
    plan = gg.cake_gg_plan("wgrad", 4, 4 * 8192 + 5, 3072, 4096, "bf16", 1)
    assert plan.tail_splits > 1
    spread = [0.0, 0.01, 0.05, 0.2, 0.5, 0.9][seed % 6]
    sizes = [max(0, int(8192 * (1 + spread * rng.uniform(-1, 1)))) for _ in range(4)]
    scale = (4 * 8192) / max(1, sum(sizes))
    sizes = [int(x * scale) for x in sizes]
    tiles = gg.cake_gg_tile_walk(plan, wl.offsets_from_sizes(sizes))
    has_pieces = bool((tiles[:, 4] > 1).any())
    assert has_pieces == (not _slack_rule_reference(sizes, plan)), sizes


# ---- FP32 router GEMM (BF16x3) planning, host side -----------------------------------------


def test_router_plan_validates_and_sizes_its_workspace():
    """cake_gg_router_plan: R and K multiples of 8, T >= 0; the workspace is the kernel header,
    the one-expert offsets and W' [R, 2K] in BF16; the plan it runs is the one-expert forward
    pass over the original K (the router kernel splits X itself)."""
    for args, code in [((16, 250, 64), gg.CAKE_GG_ERR_ALIGNMENT), ((16, 256, 60), gg.CAKE_GG_ERR_ALIGNMENT),
                       ((-1, 256, 64), gg.CAKE_GG_ERR_INVALID_ARG), ((16, 0, 64), gg.CAKE_GG_ERR_INVALID_ARG),
                       ((16, 256, 64, -1), gg.CAKE_GG_ERR_INVALID_ARG)]:
        with pytest.raises(gg.CakeGGError) as ei:
            gg.cake_gg_router_plan(*args)
        assert ei.value.code == code, args
    rp = gg.cake_gg_router_plan(16384, 256, 4096)
    assert (rp.T, rp.R, rp.K) == (16384, 256, 4096)
    g = rp.gemm
    assert (g.E, g.N, g.K, g.M_max, g.pass_) == (1, 256, 4096, 16384, gg.CAKE_GG_FWD)
    assert g.out_dtype == gg.CAKE_GG_FP32 and g.deterministic == 1
    assert (g.tile_n, g.tile_k, g.pair) == (256, 64, 2) and g.stages >= 2
    hdr = (int(g.workspace_bytes) + 255) // 256 * 256
    assert rp.workspace_bytes == hdr + 256 + (256 * 2 * 4096 * 2 + 255) // 256 * 256
    # small router widths run single CTAs on 64-wide tiles
    small = gg.cake_gg_router_plan(300, 16, 64)
    assert (small.gemm.tile_n, small.gemm.pair) == (64, 1)
    # no dependence on max_sms beyond the field itself
    capped = gg.cake_gg_router_plan(16384, 256, 4096, 10)
    assert capped.workspace_bytes == rp.workspace_bytes and capped.gemm.stages == g.stages


def test_router_plans_fit_the_kernels_tensor_memory():
    """The router kernel keeps its accumulator in TMEM columns 0..tile_n-1 and each stage's
    split A tile (32 columns of BF16 high parts, 32 of low parts) at 256 + 64 * stage, in a
    512-column allocation: every plan has tile_n <= 256 and 2..4 stages of 64-deep k-blocks,
    pairs only on tiles whose half is a whole number of 64-row W boxes."""
    for R in (8, 16, 24, 64, 120, 128, 136, 192, 248, 256, 264, 512, 1024):
        for K in (8, 64, 1096, 4096):
            g = gg.cake_gg_router_plan(1000, R, K).gemm
            assert g.tile_n <= 256 and g.tile_n % 64 == 0 and g.tile_n >= min(R, 256), (R, K)
            assert 256 + 64 * g.stages <= 512 and g.stages >= 2, (R, K)
            assert g.tile_k == 64
            assert g.pair in (1, 2) and (g.pair == 1 or (g.tile_n // 2) % 64 == 0), (R, K)


def test_router_plan_struct_layout():
    """The ctypes mirror of cake_gg_router_plan_t: 8-byte aligned fields, the nested forward plan last."""
    assert gg.CakeGGRouterPlan.gemm.offset % 8 == 0
    assert gg.CakeGGRouterPlan.workspace_bytes.offset == 24
    assert ctypes.sizeof(gg.CakeGGRouterPlan) == 32 + ctypes.sizeof(gg.CakeGGPlan)


def test_router_call_rejects_bad_arguments_before_any_cuda_call():
    """cake_gg_router_fp32's host checks (null, misaligned, workspace) run before any CUDA call."""
    lib = gg.load_library()
    rp = gg.cake_gg_router_plan(256, 64, 128)
    good, nb = 1 << 20, int(rp.workspace_bytes)
    call = lambda x, w, y, ws, n: lib.cake_gg_router_fp32(ctypes.byref(rp), x, w, y, ws, n, None)
    assert call(0, good, good, good, nb) == gg.CAKE_GG_ERR_INVALID_ARG          # null X
    assert call(good, good, good, 0, nb) == gg.CAKE_GG_ERR_INVALID_ARG          # null workspace
    assert call(good + 4, good, good, good, nb) == gg.CAKE_GG_ERR_ALIGNMENT     # misaligned X
    assert call(good, good, good, good, nb - 1) == gg.CAKE_GG_ERR_WORKSPACE     # workspace too small
    bad = gg.CakeGGRouterPlan.from_buffer_copy(rp)
    bad.gemm.K = 3 * rp.K                                                       # plan / call mismatch
    assert lib.cake_gg_router_fp32(ctypes.byref(bad), good, good, good, good, nb, None) == gg.CAKE_GG_ERR_INVALID_ARG
    # a tile shape or ring depth other than the planner's (the kernel's tensor-memory
    # A slots and shared-memory layout follow them)
    for field, value in (("stages", rp.gemm.stages - 1), ("tile_n", 128), ("pair", 3 - rp.gemm.pair),
                         ("tile_k", 128)):
        bad = gg.CakeGGRouterPlan.from_buffer_copy(rp)
        setattr(bad.gemm, field, value)
        assert lib.cake_gg_router_fp32(ctypes.byref(bad), good, good, good, good, nb, None) == \
            gg.CAKE_GG_ERR_INVALID_ARG, field


C_PROGRAM = r"""
#include <stddef.h>
#include <stdio.h>
#include "cake_gg.h"

int main(void)
{
    cake_gg_plan_t plan;
    cake_gg_router_plan_t rp;
    int rc = cake_gg_plan(&plan, CAKE_GG_WGRAD, 8, 131072, 3072, 4096, CAKE_GG_BF16, 1, 0);
    if (rc != CAKE_GG_OK) {
        printf("error %d %s\n", rc, cake_gg_strerror(rc));
        return 1;
    }
    rc = cake_gg_router_plan(&rp, 16384, 256, 4096, 0);
    if (rc != CAKE_GG_OK) return 2;
    printf("%u %u %u %u %u %u %u\n", (unsigned)sizeof(cake_gg_plan_t), (unsigned)offsetof(cake_gg_plan_t, M_max),
           (unsigned)offsetof(cake_gg_plan_t, timeout_ns), (unsigned)offsetof(cake_gg_plan_t, workspace_bytes),
           (unsigned)offsetof(cake_gg_plan_t, staging_bufs), (unsigned)sizeof(cake_gg_router_plan_t),
           (unsigned)offsetof(cake_gg_router_plan_t, gemm));
    printf("%d %d %d %d %d %d %llu %llu\n", plan.tile_n, plan.tile_k, plan.stages, plan.pair, plan.split_chunk,
           plan.tail_splits, (unsigned long long)plan.workspace_bytes, (unsigned long long)rp.workspace_bytes);
    return 0;
}
"""


def test_header_compiles_as_c99_and_layouts_match(tmp_path):
    """A strict C99 program includes the header, links the library and plans on the host: the
    ABI is plain C, its struct layouts are the ctypes mirrors', and C callers get the same plan."""
    import shutil
    import subprocess
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    src = tmp_path / "abi.c"
    src.write_text(C_PROGRAM)
    exe = tmp_path / "abi"
    libdir = os.path.dirname(gg.LIB_PATH)
    r = subprocess.run([cc, "-std=c99", "-Wall", "-Wextra", "-Werror", "-pedantic", "-I",
                        os.path.join(ROOT, "include"), str(src), "-o", str(exe), "-L", libdir, "-lcake_gg",
                        f"-Wl,-rpath,{libdir}"], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    run = subprocess.run([str(exe)], capture_output=True, text=True, timeout=60)
    assert run.returncode == 0, run.stdout + run.stderr
    layout, fields = [line.split() for line in run.stdout.strip().splitlines()]
    P, R = gg.CakeGGPlan, gg.CakeGGRouterPlan
    assert [int(v) for v in layout] == [ctypes.sizeof(P), P.M_max.offset, P.timeout_ns.offset,
                                        P.workspace_bytes.offset, P.staging_bufs.offset, ctypes.sizeof(R),
                                        R.gemm.offset]
    plan = gg.cake_gg_plan("wgrad", 8, 131072, 3072, 4096, "bf16", 1)
    rp = gg.cake_gg_router_plan(16384, 256, 4096)
    assert [int(v) for v in fields] == [plan.tile_n, plan.tile_k, plan.stages, plan.pair, plan.split_chunk,
                                        plan.tail_splits, plan.workspace_bytes, rp.workspace_bytes]
