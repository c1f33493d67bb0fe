"""Parity at the full configured sizes, in the launch configuration the benchmark uses.

Inputs are drawn on the GPU by a seeded generator (the benchmark's recipe) and
copied to the host for the FP64 oracle, which evaluates sampled outputs one by
one.  The sample is stratified by output tile: one random element from every
128-row x 64-column block of every output (forward / data gradient: blocks of
each expert's own rows, starting at its first row, so every tile any launch
shape takes is hit, including every piece of a split tail and every 64-column
slice a split finish reduces; weight gradient: blocks of every expert's dW,
empty experts included), plus uniform random elements, every expert's first
and last rows and the tile edges.  Each sample must satisfy the parity bound
|gpu - ref| <= 2^-8 |ref| + 2^-18 L max|a| max|b|.

Workloads (E experts, M routed rows, K, N):
  dense projection   E=1, T=16384, d_in in {4096, 5120}, d_out in {48, 64, 512, 1024, 4096}
  MoE gate_up        E=8, M=131072 balanced, K=4096, N=3072
  MoE down           E=32, M=131072 multinomial (seed 0), K=1536, N=4096
  skewed MoE         E=4, M=136064 Zipf(1.2) ascending with an empty expert, (K,N) = (4096,3072), (3072,4096)
  the pages' grid    gate_up N=4096 K=6144 and down N=6144 K=2048 with balanced, Zipf-skewed,
                     one-empty and lognormal group sizes (a few representative rows)
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


_cache = {}


def inputs(wk):
    """Device tensors and host bits of a workload (cached per module run)."""
    import torch
    if wk.name not in _cache:
        _cache.clear()
        torch.cuda.empty_cache()
        X, W, G = wk.make_torch(seed=0, device="cuda")
        bits = tuple(wl.torch_bf16_to_bits(t) for t in (X, W, G))
        _cache[wk.name] = (X, W, G, bits)
    return _cache[wk.name]


def tile_strata_rows_cols(off, n_out, rng):
    """One random (row, col) in every 128-row x 64-column block of each expert's rows."""
    rows, cols = [], []
    ncb = (n_out + 63) // 64
    c0 = np.arange(ncb, dtype=np.int64) * 64
    clen = np.minimum(64, n_out - c0)
    for e in range(len(off) - 1):
        r0, r1 = int(off[e]), int(off[e + 1])
        if r1 <= r0:
            continue
        starts = np.arange(r0, r1, 128, dtype=np.int64)
        lens = np.minimum(128, r1 - starts)
        rs = np.repeat(starts, ncb) + (rng.random(starts.size * ncb) * np.repeat(lens, ncb)).astype(np.int64)
        cs = np.tile(c0, starts.size) + (rng.random(starts.size * ncb) * np.tile(clen, starts.size)).astype(np.int64)
        rows.append(rs)
        cols.append(cs)
    return np.concatenate(rows), np.concatenate(cols)


def tile_strata_wgrad(E, N, K, rng):
    """One random (e, n, k) in every 128 x 64 block of every expert's dW [N, K]."""
    n0 = np.arange(0, N, 128, dtype=np.int64)
    k0 = np.arange(0, K, 64, dtype=np.int64)
    nn, kk = np.meshgrid(n0, k0, indexing="ij")
    nn, kk = nn.ravel(), kk.ravel()
    es = np.repeat(np.arange(E, dtype=np.int64), nn.size)
    nb = np.tile(nn, E)
    kb = np.tile(kk, E)
    ns = nb + (rng.random(nb.size) * np.minimum(128, N - nb)).astype(np.int64)
    ks = kb + (rng.random(kb.size) * np.minimum(64, K - kb)).astype(np.int64)
    return es, ns, ks


def sample_rows_cols(off, n_out, rng, n=384):
    M = int(off[-1])
    rows = list(rng.integers(0, M, n))
    for e in range(len(off) - 1):
        if off[e + 1] > off[e]:
            rows += [int(off[e]), int(off[e + 1]) - 1, min(int(off[e]) + 127, int(off[e + 1]) - 1),
                     min(int(off[e]) + 128, int(off[e + 1]) - 1)]
    rows = np.array(rows, np.int64)
    cols = rng.integers(0, n_out, rows.shape[0])
    edge = np.array([0, n_out - 1, min(63, n_out - 1), min(64, n_out - 1), min(255, n_out - 1),
                     min(256, n_out - 1)], np.int64)
    cols[:edge.shape[0]] = edge
    sr, sc = tile_strata_rows_cols(off, n_out, rng)
    return np.concatenate([rows, sr]), np.concatenate([cols, sc])


def run_and_check(wk, pass_, out_dtype, det, rng, env=None, monkeypatch=None):
    import torch
    if env:
        for k, v in env.items():
            monkeypatch.setenv(k, v)
    X, W, G, (Xb, Wb, Gb) = inputs(wk)
    off = wk.offsets
    offs = torch.from_numpy(off).cuda()
    a, b = {"fwd": (X, W), "dgrad": (G, W), "wgrad": (G, X)}[pass_]
    out = gg.grouped_gemm(pass_, a, b, offs, out_dtype=out_dtype, deterministic=det)
    torch.cuda.synchronize()
    f = lambda t: float(np.abs(oracle.bf16_bits_to_f64(t)).max())
    M = int(off[-1])
    if pass_ == "wgrad":
        sizes = np.diff(off)
        es = list(rng.integers(0, wk.E, 384)) + list(range(wk.E)) * 4
        es = np.array(es, np.int64)
        ns = rng.integers(0, wk.N, es.shape[0])
        ks = rng.integers(0, wk.K, es.shape[0])
        ns[:4], ks[:4] = [0, wk.N - 1, 0, wk.N - 1], [0, wk.K - 1, wk.K - 1, 0]
        se, sn, sk = tile_strata_wgrad(wk.E, wk.N, wk.K, rng)
        es, ns, ks = np.concatenate([es, se]), np.concatenate([ns, sn]), np.concatenate([ks, sk])
        ref = oracle.wgrad_at(Gb, Xb, off, wk.E, es, ns, ks)
        idx = torch.from_numpy(es * wk.N * wk.K + ns * wk.K + ks).cuda()
        got_t = out.view(-1)[idx]
        L = sizes[es].astype(np.float64)
        ma, mb = f(Gb[:M]), f(Xb[:M])
    else:
        n_out = wk.N if pass_ == "fwd" else wk.K
        rows, cols = sample_rows_cols(off, n_out, rng)
        if pass_ == "fwd":
            ref = oracle.fwd_at(Xb, Wb, off, rows, cols)
            ma, mb, L = f(Xb[:M]), f(Wb), float(wk.K)
        else:
            ref = oracle.dgrad_at(Gb, Wb, off, rows, cols)
            ma, mb, L = f(Gb[:M]), f(Wb), float(wk.N)
        idx = torch.from_numpy(rows * n_out + cols).cuda()
        got_t = out.view(-1)[idx]
    if got_t.dtype == torch.bfloat16:
        got = oracle.bf16_bits_to_f64(wl.torch_bf16_to_bits(got_t))
    else:
        got = got_t.double().cpu().numpy()
    tol = oracle.tolerance(ref, L, ma, mb)
    bad = ~(np.abs(got - ref) <= tol)
    assert not bad.any(), (f"{wk.name} {pass_} {out_dtype} det={det}: {int(bad.sum())}/{bad.size} samples "
                           f"outside the bound; e.g. got {got[bad][:3]} ref {ref[bad][:3]}")
    del out


DENSE = [(4096, 48), (4096, 64), (5120, 48), (5120, 64), (4096, 512), (5120, 512),
         (4096, 1024), (5120, 1024), (4096, 4096), (5120, 4096)]


@pytest.mark.parametrize("d_in,d_out", DENSE)
def test_dense_projection(d_in, d_out, monkeypatch):
    wk = wl.dense_projection(d_in, d_out)
    rng = np.random.default_rng(d_in + d_out)
    run_and_check(wk, "wgrad", "fp32", 1, rng)
    run_and_check(wk, "wgrad", "fp32", 0, rng)
    run_and_check(wk, "fwd", "bf16", 1, rng)
    run_and_check(wk, "dgrad", "bf16", 1, rng)


@pytest.mark.parametrize("pass_", ["fwd", "dgrad", "wgrad"])
def test_moe_gate_up(pass_):
    run_and_check(wl.moe_gate_up(), pass_, "bf16", 1, np.random.default_rng(3))


@pytest.mark.parametrize("pass_", ["fwd", "dgrad"])
def test_moe_gate_up_fp32_output(pass_):
    """FP32 output of the forward and data gradient at full size (the FP32 accumulator stored as is)."""
    run_and_check(wl.moe_gate_up(), pass_, "fp32", 1, np.random.default_rng(4))


@pytest.mark.parametrize("out_dtype", ["fp32", "bf16"])
@pytest.mark.parametrize("det,env", [(1, None), (0, None), (1, {"CAKE_GG_SPLIT_CHUNK": "16"}),
                                     (0, {"CAKE_GG_SPLIT_CHUNK": "16"})])
def test_moe_down_weight_gradient(out_dtype, det, env, monkeypatch):
    run_and_check(wl.moe_down(), "wgrad", out_dtype, det, np.random.default_rng(4), env, monkeypatch)


@pytest.mark.parametrize("transposed", [False, True])
@pytest.mark.parametrize("pass_", ["fwd", "dgrad", "wgrad"])
def test_moe_skewed(transposed, pass_):
    run_and_check(wl.moe_skewed(transposed), pass_, "bf16", 1, np.random.default_rng(5))


@pytest.mark.parametrize("pass_", ["fwd", "dgrad", "wgrad"])
def test_skewed_deterministic_bitwise_runs_and_sm_caps(pass_):
    """Deterministic mode on the skewed workload: 20 runs and 100 / 148 SM caps, all bitwise equal."""
    import torch
    wk = wl.moe_skewed(False)
    X, W, G, _ = inputs(wk)
    offs = torch.from_numpy(wk.offsets).cuda()
    a, b = {"fwd": (X, W), "dgrad": (G, W), "wgrad": (G, X)}[pass_]
    ref = gg.grouped_gemm(pass_, a, b, offs, out_dtype="bf16", deterministic=1)
    M = int(wk.offsets[-1])
    view = (lambda t: t[:M]) if pass_ != "wgrad" else (lambda t: t)
    ref_v = view(ref).contiguous().view(torch.int16)
    out = torch.empty_like(ref)
    for i in range(20):
        gg.grouped_gemm(pass_, a, b, offs, out_dtype="bf16", deterministic=1, out=out)
        assert torch.equal(view(out).contiguous().view(torch.int16), ref_v), f"run {i}"
    for cap in (100, 148):
        gg.grouped_gemm(pass_, a, b, offs, out_dtype="bf16", deterministic=1, max_sms=cap, out=out)
        assert torch.equal(view(out).contiguous().view(torch.int16), ref_v), f"max_sms={cap}"


@pytest.mark.parametrize("shape,passes", [
    ("gate_up E4 M136064 1-empty asc", ("wgrad", "fwd", "dgrad")),
    ("gate_up E4 M112576 skew", ("wgrad",)),
    ("gate_up E32 M131072 random", ("wgrad",)),
    ("down E4 M112576 bal fp32", ("wgrad",)),
    ("down E8 M131072 random", ("wgrad", "fwd", "dgrad")),
])
def test_pages_grid_rows(shape, passes):
    """Shapes of the pages' GB300 latency table (weight gradient in its stated output dtype;
    the checkpointed rows' forward and data gradient in BF16)."""
    wk, od = wl.pages_workload(shape)
    rng = np.random.default_rng(7)
    for p in passes:
        run_and_check(wk, p, od if p == "wgrad" else "bf16", 1, rng)


TAIL = wl.Workload("tail_E4_M32792_K4096_N3072", 4, 3072, 4096, [8300, 8200, 8192, 8100])


@pytest.mark.parametrize("det,out_dtype", [(1, "fp32"), (0, "bf16"), (1, "bf16")])
def test_split_tail(det, out_dtype):
    """384 pair units of 256 x 512 = 5 waves of 76 + 4: the last 4 (the lightest expert's, 8100
    rows, its last k-block partial) run as 8 pieces each; sampled outputs against the oracle."""
    plan = gg.cake_gg_plan("wgrad", TAIL.E, TAIL.M, TAIL.N, TAIL.K, out_dtype, det)
    assert (plan.tile_n, plan.tail_units, plan.tail_splits) == (512, 4, 8)
    run_and_check(TAIL, "wgrad", out_dtype, det, np.random.default_rng(8))


def test_split_tail_bitwise_across_sm_caps():
    import torch
    X, W, G, _ = inputs(TAIL)
    offs = torch.from_numpy(TAIL.offsets).cuda()
    ref = gg.grouped_gemm("wgrad", G, X, offs, out_dtype="fp32", deterministic=1)
    for cap in (100, 148, 7, 0):
        out = gg.grouped_gemm("wgrad", G, X, offs, out_dtype="fp32", deterministic=1, max_sms=cap)
        assert torch.equal(out.view(torch.int32), ref.view(torch.int32)), f"max_sms={cap}"


def test_pair_cluster_split_bitwise_across_reductions_and_sm_caps(monkeypatch):
    """4096 -> 512 at T = 16384: 32 pair tiles, each split in two by a cluster of two pairs that
    reduces on chip; the same bits as the workspace-slot reduction of the same splits, and under
    SM caps that leave fewer clusters than tiles."""
    import torch
    wk = wl.dense_projection(4096, 512)
    X, W, G, _ = inputs(wk)
    offs = torch.from_numpy(wk.offsets).cuda()
    plan = gg.cake_gg_plan("wgrad", 1, wk.M, wk.N, wk.K, "fp32", 1)
    assert plan.pair == 2 and plan.cluster_splits == 2
    ref = gg.grouped_gemm("wgrad", G, X, offs, out_dtype="fp32", deterministic=1)
    for cap in (100, 148, 8):
        out = gg.grouped_gemm("wgrad", G, X, offs, out_dtype="fp32", deterministic=1, max_sms=cap)
        assert torch.equal(out.view(torch.int32), ref.view(torch.int32)), f"max_sms={cap}"
    monkeypatch.setenv("CAKE_GG_CSPLIT", "0")
    slots = gg.grouped_gemm("wgrad", G, X, offs, out_dtype="fp32", deterministic=1)
    assert torch.equal(slots.view(torch.int32), ref.view(torch.int32))


def test_nsplit_tail_two_experts(monkeypatch):
    """Two experts of 16384 rows, 3072 x 4096, with the N-split tail rule on: a last wave of 40
    of 76 pair units runs as 160 column pieces of 128; sampled against the oracle (every output
    tile), and bitwise the plan without a tail split, also under SM caps."""
    import torch
    monkeypatch.setenv("CAKE_GG_NTAIL", "1")
    wk = wl.Workload("moe_gate_up_E2_M32768_K4096_N3072", 2, 3072, 4096, wl.balanced_sizes(2, 32768))
    plan = gg.cake_gg_plan("wgrad", wk.E, wk.M, wk.N, wk.K, "bf16", 1)
    assert plan.tail_nsplit == 4 and plan.tail_units == 40
    run_and_check(wk, "wgrad", "bf16", 1, np.random.default_rng(35))
    X, W, G, _ = inputs(wk)
    offs = torch.from_numpy(wk.offsets).cuda()
    ref = gg.grouped_gemm("wgrad", G, X, offs, out_dtype="bf16", deterministic=1)
    for cap in (100, 0):
        out = gg.grouped_gemm("wgrad", G, X, offs, out_dtype="bf16", deterministic=1, max_sms=cap)
        assert torch.equal(out.view(torch.int16), ref.view(torch.int16)), f"max_sms={cap}"
    monkeypatch.setenv("CAKE_GG_TAIL", "0")
    whole = gg.grouped_gemm("wgrad", G, X, offs, out_dtype="bf16", deterministic=1)
    assert torch.equal(whole.view(torch.int16), ref.view(torch.int16))
