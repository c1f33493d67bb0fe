"""Pins for the FP64 oracle: checks against things other than the oracle itself.

Each test ties the oracle to a fact fixed by the pages or by mathematics:
a hand-worked example (tests/golden), the E = 1 case that is one dense GEMM
(numpy's matmul), per-expert blocks that are dense GEMMs, the identity
sum_e dW_e = G^T X, exact integer arithmetic, one-hot and all-zero inputs,
the empty expert, and a pure-Python brute force on tiny inputs.  Formulas:
flashinfer PR #8258, opening summary (Y = X W^T, dX = G W, dW = G^T X over
ragged expert row groups).
"""
import os

import numpy as np
import pytest

import oracle
from moe_ragged_grouped_gb300 import workloads as wl

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _f64(bits):
    return oracle.bf16_bits_to_f64(bits)


def _rand_problem(sizes, N, K, seed, extra_rows=0):
    rng = np.random.default_rng(seed)
    E = len(sizes)
    M = sum(sizes) + extra_rows
    X = wl.randn_bf16((M, K), 1.0, rng)
    W = wl.randn_bf16((E, N, K), 1.0 / np.sqrt(K), rng)
    G = wl.randn_bf16((M, N), 1.0, rng)
    return X, W, G, wl.offsets_from_sizes(sizes)


def _load_golden(name):
    data, lines = {}, open(os.path.join(GOLDEN, name)).read().splitlines()
    lines = [ln for ln in lines if ln.strip() and not ln.startswith("#")]
    i = 0
    while i < len(lines):
        parts = lines[i].split()
        key = parts[0]
        if key in ("E", "N", "K"):
            data[key] = int(parts[1]); i += 1
        elif key == "offsets":
            data[key] = np.array([int(v) for v in parts[1:]], dtype=np.int32); i += 1
        else:
            rows, cols = int(parts[1]), int(parts[2])
            vals = [[float(v) for v in lines[i + 1 + r].split()] for r in range(rows)]
            data[key] = np.array(vals, dtype=np.float64); i += 1 + rows
    return data


def test_hand_worked_golden(oracle_lib):
    d = _load_golden("hand_worked_E3_N2_K2.txt")
    E, N, K = d["E"], d["N"], d["K"]
    X = wl.f32_to_bf16_bits(d["X"].astype(np.float32))
    W = wl.f32_to_bf16_bits(d["W"].astype(np.float32)).reshape(E, N, K)
    G = wl.f32_to_bf16_bits(d["G"].astype(np.float32))
    off = d["offsets"]
    np.testing.assert_array_equal(oracle.fwd(X, W, off, oracle_lib), d["Y"])
    np.testing.assert_array_equal(oracle.dgrad(G, W, off, oracle_lib), d["dX"])
    np.testing.assert_array_equal(oracle.wgrad(G, X, off, E, oracle_lib).reshape(E * N, K), d["dW"])


@pytest.mark.parametrize("N,K,T", [(48, 64, 37), (16, 40, 130), (64, 24, 1)])
def test_e1_is_one_dense_gemm(oracle_lib, N, K, T):
    """E = 1 reduces to a single dense GEMM (numpy float64 matmul)."""
    X, W, G, off = _rand_problem([T], N, K, seed=N + K + T)
    Xf, Wf, Gf = _f64(X), _f64(W)[0], _f64(G)
    np.testing.assert_allclose(oracle.fwd(X, W, off, oracle_lib), Xf @ Wf.T, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(oracle.dgrad(G, W, off, oracle_lib), Gf @ Wf, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(oracle.wgrad(G, X, off, 1, oracle_lib)[0], Gf.T @ Xf, rtol=1e-12, atol=1e-12)


def test_per_expert_blocks_are_dense_gemms(oracle_lib):
    """Each expert's rows are an independent dense GEMM with that expert's W."""
    sizes = [3, 0, 17, 9, 1]
    N, K = 24, 40
    X, W, G, off = _rand_problem(sizes, N, K, seed=7, extra_rows=5)
    Y = oracle.fwd(X, W, off, oracle_lib)
    dX = oracle.dgrad(G, W, off, oracle_lib)
    dW = oracle.wgrad(G, X, off, len(sizes), oracle_lib)
    Xf, Wf, Gf = _f64(X), _f64(W), _f64(G)
    for e in range(len(sizes)):
        r0, r1 = off[e], off[e + 1]
        np.testing.assert_allclose(Y[r0:r1], Xf[r0:r1] @ Wf[e].T, rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(dX[r0:r1], Gf[r0:r1] @ Wf[e], rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(dW[e], Gf[r0:r1].T @ Xf[r0:r1], rtol=1e-12, atol=1e-12)


def test_wgrad_sum_over_experts_identity(oracle_lib):
    """sum_e dW_e equals G^T X over all routed rows (rows beyond off[E] excluded)."""
    sizes = [5, 11, 0, 32, 2]
    X, W, G, off = _rand_problem(sizes, 16, 24, seed=11, extra_rows=9)
    dW = oracle.wgrad(G, X, off, len(sizes), oracle_lib)
    M = off[-1]
    np.testing.assert_allclose(dW.sum(axis=0), _f64(G)[:M].T @ _f64(X)[:M], rtol=1e-12, atol=1e-11)


def test_exact_integer_inputs(oracle_lib):
    """Small-integer inputs: every sum is exact, so the oracle equals integer matmul."""
    rng = np.random.default_rng(3)
    sizes = [7, 0, 33, 12]
    E, N, K = len(sizes), 32, 48
    M = sum(sizes)
    X = wl.small_int_bf16((M, K), rng)
    W = wl.small_int_bf16((E, N, K), rng)
    G = wl.small_int_bf16((M, N), rng)
    off = wl.offsets_from_sizes(sizes)
    Xi, Wi, Gi = (_f64(a).astype(np.int64) for a in (X, W, G))
    Y = oracle.fwd(X, W, off, oracle_lib)
    dX = oracle.dgrad(G, W, off, oracle_lib)
    dW = oracle.wgrad(G, X, off, E, oracle_lib)
    for e in range(E):
        r0, r1 = off[e], off[e + 1]
        np.testing.assert_array_equal(Y[r0:r1], Xi[r0:r1] @ Wi[e].T)
        np.testing.assert_array_equal(dX[r0:r1], Gi[r0:r1] @ Wi[e])
        np.testing.assert_array_equal(dW[e], Gi[r0:r1].T @ Xi[r0:r1])


def test_one_hot_inputs_select_weights(oracle_lib):
    """One-hot X rows pick a column of W_e; one-hot G rows pick a row of W_e."""
    sizes = [4, 6]
    E, N, K = 2, 16, 24
    rng = np.random.default_rng(5)
    W = wl.randn_bf16((E, N, K), 1.0, rng)
    off = wl.offsets_from_sizes(sizes)
    M = sum(sizes)
    one = wl.f32_to_bf16_bits(np.ones(1, np.float32))[0]
    X = np.zeros((M, K), np.uint16)
    G = np.zeros((M, N), np.uint16)
    kstar = [(3 * r + 1) % K for r in range(M)]
    nstar = [(5 * r + 2) % N for r in range(M)]
    for r in range(M):
        X[r, kstar[r]] = one
        G[r, nstar[r]] = one
    Y = oracle.fwd(X, W, off, oracle_lib)
    dX = oracle.dgrad(G, W, off, oracle_lib)
    Wf = _f64(W)
    for r in range(M):
        e = 0 if r < off[1] else 1
        np.testing.assert_array_equal(Y[r], Wf[e][:, kstar[r]])
        np.testing.assert_array_equal(dX[r], Wf[e][nstar[r], :])
    # one row per expert carrying a one-hot pair: dW_e has a single 1 at (n*, k*)
    dW = oracle.wgrad(G, X, np.array([0, 1, 2], np.int32), 2, oracle_lib)
    for e in range(2):
        expect = np.zeros((N, K))
        expect[nstar[e], kstar[e]] = 1.0
        np.testing.assert_array_equal(dW[e], expect)


def test_zero_inputs_and_empty_expert(oracle_lib):
    sizes = [0, 9, 0]
    E, N, K = 3, 8, 16
    M = 9
    zX = np.zeros((M, K), np.uint16)
    zG = np.zeros((M, N), np.uint16)
    rng = np.random.default_rng(0)
    W = wl.randn_bf16((E, N, K), 1.0, rng)
    off = wl.offsets_from_sizes(sizes)
    assert not oracle.fwd(zX, W, off, oracle_lib).any()
    assert not oracle.dgrad(zG, W, off, oracle_lib).any()
    X = wl.randn_bf16((M, K), 1.0, rng)
    G = wl.randn_bf16((M, N), 1.0, rng)
    dW = oracle.wgrad(G, X, off, E, oracle_lib)
    assert not dW[0].any() and not dW[2].any()
    assert dW[1].any()


def test_rows_beyond_last_offset_do_not_contribute(oracle_lib):
    """NaN rows after off[E] never reach any output."""
    sizes = [5, 3]
    X, W, G, off = _rand_problem(sizes, 16, 16, seed=2, extra_rows=4)
    nan = wl.f32_to_bf16_bits(np.array([np.nan], np.float32))[0]
    X[8:] = nan
    G[8:] = nan
    assert np.isfinite(oracle.fwd(X, W, off, oracle_lib)).all()
    assert np.isfinite(oracle.dgrad(G, W, off, oracle_lib)).all()
    assert np.isfinite(oracle.wgrad(G, X, off, 2, oracle_lib)).all()


def test_pure_python_brute_force(oracle_lib):
    """A direct triple loop in Python (exact rational-free float sums) on tiny inputs."""
    sizes = [2, 0, 3]
    E, N, K = 3, 3, 4
    X, W, G, off = _rand_problem(sizes, N, K, seed=9)
    Xf, Wf, Gf = _f64(X), _f64(W), _f64(G)
    Y = oracle.fwd(X, W, off, oracle_lib)
    dX = oracle.dgrad(G, W, off, oracle_lib)
    dW = oracle.wgrad(G, X, off, E, oracle_lib)
    for e in range(E):
        for r in range(off[e], off[e + 1]):
            for n in range(N):
                s = 0.0
                for k in range(K):
                    s += float(Xf[r, k]) * float(Wf[e, n, k])
                assert Y[r, n] == s
            for k in range(K):
                s = 0.0
                for n in range(N):
                    s += float(Gf[r, n]) * float(Wf[e, n, k])
                assert dX[r, k] == s
        for n in range(N):
            for k in range(K):
                s = 0.0
                for r in range(off[e], off[e + 1]):
                    s += float(Gf[r, n]) * float(Xf[r, k])
                assert dW[e, n, k] == s


def test_dgrad_is_forward_with_transposed_weights(oracle_lib):
    """dX = G W equals the forward pass with W'_e = W_e^T stored [E, K, N]."""
    sizes = [6, 10]
    X, W, G, off = _rand_problem(sizes, 16, 24, seed=4)
    Wt = np.ascontiguousarray(np.transpose(W, (0, 2, 1)))
    np.testing.assert_array_equal(oracle.dgrad(G, W, off, oracle_lib), oracle.fwd(G, Wt, off, oracle_lib))


def test_sampled_entry_points_match_full(oracle_lib):
    sizes = [13, 0, 29, 4]
    E, N, K = 4, 24, 32
    X, W, G, off = _rand_problem(sizes, N, K, seed=8, extra_rows=3)
    rng = np.random.default_rng(1)
    M = off[-1]
    rows = rng.integers(0, M, 50)
    Y = oracle.fwd(X, W, off, oracle_lib)
    dX = oracle.dgrad(G, W, off, oracle_lib)
    dW = oracle.wgrad(G, X, off, E, oracle_lib)
    cn = rng.integers(0, N, 50)
    ck = rng.integers(0, K, 50)
    es = rng.integers(0, E, 50)
    np.testing.assert_array_equal(oracle.fwd_at(X, W, off, rows, cn, oracle_lib), Y[rows, cn])
    np.testing.assert_array_equal(oracle.dgrad_at(G, W, off, rows, ck, oracle_lib), dX[rows, ck])
    np.testing.assert_array_equal(oracle.wgrad_at(G, X, off, E, es, cn, ck, oracle_lib), dW[es, cn, ck])


@pytest.mark.parametrize("bad", [[1, 3, 5], [0, 4, 3], [0, 2, 99]])
def test_invalid_offsets_rejected(oracle_lib, bad):
    X, W, G, _ = _rand_problem([2, 3], 8, 8, seed=0)
    with pytest.raises(ValueError):
        oracle.fwd(X, W, np.array(bad, np.int32), oracle_lib)
    with pytest.raises(ValueError):
        oracle.wgrad(G, X, np.array(bad, np.int32), 2, oracle_lib)


def test_bf16_widening_is_exact():
    bits = np.array([0x3F80, 0xBF80, 0x0001, 0x7F7F, 0x4049], np.uint16)
    got = oracle.bf16_bits_to_f64(bits)
    assert got[0] == 1.0 and got[1] == -1.0
    assert got[2] == 2.0 ** -133          # smallest BF16 subnormal
    assert got[3] == (2 - 2 ** -7) * 2.0 ** 127
    assert got[4] == 3.140625
