"""Pins for the oracle's FP32 router GEMM (BF16x3 emulation), on the CPU.

The dense projection family's FP32 router GEMM (flashinfer PR #8438,
"Summary", which names a router GEMM over 256 experts in FP32 emulated with
three BF16 products) computes logits Y = X W^T from FP32 X [T, K] and router weights W [R, K].  The reading
taken: v = hi + lo with hi = bf16(v) and lo = bf16(v - hi), round to nearest
even, and Y ~= sum_k x_hi w_hi + x_hi w_lo + x_lo w_hi.  These tests tie the
oracle to facts other than itself: the rounding rule at hand-picked ties and
overflow, a hand-worked product whose exact value is known, the special case
of BF16-representable inputs (the emulation is then exact), the emulation's
error bound, and a pure-Python restatement on tiny inputs.
"""
import math
import struct

import numpy as np
import pytest

import oracle


def _f32(v):
    return struct.unpack("<f", struct.pack("<f", v))[0]


@pytest.mark.parametrize("v,expect", [
    (1.0 + 2.0 ** -8, 1.0),                        # exact tie, kept part even: down
    (1.0 + 3 * 2.0 ** -8, 1.0 + 2.0 ** -6),        # exact tie, kept part odd: up to even
    (1.0 + 2.0 ** -8 + 2.0 ** -20, 1.0 + 2.0 ** -7),  # just above the tie: up
    (1.0 + 2.0 ** -8 - 2.0 ** -20, 1.0),           # just below the tie: down
    (-(1.0 + 3 * 2.0 ** -8), -(1.0 + 2.0 ** -6)),  # sign symmetric
    (2.0 ** 100 * (1.0 + 2.0 ** -9), 2.0 ** 100),  # exponent carried through
    (2.0 ** -133, 2.0 ** -133),                    # BF16 subnormal stays
    (1.5, 1.5),                                    # representable: unchanged
])
def test_round_bf16_nearest_even(v, expect, oracle_lib):
    assert oracle.round_bf16(_f32(v), oracle_lib) == expect


def test_round_bf16_overflow_and_nan(oracle_lib):
    flt_max = float(np.finfo(np.float32).max)
    assert oracle.round_bf16(flt_max, oracle_lib) == math.inf   # past the largest BF16's half-ulp
    assert oracle.round_bf16(math.inf, oracle_lib) == math.inf
    assert math.isnan(oracle.round_bf16(math.nan, oracle_lib))


def test_hand_worked_product(oracle_lib):
    """x = 1 + 2^-10, w = 1 + 2^-12 (K = 1): x_hi = w_hi = 1, x_lo = 2^-10, w_lo = 2^-12.
    The emulation keeps 1 + 2^-12 + 2^-10 and drops x_lo w_lo = 2^-22."""
    X = np.array([[1.0 + 2.0 ** -10]], dtype=np.float32)
    W = np.array([[1.0 + 2.0 ** -12]], dtype=np.float32)
    assert oracle.router_bf16x3(X, W, oracle_lib)[0, 0] == 1.0 + 2.0 ** -10 + 2.0 ** -12
    assert oracle.router_exact(X, W, oracle_lib)[0, 0] == 1.0 + 2.0 ** -10 + 2.0 ** -12 + 2.0 ** -22


def test_bf16_representable_inputs_are_exact(oracle_lib):
    """When every value is a BF16 number its low part is 0: emulation == definition, bitwise."""
    rng = np.random.default_rng(41)
    X = (rng.integers(-128, 128, (9, 40)) / 16.0).astype(np.float32)   # 8-bit integers / 16
    W = (rng.integers(-128, 128, (5, 40)) / 64.0).astype(np.float32)
    np.testing.assert_array_equal(oracle.router_bf16x3(X, W, oracle_lib), oracle.router_exact(X, W, oracle_lib))
    # and both equal the exact integer arithmetic
    exact = (X.astype(np.float64) * 16).round() @ (W.astype(np.float64) * 64).round().T / 1024.0
    np.testing.assert_array_equal(oracle.router_exact(X, W, oracle_lib), exact)


def test_emulation_error_bound(oracle_lib):
    """|emulation - definition| <= 3 * 2^-16 * sum_k |x_k w_k|, and the dropped term is not zero."""
    rng = np.random.default_rng(42)
    X = rng.standard_normal((16, 256)).astype(np.float32)
    W = (rng.standard_normal((8, 256)) / 16.0).astype(np.float32)
    emu = oracle.router_bf16x3(X, W, oracle_lib)
    ref = oracle.router_exact(X, W, oracle_lib)
    abs_dot = np.abs(X).astype(np.float64) @ np.abs(W).astype(np.float64).T
    err = np.abs(emu - ref)
    assert np.all(err <= oracle.router_emulation_bound(abs_dot))
    assert np.max(err / abs_dot) > 2.0 ** -30   # the approximation is visible


def _py_round_bf16(v):
    """Pure-Python RNE to BF16 through integer arithmetic on the significand."""
    if v == 0.0 or math.isinf(v) or math.isnan(v):
        return v
    m, e = math.frexp(v)            # v = m * 2^e, 0.5 <= |m| < 1
    scaled = m * 256.0              # 8 significant bits above the binary point
    q = math.floor(abs(scaled))
    rem = abs(scaled) - q
    if rem > 0.5 or (rem == 0.5 and q % 2 == 1):
        q += 1
    return math.copysign(q, v) * 2.0 ** (e - 8)


def test_pure_python_restatement(oracle_lib):
    """Tiny inputs: the split and the three products restated in plain Python floats."""
    rng = np.random.default_rng(43)
    X = rng.standard_normal((3, 7)).astype(np.float32)
    W = rng.standard_normal((2, 7)).astype(np.float32)
    got = oracle.router_bf16x3(X, W, oracle_lib)
    for t in range(3):
        for r in range(2):
            s = 0.0
            for k in range(7):
                x, w = float(X[t, k]), float(W[r, k])
                xh = _py_round_bf16(x); xl = _py_round_bf16(x - xh)
                wh = _py_round_bf16(w); wl = _py_round_bf16(w - wh)
                s += xh * wh
                s += xh * wl
                s += xl * wh
            assert got[t, r] == s


def test_sampled_entry_matches_full(oracle_lib):
    rng = np.random.default_rng(44)
    X = rng.standard_normal((11, 33)).astype(np.float32)
    W = rng.standard_normal((6, 33)).astype(np.float32)
    full = oracle.router_bf16x3(X, W, oracle_lib)
    ts = np.array([0, 10, 5, 3]); rs = np.array([5, 0, 2, 4])
    np.testing.assert_array_equal(oracle.router_bf16x3_at(X, W, ts, rs, oracle_lib), full[ts, rs])
