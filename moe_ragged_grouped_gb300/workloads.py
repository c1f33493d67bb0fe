"""Seeded synthetic inputs for the ragged grouped GEMM (no GEMM arithmetic here).

This module only draws random numbers and lays out group sizes; both the tests
(for the FP64 oracle and the CUDA path) and the benchmark take their inputs
from it.  It holds none of the method's arithmetic.

Workload shapes follow the pages' vocabulary (flashinfer PR #8258,
"Operations and shapes": E experts, M total routed rows, balanced / skewed /
one-empty group sizes) and the dense projection family of PR #8363 (E = 1,
T tokens, d_in -> d_out).  ``N(0, s)`` is read as mean 0 and *variance* s.

BF16 values are produced by round-to-nearest-even from float32 draws and are
returned as raw uint16 bit patterns (numpy) or as torch.bfloat16 tensors.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np

# ---------------------------------------------------------------------------
# Group sizes
# ---------------------------------------------------------------------------


def balanced_sizes(E: int, M: int) -> list[int]:
    """Split M rows as evenly as possible over E experts (first ones get +1)."""
    q, r = divmod(M, E)
    return [q + (1 if e < r else 0) for e in range(E)]


def multinomial_sizes(E: int, M: int, seed: int = 0) -> list[int]:
    """Group sizes drawn multinomially with uniform probabilities."""
    rng = np.random.default_rng(seed)
    return [int(v) for v in rng.multinomial(M, [1.0 / E] * E)]


def zipf_sizes_one_empty(E: int, M: int, s: float = 1.2) -> list[int]:
    """Zipf(s) sizes over E-1 non-empty experts plus one empty expert, ascending.

    Weights i^-s for i = 1..E-1, rounded to integers that sum to M by largest
    remainder; the empty expert comes first and the rest are sorted ascending.
    """
    w = np.array([i ** -s for i in range(1, E)], dtype=np.float64)
    exact = w / w.sum() * M
    base = np.floor(exact).astype(np.int64)
    rem = M - int(base.sum())
    order = np.argsort(-(exact - base), kind="stable")
    base[order[:rem]] += 1
    return [0] + sorted(int(v) for v in base)


def lognormal_sizes(E: int, M: int, cv: float = 0.35, seed: int = 0) -> list[int]:
    """Lognormal group sizes with coefficient of variation cv, in drawn order."""
    rng = np.random.default_rng(seed)
    sigma = math.sqrt(math.log(1.0 + cv * cv))
    w = rng.lognormal(mean=0.0, sigma=sigma, size=E)
    exact = w / w.sum() * M
    base = np.floor(exact).astype(np.int64)
    rem = M - int(base.sum())
    order = np.argsort(-(exact - base), kind="stable")
    base[order[:rem]] += 1
    return [int(v) for v in base]


def offsets_from_sizes(sizes) -> np.ndarray:
    """int32 offsets[E+1] with offsets[0] = 0 (the ragged group layout)."""
    off = np.zeros(len(sizes) + 1, dtype=np.int64)
    off[1:] = np.cumsum(np.asarray(sizes, dtype=np.int64))
    if off[-1] >= 2 ** 31:
        raise ValueError("total rows must fit in int32")
    return off.astype(np.int32)


# ---------------------------------------------------------------------------
# BF16 tensors
# ---------------------------------------------------------------------------


def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round float32 values to BF16 (round to nearest, ties to even); uint16 bits."""
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32).astype(np.uint64)
    rounded = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return rounded.astype(np.uint16)


def randn_bf16(shape, std: float, rng: np.random.Generator) -> np.ndarray:
    """N(0, std^2) draws rounded to BF16, as uint16 bit patterns."""
    x = rng.standard_normal(size=shape, dtype=np.float32)
    if std != 1.0:
        x *= np.float32(std)
    return f32_to_bf16_bits(x)


def small_int_bf16(shape, rng: np.random.Generator, lo: int = -2, hi: int = 2) -> np.ndarray:
    """Integers drawn uniformly from [lo, hi], exactly representable in BF16."""
    x = rng.integers(lo, hi + 1, size=shape).astype(np.float32)
    return f32_to_bf16_bits(x)


def to_torch_bf16(bits: np.ndarray, device="cpu"):
    """View uint16 BF16 bit patterns as a torch.bfloat16 tensor on ``device``."""
    import torch
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16)
    return t.to(device) if str(device) != "cpu" else t


def torch_bf16_to_bits(t) -> np.ndarray:
    """Copy a torch.bfloat16 tensor to host uint16 bit patterns."""
    import torch
    return t.detach().to("cpu").contiguous().view(torch.int16).numpy().view(np.uint16)


def randn_bf16_torch(shape, std: float, generator, device):
    """N(0, std^2) float32 draws from a seeded torch generator, rounded to BF16."""
    import torch
    x = torch.randn(shape, generator=generator, device=device, dtype=torch.float32)
    if std != 1.0:
        x.mul_(std)
    return x.to(torch.bfloat16)


# ---------------------------------------------------------------------------
# Named workloads
# ---------------------------------------------------------------------------


@dataclass
class Workload:
    """One grouped-GEMM problem: E experts, group sizes, N, K and input scales."""
    name: str
    E: int
    N: int
    K: int
    sizes: list
    x_std: float = 1.0
    w_std: float | None = None  # default 1/sqrt(K)
    g_std: float = 1.0
    passes: tuple = ("fwd", "dgrad", "wgrad")
    notes: dict = field(default_factory=dict)

    @property
    def M(self) -> int:
        return int(sum(self.sizes))

    @property
    def offsets(self) -> np.ndarray:
        return offsets_from_sizes(self.sizes)

    @property
    def wstd(self) -> float:
        return self.w_std if self.w_std is not None else 1.0 / math.sqrt(self.K)

    def flops(self, npasses: int = 1) -> float:
        return 2.0 * self.M * self.N * self.K * npasses

    def algorithmic_bytes(self, pass_: str, out_bytes: int = 2) -> float:
        """Bytes one pass must move at least: each operand read once, the output written once.

        fwd reads X [M,K] and W [E,N,K] and writes Y [M,N]; dgrad reads G and W and writes
        dX [M,K]; wgrad reads G and X and writes dW [E,N,K] (BF16 inputs, ``out_bytes``
        per output element).
        """
        M, N, K, E = self.M, self.N, self.K, self.E
        if pass_ == "fwd":
            return 2.0 * M * K + 2.0 * E * N * K + out_bytes * M * N
        if pass_ == "dgrad":
            return 2.0 * M * N + 2.0 * E * N * K + out_bytes * M * K
        if pass_ == "wgrad":
            return 2.0 * M * N + 2.0 * M * K + out_bytes * E * N * K
        raise ValueError(pass_)

    def make_numpy(self, seed: int = 0, M_alloc: int | None = None):
        """(X, W, G) uint16 BF16 bits, generated in the order X, W, G.

        Rows beyond sum(sizes) (up to M_alloc) are filled too, so that code
        reading past the last expert would see non-zero data.
        """
        rng = np.random.default_rng(seed)
        M = self.M if M_alloc is None else M_alloc
        X = randn_bf16((M, self.K), self.x_std, rng)
        W = randn_bf16((self.E, self.N, self.K), self.wstd, rng)
        G = randn_bf16((M, self.N), self.g_std, rng)
        return X, W, G

    def make_torch(self, seed: int = 0, device="cuda", M_alloc: int | None = None):
        """(X, W, G) torch.bfloat16 tensors drawn on ``device`` by a seeded generator."""
        import torch
        gen = torch.Generator(device=device)
        gen.manual_seed(seed)
        M = self.M if M_alloc is None else M_alloc
        X = randn_bf16_torch((M, self.K), self.x_std, gen, device)
        W = randn_bf16_torch((self.E, self.N, self.K), self.wstd, gen, device)
        G = randn_bf16_torch((M, self.N), self.g_std, gen, device)
        return X, W, G


def tiny() -> Workload:
    """E=4 experts x 128 rows, K=256, N=128; X~N(0,1), W~N(0,1/K), G~N(0,1)."""
    return Workload("tiny_E4_M512_K256_N128", 4, 128, 256, [128] * 4)


def dense_projection(d_in: int, d_out: int, T: int = 16384) -> Workload:
    """E=1 dense projection: X [T, d_in], W [d_out, d_in], G [T, d_out] with G~N(0, 1e-2)."""
    return Workload(f"dense_T{T}_{d_in}to{d_out}", 1, d_out, d_in, [T], g_std=0.1)


def moe_gate_up() -> Workload:
    """E=8, M=131072 balanced, K=4096 hidden, N=3072 (2 x 1536)."""
    return Workload("moe_gate_up_E8_M131072_K4096_N3072", 8, 3072, 4096,
                    balanced_sizes(8, 131072))


def moe_down() -> Workload:
    """E=32, M=131072 multinomial (uniform probabilities, seed 0), K=1536, N=4096."""
    return Workload("moe_down_E32_M131072_K1536_N4096", 32, 4096, 1536,
                    multinomial_sizes(32, 131072, 0), passes=("wgrad",))


def moe_skewed(transposed: bool = False) -> Workload:
    """E=4, M=136064, Zipf(1.2) sizes ascending with one empty expert."""
    K, N = (3072, 4096) if transposed else (4096, 3072)
    return Workload(f"moe_skew_E4_M136064_K{K}_N{N}", 4, N, K,
                    zipf_sizes_one_empty(4, 136064, 1.2))


DENSE_SHAPES = [(d_in, d_out) for d_in in (4096, 5120) for d_out in (48, 64, 512, 1024, 4096)]
