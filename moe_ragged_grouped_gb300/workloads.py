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


def zipf_sizes(E: int, M: int, s: float = 1.2, one_empty: bool = False, ascending: bool = False) -> list[int]:
    """Zipf(s) group sizes: weights i^-s (i = 1..E, or 1..E-1 plus one empty group),
    rounded to integers summing to M by largest remainder; descending (the empty
    group last) or ascending (the empty group first)."""
    n = E - 1 if one_empty else E
    w = np.array([i ** -s for i in range(1, n + 1)], dtype=np.float64)
    exact = w / w.sum() * M
    base = np.floor(exact).astype(np.int64)
    rem = M - int(base.sum())
    order = np.argsort(-(exact - base), kind="stable")
    base[order[:rem]] += 1
    sizes = sorted((int(v) for v in base), reverse=True) + ([0] if one_empty else [])
    return sizes[::-1] if ascending else sizes


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


# ---------------------------------------------------------------------------
# The pages' GB300 measurement grid
# ---------------------------------------------------------------------------

# GB300 (sm_103a, 152 SMs) rows of the per-row latency table of flashinfer PR
# #8269 ("perf(cake_moe_grouped_gemm): run the split k512 wgrad tail whole on
# the least-loaded clusters on sm_100a and sm_103a", the GB300 table): shape,
# operation, deterministic-variant ms, non-Cake SOTA ms and its key (t =
# torch._grouped_mm, c = per-expert cuBLAS loop), new non-deterministic ms.
# CUPTI GPU time of one call, cold L2, eager.
PAGES_GB300_ROWS = [
    ("gate_up E4 M112576 bal", "dW", 3.1664, 3.3368, "c", 3.1727),
    ("gate_up E4 M112576 skew", "dW", 3.2938, 3.3325, "c", 3.2940),
    ("gate_up E4 M112576 1-empty", "dW", 3.2723, 3.2834, "c", 3.2754),
    ("gate_up E4 M112576 bal fp32", "dW", 3.2252, 3.3082, "c", 3.2008),
    ("gate_up E4 M136064 bal", "dW", 3.8339, 4.0270, "c", 3.8366),
    ("gate_up E4 M136064 skew", "dW", 3.9911, 4.0418, "c", 3.9970),
    ("gate_up E4 M136064 1-empty", "dW", 3.9701, 4.0361, "c", 3.9598),
    ("gate_up E4 M136064 bal fp32", "dW", 3.9346, 4.0701, "c", 3.9356),
    ("gate_up E8 M131072 bal", "dW", 3.7203, 3.9216, "c", 3.7105),
    ("gate_up E16 M131072 bal", "dW", 3.6980, 3.8986, "t", 3.7095),
    ("gate_up E32 M131072 bal", "dW", 3.6352, 3.7648, "t", 3.6531),
    ("gate_up E4 M112576 skew asc", "dW", 3.2793, 3.3505, "c", 3.2955),
    ("gate_up E4 M112576 1-empty asc", "dW", 3.2443, 3.3886, "c", 3.2818),
    ("gate_up E4 M136064 skew asc", "dW", 3.9035, 4.0407, "c", 3.9712),
    ("gate_up E4 M136064 1-empty asc", "dW", 4.0163, 4.1055, "c", 4.0460),
    ("gate_up E8 M131072 random", "dW", 3.8180, 3.8463, "c", 3.6891),
    ("gate_up E16 M131072 random", "dW", 3.9325, 4.0392, "c", 3.7601),
    ("gate_up E32 M131072 random", "dW", 3.8478, 3.9913, "t", 3.7896),
    ("down E4 M112576 bal", "dW", 1.5830, 1.6822, "c", 1.5775),
    ("down E4 M112576 skew", "dW", 1.6370, 1.6920, "c", 1.6184),
    ("down E4 M112576 1-empty", "dW", 1.5785, 1.6550, "c", 1.5867),
    ("down E4 M112576 bal fp32", "dW", 1.5961, 1.6638, "c", 1.5916),
    ("down E4 M136064 bal", "dW", 1.9327, 2.0381, "c", 1.9244),
    ("down E4 M136064 skew", "dW", 2.0012, 2.0400, "c", 1.9730),
    ("down E4 M136064 1-empty", "dW", 1.9253, 2.0177, "c", 1.9195),
    ("down E4 M136064 bal fp32", "dW", 1.9469, 2.0505, "c", 1.9476),
    ("down E8 M131072 bal", "dW", 1.8187, 1.9639, "c", 1.8148),
    ("down E16 M131072 bal", "dW", 1.8721, 2.0858, "c", 1.8699),
    ("down E32 M131072 bal", "dW", 1.8647, 1.9556, "t", 1.8786),
    ("down E4 M112576 skew asc", "dW", 1.6412, 1.6908, "c", 1.5861),
    ("down E4 M112576 1-empty asc", "dW", 1.7711, 1.7099, "c", 1.6029),
    ("down E4 M136064 skew asc", "dW", 2.0348, 2.0424, "c", 1.9711),
    ("down E4 M136064 1-empty asc", "dW", 2.1324, 2.0732, "c", 1.9147),
    ("down E8 M131072 random", "dW", 2.0384, 1.9910, "c", 1.8844),
    ("down E16 M131072 random", "dW", 2.1025, 2.0670, "c", 1.9089),
    ("down E32 M131072 random", "dW", 1.9379, 2.0551, "t", 1.8630),
    ("gate_up E4 M112576 bal", "ckpt", 12.6579, 15.5120, "t", 12.6513),
    ("gate_up E4 M112576 skew", "ckpt", 12.8493, 15.7940, "t", 12.8874),
    ("gate_up E4 M112576 1-empty", "ckpt", 12.6127, 15.5400, "t", 12.6125),
    ("gate_up E4 M136064 bal", "ckpt", 15.2573, 18.8586, "t", 15.2624),
    ("gate_up E4 M136064 skew", "ckpt", 15.5979, 19.2668, "t", 15.6181),
    ("gate_up E4 M136064 1-empty", "ckpt", 15.4011, 18.8718, "t", 15.3635),
    ("gate_up E8 M131072 bal", "ckpt", 14.7011, 17.5611, "t", 14.7249),
    ("gate_up E16 M131072 bal", "ckpt", 15.0497, 16.6615, "t", 14.9718),
    ("gate_up E32 M131072 bal", "ckpt", 14.7770, 15.2884, "t", 14.8132),
    ("gate_up E4 M112576 skew asc", "ckpt", 12.6952, 15.7037, "t", 12.7579),
    ("gate_up E4 M112576 1-empty asc", "ckpt", 12.9375, 16.1023, "t", 12.8959),
    ("gate_up E4 M136064 skew asc", "ckpt", 15.3430, 18.9009, "t", 15.3180),
    ("gate_up E4 M136064 1-empty asc", "ckpt", 15.4231, 19.3197, "t", 15.5385),
    ("gate_up E8 M131072 random", "ckpt", 15.1947, 18.3366, "t", 15.0282),
    ("gate_up E16 M131072 random", "ckpt", 15.0851, 16.8810, "t", 14.9818),
    ("gate_up E32 M131072 random", "ckpt", 15.4443, 16.1078, "t", 15.4361),
    ("down E4 M112576 bal", "ckpt", 6.2910, 7.5948, "t", 6.2707),
    ("down E4 M112576 skew", "ckpt", 6.4125, 7.9380, "t", 6.3908),
    ("down E4 M112576 1-empty", "ckpt", 6.2826, 7.7901, "t", 6.2811),
    ("down E4 M136064 bal", "ckpt", 7.6785, 9.3028, "t", 7.6777),
    ("down E4 M136064 skew", "ckpt", 7.8223, 9.7387, "t", 7.7981),
    ("down E4 M136064 1-empty", "ckpt", 7.6135, 9.5114, "t", 7.5951),
    ("down E8 M131072 bal", "ckpt", 7.4072, 8.4058, "t", 7.4073),
    ("down E16 M131072 bal", "ckpt", 7.4652, 8.2022, "t", 7.4943),
    ("down E32 M131072 bal", "ckpt", 7.4224, 7.7417, "t", 7.4310),
    ("down E4 M112576 skew asc", "ckpt", 6.4784, 7.9554, "t", 6.4242),
    ("down E4 M112576 1-empty asc", "ckpt", 6.4520, 7.8480, "t", 6.2790),
    ("down E4 M136064 skew asc", "ckpt", 7.7877, 9.5875, "t", 7.7600),
    ("down E4 M136064 1-empty asc", "ckpt", 7.9959, 9.8420, "t", 7.7823),
    ("down E8 M131072 random", "ckpt", 7.5057, 8.5003, "t", 7.3713),
    ("down E16 M131072 random", "ckpt", 7.6812, 8.3222, "t", 7.5734),
    ("down E32 M131072 random", "ckpt", 7.8150, 8.3989, "t", 7.7680),
    ("gate_up E4 M112576 bal", "ckpt ES", 9.3663, 11.4013, "t", 9.3447),
    ("gate_up E4 M112576 skew", "ckpt ES", 9.5468, 11.5057, "t", 9.5800),
    ("gate_up E4 M112576 1-empty", "ckpt ES", 9.6244, 11.7650, "t", 9.6418),
    ("gate_up E4 M136064 bal", "ckpt ES", 11.3815, 13.8066, "t", 11.3533),
    ("gate_up E4 M136064 skew", "ckpt ES", 11.7204, 14.3336, "t", 11.6077),
    ("gate_up E4 M136064 1-empty", "ckpt ES", 11.6324, 14.3628, "t", 11.5513),
    ("gate_up E8 M131072 bal", "ckpt ES", 10.7533, 12.8192, "t", 10.8549),
    ("gate_up E16 M131072 bal", "ckpt ES", 11.0500, 11.9749, "t", 11.0566),
    ("gate_up E32 M131072 bal", "ckpt ES", 11.3156, 12.0762, "t", 11.3186),
    ("gate_up E4 M112576 skew asc", "ckpt ES", 9.4904, 11.5859, "t", 9.4971),
    ("gate_up E4 M112576 1-empty asc", "ckpt ES", 9.5237, 11.6802, "t", 9.5470),
    ("gate_up E4 M136064 skew asc", "ckpt ES", 11.7361, 14.3327, "t", 11.6922),
    ("gate_up E4 M136064 1-empty asc", "ckpt ES", 11.5073, 14.1531, "t", 11.4805),
    ("gate_up E8 M131072 random", "ckpt ES", 11.2200, 13.2241, "t", 11.1049),
    ("gate_up E16 M131072 random", "ckpt ES", 11.5895, 12.8866, "t", 11.3570),
    ("gate_up E32 M131072 random", "ckpt ES", 11.4684, 11.8086, "t", 11.4100),
    ("down E4 M112576 bal", "ckpt ES", 4.6835, 5.6540, "t", 4.6771),
    ("down E4 M112576 skew", "ckpt ES", 4.6944, 5.8074, "t", 4.7181),
    ("down E4 M112576 1-empty", "ckpt ES", 4.7842, 5.9623, "t", 4.7729),
    ("down E4 M136064 bal", "ckpt ES", 5.6247, 6.8500, "t", 5.6219),
    ("down E4 M136064 skew", "ckpt ES", 5.7158, 7.0419, "t", 5.7121),
    ("down E4 M136064 1-empty", "ckpt ES", 5.8110, 7.2810, "t", 5.8082),
    ("down E8 M131072 bal", "ckpt ES", 5.4216, 6.3190, "t", 5.4276),
    ("down E16 M131072 bal", "ckpt ES", 5.4970, 6.0144, "t", 5.4857),
    ("down E32 M131072 bal", "ckpt ES", 5.6244, 6.0064, "t", 5.6179),
    ("down E4 M112576 skew asc", "ckpt ES", 4.7019, 5.8377, "t", 4.6960),
    ("down E4 M112576 1-empty asc", "ckpt ES", 4.9442, 5.9699, "t", 4.7619),
    ("down E4 M136064 skew asc", "ckpt ES", 5.7645, 7.1457, "t", 5.7020),
    ("down E4 M136064 1-empty asc", "ckpt ES", 5.8676, 7.1629, "t", 5.7041),
    ("down E8 M131072 random", "ckpt ES", 5.7750, 6.6888, "t", 5.6299),
    ("down E16 M131072 random", "ckpt ES", 5.6758, 6.2531, "t", 5.5429),
    ("down E32 M131072 random", "ckpt ES", 5.7573, 6.1208, "t", 5.6771),
]

PAGES_SHAPES = {"gate_up": (4096, 6144), "down": (6144, 2048)}   # (N, K)
# a checkpointed grouped GEMM: forward, then forward again and the backward
PAGES_OPS = {"dW": ("wgrad",), "ckpt": ("fwd", "fwd", "dgrad", "wgrad"), "ckpt ES": ("fwd", "dgrad", "wgrad")}


def pages_workload(shape: str) -> tuple:
    """(Workload, dW output dtype) for a shape name of the pages' grid, e.g.
    "gate_up E4 M112576 skew asc" or "down E4 M136064 bal fp32".

    bal = balanced; skew = Zipf(1.2) over all groups; 1-empty = Zipf(1.2) over
    E-1 groups plus one empty group; both descending unless "asc"; random =
    lognormal sizes (CV 0.35, seed 0) in drawn order; fp32 = FP32 dW output.
    """
    parts = shape.split()
    N, K = PAGES_SHAPES[parts[0]]
    E, M = int(parts[1][1:]), int(parts[2][1:])
    kind = parts[3]
    asc = "asc" in parts[4:]
    if kind == "bal":
        sizes = balanced_sizes(E, M)
    elif kind == "skew":
        sizes = zipf_sizes(E, M, 1.2, one_empty=False, ascending=asc)
    elif kind == "1-empty":
        sizes = zipf_sizes(E, M, 1.2, one_empty=True, ascending=asc)
    elif kind == "random":
        sizes = lognormal_sizes(E, M, 0.35, 0)
    else:
        raise ValueError(shape)
    od = "fp32" if "fp32" in parts[4:] else "bf16"
    return Workload(shape.replace(" ", "_"), E, N, K, sizes), od


# ---------------------------------------------------------------------------
# FP32 router GEMM inputs (dense projection family, flashinfer PR #8438,
# "Summary": an FP32 router GEMM over 256 experts)
# ---------------------------------------------------------------------------

ROUTER_T, ROUTER_K, ROUTER_R = 16384, 4096, 256


def router_inputs(T: int, K: int, R: int, seed: int = 0):
    """(X [T, K], W [R, K]) float32 numpy arrays: X ~ N(0, 1), W ~ N(0, 1/K), generation order X, W."""
    rng = np.random.default_rng(seed)
    X = rng.standard_normal((T, K), dtype=np.float32)
    W = (rng.standard_normal((R, K), dtype=np.float32) * np.float32(1.0 / math.sqrt(K))).astype(np.float32)
    return X, W


def router_inputs_torch(T: int, K: int, R: int, seed: int = 0, device="cuda"):
    """(X, W) float32 torch tensors drawn on ``device`` by a seeded generator (large sizes)."""
    import torch
    gen = torch.Generator(device=device)
    gen.manual_seed(seed)
    X = torch.randn((T, K), generator=gen, device=device, dtype=torch.float32)
    W = torch.randn((R, K), generator=gen, device=device, dtype=torch.float32) * (1.0 / math.sqrt(K))
    return X, W
