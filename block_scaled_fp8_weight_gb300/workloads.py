"""Seeded synthetic inputs for the block-scaled FP8 weight GEMM and its twin quantizer.

This module draws random numbers and nothing else: it holds none of the method's
arithmetic (no dequantisation, no GEMM, no quantisation), so both the CUDA path and the
CPU oracle can be fed from it.  bf16 values are returned as uint16 bit patterns; the
only rounding done here is torch's float32 -> bfloat16 cast of the N(0,1) activations.

The shapes follow the deployments described on the pages
"recipes/docker-images/mia-tp4/adapter/wo_a_w8.py" (wo_a: G groups of [1024, 4096],
G = 2 at TP4, 4 at padded TP3, rows 2..8 and 9..192) and
"recipes/docker-images/mia-tp4/adapter/shared_pad_k.py" (shared-expert down_proj
N = 5120, K = 576 padded to 640, M = 6).  The pages measure on a live model that is not
available here; these seeded tensors stand in for its weights and activations.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

# Every finite, non-NaN e4m3 byte: 0x00..0x7E and 0x80..0xFE (254 patterns).
FINITE_CODES = np.concatenate([np.arange(0x00, 0x7F), np.arange(0x80, 0xFF)]).astype(np.uint8)


def rng(seed: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(int(seed)))


def codes(r: np.random.Generator, shape) -> np.ndarray:
    """e4m3 codes drawn uniformly over the 254 finite byte patterns."""
    return FINITE_CODES[r.integers(0, FINITE_CODES.size, size=shape)]


def exponents(r: np.random.Generator, shape, lo: int, hi: int) -> np.ndarray:
    """Exponent bytes (ue8m0, byte = e + 127) uniform in [lo, hi] inclusive."""
    return r.integers(lo, hi + 1, size=shape).astype(np.uint8)


def activations(r: np.random.Generator, M: int, cols: int) -> np.ndarray:
    """bf16 bit patterns of N(0,1) samples, shape [M, cols] (torch's RNE cast)."""
    import torch

    f = r.standard_normal(size=(M, cols)).astype(np.float32)
    return torch.from_numpy(f).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16).copy()


def nudge_sites(r: np.random.Generator, G: int, N: int, K: int, frac: float = 0.01):
    """Pick max(1, round(frac * #blocks)) distinct 32x32 blocks and one element in each.

    Returns a list of flat element indices into a [G, N, K] array.
    """
    nb, kb = N // 32, K // 32
    nblocks = G * nb * kb
    count = max(1, int(round(frac * nblocks)))
    blocks = r.choice(nblocks, size=count, replace=False)
    sites = []
    for b in blocks:
        g, rem = divmod(int(b), nb * kb)
        bi, bj = divmod(rem, kb)
        rr, cc = r.integers(0, 32, size=2)
        sites.append(((g * N) + bi * 32 + int(rr)) * K + bj * 32 + int(cc))
    return sites


def apply_nudge(w_bits: np.ndarray, sites) -> np.ndarray:
    """Add one to the bf16 bit pattern at every site (one bf16 ulp away from zero)."""
    out = np.array(w_bits, dtype=np.uint16, copy=True)
    flat = out.reshape(-1)
    for s in sites:
        flat[s] = np.uint16((int(flat[s]) + 1) & 0xFFFF)
    return out


@dataclass
class Workload:
    """One seeded GEMM problem: y[m,g,n] = sum_k x[m, g*K+k] * W[g,n,k]."""

    name: str
    G: int
    N: int
    K: int
    M: int
    exp_lo: int
    exp_hi: int
    split_k: int = 0
    copies: int = 1
    seed: int = 0
    notes: str = ""
    extra: dict = field(default_factory=dict)

    @property
    def weight_bytes(self) -> int:
        """e4m3 bytes plus exponent bytes streamed per call."""
        return self.G * self.N * self.K + self.G * (self.N // 32) * (self.K // 32)

    @property
    def algorithmic_bytes(self) -> int:
        """Weight stream plus the bf16 activations read and the bf16 outputs written."""
        return self.weight_bytes + self.M * self.G * self.K * 2 + self.M * self.G * self.N * 2

    @property
    def flops(self) -> int:
        return 2 * self.M * self.G * self.N * self.K

    def weights(self, copy: int = 0):
        r = rng(self.seed * 1000003 + copy)
        w8 = codes(r, (self.G, self.N, self.K))
        ex = exponents(r, (self.G, self.N // 32, self.K // 32), self.exp_lo, self.exp_hi)
        return w8, ex

    def x(self, copy: int = 0, M: int | None = None) -> np.ndarray:
        r = rng(self.seed * 1000003 + 500009 + copy)
        return activations(r, self.M if M is None else M, self.G * self.K)


# The five workloads.  Exponent ranges: [115, 127] for wo_a-shaped weights, [118, 127]
# for the down_proj, as the scale ranges of those checkpoints.
TINY = Workload("tiny G=1 N=256 K=512 M=4", G=1, N=256, K=512, M=4, exp_lo=115, exp_hi=127,
                seed=11)
WO_A = Workload("wo_a G=2 N=1024 K=4096 M=6 split_k=8", G=2, N=1024, K=4096, M=6,
                exp_lo=115, exp_hi=127, split_k=8, copies=43, seed=22)
DOWN_PROJ = Workload("down_proj N=5120 K=576 M=6", G=1, N=5120, K=576, M=6,
                     exp_lo=118, exp_hi=127, split_k=1, copies=43, seed=33)
MID = Workload("mid G=4 N=1024 K=4096", G=4, N=1024, K=4096, M=64, exp_lo=115, exp_hi=127,
               copies=43, seed=44)
GATE_UP = Workload("gate_up-like N=1152 K=5120", G=1, N=1152, K=5120, M=6, exp_lo=115,
                   exp_hi=127, copies=43, seed=55)
HEAD = Workload("head-like N=32768 K=5120", G=1, N=32768, K=5120, M=6, exp_lo=115,
                exp_hi=127, copies=1, seed=66)

WO_A_ROWS = (2, 4, 6, 8)
MID_ROWS = (9, 16, 32, 64, 96, 128, 192)
MID_SPLITS = (1, 2, 4, 8)
SWEEP_ROWS = (1, 2, 6, 16, 64, 128)
