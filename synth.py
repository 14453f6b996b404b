"""Seeded synthetic inputs for the k-quant prefill matmul.

This module is shared by the tests, the benchmark and the smoke check, and
serves the CUDA path and the CPU oracle alike.  It holds none of the method's
arithmetic: it draws random bytes and numbers and places them at the byte
offsets of the block formats.  Quantization, packing of fields, unpacking and
the matmul live in the oracle and in the CUDA library, separately.

Generator: SplitMix64 (Steele, Lea and Flood, "Fast splittable pseudorandom
number generators", OOPSLA 2014), used counter-style -- output i of stream s
is mix(s + (i + 1) * 0x9E3779B97F4A7C15) -- so any slice can be drawn without
drawing what precedes it.  Normals are Box-Muller pairs of 53-bit uniforms.

Field distributions (the benchmark workloads):
  Q4_K  qs uniform 0..15, 6-bit scales and mins uniform 0..63 (uniform random
        bytes give exactly that, whatever the bit packing), d and dmin fp16
        drawn uniform in [1e-4, 1e-3] and rounded to nearest fp16.
  Q6_K  ql 4-bit and qh 2-bit uniform (uniform random bytes), int8 sub-scales
        uniform in [-32, 31] (or, for the full-scale workload, in [-128, 127]),
        d fp16 uniform in [1e-4, 1e-3].
  X     fp32 sigma * N(0, 1); optionally a seeded 1% of the columns scaled x8
        (the same columns for every row).
"""
from __future__ import annotations

import dataclasses

import numpy as np

GAMMA = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)

Q4K_BYTES = 144
Q6K_BYTES = 210


def splitmix64(seed: int, n: int, start: int = 0) -> np.ndarray:
    """Outputs start .. start+n-1 of the SplitMix64 stream seeded by `seed`."""
    i = np.arange(start + 1, start + n + 1, dtype=np.uint64)
    with np.errstate(over="ignore"):
        z = np.uint64(seed & 0xFFFFFFFFFFFFFFFF) + i * GAMMA
        z = (z ^ (z >> np.uint64(30))) * _M1
        z = (z ^ (z >> np.uint64(27))) * _M2
    return z ^ (z >> np.uint64(31))


def uniform01(seed: int, n: int) -> np.ndarray:
    """n doubles uniform in [0, 1) (53-bit)."""
    return (splitmix64(seed, n) >> np.uint64(11)).astype(np.float64) * (2.0 ** -53)


def normal(seed: int, n: int) -> np.ndarray:
    """n standard normal doubles (Box-Muller on consecutive pairs)."""
    npair = (n + 1) // 2
    z = splitmix64(seed, 2 * npair)
    u1 = ((z[0::2] >> np.uint64(11)).astype(np.float64) + 1.0) * (2.0 ** -53)  # (0, 1]
    u2 = (z[1::2] >> np.uint64(11)).astype(np.float64) * (2.0 ** -53)
    r = np.sqrt(-2.0 * np.log(u1))
    out = np.empty(2 * npair)
    out[0::2] = r * np.cos(2.0 * np.pi * u2)
    out[1::2] = r * np.sin(2.0 * np.pi * u2)
    return out[:n]


def random_bytes(seed: int, n: int) -> np.ndarray:
    nw = (n + 7) // 8
    return splitmix64(seed, nw).view(np.uint8)[:n].copy()


def fp16_uniform_bits(seed: int, n: int, lo: float = 1e-4, hi: float = 1e-3) -> np.ndarray:
    """n fp16 bit patterns of values drawn uniform in [lo, hi] (fp32, then RNE to fp16)."""
    u = uniform01(seed, n)
    v = (np.float32(lo) + (np.float32(hi) - np.float32(lo)) * u.astype(np.float32)).astype(np.float32)
    return v.astype(np.float16).view(np.uint16)


def gen_q4k(N: int, K: int, seed: int) -> np.ndarray:
    """Q4_K weights, uint8 [N, (K/256)*144]: d @0, dmin @2, scales @4..16, qs @16..144."""
    assert K % 256 == 0
    nb = K // 256
    w = random_bytes(seed * 4 + 1, N * nb * Q4K_BYTES).reshape(N * nb, Q4K_BYTES)
    d = fp16_uniform_bits(seed * 4 + 2, N * nb)
    dmin = fp16_uniform_bits(seed * 4 + 3, N * nb)
    w[:, 0:2] = d.view(np.uint8).reshape(-1, 2)
    w[:, 2:4] = dmin.view(np.uint8).reshape(-1, 2)
    return w.reshape(N, nb * Q4K_BYTES)


def gen_q6k(N: int, K: int, seed: int, full_scales: bool = False) -> np.ndarray:
    """Q6_K weights, uint8 [N, (K/256)*210]: ql @0, qh @128, scales @192, d @208.
    Sub-scales uniform in [-32, 31], or with full_scales over the whole int8
    range [-128, 127] (as quantizers that scale a block's largest sub-block to
    the int8 limit produce)."""
    assert K % 256 == 0
    nb = K // 256
    w = random_bytes(seed * 4 + 1, N * nb * Q6K_BYTES).reshape(N * nb, Q6K_BYTES)
    bits = 8 if full_scales else 6
    sc = (splitmix64(seed * 4 + 2, N * nb * 16) >> np.uint64(64 - bits)).astype(np.int64) - (1 << (bits - 1))
    w[:, 192:208] = sc.astype(np.int8).view(np.uint8).reshape(-1, 16)
    d = fp16_uniform_bits(seed * 4 + 3, N * nb)
    w[:, 208:210] = d.view(np.uint8).reshape(-1, 2)
    return w.reshape(N, nb * Q6K_BYTES)


PTQ1_BYTES = 28


def gen_ptq1(N: int, K: int, seed: int) -> np.ndarray:
    """PTQ1_0 weights, uint8 [N, (K/128)*28]: 24 qs bytes drawn uniform over the
    243 five-trit values, 2 qh bytes over the 81 four-trit values, fp16 d @26
    drawn uniform in [1e-3, 1e-2] (each valid byte value is equally likely, so
    every trit is uniform over {0, 1, 2})."""
    assert K % 256 == 0
    nb = K // 128
    qs = (splitmix64(seed * 4 + 1, N * nb * 24) % np.uint64(243)).astype(np.uint8).reshape(N * nb, 24)
    qh = (splitmix64(seed * 4 + 2, N * nb * 2) % np.uint64(81)).astype(np.uint8).reshape(N * nb, 2)
    d = fp16_uniform_bits(seed * 4 + 3, N * nb, 1e-3, 1e-2)
    w = np.concatenate([qs, qh, d.view(np.uint8).reshape(-1, 2)], axis=1)
    return np.ascontiguousarray(w.reshape(N, nb * PTQ1_BYTES))


def outlier_columns(K: int, seed: int, frac: float = 0.01) -> np.ndarray:
    """round(frac*K) distinct column indices, chosen by a seeded shuffle."""
    k = int(round(frac * K))
    keys = splitmix64(seed * 4 + 3, K)
    return np.sort(np.argsort(keys, kind="stable")[:k])


def gen_x(M: int, K: int, seed: int, sigma: float = 1.0, outlier_frac: float = 0.0,
          outlier_scale: float = 8.0) -> np.ndarray:
    """Activations fp32 [M, K] ~ sigma * N(0,1), optional outlier columns."""
    x = (sigma * normal(seed * 4 + 1, M * K)).astype(np.float32).reshape(M, K)
    if outlier_frac > 0.0:
        cols = outlier_columns(K, seed, outlier_frac)
        x[:, cols] *= np.float32(outlier_scale)
    return x


def gen_ids(M: int, top_k: int, E: int, seed: int, skew: float = 0.0) -> np.ndarray:
    """Expert ids int32 [M, top_k] of a synthetic router: per token, top_k
    distinct experts drawn without replacement with weights (e+1)^-skew
    (skew 0: uniform), by the keys u^(1/weight) of seeded uniforms u."""
    assert 1 <= top_k <= E
    u = uniform01(seed * 4 + 2, M * E).reshape(M, E)
    wts = (np.arange(1, E + 1, dtype=np.float64)) ** (-skew)
    keys = np.log(np.maximum(u, 1e-300)) / wts          # log of u^(1/w): order-preserving
    order = np.argsort(-keys, axis=1, kind="stable")
    return np.ascontiguousarray(order[:, :top_k]).astype(np.int32)


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    wtype: int          # 4 = Q4_K, 6 = Q6_K
    M: int
    K: int
    N: int
    w_seed: int
    x_seed: int
    sigma: float = 1.0
    outlier_frac: float = 0.0
    full_scales: bool = False   # Q6_K: sub-scales over the whole int8 range

    def weights(self) -> np.ndarray:
        if self.wtype == 6:
            return gen_q6k(self.N, self.K, self.w_seed, self.full_scales)
        gen = {4: gen_q4k, 1: gen_ptq1}[self.wtype]
        return gen(self.N, self.K, self.w_seed)

    def x(self) -> np.ndarray:
        return gen_x(self.M, self.K, self.x_seed, self.sigma, self.outlier_frac)

    @property
    def block_bytes(self) -> int:
        """Weight bytes per 256 weights of a row."""
        return {4: Q4K_BYTES, 6: Q6K_BYTES, 1: 2 * PTQ1_BYTES}[self.wtype]


def _c(i: int, name: str, wtype: int, M: int, K: int, N: int, **kw) -> Workload:
    seed = 1000 + i
    return Workload(name, wtype, M, K, N, w_seed=seed, x_seed=seed * 100 + 7, **kw)


# The benchmark workloads (LLaMA-like FFN projection shapes).
C0 = _c(0, "q4k_m64_k2048_n2048", 4, 64, 2048, 2048)
C1 = _c(1, "q4k_m512_k2048_n11008_outliers", 4, 512, 2048, 11008, outlier_frac=0.01)
C2 = _c(2, "q6k_m512_k11008_n2048", 6, 512, 11008, 2048)
C3 = _c(3, "q4k_m2048_k4096_n14336", 4, 2048, 4096, 14336, sigma=0.5)
SWEEP_M = (1, 4, 8, 64, 512, 2048, 8192)


def sweep(M: int) -> Workload:
    """Q4_K K = N = 5120 sweep point; weights shared across M, X seeded per M."""
    return Workload(f"q4k_sweep_m{M}_k5120_n5120", 4, M, 5120, 5120,
                    w_seed=1004, x_seed=1004 * 100 + M)


CONFIGS = (C0, C1, C2, C3) + tuple(sweep(m) for m in SWEEP_M)

# The Q6_K shape with sub-scales over the whole int8 range (real Q6_K tensors
# use it): the cost of the tile path's exact hi/lo split, measured beside C2.
F2 = Workload("q6k_fullscale_m512_k11008_n2048", 6, 512, 11008, 2048, w_seed=1002, x_seed=100207,
              full_scales=True)
FULLSCALE_CONFIGS = (F2,)

# PTQ1_0 ternary weights at the K = 5120 projection shape the pages measure
# PTQ1_0 prefill on (a 2048-token prompt).
T0 = Workload("ptq1_m2048_k5120_n5120", 1, 2048, 5120, 5120, w_seed=3000, x_seed=300007)
PTQ1_CONFIGS = (T0,)


@dataclasses.dataclass(frozen=True)
class RoutedWorkload:
    """Expert-routed (MUL_MAT_ID) workload: E experts of N rows stacked, top_k
    experts per token from the synthetic router (gen_ids)."""
    name: str
    wtype: int
    M: int
    K: int
    N: int
    E: int
    top_k: int
    w_seed: int
    x_seed: int
    ids_seed: int
    sigma: float = 1.0
    skew: float = 0.0

    def weights(self) -> np.ndarray:
        return (gen_q4k if self.wtype == 4 else gen_q6k)(self.E * self.N, self.K, self.w_seed)

    def x(self) -> np.ndarray:
        return gen_x(self.M, self.K, self.x_seed, self.sigma)

    def ids(self) -> np.ndarray:
        return gen_ids(self.M, self.top_k, self.E, self.ids_seed, self.skew)

    @property
    def block_bytes(self) -> int:
        return Q4K_BYTES if self.wtype == 4 else Q6K_BYTES


# A mixture-of-experts FFN projection (LLaMA-like expert shape): 8 experts,
# 2 per token, 512 tokens -> 1024 routed rows, about 128 per expert.
R0 = RoutedWorkload("q4k_moe_e8_top2_m512_k4096_n14336", 4, 512, 4096, 14336, 8, 2,
                    w_seed=2000, x_seed=200007, ids_seed=2001, sigma=0.5)
ROUTED_CONFIGS = (R0,)
