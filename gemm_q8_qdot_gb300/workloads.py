"""Seeded synthetic inputs for the Q8_0 workloads.

This module only draws f32 arrays from a seeded generator.  It holds none of
the quantizer's or of qdot_t's arithmetic, so the oracle side and the CUDA
side can both take their inputs from it.

Shapes are decode and prompt projections of a model with hidden size 4096
(intermediate 14336 or 11008); the value distributions are:

* activations ~ N(0, 1); for the small-batch case each row is multiplied by a
  scale drawn log-uniformly in [0.1, 10]; for the prompt case 0.5% of the K
  channels (a seeded choice of columns) are multiplied by 50;
* weights ~ N(0, 0.02); for the decode FFN shapes 1% of the entries (a
  seeded Bernoulli mask) are multiplied by 20;
* the smallest (parity) case uses N(0, 1) for both;
* the Q5_0 decode case (q50_qdot_t) draws its weight blocks directly: every
  byte uniform in [0, 255] (so every element q - 16 is uniform in [-16, 15])
  and the f32 block scales log-uniform in [1e-3, 1e-2], the range a Q5_0
  encoding of N(0, 0.02) weights has (the pages define no Q5_0 encoder).

Every workload is seeded with 20261202 + its index, drawn with numpy's PCG64.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

SEED_BASE = 20261202


@dataclass(frozen=True)
class Workload:
    name: str
    M: int
    N: int
    K: int
    index: int
    x_dist: str = "normal"        # normal | row_loguniform | outlier_channels
    w_std: float = 0.02
    w_outliers: bool = False
    w_format: str = "q8_0"        # q8_0 | q5_0 (q50_qdot_t)
    extra: dict = field(default_factory=dict, compare=False, hash=False)

    @property
    def seed(self) -> int:
        return SEED_BASE + self.index

    @property
    def weight_bytes(self) -> int:
        """Stored bytes of W: Q8_0 N*K int8 values, or Q5_0 20 bytes per 32 elements,
        plus N*K/32 f32 scales."""
        data = self.N * (self.K // 32) * 20 if self.w_format == "q5_0" else self.N * self.K
        return data + 4 * self.N * (self.K // 32)

    @property
    def ops(self) -> int:
        """2*M*N*K integer multiply-add operations."""
        return 2 * self.M * self.N * self.K


WORKLOADS = {
    "parity_m1_k256_n64": Workload("parity_m1_k256_n64", 1, 64, 256, 0, w_std=1.0),
    "decode_m1_k4096_n4096": Workload("decode_m1_k4096_n4096", 1, 4096, 4096, 1),
    "ffn_up_m1_k4096_n14336": Workload("ffn_up_m1_k4096_n14336", 1, 14336, 4096, 2, w_outliers=True),
    "ffn_down_m1_k14336_n4096": Workload("ffn_down_m1_k14336_n4096", 1, 4096, 14336, 2, w_outliers=True),
    "smallm_m4_k4096_n11008": Workload("smallm_m4_k4096_n11008", 4, 11008, 4096, 3, x_dist="row_loguniform"),
    "smallm_m16_k4096_n11008": Workload("smallm_m16_k4096_n11008", 16, 11008, 4096, 3, x_dist="row_loguniform"),
    "smallm_m64_k4096_n11008": Workload("smallm_m64_k4096_n11008", 64, 11008, 4096, 3, x_dist="row_loguniform"),
    "prompt_m512_k4096_n14336": Workload("prompt_m512_k4096_n14336", 512, 14336, 4096, 4, x_dist="outlier_channels"),
    "q50_decode_m1_k4096_n4096": Workload("q50_decode_m1_k4096_n4096", 1, 4096, 4096, 5, w_format="q5_0"),
    "q50_prompt_m512_k4096_n14336": Workload("q50_prompt_m512_k4096_n14336", 512, 14336, 4096, 6,
                                             x_dist="outlier_channels", w_format="q5_0"),
}

# the workloads whose weights are Q8_0 (qdot_t proper)
Q8_WORKLOADS = {n: w for n, w in WORKLOADS.items() if w.w_format == "q8_0"}


def _rng(seed: int, stream: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64([seed, stream]))


def activations(wl: Workload, M: int | None = None, K: int | None = None) -> np.ndarray:
    """f32 [M, K] activations of a workload (shape overridable for scaled-down cases)."""
    M = wl.M if M is None else M
    K = wl.K if K is None else K
    rng = _rng(wl.seed, 1)
    x = rng.standard_normal((M, K), dtype=np.float32)
    if wl.x_dist == "row_loguniform":
        s = np.exp(rng.uniform(np.log(0.1), np.log(10.0), size=(M, 1))).astype(np.float32)
        x *= s
    elif wl.x_dist == "outlier_channels":
        n_out = max(1, int(round(0.005 * K)))
        cols = rng.permutation(K)[:n_out]
        x[:, cols] *= np.float32(50.0)
    return x


def weights(wl: Workload, N: int | None = None, K: int | None = None) -> np.ndarray:
    """f32 [N, K] weights of a workload (shape overridable for scaled-down cases)."""
    N = wl.N if N is None else N
    K = wl.K if K is None else K
    rng = _rng(wl.seed, 2 if wl.name != "ffn_down_m1_k14336_n4096" else 3)
    w = rng.standard_normal((N, K), dtype=np.float32)
    w *= np.float32(wl.w_std)
    if wl.w_outliers:
        mask = rng.random((N, K), dtype=np.float32) < np.float32(0.01)
        w[mask] *= np.float32(20.0)
    return w


def random_int8(rng: np.random.Generator, shape, lo: int = -128, hi: int = 127) -> np.ndarray:
    """Uniform int8 values in [lo, hi] (edge-case operand for qdot_t)."""
    return rng.integers(lo, hi + 1, size=shape, dtype=np.int16).astype(np.int8)


def random_scales(rng: np.random.Generator, shape, lo: float = 1e-4, hi: float = 1.0) -> np.ndarray:
    """Positive f32 scales, log-uniform in [lo, hi]."""
    return np.exp(rng.uniform(np.log(lo), np.log(hi), size=shape)).astype(np.float32)


def q50_weights(wl: Workload, N: int | None = None, K: int | None = None):
    """Q5_0 weight blocks uint8 [N, K/32 * 20] and f32 scales [N, K/32] of a workload."""
    N = wl.N if N is None else N
    K = wl.K if K is None else K
    rng = _rng(wl.seed, 4)
    w5 = rng.integers(0, 256, size=(N, K // 32 * 20), dtype=np.uint8)
    ws = random_scales(rng, (N, K // 32), 1e-3, 1e-2)
    return w5, ws
