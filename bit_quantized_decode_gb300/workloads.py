"""Workload shapes and seeded synthetic inputs.

This module holds no arithmetic of the method: only the matrix shapes of the
decode linears the source pages run, and seeded random-number draws that
stand in for real model weights and activations.  Tests, the benchmark and
the smoke check draw inputs here and hand the same arrays to the GPU library
and to the CPU oracle.

Shapes:
  * 7B decode linears ("Jetson Orin AGX INT4 推理优化实践", §模型尺寸和 decode 的真实瓶颈):
    N_LAYERS 28, HIDDEN 3584, KV_DIM 512, INTERMEDIATE 18944, VOCAB 152064.
    Fused shards: QKV = [3584, 512, 512] rows, gate/up = [18944, 18944] rows.
  * Gemma4-E2B decode linears ("在香橙派上跑 Gemma4", §一 网络结构简介 and §3.1):
    hidden 1536, FFN 6144, 8 query heads of 256 and one KV head of 256, vocab 262144.

Distributions: weights N(0, sigma) with sigma 0.02 (7B, lm_head) or 0.03
(Gemma), activations N(0, 1), bias N(0, 0.01); the single-GEMV workload also
scales 0.1% of the activation entries (seeded choice) by 20 to plant outliers.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

# ------------------------------------------------------------------ shapes
QWEN7B_HIDDEN = 3584
QWEN7B_KV_DIM = 512
QWEN7B_INTERMEDIATE = 18944
QWEN7B_VOCAB = 152064
QWEN7B_LAYERS = 28

GEMMA_HIDDEN = 1536
GEMMA_FFN = 6144
GEMMA_QKV = 8 * 256 + 256 + 256
GEMMA_VOCAB = 262144


@dataclass(frozen=True)
class Linear:
    """One (possibly shard-fused) decode linear: y[M][N] = W[N][K] x[M][K] + b."""

    name: str
    shards: tuple          # rows of each shard, concatenated in order
    K: int
    fmt: str = "w4"        # "w4" per-row INT4, "q4_0", "i8g32"
    bias: bool = True
    sigma: float = 0.02

    @property
    def N(self) -> int:
        return int(sum(self.shards))


def qwen7b_layer() -> list:
    H, KV, F = QWEN7B_HIDDEN, QWEN7B_KV_DIM, QWEN7B_INTERMEDIATE
    return [
        Linear("qkv", (H, KV, KV), H),
        Linear("o", (H,), H),
        Linear("gate_up", (F, F), H),
        Linear("down", (H,), F),
    ]


def qwen7b_lm_head() -> Linear:
    return Linear("lm_head", (QWEN7B_VOCAB,), QWEN7B_HIDDEN)


def gemma_layer_q4_0() -> list:
    return [
        Linear("qkv", (8 * 256, 256, 256), GEMMA_HIDDEN, fmt="q4_0", bias=False, sigma=0.03),
        Linear("gate_up", (GEMMA_FFN, GEMMA_FFN), GEMMA_HIDDEN, fmt="q4_0", bias=False, sigma=0.03),
        Linear("down", (GEMMA_HIDDEN,), GEMMA_FFN, fmt="q4_0", bias=False, sigma=0.03),
    ]


def gemma_lm_head_i8g32() -> Linear:
    return Linear("lm_head_i8g32", (GEMMA_VOCAB,), GEMMA_HIDDEN, fmt="i8g32", bias=True, sigma=0.02)


def gemma_lm_head_q6g32() -> Linear:
    """The same 6-bit lm_head values packed in 6 bits instead of widened to int8."""
    return Linear("lm_head_q6g32", (GEMMA_VOCAB,), GEMMA_HIDDEN, fmt="q6g32", bias=True, sigma=0.02)


@dataclass(frozen=True)
class Workload:
    name: str
    linears: tuple
    M: int = 1
    repeat: int = 1                      # how many times the linear list repeats (layers)
    tail: tuple = field(default=())      # linears after the repeated block (lm_head)
    outliers: bool = False

    def sequence(self):
        for layer in range(self.repeat):
            for lin in self.linears:
                yield layer, lin
        for lin in self.tail:
            yield self.repeat, lin


def workload(name: str, M: int = 1) -> Workload:
    """The five named workloads, smallest first."""
    if name == "w4a8_single":
        return Workload(name, (Linear("single", (512,), QWEN7B_HIDDEN),), M=M, outliers=True)
    if name == "qwen7b_layer":
        return Workload(name, tuple(qwen7b_layer()), M=M)
    if name == "gemma_q4_0":
        return Workload(name, tuple(gemma_layer_q4_0()), M=M)
    if name == "lm_head":
        return Workload(name, (qwen7b_lm_head(), gemma_lm_head_i8g32()), M=M)
    if name == "qwen7b_step":
        return Workload(name, tuple(qwen7b_layer()), M=M, repeat=QWEN7B_LAYERS,
                        tail=(qwen7b_lm_head(),))
    raise KeyError(name)


WORKLOADS = ("w4a8_single", "qwen7b_layer", "gemma_q4_0", "lm_head", "qwen7b_step")


# ------------------------------------------------------- host (numpy) draws
def rng(seed: int = 0) -> np.random.Generator:
    return np.random.default_rng(seed)


def weights(g: np.random.Generator, N: int, K: int, sigma: float = 0.02) -> np.ndarray:
    return (g.standard_normal((N, K), dtype=np.float64) * sigma).astype(np.float32)


def activations(g: np.random.Generator, M: int, K: int, outliers: bool = False) -> np.ndarray:
    x = g.standard_normal((M, K), dtype=np.float64).astype(np.float32)
    if outliers:
        n_out = max(1, (M * K) // 1000)
        idx = g.choice(M * K, size=n_out, replace=False)
        x.reshape(-1)[idx] *= np.float32(20.0)
    return x


def bias(g: np.random.Generator, N: int) -> np.ndarray:
    return (g.standard_normal(N, dtype=np.float64) * 0.01).astype(np.float32)


def norm_weight(g: np.random.Generator, K: int) -> np.ndarray:
    """RMSNorm weight: 1 + N(0, 0.1) per channel, with 0.5% of the channels
    scaled by 8 (trained norm weights carry a few large channels)."""
    w = 1.0 + 0.1 * g.standard_normal(K, dtype=np.float64)
    idx = g.choice(K, size=max(1, K // 200), replace=False)
    w[idx] *= 8.0
    return w.astype(np.float32)


def residual_stream(g: np.random.Generator, M: int, K: int, scale: float = 4.0) -> np.ndarray:
    """Decoder residual stream h: N(0, scale^2), the magnitude a few dozen
    residual adds leave it at."""
    return (g.standard_normal((M, K), dtype=np.float64) * scale).astype(np.float32)


def int_codes(g: np.random.Generator, shape, lo: int, hi: int) -> np.ndarray:
    """Uniform integers in [lo, hi], int8."""
    return g.integers(lo, hi + 1, size=shape, dtype=np.int64).astype(np.int8)


def positive_scales(g: np.random.Generator, n: int, lo: float = 1e-3, hi: float = 1e-1) -> np.ndarray:
    return g.uniform(lo, hi, size=n).astype(np.float32)


# ------------------------------------------------------- device (torch) draws
def torch_normal(shape, std: float, seed: int, device="cuda"):
    """N(0, std) float32 tensor drawn on `device` from a seeded torch generator."""
    import torch

    gen = torch.Generator(device=device)
    gen.manual_seed(int(seed))
    t = torch.randn(*shape, generator=gen, device=device, dtype=torch.float32)
    if std != 1.0:
        t.mul_(std)
    return t
