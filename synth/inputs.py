"""Seeded generators for the five synthetic workloads.

Every generator takes an integer ``seed`` and a ``stream`` label so that each
tensor of a workload has its own independent random stream
(``numpy.random.SeedSequence([seed, stream])`` feeding PCG64).

Weights are generated as ``[K, N]`` fp32 matrices (K = input features, the
dimension the quantization groups run along).  Activations are ``[M, K]``
matrices drawn in fp32 from N(0, 1) and then rounded once (round-to-nearest-
even) to fp16 or bf16 by torch's dtype conversion; the rounded values are the
activations both sides consume.
"""

from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

# Stream labels: one independent random stream per tensor role.
_STREAM_W = 1
_STREAM_SALIENT = 2
_STREAM_PERM = 3
_STREAM_X = 4


def _rng(seed: int, stream: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence([int(seed), int(stream)])))


def gaussian_weights(K: int, N: int, sigma: float = 0.02, seed: int = 0) -> np.ndarray:
    """W ~ N(0, sigma^2), fp32, shape [K, N]."""
    g = _rng(seed, _STREAM_W)
    W = g.standard_normal((K, N), dtype=np.float32)
    W *= np.float32(sigma)
    return W


def student_t_weights(K: int, N: int, df: float = 5.0, scale: float = 0.01, seed: int = 0) -> np.ndarray:
    """W ~ scale * Student-t(df), fp32, shape [K, N]."""
    g = _rng(seed, _STREAM_W)
    W = g.standard_t(df, size=(K, N)).astype(np.float32)
    W *= np.float32(scale)
    return W


def salient_rows(K: int, frac: float = 0.01, seed: int = 0) -> np.ndarray:
    """round(frac*K) distinct input-channel (K-row) indices, sorted, int64."""
    g = _rng(seed, _STREAM_SALIENT)
    n = int(round(frac * K))
    return np.sort(g.choice(K, size=n, replace=False))


def act_order_g_idx(K: int, group_size: int = 128, seed: int = 0) -> np.ndarray:
    """Random act-order row->group map, int32[K].

    A seeded permutation ``perm`` of the K rows gives the order in which rows
    are grouped; the j-th row in that order joins group j // group_size.  Every
    group therefore holds exactly ``group_size`` rows scattered over K, while
    the weight rows themselves stay in their original order.
    """
    if K % group_size:
        raise ValueError("K must be a multiple of group_size")
    g = _rng(seed, _STREAM_PERM)
    perm = g.permutation(K)
    g_idx = np.empty(K, dtype=np.int32)
    g_idx[perm] = (np.arange(K) // group_size).astype(np.int32)
    return g_idx


def activations(M: int, K: int, dtype: str = "bf16", seed: int = 0):
    """X ~ N(0, 1) drawn in fp32 then rounded once to ``dtype``; torch CPU tensor [M, K]."""
    import torch

    g = _rng(seed, _STREAM_X)
    x32 = torch.from_numpy(g.standard_normal((M, K), dtype=np.float32))
    tdt = {"bf16": torch.bfloat16, "f16": torch.float16}[dtype]
    return x32.to(tdt)


@dataclass(frozen=True)
class Workload:
    """One synthetic workload: shapes, token counts, weight distribution, dtype."""

    name: str
    shapes: tuple  # ((K, N), ...)
    Ms: tuple
    dtype: str  # activation / output dtype: "f16" or "bf16"
    fmt: str  # "int4" or "nf4"
    dist: str  # "normal", "normal_salient", "t5"
    act_order: bool = False
    group_size: int = 128
    blocksize: int = 64
    labels: tuple = field(default_factory=tuple)


WORKLOADS = {
    "single_linear": Workload(
        name="single W4A16 linear 4096x4096, M=16, fp16",
        shapes=((4096, 4096),), Ms=(16,), dtype="f16", fmt="int4", dist="normal"),
    "decode_sweep": Workload(
        name="Llama-7B-shaped decode sweep, M in {1,4,16}, bf16, 1% salient input channels x10",
        shapes=((4096, 12288), (4096, 4096), (4096, 22016), (11008, 4096)),
        Ms=(1, 4, 16), dtype="bf16", fmt="int4", dist="normal_salient",
        labels=("qkv", "o", "gate_up", "down")),
    "act_order": Workload(
        name="70B-style MLP with act-order g_idx, M in {1,16,64}, fp16, W ~ 0.01*t5",
        shapes=((8192, 28672), (28672, 8192)), Ms=(1, 16, 64), dtype="f16", fmt="int4",
        dist="t5", act_order=True, labels=("up", "down")),
    "qwen32b": Workload(
        name="Qwen2.5-32B-shaped linears, M in {1,256,1024,4096}, bf16",
        shapes=((5120, 7168), (5120, 5120), (5120, 55296), (27648, 5120)),
        Ms=(1, 256, 1024, 4096), dtype="bf16", fmt="int4", dist="normal",
        labels=("qkv", "o", "gate_up", "down")),
    "nf4": Workload(
        name="NF4 blockwise 8192x8192, block 64, M in {1,64,1024}, bf16",
        shapes=((8192, 8192),), Ms=(1, 64, 1024), dtype="bf16", fmt="nf4", dist="normal"),
}


def weights_for(wl: Workload, K: int, N: int, seed: int = 0) -> np.ndarray:
    """fp32 [K, N] weights drawn with the workload's distribution."""
    if wl.dist == "normal":
        return gaussian_weights(K, N, 0.02, seed)
    if wl.dist == "normal_salient":
        W = gaussian_weights(K, N, 0.02, seed)
        W[salient_rows(K, 0.01, seed)] *= np.float32(10.0)
        return W
    if wl.dist == "t5":
        return student_t_weights(K, N, 5.0, 0.01, seed)
    raise ValueError(wl.dist)
