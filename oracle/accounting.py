"""Byte counts of the packed checkpoint tensors.

"LLM量化技术深度对比:GPTQ vs AWQ vs bitsandbytes 2026基准全解析", key-data
item 3: one forward of Qwen2.5-32B moves 64 GB of weights at FP16 and 16 GB
at 4 bit; cloud.tencent.com/developer/article/2726413 §2.3: 4-bit needs about
a quarter of FP16's memory.  These functions count the bytes a decode step
must stream for the formats here.
"""

from __future__ import annotations


def int4_bytes(K: int, N: int, group_size: int = 128, act_order: bool = False) -> int:
    """qweight (K*N/2) + fp16 scales + packed 4-bit zeros (+ int32 g_idx)."""
    G = K // group_size
    b = K * N // 2 + G * N * 2 + G * N // 2
    if act_order:
        b += 4 * K
    return b


def nf4_bytes(K: int, N: int, blocksize: int = 64) -> int:
    """qweight (K*N/2) + fp32 absmax per block."""
    return K * N // 2 + (K // blocksize) * N * 4


def fp16_bytes(K: int, N: int) -> int:
    return 2 * K * N


def bits_per_weight(K: int, N: int, group_size: int = 128) -> float:
    return 8.0 * int4_bytes(K, N, group_size) / (K * N)
