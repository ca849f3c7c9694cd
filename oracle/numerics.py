"""Round-to-nearest-even conversion to the 16-bit storage types.

The pages store scales in fp16 and compute in fp16 or bf16
(cloud.tencent.com/developer/article/2726413 §3.3 loads checkpoints whose
scales are fp16; "GPTQ与bitsandbytes对比" bitsandbytes section sets
``bnb_4bit_compute_dtype=torch.bfloat16``).  They do not spell out the
rounding; IEEE 754 round-to-nearest, ties-to-even, is the reading taken here.

fp16: numpy's float64 -> float16 conversion rounds once, directly from the
double (no intermediate float32), with ties to even.  The tests pin this
against exact rational arithmetic.

bf16: numpy has no bf16 type, so the rounding is written from its
definition: bf16 keeps the upper 16 bits of an fp32 pattern; the dropped 16
bits are rounded to nearest, ties to the even upper half.
"""

from __future__ import annotations

import numpy as np


def to_f16(x) -> np.ndarray:
    """RNE of float64 (or float32) values to fp16; returns float16 array."""
    with np.errstate(over="ignore"):
        return np.asarray(x, dtype=np.float64).astype(np.float16)


def f32_to_bf16_bits(x) -> np.ndarray:
    """RNE of float32 values to bf16; returns the uint16 bit patterns.

    Finite inputs only (the quantized weights never hold NaN).  Overflow past
    the largest bf16 rounds to infinity, as IEEE requires.
    """
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    lsb = (u >> np.uint64(16)) & np.uint64(1)
    r = (u + np.uint64(0x7FFF) + lsb) >> np.uint64(16)
    return r.astype(np.uint16)


def bf16_bits_to_f64(b) -> np.ndarray:
    """Exact value of bf16 bit patterns, as float64."""
    u = np.asarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return u.view(np.float32).astype(np.float64)


def f16_bits_to_f64(b) -> np.ndarray:
    """Exact value of fp16 bit patterns, as float64."""
    return np.asarray(b, dtype=np.uint16).view(np.float16).astype(np.float64)


def round_to_dtype_bits(x, dtype: str) -> np.ndarray:
    """RNE of (exactly fp32-representable) values to ``dtype``; uint16 bits."""
    if dtype == "f16":
        return to_f16(x).view(np.uint16)
    if dtype == "bf16":
        return f32_to_bf16_bits(np.asarray(x, dtype=np.float32))
    raise ValueError(dtype)


def dtype_bits_to_f64(b, dtype: str) -> np.ndarray:
    if dtype == "f16":
        return f16_bits_to_f64(b)
    if dtype == "bf16":
        return bf16_bits_to_f64(b)
    raise ValueError(dtype)
