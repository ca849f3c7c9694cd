"""NF4 ("normal float 4") blockwise quantization, as bitsandbytes uses it.

Sources (page title / section):

* "LLM量化技术深度对比:GPTQ vs AWQ vs bitsandbytes 2026基准全解析", key-data
  item 2: NF4 places its 16 representable values near zero, where LLM weights
  concentrate, and the format is dequantized back to 16-bit on every forward.
* "GPTQ、AWQ与Bitsandbytes：大模型量化三大技术路径深度对比" §2.3 / §3.3:
  bitsandbytes ``load_in_4bit`` quantizes block-wise, calibration-free, with
  the NF4 type; ``bnb_4bit_compute_dtype`` picks the dtype of the product.
* "GPTQ与bitsandbytes对比" bitsandbytes section: ``bnb_4bit_quant_type="nf4"``,
  ``bnb_4bit_compute_dtype=torch.bfloat16``.

Readings where the pages are silent or garbled (each listed in the design
notes):

1. Codebook: 16 ascending fp32 values, C[7] = 0 exactly, C[8..15] the
   standard-normal quantiles of 8 evenly spaced probabilities from ``delta``
   down to (but excluding) 0.5, C[0..6] the negated quantiles of 7 evenly
   spaced probabilities from ``delta`` down to (excluding) 0.5, all divided by
   the quantile of ``delta`` so that C[0] = -1 and C[15] = +1.  ``delta`` is
   1 - (1/30 + 1/32) / 2.  (The first page's "inverse CDF of i/15, code 0000
   -> -3.0" cannot be right -- the quantile of 0 is infinite and it
   contradicts normalisation to [-1, 1] -- so it is not used.)
2. Blocks: 64 consecutive K rows of one output column share an fp32 absmax
   (the first page's "64x64 blocks" is not used).
3. Code: ``v = fl32(w / absmax)``; ``q = argmin_i |C[i] - v|`` evaluated
   exactly, ties to the lower index; an all-zero block gets code 7.
4. Dequantization: ``w_hat = RNE_dtype(fl32(C[q] * absmax))`` -- an fp32
   product, then one rounding to the compute dtype.

Equality of this codebook with the table bitsandbytes ships is parity
unpinned: the pages do not print that table.

Double quantization ("GPTQ、AWQ与Bitsandbytes" §3.3 sets
``bnb_4bit_use_double_quant=True``; its pitfall list in §4.3 explains that
double quantization stores a scale of the scale).  Reading, where the pages
stop there:

5. The fp32 absmax values are themselves quantized to 8-bit unsigned codes
   (absmax >= 0), in blocks of 256 consecutive values of one absmax row
   (256 consecutive output columns of one 64-row block), each block with one
   fp32 second-level scale ``s2 = fl32(max / 255)`` (a zero scale becomes 1),
   ``code = clamp(rint(absmax / s2), 0, 255)`` (division in fp64).
6. The stored absmax is then ``absmax_hat = fl32(code * s2)`` (one fp32
   rounding of the exact product), and the weights' 4-bit codes are those of
   the first level, computed with the original absmax; dequantization uses
   ``absmax_hat`` in place of absmax.

Equality of this second level with bitsandbytes' own (which the pages do not
describe) is parity unpinned.
"""

from __future__ import annotations

import math

import numpy as np
from scipy.special import ndtri

from . import int4, numerics

DELTA = 1.0 - 0.5 * (1.0 / 30.0 + 1.0 / 32.0)


def codebook(delta: float = DELTA) -> np.ndarray:
    """The 16-entry NF4 codebook, float32, ascending."""
    p_pos = delta - (delta - 0.5) * np.arange(8) / 8.0  # 8 values, delta .. >0.5
    p_neg = delta - (delta - 0.5) * np.arange(7) / 7.0  # 7 values, delta .. >0.5
    scale = ndtri(delta)
    pos = ndtri(p_pos) / scale
    neg = -ndtri(p_neg) / scale
    c = np.sort(np.concatenate([neg, [0.0], pos]))
    return c.astype(np.float32)


def normal_quantile_bisect(p: float) -> float:
    """Standard-normal quantile by bisection on Phi(x) = erfc(-x / sqrt 2) / 2.

    Independent of ``scipy.special.ndtri``; used only to pin the codebook.
    """
    lo, hi = -40.0, 40.0
    for _ in range(200):
        mid = 0.5 * (lo + hi)
        if 0.5 * math.erfc(-mid / math.sqrt(2.0)) < p:
            lo = mid
        else:
            hi = mid
    return 0.5 * (lo + hi)


def nf4_quantize(W: np.ndarray, cb: np.ndarray, blocksize: int = 64):
    """Quantize fp32 ``W[K, N]``: returns ``(codes uint8[K, N], absmax float32[K/bs, N])``."""
    W = np.asarray(W, dtype=np.float32)
    K, N = W.shape
    if K % blocksize:
        raise ValueError("K must be a multiple of blocksize")
    cb64 = np.asarray(cb, dtype=np.float32).astype(np.float64)
    nb = K // blocksize
    codes = np.empty((K, N), dtype=np.uint8)
    absmax = np.empty((nb, N), dtype=np.float32)
    for b in range(nb):
        Wb = W[b * blocksize:(b + 1) * blocksize]
        am = np.abs(Wb).max(axis=0)
        absmax[b] = am
        zero = am == 0
        safe = np.where(zero, np.float32(1.0), am)
        v = (Wb / safe[None, :]).astype(np.float32)  # fp32 division
        # exact distances (differences of two fp32 values are exact in fp64)
        d = np.abs(cb64[:, None, None] - v.astype(np.float64)[None, :, :])
        q = np.argmin(d, axis=0)  # first minimum -> ties go to the lower index
        q[:, zero] = 7
        codes[b * blocksize:(b + 1) * blocksize] = q.astype(np.uint8)
    return codes, absmax


def nf4_dequant(codes, absmax, cb, dtype: str = "bf16", blocksize: int = 64) -> np.ndarray:
    """``RNE_dtype(fl32(C[q] * absmax))`` as uint16 bit patterns ``[K, N]``."""
    codes = np.asarray(codes)
    K, N = codes.shape
    am = np.repeat(np.asarray(absmax, dtype=np.float32), blocksize, axis=0)
    c = np.asarray(cb, dtype=np.float32)[codes]
    prod = (c * am).astype(np.float32)  # one fp32 rounding
    return numerics.round_to_dtype_bits(prod, dtype)


DQ_BLOCK = 256


def double_quantize_absmax(absmax: np.ndarray, dq_block: int = DQ_BLOCK):
    """Second-level quantization of fp32 ``absmax[B, N]`` (readings 5 and 6):
    ``(codes uint8[B, N], s2 float32[B, ceil(N / dq_block)])``."""
    am = np.asarray(absmax, dtype=np.float32)
    B, N = am.shape
    nc = -(-N // dq_block)
    codes = np.empty((B, N), dtype=np.uint8)
    s2 = np.empty((B, nc), dtype=np.float32)
    for c in range(nc):
        blk = am[:, c * dq_block:(c + 1) * dq_block].astype(np.float64)
        s = (blk.max(axis=1) / 255.0).astype(np.float32)  # one rounding of the fp64 quotient
        s[s == 0] = np.float32(1.0)
        s2[:, c] = s
        codes[:, c * dq_block:(c + 1) * dq_block] = np.clip(
            np.rint(blk / s.astype(np.float64)[:, None]), 0, 255).astype(np.uint8)
    return codes, s2


def absmax_from_double_quant(codes: np.ndarray, s2: np.ndarray, dq_block: int = DQ_BLOCK) -> np.ndarray:
    """``absmax_hat = fl32(code * s2)`` as float32 ``[B, N]``."""
    codes = np.asarray(codes)
    B, N = codes.shape
    s = np.repeat(np.asarray(s2, dtype=np.float32), dq_block, axis=1)[:, :N]
    # code (<= 255) and s2 are exact in fp64, so the fp64 product is exact and
    # its conversion to float32 is the single rounding
    return (codes.astype(np.float64) * s.astype(np.float64)).astype(np.float32)


def nf4_quantize_packed(W, cb, blocksize: int = 64):
    """Quantize and pack: ``(qweight uint32[K/8, N], absmax f32[K/bs, N], codes)``."""
    codes, absmax = nf4_quantize(W, cb, blocksize)
    return int4.pack_along_k(codes), absmax, codes
