"""Asymmetric INT4 round-to-nearest quantization, packing and dequantization.

Sources (page title / section):

* cloud.tencent.com/developer/article/2726413 §2.1: asymmetric quantization
  maps a float range onto an integer range that is not centred on zero and
  stores a zero point beside the scale; §2.2: group-wise granularity, one
  scale shared by each group of e.g. 128 elements; §2.3: 4-bit, 16 levels.
* "模型量化实践：GPTQ 与 AWQ 在生产环境的精度与速度权衡" §3.1: the GPTQ
  config ``bits=4, group_size=128, desc_act=True`` and the AWQ config
  ``zero_point=True, q_group_size=128, w_bit=4``.
* "GPTQ与bitsandbytes对比：谁是2024年大模型量化的终极选择？" (GPTQ section):
  round-to-nearest (RTN) is the plain baseline quantizer; ``--act-order``
  quantizes columns in order of activation size, so a group's rows are
  scattered over K (the row->group map ``g_idx``).

Readings where the pages are silent (each listed in the design notes):

1. Range: ``mn = min(min w, 0)``, ``mx = max(max w, 0)`` over a group's rows
   of one output column (zero always representable).
2. Scale: ``s = fp16_RNE((mx - mn) / 15)`` with the division in fp64; a zero
   scale becomes 1.
3. Zero point: ``z = clamp(rint(-mn / s), 0, 15)`` using the stored fp16 ``s``;
   ``rint`` rounds half to even.
4. Code: ``q = clamp(rint(w / s) + z, 0, 15)``, division in fp64.
5. Packing: 8 codes per little-endian uint32 along K, code of row ``8i + j``
   in bits ``4j .. 4j+3`` of word ``[i, n]``; zero points packed the same way
   along N: zero of column ``8c + j`` in bits ``4j ..`` of word ``[g, c]``.
   The stored zero is ``z`` itself (no offset).
6. Dequantization: ``w_hat = (q - z) * s`` is exact in fp32 (|q - z| <= 15
   has 4 bits, ``s`` 11); the value used by the product is that exact value
   rounded once to the compute dtype.
7. Symmetric quantization (cloud.tencent.com/developer/article/2726413 §2.1:
   the float range is mapped symmetrically onto the integer range and the
   zero point is fixed at 0): signed 4-bit codes ``c`` in [-8, 7] with
   ``s = fp16_RNE(max |w| / 7)`` (a zero scale becomes 1) and
   ``c = clamp(rint(w / s), -8, 7)``, stored in the same unsigned nibble as
   ``q = c + 8``; so the stored format is the asymmetric one with every zero
   point equal to 8, and no zero points need to be stored.
"""

from __future__ import annotations

import numpy as np

from . import numerics


def row_groups(K: int, group_size: int, g_idx=None) -> np.ndarray:
    """Group index of each of the K rows: ``g_idx`` if given, else ``k // group_size``."""
    if g_idx is None:
        if K % group_size:
            raise ValueError("K must be a multiple of group_size")
        return (np.arange(K) // group_size).astype(np.int64)
    g = np.asarray(g_idx).astype(np.int64)
    if g.shape != (K,):
        raise ValueError("g_idx must have K entries")
    return g


def rtn_quantize(W: np.ndarray, group_size: int = 128, g_idx=None):
    """Quantize fp32 ``W[K, N]``.

    Returns ``(q uint8[K, N], scales float16[G, N], zeros uint8[G, N])`` with
    ``G = K // group_size``.  Each group ``gi`` holds the rows ``k`` whose
    group index is ``gi``; the statistics are taken per output column.
    """
    W = np.asarray(W, dtype=np.float32)
    K, N = W.shape
    gid = row_groups(K, group_size, g_idx)
    G = K // group_size
    q = np.empty((K, N), dtype=np.uint8)
    scales = np.empty((G, N), dtype=np.float16)
    zeros = np.empty((G, N), dtype=np.uint8)
    for gi in range(G):
        rows = np.nonzero(gid == gi)[0]
        Wg = W[rows].astype(np.float64)
        mn = np.minimum(Wg.min(axis=0), 0.0)
        mx = np.maximum(Wg.max(axis=0), 0.0)
        s16 = numerics.to_f16((mx - mn) / 15.0)
        s16[s16 == 0] = np.float16(1.0)
        s = s16.astype(np.float64)
        z = np.clip(np.rint(-mn / s), 0, 15)
        qg = np.clip(np.rint(Wg / s) + z, 0, 15)
        q[rows] = qg.astype(np.uint8)
        scales[gi] = s16
        zeros[gi] = z.astype(np.uint8)
    return q, scales, zeros


SYM_ZERO = 8


def rtn_quantize_sym(W: np.ndarray, group_size: int = 128, g_idx=None):
    """Symmetric RTN quantization of fp32 ``W[K, N]`` (reading 7).

    Returns ``(q uint8[K, N], scales float16[G, N])``; the zero point of every
    group is ``SYM_ZERO`` (8).
    """
    W = np.asarray(W, dtype=np.float32)
    K, N = W.shape
    gid = row_groups(K, group_size, g_idx)
    G = K // group_size
    q = np.empty((K, N), dtype=np.uint8)
    scales = np.empty((G, N), dtype=np.float16)
    for gi in range(G):
        rows = np.nonzero(gid == gi)[0]
        Wg = W[rows].astype(np.float64)
        amax = np.abs(Wg).max(axis=0)
        s16 = numerics.to_f16(amax / 7.0)
        s16[s16 == 0] = np.float16(1.0)
        s = s16.astype(np.float64)
        c = np.clip(np.rint(Wg / s), -8, 7)
        q[rows] = (c + SYM_ZERO).astype(np.uint8)
        scales[gi] = s16
    return q, scales


def sym_zeros(G: int, N: int) -> np.ndarray:
    """The zero points a symmetric checkpoint implies: 8 everywhere."""
    return np.full((G, N), SYM_ZERO, dtype=np.uint8)


def pack_along_k(q: np.ndarray) -> np.ndarray:
    """uint8 codes ``[K, N]`` (values 0..15) -> uint32 ``[K/8, N]``."""
    q = np.asarray(q, dtype=np.uint32)
    K, N = q.shape
    if K % 8:
        raise ValueError("K must be a multiple of 8")
    q3 = q.reshape(K // 8, 8, N)
    out = np.zeros((K // 8, N), dtype=np.uint32)
    for j in range(8):
        out |= q3[:, j, :] << np.uint32(4 * j)
    return out


def unpack_along_k(packed: np.ndarray) -> np.ndarray:
    """uint32 ``[K/8, N]`` -> uint8 codes ``[K, N]``."""
    p = np.asarray(packed, dtype=np.uint32)
    R, N = p.shape
    out = np.empty((R, 8, N), dtype=np.uint8)
    for j in range(8):
        out[:, j, :] = ((p >> np.uint32(4 * j)) & np.uint32(0xF)).astype(np.uint8)
    return out.reshape(R * 8, N)


def pack_zeros(z: np.ndarray) -> np.ndarray:
    """uint8 zero points ``[G, N]`` -> uint32 ``[G, N/8]`` (packed along N)."""
    z = np.asarray(z, dtype=np.uint32)
    G, N = z.shape
    if N % 8:
        raise ValueError("N must be a multiple of 8")
    z3 = z.reshape(G, N // 8, 8)
    out = np.zeros((G, N // 8), dtype=np.uint32)
    for j in range(8):
        out |= z3[:, :, j] << np.uint32(4 * j)
    return out


def unpack_zeros(packed: np.ndarray) -> np.ndarray:
    """uint32 ``[G, N/8]`` -> uint8 zero points ``[G, N]``."""
    p = np.asarray(packed, dtype=np.uint32)
    G, C = p.shape
    out = np.empty((G, C, 8), dtype=np.uint8)
    for j in range(8):
        out[:, :, j] = ((p >> np.uint32(4 * j)) & np.uint32(0xF)).astype(np.uint8)
    return out.reshape(G, C * 8)


def dequant_exact(q, scales, zeros, group_size: int = 128, g_idx=None) -> np.ndarray:
    """``(q - z) * s`` for every element, float64 ``[K, N]`` (exact)."""
    q = np.asarray(q)
    K, N = q.shape
    gid = row_groups(K, group_size, g_idx)
    s = np.asarray(scales, dtype=np.float16).astype(np.float64)[gid]
    z = np.asarray(zeros).astype(np.float64)[gid]
    return (q.astype(np.float64) - z) * s


def dequant(q, scales, zeros, dtype: str, group_size: int = 128, g_idx=None) -> np.ndarray:
    """Dequantized weights in ``dtype`` (uint16 bit patterns ``[K, N]``).

    The exact product is representable in fp32, so rounding it from fp32 to
    the 16-bit type is a single rounding of the exact value.
    """
    w = dequant_exact(q, scales, zeros, group_size, g_idx).astype(np.float32)
    return numerics.round_to_dtype_bits(w, dtype)


def quantize_packed(W, group_size: int = 128, g_idx=None):
    """Quantize and pack: ``(qweight uint32[K/8,N], scales f16[G,N], qzeros uint32[G,N/8], q, zeros)``."""
    q, scales, zeros = rtn_quantize(W, group_size, g_idx)
    return pack_along_k(q), scales, pack_zeros(zeros), q, zeros
