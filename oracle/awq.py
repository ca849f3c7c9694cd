"""The AWQ checkpoint layout and its conversion to this library's layout.

TEST INFRASTRUCTURE ONLY (see the package docstring).

Sources (page title / section):

* "模型量化实践：GPTQ 与 AWQ 在生产环境的精度与速度权衡" §3.1: the AWQ config
  ``zero_point=True, q_group_size=128, w_bit=4, version="GEMM"`` -- an
  asymmetric 4-bit checkpoint with a zero point per group, in the layout of
  AWQ's GEMM kernels.
* "LLM量化技术深度对比:GPTQ vs AWQ vs bitsandbytes 2026基准全解析" §5: AWQ
  checkpoints are served by the Marlin kernel (the top row of its H200 table),
  i.e. the same weights can be re-laid out for a faster kernel.

Reading (the pages do not print the packing; this is AWQ's published GEMM
layout, so equality with files written by AWQ's own tools is *parity
unpinned*):

* ``qweight int32 [K, N/8]``: word ``[k, c]`` holds the codes of row k,
  columns 8c .. 8c+7 -- packed along N, not along K -- with column
  ``8c + ORDER[j]`` in bits ``4j .. 4j+3``, ``ORDER = (0, 2, 4, 6, 1, 3, 5, 7)``.
* ``qzeros int32 [G, N/8]``: the zero points packed the same way.
* ``scales fp16 [G, N]``: as in this library.
* The stored zero is z (w_hat = (q - z) * s), as in this library.

Converting to this library's layout is a pure re-arrangement of nibbles:
codes packed 8 per word along K, zero points packed along N in natural order.
"""

from __future__ import annotations

import numpy as np

from . import int4

ORDER = (0, 2, 4, 6, 1, 3, 5, 7)


def pack_awq(v: np.ndarray) -> np.ndarray:
    """uint8 nibbles ``[R, N]`` -> uint32 ``[R, N/8]`` in the AWQ column order."""
    v = np.asarray(v, dtype=np.uint32)
    R, N = v.shape
    if N % 8:
        raise ValueError("N must be a multiple of 8")
    v3 = v.reshape(R, N // 8, 8)
    out = np.zeros((R, N // 8), dtype=np.uint32)
    for j in range(8):
        out |= v3[:, :, ORDER[j]] << np.uint32(4 * j)
    return out


def unpack_awq(packed: np.ndarray) -> np.ndarray:
    """uint32 ``[R, N/8]`` in the AWQ column order -> uint8 nibbles ``[R, N]``."""
    p = np.asarray(packed, dtype=np.uint32)
    R, C = p.shape
    out = np.empty((R, C, 8), dtype=np.uint8)
    for j in range(8):
        out[:, :, ORDER[j]] = ((p >> np.uint32(4 * j)) & np.uint32(0xF)).astype(np.uint8)
    return out.reshape(R, C * 8)


def awq_checkpoint(W: np.ndarray, group_size: int = 128):
    """Quantize fp32 ``W[K, N]`` (this library's asymmetric RTN reading) and lay
    it out as an AWQ checkpoint: ``(qweight_awq, scales, qzeros_awq, q, zeros)``."""
    q, scales, zeros = int4.rtn_quantize(W, group_size)
    return pack_awq(q), scales, pack_awq(zeros), q, zeros


def to_library_layout(qweight_awq: np.ndarray, qzeros_awq: np.ndarray):
    """AWQ ``(qweight [K, N/8], qzeros [G, N/8])`` -> this library's
    ``(qweight [K/8, N] packed along K, qzeros [G, N/8] in natural order)``."""
    q = unpack_awq(qweight_awq)
    z = unpack_awq(qzeros_awq)
    return int4.pack_along_k(q), int4.pack_zeros(z)
