"""Host checks of the arithmetic facts the kernels' exact dequantization routes
rest on, over every finite fp16 scale, every code and every zero point.

The value both routes must produce is w_hat = RNE_dtype((q - z) * s)
(cloud.tencent.com/developer/article/2726413 §2.1: asymmetric quantization
with a stored zero point).  These checks do the routes' steps in exact fp64 arithmetic
(every product and sum below is exact in fp64) and assert that each rounding
the hardware performs is exact except the final one.  They run no kernel and
use no oracle code; the GPU tests pin the kernels themselves against the
oracle.
"""

import numpy as np


def _finite_f16_scales():
    s = np.arange(0x10000, dtype=np.uint32).astype(np.uint16).view(np.float16).astype(np.float64)
    return s[np.isfinite(s)]


def _is_f32(x):
    with np.errstate(over="ignore"):
        return np.array_equal(x.astype(np.float32).astype(np.float64), x)


def _is_bf16(x):
    return _is_f32(x) and not np.any(x.astype(np.float32).view(np.uint32) & 0xFFFF)


def test_magic_codes():
    # fp16 0x6400 | q is 1024 + q; 0x5400 | (q << 4) is 64 + q; bf16 0x4300 | q is 128 + q
    q = np.arange(16, dtype=np.uint16)
    assert np.array_equal((0x6400 | q).view(np.float16).astype(np.float64), 1024.0 + q)
    assert np.array_equal((0x5400 | (q << 4)).view(np.float16).astype(np.float64), 64.0 + q)
    bf = ((0x4300 | q).astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    assert np.array_equal(bf, 128.0 + q)


def test_fp32_fma_route_is_exact_for_every_scale():
    # fma(bias + q, s, -(bias + z) * s): the fp32 addend is exact (<= 22
    # significant bits), the FMA's single rounding lands on the exact
    # (q - z) * s (<= 15 bits), so the one conversion to bf16 is the only
    # rounding of the exact product
    s = _finite_f16_scales()
    for bias in (1024.0, 64.0):
        for z in range(16):
            addend = -(bias + z) * s
            assert _is_f32(addend), (bias, z)
            for q in range(16):
                exact_sum = (bias + q) * s + addend
                assert np.array_equal(exact_sum, (q - z) * s)
                assert _is_f32(exact_sum), (bias, z, q)


def test_packed_bf16_route_is_exact_for_every_scale():
    # s = s_hi + s_lo with s_hi the first 8 significant bits of s: both parts
    # are bf16 numbers, (q - z) * s_lo is exact in bf16, and
    # fma(q - z, s_hi, (q - z) * s_lo) rounds the exact (q - z) * s once
    s = _finite_f16_scales()
    bits = s.astype(np.float32).view(np.uint32)
    s_hi = (bits & 0xFFFF0000).view(np.float32).astype(np.float64)
    s_lo = s - s_hi
    assert _is_bf16(s_hi) and _is_bf16(s_lo)
    for v in range(-15, 16):
        assert _is_bf16(v * s_lo), v
        assert np.array_equal(v * s_hi + v * s_lo, v * s)
