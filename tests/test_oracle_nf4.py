"""Pins for the oracle's NF4 codebook, quantizer and dequantization."""

from fractions import Fraction

import numpy as np

from oracle import nf4, numerics
from synth import gaussian_weights


def test_codebook_invariants():
    c = nf4.codebook()
    assert c.dtype == np.float32 and c.shape == (16,)
    assert c[0] == -1.0 and c[7] == 0.0 and c[15] == 1.0
    assert np.all(np.diff(c) > 0)
    assert np.sum(c < 0) == 7 and np.sum(c > 0) == 8
    # values concentrate near zero: the steps grow away from the centre
    pos = np.diff(c[7:])
    neg = np.diff(c[:8])
    assert np.all(np.diff(pos) > 0)
    assert np.all(np.diff(neg) < 0)


def test_codebook_against_bisection_quantiles():
    # each entry equals an independent inverse-CDF evaluation (bisection on
    # erfc) to within one fp32 ulp
    d = nf4.DELTA
    scale = nf4.normal_quantile_bisect(d)
    pos = [nf4.normal_quantile_bisect(d - (d - 0.5) * i / 8) / scale for i in range(8)]
    neg = [-nf4.normal_quantile_bisect(d - (d - 0.5) * j / 7) / scale for j in range(7)]
    want = np.sort(np.array(neg + [0.0] + pos)).astype(np.float32)
    got = nf4.codebook()
    ulp = np.spacing(np.abs(want).astype(np.float32))
    assert np.all(np.abs(got.astype(np.float64) - want.astype(np.float64)) <= ulp)


def test_quantize_is_nearest_code_brute_force():
    cb = nf4.codebook()
    rng = np.random.default_rng(1)
    K, N = 64, 6
    W = (rng.standard_normal((K, N)) * 0.02).astype(np.float32)
    codes, absmax = nf4.nf4_quantize(W, cb, 64)
    assert np.array_equal(absmax[0], np.abs(W).max(axis=0))
    for k in range(K):
        for n in range(N):
            v = Fraction(float(np.float32(W[k, n]) / np.float32(absmax[0, n])))
            best = min(range(16), key=lambda i: (abs(Fraction(float(cb[i])) - v), i))
            assert codes[k, n] == best


def test_quantize_ties_go_low_and_zero_block():
    # an evenly spaced test codebook (the quantizer takes any ascending table)
    # whose midpoints are exact in fp32: a value exactly halfway between two
    # codes (after dividing by absmax = 1) takes the lower code
    cb = ((np.arange(16) - 7) / 8).astype(np.float32)
    W = np.zeros((64, 2), dtype=np.float32)
    W[0, 0] = 1.0
    W[1, 0] = 5.0 / 16.0  # halfway between 2/8 (code 9) and 3/8 (code 10)
    W[2, 0] = np.nextafter(np.float32(5.0 / 16.0), np.float32(1))
    codes, absmax = nf4.nf4_quantize(W, cb, 64)
    assert codes[1, 0] == 9 and codes[2, 0] == 10
    assert np.all(codes[:, 1] == 7) and absmax[0, 1] == 0.0  # all-zero block
    assert codes[0, 0] == 15


def test_reconstruction_bound():
    cb = nf4.codebook()
    K, N = 512, 64
    W = gaussian_weights(K, N, 0.02, 2)
    codes, absmax = nf4.nf4_quantize(W, cb, 64)
    w_hat = numerics.bf16_bits_to_f64(nf4.nf4_dequant(codes, absmax, cb, "bf16"))
    am = np.repeat(absmax.astype(np.float64), 64, axis=0)
    gap = np.max(np.diff(cb.astype(np.float64))) / 2
    err = np.abs(W.astype(np.float64) - w_hat)
    # half the widest codebook step, plus the fp32 division and the bf16 rounding
    assert np.all(err <= am * (gap + 2.0 ** -22) + np.abs(w_hat) * 2.0 ** -8)
    # the block maximum is reproduced to bf16 precision (code +-1 -> +-absmax)
    top = np.argmax(np.abs(W.reshape(8, 64, N)), axis=1)
    for b in range(8):
        for n in range(N):
            k = 64 * b + top[b, n]
            assert codes[k, n] in (0, 15)


def test_dequant_is_fp32_product_then_one_rounding():
    cb = nf4.codebook()
    rng = np.random.default_rng(5)
    codes = rng.integers(0, 16, size=(128, 32)).astype(np.uint8)
    absmax = (rng.uniform(0.01, 0.2, size=(2, 32))).astype(np.float32)
    got = nf4.nf4_dequant(codes, absmax, cb, "bf16")
    am = np.repeat(absmax, 64, axis=0)
    for k in range(0, 128, 17):
        for n in range(32):
            p = np.float32(cb[codes[k, n]]) * np.float32(am[k, n])  # fp32 product
            # nearest bf16 to p, ties to even, by exhaustive neighbour search
            b = int(np.float32(p).view(np.uint32)) >> 16
            cands = [b, b + 1]
            vals = [Fraction(float(np.uint32(c << 16).view(np.float32))) for c in cands]
            pv = Fraction(float(p))
            best = min(zip(vals, cands), key=lambda t: (abs(t[0] - pv), t[1] % 2))[1]
            assert got[k, n] == best


# ----------------------------------------------------- double quantization
def test_double_quant_exact_grid_recovered():
    # absmax values on the second-level grid k * s2, with each 256-column
    # block's maximum at 255 * s2 (s2 = 2^-12, exact), come back unchanged:
    # s2 = max / 255 exactly, codes k, absmax_hat = absmax
    s2 = 2.0 ** -12
    rng = np.random.default_rng(2)
    B, N = 6, 600  # three second-level blocks per row, the last one ragged
    k = rng.integers(0, 256, size=(B, N))
    k[:, 0] = 255
    k[:, 256] = 255
    k[:, 512] = 255
    am = (k * s2).astype(np.float32)
    codes, sc = nf4.double_quantize_absmax(am)
    assert sc.shape == (B, 3) and np.all(sc == np.float32(s2))
    assert np.array_equal(codes.astype(int), k)
    assert np.array_equal(nf4.absmax_from_double_quant(codes, sc), am)


def test_double_quant_half_step_and_blocks():
    W = gaussian_weights(1024, 520, 0.02, 4)
    cb = nf4.codebook()
    _, am = nf4.nf4_quantize(W, cb)
    codes, sc = nf4.double_quantize_absmax(am)
    hat = nf4.absmax_from_double_quant(codes, sc).astype(np.float64)
    s_cols = np.repeat(sc.astype(np.float64), 256, axis=1)[:, :am.shape[1]]
    # rint to the nearest step, then one fp32 rounding of code * s2
    err = np.abs(hat - am.astype(np.float64))
    assert np.all(err <= s_cols / 2 + np.spacing(hat.astype(np.float32)).astype(np.float64))
    # each block's largest absmax takes code 255; the scale is per block of 256
    # consecutive columns of one row: a change in one block moves only its s2
    for c in range(sc.shape[1]):
        blk = codes[:, c * 256:(c + 1) * 256]
        assert np.all(blk.max(axis=1) == 255)
    am2 = am.copy()
    am2[3, 10] *= 2
    _, sc2 = nf4.double_quantize_absmax(am2)
    diff = np.argwhere(sc2 != sc)
    assert diff.tolist() == [[3, 0]]


def test_double_quant_zero_block():
    am = np.zeros((2, 256), dtype=np.float32)
    am[1, 5] = 0.5
    codes, sc = nf4.double_quantize_absmax(am)
    assert sc[0, 0] == 1.0 and np.all(codes[0] == 0)  # a zero scale becomes 1
    hat = nf4.absmax_from_double_quant(codes, sc)
    assert np.all(hat[0] == 0.0) and hat[1, 5] == np.float32(np.float32(0.5 / 255) * 255)
