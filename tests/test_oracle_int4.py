"""Pins for the oracle's INT4 asymmetric RTN quantizer, packing and dequantization.

Each test checks a property the pages or the mathematics fix, chosen so that a
plausible slip (a dropped zero point, a wrong sign, a swapped nibble order, a
group index taken along the wrong axis) fails at least one of them.
"""

import numpy as np
import pytest

from oracle import int4, numerics
from synth import act_order_g_idx, gaussian_weights, student_t_weights


def _quant(W, g_idx=None, gs=128):
    q, s, z = int4.rtn_quantize(W, gs, g_idx)
    return q, s, z


@pytest.mark.parametrize("dist", ["normal", "t5"])
def test_grid_invariant_and_levels(dist):
    K, N = 512, 96
    W = gaussian_weights(K, N, 0.02, 1) if dist == "normal" else student_t_weights(K, N, 5, 0.01, 1)
    q, s, z = _quant(W)
    assert q.max() <= 15 and z.max() <= 15  # 16 levels
    w_hat = int4.dequant_exact(q, s, z)
    s_rows = s.astype(np.float64)[np.arange(K) // 128]
    z_rows = z.astype(np.float64)[np.arange(K) // 128]
    ratio = w_hat / s_rows
    # every reconstruction sits exactly on the integer grid (q - z) * s
    assert np.array_equal(ratio, np.round(ratio))
    assert np.all(ratio >= -z_rows) and np.all(ratio <= 15 - z_rows)


def test_zero_is_exactly_representable():
    # asymmetric quantization stores the zero point so that 0.0 maps to an
    # integer code and reconstructs to exactly 0
    W = gaussian_weights(256, 64, 0.02, 5)
    W[::7, ::3] = 0.0
    q, s, z = _quant(W)
    w_hat = int4.dequant_exact(q, s, z)
    assert np.all(w_hat[::7, ::3] == 0.0)


def test_half_step_error_bound():
    K, N = 1024, 128
    W = student_t_weights(K, N, 5, 0.01, 2)
    q, s, z = _quant(W)
    w_hat = int4.dequant_exact(q, s, z)
    s_rows = s.astype(np.float64)[np.arange(K) // 128]
    err = np.abs(W.astype(np.float64) - w_hat)
    clamped = (q == 0) | (q == 15)
    # nearest-grid rounding: at most half a step away, wherever no clamp acted
    interior = ~clamped
    assert np.all(err[interior] <= s_rows[interior] / 2)
    # at the ends the fp16 rounding of s can push min/max just outside the
    # 15-step grid; the bound there is (1/2 + 15 * 2^-11 * (1 + 2^-11)) * s
    bound = (0.5 + 15 * 2.0 ** -11 * (1 + 2.0 ** -11)) * s_rows
    assert np.all(err <= bound)


def test_lossless_on_exact_grid():
    # weights built on a grid the quantizer can represent exactly must come back
    # unchanged, with the grid's own scale, zero point and codes
    rng = np.random.default_rng(11)
    K, N = 256, 40
    s0 = 2.0 ** -6
    z0 = rng.integers(0, 16, size=(K // 128, N))
    q0 = rng.integers(0, 16, size=(K, N))
    q0[::128] = 0  # each group-column holds code 0 and code 15, so min/max
    q0[1::128] = 15  # span exactly 15 steps
    zr = z0[np.arange(K) // 128]
    W = ((q0 - zr) * s0).astype(np.float32)
    # groups with z0 == 0 or 15 have a zero end point already; others include 0
    q, s, z = _quant(W)
    assert np.all(s.astype(np.float64) == s0)
    assert np.array_equal(z, z0.astype(np.uint8))
    assert np.array_equal(q, q0.astype(np.uint8))
    assert np.array_equal(int4.dequant_exact(q, s, z), W.astype(np.float64))


def test_monotone_in_w_within_group():
    K, N = 128, 64
    W = gaussian_weights(K, N, 0.02, 9)
    q, s, z = _quant(W)
    order = np.argsort(W, axis=0, kind="stable")
    qs = np.take_along_axis(q.astype(int), order, axis=0)
    assert np.all(np.diff(qs, axis=0) >= 0)


def test_pack_unpack_roundtrip_exhaustive_positions():
    # every code value at every nibble position of a word
    K, N = 8 * 16, 8
    q = np.zeros((K, N), dtype=np.uint8)
    for v in range(16):
        for j in range(8):
            q[8 * v + j, j] = v
    p = int4.pack_along_k(q)
    assert np.array_equal(int4.unpack_along_k(p), q)
    rng = np.random.default_rng(0)
    words = rng.integers(0, 2 ** 32, size=(64, 24), dtype=np.uint64).astype(np.uint32)
    assert np.array_equal(int4.pack_along_k(int4.unpack_along_k(words)), words)
    zw = rng.integers(0, 2 ** 32, size=(5, 3), dtype=np.uint64).astype(np.uint32)
    assert np.array_equal(int4.pack_zeros(int4.unpack_zeros(zw)), zw)


def test_pack_nibble_order():
    # row 8i+j of a column lands in bits 4j..4j+3 of word [i, n]; zero point of
    # column 8c+j lands in bits 4j.. of word [g, c]
    q = np.arange(8, dtype=np.uint8).reshape(8, 1)
    assert int4.pack_along_k(q)[0, 0] == 0x76543210
    z = (np.arange(8, dtype=np.uint8) + 1).reshape(1, 8)
    assert int4.pack_zeros(z)[0, 0] == 0x87654321


def test_dequant_single_rounding():
    # the dtype value is the exact (q - z) * s rounded once; forming
    # q*s - z*s in the dtype instead differs on some inputs
    rng = np.random.default_rng(4)
    K, N = 128, 512
    q = rng.integers(0, 16, size=(K, N)).astype(np.uint8)
    z = rng.integers(0, 16, size=(1, N)).astype(np.uint8)
    s = numerics.to_f16(rng.uniform(1e-4, 0.1, size=(1, N)))
    for dt in ("f16", "bf16"):
        bits = int4.dequant(q, s, z, dt)
        exact = int4.dequant_exact(q, s, z)
        back = numerics.dtype_bits_to_f64(bits, dt)
        # nearest representable: no other dtype value is closer
        nxt = numerics.dtype_bits_to_f64(bits + np.uint16(1), dt)
        prv = numerics.dtype_bits_to_f64(bits - np.uint16(1), dt)
        err = np.abs(back - exact)
        pos = back > 0
        assert np.all(err[pos] <= np.abs(nxt[pos] - exact[pos]))
        assert np.all(err[pos] <= np.abs(prv[pos] - exact[pos]))


def test_act_order_equals_physical_regroup():
    # quantizing with a scattered row->group map must give the same codes as
    # first moving each group's rows together and quantizing contiguous groups
    K, N = 1024, 48
    W = student_t_weights(K, N, 5, 0.01, 3)
    g_idx = act_order_g_idx(K, 128, 3)
    q, s, z = _quant(W, g_idx)
    order = np.argsort(g_idx, kind="stable")  # rows sorted by group
    q2, s2, z2 = _quant(W[order])
    assert np.array_equal(q[order], q2)
    assert np.array_equal(s, s2) and np.array_equal(z, z2)
    # and dequantization follows the map row by row
    w1 = int4.dequant_exact(q, s, z, 128, g_idx)
    w2 = int4.dequant_exact(q2, s2, z2)
    assert np.array_equal(w1[order], w2)


def test_g_idx_groups_have_group_size_rows():
    g = act_order_g_idx(4096, 128, 0)
    assert np.all(np.bincount(g) == 128)
    assert not np.array_equal(g, np.arange(4096) // 128)


@pytest.mark.parametrize("gs", [32, 64, 1024])
def test_other_group_sizes(gs):
    # the quantizer and dequantizer take the group size as a parameter (a
    # finer grouping, or one group per column when it equals K); the grid
    # invariant, the half-step bound and exact recovery of an exact grid
    # must hold at every size, with the statistics taken per group of gs rows
    K, N = 1024, 48
    W = student_t_weights(K, N, 5, 0.01, gs)
    q, s, z = _quant(W, gs=gs)
    assert s.shape == (K // gs, N) and z.shape == (K // gs, N)
    w_hat = int4.dequant_exact(q, s, z, gs)
    s_rows = s.astype(np.float64)[np.arange(K) // gs]
    z_rows = z.astype(np.float64)[np.arange(K) // gs]
    ratio = w_hat / s_rows
    assert np.array_equal(ratio, np.round(ratio))
    assert np.all(ratio >= -z_rows) and np.all(ratio <= 15 - z_rows)
    err = np.abs(W.astype(np.float64) - w_hat)
    interior = (q != 0) & (q != 15)
    assert np.all(err[interior] <= s_rows[interior] / 2)
    assert np.all(err <= (0.5 + 15 * 2.0 ** -11 * (1 + 2.0 ** -11)) * s_rows)
    # each group's scale comes from that group's own range: the range of the
    # first group of column 0 is 15 steps of its scale to within fp16 rounding
    g0 = W[:gs, 0].astype(np.float64)
    rng_ = max(g0.max(), 0.0) - min(g0.min(), 0.0)
    assert abs(float(s[0, 0]) * 15 - rng_) <= 15 * float(s[0, 0]) * 2.0 ** -10
    # exact grid, recovered unchanged
    rng = np.random.default_rng(gs)
    z0 = rng.integers(0, 16, size=(K // gs, N))
    q0 = rng.integers(0, 16, size=(K, N))
    q0[::gs] = 0
    q0[1::gs] = 15
    s0 = 2.0 ** -7
    Wg = ((q0 - z0[np.arange(K) // gs]) * s0).astype(np.float32)
    q1, s1, z1 = _quant(Wg, gs=gs)
    assert np.all(s1.astype(np.float64) == s0)
    assert np.array_equal(z1, z0.astype(np.uint8)) and np.array_equal(q1, q0.astype(np.uint8))
    # a different group size on the same weights gives different statistics
    q2, s2, _ = _quant(W, gs=128 if gs != 128 else 64)
    assert s2.shape != s.shape


def test_zero_point_uses_the_stored_fp16_scale():
    # The stored format keeps s in fp16 and the zero point is z = round(-min/s)
    # with that stored s (cloud.tencent.com/developer/article/2726413 §2.1: an
    # asymmetric grid stores a scale and a zero point; the fp16 scale is the
    # stored one).  This group is built so that the fp16 rounding of s decides
    # z.  With u = 2^-7:
    #   min w = -(5.5 + 5.5 * 2^-14) * u,  max w = (9.5 + 24.5 * 2^-14) * u,
    #   (max - min) / 15 = u * (1 + 2^-13), which rounds to s = u in fp16,
    #   -min / s = 5.5 + 5.5 * 2^-14 -> z = 6,
    # while the unrounded scale would give -min / (u (1 + 2^-13)) = 5.4997...
    # -> 5.  Codes, by hand: min -> rint(-5.5003) + 6 = 0; max -> rint(9.5015)
    # + 6 = 16 -> 15; 0 -> 6; u -> 7.
    u = 2.0 ** -7
    mn = -(5.5 + 5.5 * 2.0 ** -14) * u
    mx = (9.5 + 24.5 * 2.0 ** -14) * u
    W = np.zeros((128, 8), dtype=np.float32)
    W[0, :] = mn
    W[1, :] = mx
    W[2, :] = u
    assert float(np.float32(mn)) == mn and float(np.float32(mx)) == mx  # exact in fp32
    q, s, z = _quant(W)
    assert np.all(s.astype(np.float64) == u)
    assert np.all(z == 6)
    assert np.all(q[0] == 0) and np.all(q[1] == 15) and np.all(q[2] == 7) and np.all(q[3:] == 6)
    # the zero weight reconstructs exactly through the stored z
    assert np.all(int4.dequant_exact(q, s, z)[3:] == 0.0)


def test_range_always_contains_zero():
    # An asymmetric grid with a stored zero point represents 0 exactly (same
    # passage), so the range of a group is taken with 0 included.  All-positive
    # group: w = k * u for k = 1..15 (and copies), u = 2^-7.  With 0 in range:
    # s = 15u / 15 = u, z = 0, q = k.  (Without it, s would be 14u / 15 in fp16
    # and the codes would not be k.)
    u = 2.0 ** -7
    k = (np.arange(128) % 15) + 1
    W = np.repeat((k * u).astype(np.float32)[:, None], 8, axis=1)
    q, s, z = _quant(W)
    assert np.all(s.astype(np.float64) == u)
    assert np.all(z == 0)
    assert np.array_equal(q[:, 0], k.astype(np.uint8))
    # all-negative group: w = -k * u -> s = u, z = 15, q = 15 - k
    qn, sn, zn = _quant(-W)
    assert np.all(sn.astype(np.float64) == u)
    assert np.all(zn == 15)
    assert np.array_equal(qn[:, 0], (15 - k).astype(np.uint8))
    # and in both, the weights come back exactly
    assert np.array_equal(int4.dequant_exact(q, s, z), W.astype(np.float64))
    assert np.array_equal(int4.dequant_exact(qn, sn, zn), -W.astype(np.float64))


# ---------------------------------------------------------------- symmetric
def test_symmetric_exact_grid_recovered():
    # Symmetric quantization (same passage, §2.1): the range [-max|w|, max|w|]
    # maps onto the signed integers with the zero point fixed at 0.  Weights
    # c * u with c in -7..7 and max |w| = 7u (u = 2^-8, exact in fp16) come
    # back as scale u and stored codes c + 8.
    u = 2.0 ** -8
    rng = np.random.default_rng(5)
    c0 = rng.integers(-7, 8, size=(256, 24))
    c0[0] = 7
    c0[1] = -7
    W = (c0 * u).astype(np.float32)
    q, s = int4.rtn_quantize_sym(W)
    assert np.all(s.astype(np.float64) == u)
    assert np.array_equal(q.astype(int), c0 + 8)
    z = int4.sym_zeros(*s.shape)
    assert np.array_equal(int4.dequant_exact(q, s, z), W.astype(np.float64))


def test_symmetric_scale_is_max_abs_over_7_and_zero_is_exact():
    # one group whose largest magnitude is negative: s = fp16(max|w| / 7) (here
    # |min| = 0.0875 -> 0.0125 -> fp16 6552 * 2^-19 = 0.0124969482421875), the most negative
    # weight gets code 8 - 7 = 1, and 0 gets code 8 and reconstructs to 0
    W = np.zeros((128, 8), dtype=np.float32)
    W[0] = -0.0875
    W[1] = 0.05
    q, s = int4.rtn_quantize_sym(W)
    assert np.all(s == np.float16(0.0125))
    assert float(np.float16(0.0125)) == 6552 * 2.0 ** -19
    assert np.all(q[0] == 1) and np.all(q[2:] == 8)
    # 0.05 / 0.0124969 = 4.0010 -> 4 -> code 12; -0.0875 / 0.0124969 = -7.0017 -> -7
    assert np.all(q[1] == 12)
    w_hat = int4.dequant_exact(q, s, int4.sym_zeros(*s.shape))
    assert np.all(w_hat[2:] == 0.0)


def test_symmetric_is_odd_and_within_half_a_step():
    K, N = 512, 64
    W = student_t_weights(K, N, 5, 0.01, 8)
    q, s = int4.rtn_quantize_sym(W)
    qn, sn = int4.rtn_quantize_sym(-W)
    assert np.array_equal(s, sn)
    z = int4.sym_zeros(*s.shape)
    w1 = int4.dequant_exact(q, s, z)
    w2 = int4.dequant_exact(qn, sn, z)
    assert np.array_equal(w2, -w1)  # w -> -w flips every reconstruction (rint is odd)
    s_rows = s.astype(np.float64)[np.arange(K) // 128]
    err = np.abs(W.astype(np.float64) - w1)
    # |w / s| <= 7 (1 + 2^-11) < 7.5, so no code is clamped: half a step everywhere
    assert np.all(err <= s_rows / 2)
    ratio = w1 / s_rows
    assert np.array_equal(ratio, np.round(ratio)) and np.all(np.abs(ratio) <= 7)
