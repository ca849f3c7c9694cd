"""Pins for the oracle's reference product, its tolerance check and byte accounting."""

import json
import os
from fractions import Fraction

import numpy as np
import pytest

from oracle import accounting, int4, numerics, product
from synth import WORKLOADS, activations, gaussian_weights

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "page_numbers.json")


def _exact_product(X, W):
    M, K = X.shape
    _, N = W.shape
    Y = np.empty((M, N))
    for m in range(M):
        for n in range(N):
            Y[m, n] = float(sum(Fraction(float(X[m, k])) * Fraction(float(W[k, n])) for k in range(K)))
    return Y


def test_brute_force_8x8_one_group():
    # M = N = 8, K = 128: the fp64 library product agrees with an exact
    # rational triple loop to within fp64 summation error
    W = gaussian_weights(128, 8, 0.02, 1)
    q, s, z = int4.rtn_quantize(W)
    w_hat = numerics.dtype_bits_to_f64(int4.dequant(q, s, z, "bf16"), "bf16")
    X = activations(8, 128, "bf16", 1).float().numpy().astype(np.float64)
    Y, A = product.reference(X, w_hat)
    Yx = _exact_product(X, w_hat)
    assert np.all(np.abs(Y - Yx) <= 128 * 2.0 ** -52 * A)


def test_non_square_orientation():
    # a transposed operand would not even have the right shape here, and the
    # one-hot rows of X must pick out rows of W_hat exactly
    K, N = 256, 24
    W = gaussian_weights(K, N, 0.02, 2)
    q, s, z = int4.rtn_quantize(W)
    w_hat = numerics.dtype_bits_to_f64(int4.dequant(q, s, z, "f16"), "f16")
    X = np.zeros((3, K))
    X[0, 5] = X[1, 130] = X[2, 255] = 1.0
    Y, _ = product.reference(X, w_hat)
    assert Y.shape == (3, N)
    assert np.array_equal(Y, w_hat[[5, 130, 255]])


def test_zero_when_codes_equal_zero_points():
    K, N = 256, 32
    rng = np.random.default_rng(0)
    z = rng.integers(0, 16, size=(K // 128, N)).astype(np.uint8)
    q = z[np.arange(K) // 128]
    s = numerics.to_f16(rng.uniform(1e-3, 1e-1, size=(K // 128, N)))
    w_hat = numerics.dtype_bits_to_f64(int4.dequant(q, s, z, "bf16"), "bf16")
    X = activations(4, K, "bf16", 0).float().numpy()
    Y, A = product.reference(X, w_hat)
    assert np.all(Y == 0)
    ok, m, f = product.within_tolerance(Y, Y, A)
    assert ok and m == 0 and f == 0


def test_tolerance_check_rejects_planted_errors():
    rng = np.random.default_rng(1)
    X = rng.standard_normal((4, 512))
    W = rng.standard_normal((512, 16)) * 0.02
    Y, A = product.reference(X, W)
    assert product.within_tolerance(Y, Y, A)[0]
    # bf16 rounding of the output alone stays inside the budget
    Yb = numerics.bf16_bits_to_f64(numerics.f32_to_bf16_bits(Y.astype(np.float32)))
    assert product.within_tolerance(Yb, Y, A)[0]
    # a dropped term (one K row missing) or a sign slip does not
    Yd, _ = product.reference(X[:, 1:], W[1:])
    assert not product.within_tolerance(Yd, Y, A)[0]
    assert not product.within_tolerance(-Y, Y, A)[0]


def test_byte_accounting_matches_pages():
    g = json.load(open(GOLDEN))
    wl = WORKLOADS["qwen32b"]
    per_layer = sum(accounting.int4_bytes(K, N) for K, N in wl.shapes)
    assert per_layer == 253_317_120
    stack = 64 * per_layer
    assert stack == 16_212_295_680
    fp16 = 64 * sum(accounting.fp16_bytes(K, N) for K, N in wl.shapes)
    # 16 GB at 4 bit vs 64 GB at fp16 (the pages count the whole model, the
    # stack here only its linears: agree to within a few percent)
    assert abs(stack / 1e9 - g["qwen32b_int4_weight_gb"]["value"]) / 16 < 0.05
    assert abs(fp16 / 1e9 - g["qwen32b_fp16_weight_gb"]["value"]) / 64 < 0.05
    ratio = accounting.bits_per_weight(5120, 5120) / 16
    assert abs(ratio - g["int4_fraction_of_fp16"]["value"]) < 0.02
    # Llama-7B: the decode-sweep shapes x 32 layers, plus 32000x4096
    # embedding and head, at fp16 is "about 14 GB"
    d = WORKLOADS["decode_sweep"]
    params = 32 * sum(K * N for K, N in d.shapes) + 2 * 32000 * 4096
    assert abs(2 * params / 1e9 - g["llama7b_fp16_gb"]["value"]) / 14 < 0.05
    assert g["int4_levels"]["value"] == 16
    assert g["group_size"]["value"] == 128


@pytest.mark.parametrize("name", list(WORKLOADS))
def test_workload_shapes_are_valid(name):
    wl = WORKLOADS[name]
    for K, N in wl.shapes:
        assert K % 128 == 0 and N % 8 == 0


# ------------------------------------------------------ fused SiLU * up
def test_silu_closed_forms():
    t = np.array([-50.0, -3.0, -1e-3, 0.0, 1e-3, 2.0, 60.0])
    s = product.silu(t)
    assert s[3] == 0.0
    # SiLU(t) - SiLU(-t) = t for every t (t sigma(t) + t (1 - sigma(t)))
    assert np.allclose(product.silu(t) - product.silu(-t), t, rtol=0, atol=1e-15)
    assert s[-1] == 60.0  # sigma(60) = 1 - 9e-27 rounds to 1 in fp64
    assert 0 > s[0] > -1e-19  # -50 sigma(-50) = -50 e^-50 ~ -9.6e-21
    assert abs(s[1] - (-3.0 / (1 + np.exp(3.0)))) < 1e-16
    # derivative: central differences
    h = 1e-6
    for v in (-4.0, -0.5, 0.0, 0.7, 3.0):
        fd = (product.silu(v + h) - product.silu(v - h)) / (2 * h)
        assert abs(fd - product.silu_grad(v)) < 1e-8
    assert product.silu_grad(0.0) == 0.5


def test_silu_mul_takes_gate_first_then_up():
    # K = 2, F = 3: gate columns are the first F, up the last F.  With X = [1, 0]
    # the products are the first row of W itself.
    W = np.array([[1.0, -2.0, 0.0, 3.0, 0.5, -1.0],
                  [9.0, 9.0, 9.0, 9.0, 9.0, 9.0]])
    act, A = product.silu_mul_reference(np.array([[1.0, 0.0]]), W)
    sg = product.silu(np.array([1.0, -2.0, 0.0]))
    assert np.allclose(act[0], sg * np.array([3.0, 0.5, -1.0]), rtol=1e-15, atol=0)
    # normaliser: |SiLU'(g)| |u| A_g + |SiLU(g)| A_u with A = |x| |w|
    Ag = np.array([1.0, 2.0, 0.0])
    Au = np.array([3.0, 0.5, 1.0])
    want = np.abs(product.silu_grad(np.array([1.0, -2.0, 0.0]))) * np.abs([3.0, 0.5, -1.0]) * Ag + np.abs(sg) * Au
    assert np.allclose(A[0], want, rtol=1e-15, atol=0)
