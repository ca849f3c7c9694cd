"""Pins for the oracle's AWQ layout (codes packed along N in AWQ's column
order) and its re-arrangement into this library's layout."""

import numpy as np

from oracle import awq, int4
from synth import gaussian_weights


def test_awq_word_golden():
    # column 8c + ORDER[j] lands in bits 4j..4j+3 with ORDER = (0,2,4,6,1,3,5,7):
    # columns holding their own index 0..7 pack to 0x75316420, and 1..8 to 0x86427531
    v = np.arange(8, dtype=np.uint8).reshape(1, 8)
    assert awq.pack_awq(v)[0, 0] == 0x75316420
    assert awq.pack_awq(v + 1)[0, 0] == 0x86427531


def test_awq_roundtrip_exhaustive_positions():
    v = np.zeros((16, 64), dtype=np.uint8)
    for val in range(16):
        for col in range(64):
            v[val, col] = (val + col) % 16
    assert np.array_equal(awq.unpack_awq(awq.pack_awq(v)), v)
    rng = np.random.default_rng(1)
    words = rng.integers(0, 2 ** 32, size=(9, 5), dtype=np.uint64).astype(np.uint32)
    assert np.array_equal(awq.pack_awq(awq.unpack_awq(words)), words)


def test_awq_to_library_layout_is_the_same_checkpoint():
    # the same quantized weights in both layouts dequantize to the same values
    K, N = 512, 40
    W = gaussian_weights(K, N, 0.02, 9)
    qa, sc, za, q, z = awq.awq_checkpoint(W)
    assert qa.shape == (K, N // 8) and za.shape == (K // 128, N // 8)
    qw, qz = awq.to_library_layout(qa, za)
    assert np.array_equal(qw, int4.pack_along_k(q))
    assert np.array_equal(qz, int4.pack_zeros(z))
    assert np.array_equal(int4.unpack_along_k(qw), q) and np.array_equal(int4.unpack_zeros(qz), z)
    # a layout that is not the identity: AWQ's word differs from the natural one
    assert not np.array_equal(qa[:, :1], int4.pack_zeros(q[:, :8]))
