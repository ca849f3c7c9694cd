"""GPU dequantization and quantization, bit-exact against the oracle."""

import numpy as np
import pytest
import torch

import bit_weight_only_wise_b300 as w4
from oracle import int4, nf4
from synth import WORKLOADS, act_order_g_idx, activations, gaussian_weights, student_t_weights, weights_for

import gpu_util
from gpu_util import bits, dev, to_dev, to_dev_u32

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_dequant_exhaustive_codes_zeros_scales(dtype):
    # every code q (0..15) x every zero point z (0..15) x every positive finite
    # fp16 scale, plus negative scales: the fast in-register routines must hit
    # RNE((q - z) * s) bit for bit
    s_bits = np.concatenate([np.arange(1, 0x7C00, dtype=np.uint16),
                             (np.arange(1, 0x7C00, 61, dtype=np.uint16) | 0x8000)]).astype(np.uint16)
    S = s_bits.size
    N = 16 * S
    N += (-N) % 8
    K = 128
    q = np.tile((np.arange(K) % 16).astype(np.uint8)[:, None], (1, N))
    z = (np.arange(N) % 16).astype(np.uint8)[None, :]
    sc = np.resize(np.repeat(s_bits, 16), N).view(np.float16)[None, :]
    got = bits(w4.dequant(to_dev_u32(int4.pack_along_k(q)), to_dev(sc), to_dev_u32(int4.pack_zeros(z)),
                          dtype=torch.float16 if dtype == "f16" else torch.bfloat16))
    want = int4.dequant(q, sc, z, dtype)
    bad = np.nonzero(got != want)
    assert bad[0].size == 0, f"{bad[0].size} mismatches, first at {bad[0][0]},{bad[1][0]}"


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("act", [False, True])
def test_dequant_random_checkpoint(dtype, act):
    K, N = 2048, 1032  # N not a multiple of the 256-column tile
    W = student_t_weights(K, N, 5, 0.01, 4)
    g_idx = act_order_g_idx(K, 128, 4) if act else None
    qw, sc, qz, q, z = int4.quantize_packed(W, 128, g_idx)
    got = bits(w4.dequant(to_dev_u32(qw), to_dev(sc), to_dev_u32(qz), None if g_idx is None else to_dev(g_idx),
                          dtype=torch.float16 if dtype == "f16" else torch.bfloat16))
    assert np.array_equal(got, int4.dequant(q, sc, z, dtype, 128, g_idx))


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_nf4_dequant(dtype):
    K, N = 1024, 520
    W = gaussian_weights(K, N, 0.02, 6)
    cb = nf4.codebook()
    qw, am, codes = nf4.nf4_quantize_packed(W, cb)
    got = bits(w4.nf4_dequant(to_dev_u32(qw), to_dev(am), to_dev(cb),
                              dtype=torch.float16 if dtype == "f16" else torch.bfloat16))
    assert np.array_equal(got, nf4.nf4_dequant(codes, am, cb, dtype))


@pytest.mark.parametrize("name", ["single_linear", "decode_sweep", "act_order", "qwen32b"])
def test_rtn_quantize_matches_oracle(name):
    wl = WORKLOADS[name]
    K, N = 1024, 776
    W = weights_for(wl, K, N, 8)
    qw_o, sc_o, qz_o, _, _ = int4.quantize_packed(W)
    qw, sc, qz = w4.quantize(to_dev(W))
    assert np.array_equal(qw.cpu().numpy().view(np.uint32), qw_o)
    assert np.array_equal(sc.cpu().numpy().view(np.uint16), sc_o.view(np.uint16))
    assert np.array_equal(qz.cpu().numpy().view(np.uint32), qz_o)


def test_rtn_quantize_degenerate_groups():
    # all-zero group (scale 0 -> 1), all-positive and all-negative columns
    K, N = 256, 64
    W = gaussian_weights(K, N, 0.02, 1)
    W[:128, 0] = 0.0
    W[:, 1] = np.abs(W[:, 1])
    W[:, 2] = -np.abs(W[:, 2])
    W[5, 3] = 1e-30  # tiny
    qw_o, sc_o, qz_o, _, _ = int4.quantize_packed(W)
    qw, sc, qz = w4.quantize(to_dev(W))
    assert np.array_equal(qw.cpu().numpy().view(np.uint32), qw_o)
    assert np.array_equal(sc.cpu().numpy().view(np.uint16), sc_o.view(np.uint16))
    assert np.array_equal(qz.cpu().numpy().view(np.uint32), qz_o)


def test_nf4_quantize_matches_oracle():
    K, N = 1024, 520
    W = gaussian_weights(K, N, 0.02, 2)
    W[:64, 0] = 0.0  # all-zero block
    cb = nf4.codebook()
    qw_o, am_o, _ = nf4.nf4_quantize_packed(W, cb)
    qw, am = w4.nf4_quantize(to_dev(W), to_dev(cb))
    assert np.array_equal(am.cpu().numpy(), am_o)
    assert np.array_equal(qw.cpu().numpy().view(np.uint32), qw_o)


def test_binding_codebook_matches_oracle_codebook():
    # the library builds its default table independently of the oracle (its own
    # Newton iteration on libm's erfc); the two fp32 tables are bit-identical
    got = w4.nf4_codebook(dev()).cpu().numpy()
    want = nf4.codebook()
    assert np.array_equal(got.view(np.uint32), want.view(np.uint32))


def test_nf4_null_codebook_is_the_builtin_table():
    # a NULL table in the C calls means the built-in one: quantize, dequantize
    # and both product kernels give bit-identical results with NULL and with
    # the oracle's table passed explicitly
    K, N = 512, 264
    W = gaussian_weights(K, N, 0.02, 12)
    cb = nf4.codebook()
    Wd, cbd = to_dev(W), to_dev(cb)
    qw0, am0 = w4.nf4_quantize(Wd, None)
    qw1, am1 = w4.nf4_quantize(Wd, cbd)
    assert torch.equal(qw0, qw1) and torch.equal(am0, am1)
    qw_o, am_o, codes = nf4.nf4_quantize_packed(W, cb)
    assert np.array_equal(qw0.cpu().numpy().view(np.uint32), qw_o)
    for dt in ("bf16", "f16"):
        d0 = w4.nf4_dequant(qw0, am0, None, dtype=gpu_util.TDT[dt])
        assert np.array_equal(bits(d0), nf4.nf4_dequant(codes, am_o, cb, dt))
        for M in (3, 40):
            X = activations(M, K, dt, 5).to(dev())
            y0 = w4.nf4_gemm(X, qw0, am0, None)
            y1 = w4.nf4_gemm(X, qw0, am0, cbd)
            torch.cuda.synchronize()
            assert torch.equal(y0, y1)
