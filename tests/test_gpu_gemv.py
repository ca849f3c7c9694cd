"""Decode-shape products (M <= 16) through the C ABI against the oracle."""

import numpy as np
import pytest
import torch

import bit_weight_only_wise_b300 as w4
from oracle import int4, nf4, numerics
from synth import WORKLOADS, act_order_g_idx, activations, gaussian_weights, student_t_weights, weights_for

from gpu_util import (TDT, assert_close, bits, int4_expected, nf4_expected, sample_columns, to_dev, to_dev_u32,
                      to_f64)

pytestmark = pytest.mark.gpu


def _int4_dev(W, g_idx=None):
    qw, sc, qz, q, z = int4.quantize_packed(W, 128, g_idx)
    return (to_dev_u32(qw), to_dev(sc), to_dev_u32(qz), None if g_idx is None else to_dev(g_idx)), (q, sc, z)


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("M", [1, 2, 3, 7, 8, 9, 15, 16])
@pytest.mark.parametrize("act", [False, True])
def test_gemv_small_all_columns(dtype, M, act):
    # several column tiles plus a ragged tail, several K groups, every output checked
    K, N = 1536, 776
    W = student_t_weights(K, N, 5, 0.01, M) if act else gaussian_weights(K, N, 0.02, M)
    g_idx = act_order_g_idx(K, 128, M) if act else None
    dev_t, _ = _int4_dev(W, g_idx)
    X = activations(M, K, dtype, M)
    Y = w4.gemv(X.cuda(), *dev_t[:3], g_idx=dev_t[3])
    torch.cuda.synchronize()
    Y_ref, A = int4_expected(W, X.double().numpy(), dtype, None, g_idx)
    assert_close(to_f64(Y), Y_ref, A, f"M={M} {dtype} act={act}")


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("act", [False, True])
def test_gemv_one_hot_rows_are_exact(dtype, act):
    # X = rows of the identity: each Y row must equal a row of W_hat bit for bit
    # (one product by 1.0 per output, then an exact rounding), which pins the
    # kernel's indexing of rows, columns, groups and the act-order map exactly
    K, N = 1024, 520
    W = gaussian_weights(K, N, 0.02, 3)
    g_idx = act_order_g_idx(K, 128, 3) if act else None
    dev_t, (q, sc, z) = _int4_dev(W, g_idx)
    rows = np.array([0, 1, 7, 8, 127, 128, 500, 511, 512, 640, 777, 895, 1000, 1016, 1022, 1023])
    X = torch.zeros((16, K), dtype=TDT[dtype])
    X[torch.arange(16), torch.from_numpy(rows)] = 1.0
    Y = w4.gemv(X.cuda(), *dev_t[:3], g_idx=dev_t[3])
    w_hat = int4.dequant(q, sc, z, dtype, 128, g_idx)
    assert np.array_equal(bits(Y), w_hat[rows])


def test_gemv_zero_when_codes_equal_zero_points():
    K, N = 512, 264
    rng = np.random.default_rng(0)
    z = rng.integers(0, 16, size=(K // 128, N)).astype(np.uint8)
    q = z[np.arange(K) // 128]
    sc = numerics.to_f16(rng.uniform(1e-3, 0.1, size=(K // 128, N)))
    X = activations(5, K, "bf16", 1).cuda()
    Y = w4.gemv(X, to_dev_u32(int4.pack_along_k(q)), to_dev(sc), to_dev_u32(int4.pack_zeros(z)))
    assert torch.count_nonzero(Y.float()).item() == 0


def test_gemv_deterministic_and_workspace_reuse():
    K, N = 4096, 4096
    W = gaussian_weights(K, N, 0.02, 0)
    dev_t, _ = _int4_dev(W)
    X = activations(16, K, "f16", 0).cuda()
    Y1 = w4.gemv(X, *dev_t[:3])
    Y2 = w4.gemv(X, *dev_t[:3])
    Y3 = w4.gemv(X[:3].contiguous(), *dev_t[:3])  # another M (and plan) through the same workspace
    Y4 = w4.gemv(X, *dev_t[:3])
    assert torch.equal(Y1.view(torch.int16), Y2.view(torch.int16))
    assert torch.equal(Y1.view(torch.int16), Y4.view(torch.int16))
    # a different M may split K differently: equal to within rounding
    assert torch.allclose(Y3.float(), Y1[:3].float(), rtol=1e-2, atol=1e-2)
    Y5 = w4.gemv(X[:3].contiguous(), *dev_t[:3])
    assert torch.equal(Y3.view(torch.int16), Y5.view(torch.int16))


def test_gemv_batch_equals_single_calls():
    # one w4a16_gemv_batch call over mixed items (dtypes, M, act-order,
    # symmetric groups of 64, an empty item) computes each product exactly as
    # its own w4a16_gemv call does, through one shared workspace, twice
    items, singles = [], []
    cases = [(1, 1024, 776, "bf16", False, 128, False), (5, 2048, 512, "f16", False, 128, False),
             (16, 1536, 264, "bf16", True, 128, False), (3, 1024, 520, "f16", False, 64, True),
             (0, 512, 256, "bf16", False, 128, False)]
    for i, (M, K, N, dtype, act, g, sym) in enumerate(cases):
        W = gaussian_weights(K, N, 0.02, 50 + i)
        g_idx = act_order_g_idx(K, g, i) if act else None
        if sym:
            q, sc = int4.rtn_quantize_sym(W, g)
            qw, qz = to_dev_u32(int4.pack_along_k(q)), None
        else:
            qwp, scp, qzp, _, _ = int4.quantize_packed(W, g, g_idx)
            qw, sc, qz = to_dev_u32(qwp), scp, to_dev_u32(qzp)
        gi = None if g_idx is None else to_dev(g_idx)
        X = activations(max(M, 1), K, dtype, i).cuda()[:M].contiguous()
        Y = torch.full((M, N), 7.0, dtype=TDT[dtype], device="cuda")
        items.append(dict(X=X, qweight=qw, scales=to_dev(sc), qzeros=qz, Y=Y, g_idx=gi, group_size=g))
        singles.append(w4.gemv(X, qw, to_dev(sc), qz, g_idx=gi, group_size=g) if M else None)
    batch = w4.GemvBatch(items)
    for _ in range(2):
        for it in items:
            it["Y"].fill_(7.0)
        batch()
        torch.cuda.synchronize()
        for it, Y1 in zip(items, singles):
            if Y1 is not None:
                assert torch.equal(it["Y"].view(torch.int16), Y1.view(torch.int16))


def test_gemm_entry_dispatches_small_m_to_gemv():
    K, N = 1024, 512
    W = gaussian_weights(K, N, 0.02, 1)
    dev_t, _ = _int4_dev(W)
    X = activations(16, K, "bf16", 1).cuda()
    assert torch.equal(w4.gemm(X, *dev_t[:3]).view(torch.int16), w4.gemv(X, *dev_t[:3]).view(torch.int16))


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("M", [1, 5, 16])
def test_nf4_gemv_small(dtype, M):
    K, N = 1024 + 64, 520  # K not a multiple of 128: a half chunk at the end
    W = gaussian_weights(K, N, 0.02, 7)
    cb = nf4.codebook()
    qw, am, _ = nf4.nf4_quantize_packed(W, cb)
    X = activations(M, K, dtype, 2)
    Y = w4.nf4_gemm(X.cuda(), to_dev_u32(qw), to_dev(am), to_dev(cb))
    Y_ref, A = nf4_expected(W, X.double().numpy(), cb, dtype)
    assert_close(to_f64(Y), Y_ref, A, f"nf4 M={M} {dtype}")


def _full_size_cases():
    out = []
    for name in ("single_linear", "decode_sweep", "act_order", "qwen32b"):
        wl = WORKLOADS[name]
        for (K, N) in wl.shapes:
            Ms = [m for m in wl.Ms if m <= 16]
            if Ms:
                out.append(pytest.param(name, K, N, tuple(Ms), id=f"{name}-{K}x{N}"))
    return out


@pytest.mark.parametrize("name,K,N,Ms", _full_size_cases())
def test_gemv_full_size_sampled_columns(name, K, N, Ms):
    # the workloads' full shapes, launched exactly as the bench launches them;
    # the oracle recomputes a sample of output columns (first, last, random)
    wl = WORKLOADS[name]
    W = weights_for(wl, K, N, 0)
    g_idx = act_order_g_idx(K, 128, 0) if wl.act_order else None
    cols = sample_columns(N)
    if g_idx is None:
        qw, sc, qz = w4.quantize(to_dev(W))
        qw_o, sc_o, qz_o, _, _ = int4.quantize_packed(W[:, cols])
        assert np.array_equal(qw.cpu().numpy().view(np.uint32)[:, cols], qw_o)
        gi = None
    else:
        (qw, sc, qz, gi), _ = _int4_dev(W, g_idx)
    for M in Ms:
        X = activations(M, K, wl.dtype, M)
        Y = w4.gemm(X.cuda(), qw, sc, qz, g_idx=gi)
        Y_ref, A = int4_expected(W, X.double().numpy(), wl.dtype, cols, g_idx)
        assert_close(to_f64(Y)[:, cols], Y_ref, A, f"{name} {K}x{N} M={M}")


def test_nf4_gemv_full_size_sampled_columns():
    wl = WORKLOADS["nf4"]
    K, N = wl.shapes[0]
    W = weights_for(wl, K, N, 0)
    cb = nf4.codebook()
    qw, am = w4.nf4_quantize(to_dev(W), to_dev(cb))
    cols = sample_columns(N)
    X = activations(1, K, "bf16", 1)
    Y = w4.nf4_gemm(X.cuda(), qw, am, to_dev(cb))
    Y_ref, A = nf4_expected(W, X.double().numpy(), cb, "bf16", cols)
    assert_close(to_f64(Y)[:, cols], Y_ref, A, "nf4 full M=1")


def test_gemv_workspace_shared_across_shapes():
    # one cached workspace serves calls whose split-K plans differ; a call must
    # not find stale partial sums where its tickets live
    cases = [(1024, 512), (2048, 3072), (1024, 22016), (4096, 776), (1024, 512)]
    outs = []
    for K, N in cases:
        W = gaussian_weights(K, N, 0.02, K + N)
        dev_t, _ = _int4_dev(W)
        X = activations(3, K, "bf16", 5)
        Y = w4.gemv(X.cuda(), *dev_t[:3])
        Y_ref, A = int4_expected(W, X.double().numpy(), "bf16")
        assert_close(to_f64(Y), Y_ref, A, f"{K}x{N}")
        outs.append(Y)
    assert torch.equal(outs[0].view(torch.int16), outs[-1].view(torch.int16))


@pytest.mark.parametrize("M", [4, 64])
def test_act_order_entry_out_of_range_is_reported(M):
    # a g_idx entry outside [0, K/128) is clamped by the kernels (nothing
    # outside the scale and zero arrays is read) and reported as INVALID_ARG
    from synth import act_order_g_idx

    K, N = 512, 256
    W = gaussian_weights(K, N, 0.02, 5)
    g_idx = act_order_g_idx(K, 128, 5)
    qw, sc, qz, _, _ = int4.quantize_packed(W, 128, g_idx)
    bad = g_idx.copy()
    bad[5], bad[300] = K // 128 + 7, -3
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    w4.gemm(activations(M, K, "bf16", 1).cuda(), to_dev_u32(qw), to_dev(sc), to_dev_u32(qz), g_idx=to_dev(bad),
            dev_status=st)
    torch.cuda.synchronize()
    assert st.item() == w4.ERR_INVALID_ARG
    st.zero_()
    w4.gemm(activations(M, K, "bf16", 1).cuda(), to_dev_u32(qw), to_dev(sc), to_dev_u32(qz), g_idx=to_dev(g_idx),
            dev_status=st)
    torch.cuda.synchronize()
    assert st.item() == 0


def _assert_rows_exact(got, want, dtype):
    # bit for bit, except that a weight of -0 comes out of the product as +0
    # (the exact sum -0 + 0*w + ... is +0 in IEEE arithmetic)
    gv, wv = numerics.dtype_bits_to_f64(got, dtype), numerics.dtype_bits_to_f64(want, dtype)
    bad = np.nonzero((got != want) & ~((gv == 0) & (wv == 0)))
    assert bad[0].size == 0, f"{bad[0].size} mismatches, first at {bad[0][0]},{bad[1][0]}"


def _exhaustive_scale_checkpoint(dtype):
    # every code q (0..15) x every zero point (0..15) x every positive finite
    # fp16 scale and a spread of negative ones, in one 128-row group.  For
    # fp16 outputs the scales stop where 15 * s would overflow: an infinite
    # weight times a zero activation in another row would turn the whole
    # column's sum into NaN.
    top = 0x7C00 if dtype == "bf16" else 0x6C43  # 4366 * 15 < 65504
    s_bits = np.concatenate([np.arange(1, top, dtype=np.uint16),
                             (np.arange(1, top, 61, dtype=np.uint16) | 0x8000)]).astype(np.uint16)
    N = 16 * s_bits.size
    N += (-N) % 8
    K = 128
    q = np.tile((np.arange(K) % 16).astype(np.uint8)[:, None], (1, N))
    z = (np.arange(N) % 16).astype(np.uint8)[None, :]
    sc = np.resize(np.repeat(s_bits, 16), N).view(np.float16)[None, :]
    return q, sc, z


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("M", [16, 64])
def test_fused_dequant_exact_over_every_scale(dtype, M):
    # one-hot activation rows pick weight rows out of the product, so the
    # decode kernel (M=16) and the tensor-core kernel (M=64) must reproduce
    # RNE((q - z) * s) bit for bit on every code, zero point and fp16 scale
    q, sc, z = _exhaustive_scale_checkpoint(dtype)
    K, N = q.shape
    rows = np.arange(M) % K
    X = torch.zeros((M, K), dtype=TDT[dtype])
    X[torch.arange(M), torch.from_numpy(rows)] = 1.0
    Y = w4.gemm(X.cuda(), to_dev_u32(int4.pack_along_k(q)), to_dev(sc), to_dev_u32(int4.pack_zeros(z)))
    want = int4.dequant(q, sc, z, dtype)[rows]
    _assert_rows_exact(bits(Y), want, dtype)


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("M", [16, 64])
def test_fused_nf4_dequant_exact_over_wide_absmax(dtype, M):
    # NF4 through the fused kernels, one-hot rows: RNE(fl32(C[q] * absmax))
    # bit for bit for every code and absmax values over many binades
    K = 128
    rng = np.random.default_rng(5)
    cb = nf4.codebook()
    N = 8192
    hi = 40 if dtype == "bf16" else 15  # fp16: keep every weight finite (see above)
    am = (2.0 ** rng.uniform(-40, hi, size=(K // 64, N))).astype(np.float32)
    codes = np.tile((np.arange(K) % 16).astype(np.uint8)[:, None], (1, N))
    codes = (codes + np.arange(N)[None, :]) % 16
    rows = np.arange(M) % K
    X = torch.zeros((M, K), dtype=TDT[dtype])
    X[torch.arange(M), torch.from_numpy(rows)] = 1.0
    Y = w4.nf4_gemm(X.cuda(), to_dev_u32(int4.pack_along_k(codes.astype(np.uint8))), to_dev(am), to_dev(cb))
    want = nf4.nf4_dequant(codes.astype(np.uint8), am, cb, dtype)[rows]
    _assert_rows_exact(bits(Y), want, dtype)
