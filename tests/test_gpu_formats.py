"""Group sizes, symmetric weights, act-order through the decode kernel's table,
and NF4 with double-quantized absmax: every product through the C ABI against
the oracle, every dequantized value bit for bit."""

import numpy as np
import pytest
import torch

import bit_weight_only_wise_b300 as w4
from oracle import int4, nf4, numerics, product
from synth import act_order_g_idx, activations, gaussian_weights, student_t_weights

from gpu_util import TDT, assert_close, bits, to_dev, to_dev_u32, to_f64

pytestmark = pytest.mark.gpu


def _quantize(W, g, sym, g_idx=None):
    """Oracle quantization -> (device tensors, (q, scales, zeros))."""
    if sym:
        q, sc = int4.rtn_quantize_sym(W, g, g_idx)
        z = int4.sym_zeros(*sc.shape)
        qz = None
    else:
        q, sc, z = int4.rtn_quantize(W, g, g_idx)
        qz = to_dev_u32(int4.pack_zeros(z))
    dev_t = (to_dev_u32(int4.pack_along_k(q)), to_dev(sc), qz, None if g_idx is None else to_dev(g_idx))
    return dev_t, (q, sc, z)


def _expected(q, sc, z, g, dtype, X, g_idx=None):
    w_hat = numerics.dtype_bits_to_f64(int4.dequant(q, sc, z, dtype, g, g_idx), dtype)
    return product.reference(X.double().numpy(), w_hat)


# ------------------------------------------------------------- group sizes
# (K, g): groups of 32 and 64 (several per 128-row unit, and K ending part way
# through a unit), a multiple of 128, and one group for all of K (per channel,
# also with K not a multiple of 128)
GROUPS = [(1056, 32), (1088, 64), (1024, 256), (1024, 1024), (1000, 1000)]


@pytest.mark.parametrize("K,g", GROUPS)
@pytest.mark.parametrize("sym", [False, True])
@pytest.mark.parametrize("M", [1, 5, 16, 40, 200])
def test_group_sizes_and_symmetric_products(K, g, sym, M):
    N = 520
    dtype = "bf16" if (M + g + int(sym)) % 2 else "f16"  # both dtypes on every (K, g, M)
    W = gaussian_weights(K, N, 0.02, K + g + M)
    dev_t, (q, sc, z) = _quantize(W, g, sym)
    X = activations(M, K, dtype, M)
    Y = w4.gemm(X.cuda(), *dev_t[:3], group_size=g)
    torch.cuda.synchronize()
    Y_ref, A = _expected(q, sc, z, g, dtype, X)
    assert_close(to_f64(Y), Y_ref, A, f"K={K} g={g} sym={sym} M={M} {dtype}")


@pytest.mark.parametrize("g", [32, 64, 1024])
@pytest.mark.parametrize("sym", [False, True])
@pytest.mark.parametrize("M", [16, 32])
@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_group_sizes_one_hot_rows_are_exact(g, sym, M, dtype):
    # one-hot rows reproduce rows of W_hat bit for bit, on both kernels (M = 16:
    # decode, M = 32: tensor cores), pinning which group each row reads (rows
    # 31 and 32 straddle a boundary between groups of 32)
    K, N = 1024, 264
    W = student_t_weights(K, N, 5, 0.01, g)
    dev_t, (q, sc, z) = _quantize(W, g, sym)
    rng = np.random.default_rng(g + M)
    rows = np.sort(rng.choice(K, size=M, replace=False))
    rows[:4] = [0, 31, 32, 1023]
    X = torch.zeros((M, K), dtype=TDT[dtype])
    X[torch.arange(M), torch.from_numpy(rows)] = 1.0
    Y = w4.gemm(X.cuda(), *dev_t[:3], group_size=g)
    w_hat = int4.dequant(q, sc, z, dtype, g)
    assert np.array_equal(bits(Y), w_hat[rows])


@pytest.mark.parametrize("K,g", GROUPS)
@pytest.mark.parametrize("sym", [False, True])
def test_quantize_and_dequant_match_oracle(K, g, sym):
    N = 264
    W = student_t_weights(K, N, 5, 0.01, g + 1)
    W[:, 3] = 0.0  # an all-zero column: scale 1, code at the zero point
    qw, sc, qz = w4.quantize(to_dev(W), group_size=g, symmetric=sym)
    if sym:
        q_o, sc_o = int4.rtn_quantize_sym(W, g)
        z_o = int4.sym_zeros(*sc_o.shape)
        assert qz is None
    else:
        q_o, sc_o, z_o = int4.rtn_quantize(W, g)
        assert np.array_equal(qz.cpu().numpy().view(np.uint32), int4.pack_zeros(z_o))
    assert np.array_equal(qw.cpu().numpy().view(np.uint32), int4.pack_along_k(q_o))
    assert np.array_equal(sc.cpu().numpy().view(np.uint16), sc_o.view(np.uint16))
    for dt in ("f16", "bf16"):
        d = w4.dequant(qw, sc, qz, dtype=TDT[dt], group_size=g)
        assert np.array_equal(bits(d), int4.dequant(q_o, sc_o, z_o, dt, g))


def test_group_sizes_full_size_decode():
    # Llama-7B-shaped gate+up at M = 1 with groups of 64 and 32, and symmetric
    # g = 128: sampled columns against the oracle
    K, N = 4096, 11008
    W = gaussian_weights(K, N, 0.02, 7)
    cols = np.unique(np.concatenate([np.arange(8), np.arange(N - 8, N),
                                     np.random.default_rng(1).choice(N, 128, replace=False)]))
    X = activations(1, K, "bf16", 7)
    for g, sym in ((64, False), (32, False), (128, True)):
        dev_t, _ = _quantize(W, g, sym)
        Y = w4.gemm(X.cuda(), *dev_t[:3], group_size=g)
        torch.cuda.synchronize()
        # the statistics are per column, so the sampled columns quantize alone
        _, (q, sc, z) = _quantize(W[:, cols], g, sym)
        Y_ref, A = _expected(q, sc, z, g, "bf16", X)
        assert_close(to_f64(Y)[:, cols], Y_ref, A, f"g={g} sym={sym}")


def test_unsupported_group_sizes_are_rejected():
    X = torch.zeros((4, 384), dtype=torch.bfloat16, device="cuda")
    qw = torch.zeros((48, 64), dtype=torch.int32, device="cuda")
    sc = torch.zeros((8, 64), dtype=torch.float16, device="cuda")
    with pytest.raises(w4.W4A16Error) as e:
        w4.gemm(X, qw, sc, None, group_size=48)
    assert e.value.status == w4.ERR_UNSUPPORTED


# ------------------------------------------------- act-order (stored map)
@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("M", [1, 3, 9, 16])
@pytest.mark.parametrize("g,sym", [(128, False), (64, False), (128, True)])
def test_act_order_table_kernel(dtype, M, g, sym):
    # the decode kernel's shared-memory table of every group: several column
    # blocks (one CTA crosses into the next block and reloads its table) and a
    # ragged tail, every output checked
    K, N = 2048, 776
    W = student_t_weights(K, N, 5, 0.01, M + g)
    g_idx = act_order_g_idx(K, g, M + g)
    dev_t, (q, sc, z) = _quantize(W, g, sym, g_idx)
    X = activations(M, K, dtype, M)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    Y = w4.gemv(X.cuda(), *dev_t[:3], g_idx=dev_t[3], group_size=g, dev_status=st)
    torch.cuda.synchronize()
    assert st.item() == 0
    Y_ref, A = _expected(q, sc, z, g, dtype, X, g_idx)
    assert_close(to_f64(Y), Y_ref, A, f"act-order M={M} g={g} sym={sym} {dtype}")


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_act_order_table_kernel_one_hot_exact(dtype):
    K, N = 1024, 520
    W = gaussian_weights(K, N, 0.02, 5)
    g_idx = act_order_g_idx(K, 128, 5)
    dev_t, (q, sc, z) = _quantize(W, 128, False, g_idx)
    rows = np.array([0, 1, 2, 3, 4, 5, 6, 7, 128, 255, 511, 512, 800, 1015, 1022, 1023])
    X = torch.zeros((16, K), dtype=TDT[dtype])
    X[torch.arange(16), torch.from_numpy(rows)] = 1.0
    Y = w4.gemv(X.cuda(), *dev_t[:3], g_idx=dev_t[3])
    assert np.array_equal(bits(Y), int4.dequant(q, sc, z, dtype, 128, g_idx)[rows])


def test_act_order_many_groups_fallback():
    # 384 groups (K = 12288 in groups of 32) do not fit the decode kernel's
    # table; the global-lookup kernel serves them
    K, N, g = 12288, 264, 32
    W = student_t_weights(K, N, 5, 0.01, 3)
    g_idx = act_order_g_idx(K, g, 3)
    dev_t, (q, sc, z) = _quantize(W, g, False, g_idx)
    X = activations(2, K, "bf16", 3)
    Y = w4.gemv(X.cuda(), *dev_t[:3], g_idx=dev_t[3], group_size=g)
    torch.cuda.synchronize()
    Y_ref, A = _expected(q, sc, z, g, "bf16", X, g_idx)
    assert_close(to_f64(Y), Y_ref, A, "act-order fallback")


def test_act_order_table_out_of_range_reported():
    K, N = 1024, 264
    W = gaussian_weights(K, N, 0.02, 1)
    g_idx = act_order_g_idx(K, 128, 1)
    dev_t, _ = _quantize(W, 128, False, g_idx)
    bad = g_idx.copy()
    bad[5] = 8  # one past the last group
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    X = activations(1, K, "bf16", 1).cuda()
    w4.gemv(X, *dev_t[:3], g_idx=to_dev(bad), dev_status=st)
    torch.cuda.synchronize()
    assert st.item() == w4.ERR_INVALID_ARG


# ---------------------------------------------- NF4 double quantization
def _nf4dq(W):
    cb = nf4.codebook()
    codes, am = nf4.nf4_quantize(W, cb)
    am_q, s2 = nf4.double_quantize_absmax(am)
    am_hat = nf4.absmax_from_double_quant(am_q, s2)
    return cb, codes, am, am_q, s2, am_hat


def test_double_quantize_matches_oracle():
    K, N = 2048, 600  # three second-level blocks per row, the last one ragged
    W = gaussian_weights(K, N, 0.02, 4)
    W[:64, 0:256] = 0.0  # an all-zero second-level block
    _, _, am, am_q, s2, _ = _nf4dq(W)
    q_d, s2_d = w4.nf4_double_quantize(to_dev(am))
    assert np.array_equal(q_d.cpu().numpy(), am_q)
    assert np.array_equal(s2_d.cpu().numpy().view(np.uint32), s2.view(np.uint32))


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_nf4dq_dequant_bit_exact(dtype):
    K, N = 1024, 520
    W = gaussian_weights(K, N, 0.02, 6)
    cb, codes, _, am_q, s2, am_hat = _nf4dq(W)
    d = w4.nf4dq_dequant(to_dev_u32(int4.pack_along_k(codes)), to_dev(am_q), to_dev(s2), None, dtype=TDT[dtype])
    assert np.array_equal(bits(d), nf4.nf4_dequant(codes, am_hat, cb, dtype))


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("M", [1, 7, 16, 40, 300])
def test_nf4dq_products(dtype, M):
    K, N = 1536, 776
    W = gaussian_weights(K, N, 0.02, M)
    cb, codes, _, am_q, s2, am_hat = _nf4dq(W)
    X = activations(M, K, dtype, M)
    Y = w4.nf4dq_gemm(X.cuda(), to_dev_u32(int4.pack_along_k(codes)), to_dev(am_q), to_dev(s2), to_dev(cb))
    torch.cuda.synchronize()
    w_hat = numerics.dtype_bits_to_f64(nf4.nf4_dequant(codes, am_hat, cb, dtype), dtype)
    Y_ref, A = product.reference(X.double().numpy(), w_hat)
    assert_close(to_f64(Y), Y_ref, A, f"nf4dq M={M} {dtype}")


@pytest.mark.parametrize("M", [16, 32])
def test_nf4dq_one_hot_exact(M):
    K, N = 1024, 264
    W = student_t_weights(K, N, 5, 0.01, 2)
    cb, codes, _, am_q, s2, am_hat = _nf4dq(W)
    rows = np.sort(np.random.default_rng(M).choice(K, size=M, replace=False))
    X = torch.zeros((M, K), dtype=torch.bfloat16)
    X[torch.arange(M), torch.from_numpy(rows)] = 1.0
    Y = w4.nf4dq_gemm(X.cuda(), to_dev_u32(int4.pack_along_k(codes)), to_dev(am_q), to_dev(s2), None)
    assert np.array_equal(bits(Y), nf4.nf4_dequant(codes, am_hat, cb, "bf16")[rows])


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_nf4dq_split_tail_all_outputs(dtype):
    # the tensor-core kernel on 150 column tiles (a full wave of whole tiles
    # and two tiles split along K) with double-quantized absmax converted per
    # block by the dequant warps; every output
    M, K, N = 40, 2048, 150 * 128
    W = gaussian_weights(K, N, 0.02, 12)
    cb, codes, _, am_q, s2, am_hat = _nf4dq(W)
    X = activations(M, K, dtype, 12)
    Y = w4.nf4dq_gemm(X.cuda(), to_dev_u32(int4.pack_along_k(codes)), to_dev(am_q), to_dev(s2), to_dev(cb))
    torch.cuda.synchronize()
    w_hat = numerics.dtype_bits_to_f64(nf4.nf4_dequant(codes, am_hat, cb, dtype), dtype)
    Y_ref, A = product.reference(X.double().numpy(), w_hat)
    assert_close(to_f64(Y), Y_ref, A, f"nf4dq split tail {dtype}")


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("sym", [False, True])
def test_groups_of_32_split_tail_all_outputs(dtype, sym):
    # groups of 32 rows (the tensor-core kernel's two-halves format, each
    # 64-row block carrying two groups) on 150 column tiles, two of them split
    # along K into ranges that start mid-way through the groups' K; every
    # output, and bit-equal across two runs
    M, K, N = 17, 1056, 150 * 128
    W = gaussian_weights(K, N, 0.02, 32 + int(sym))
    dev_t, (q, sc, z) = _quantize(W, 32, sym)
    X = activations(M, K, dtype, 33)
    Y1 = w4.gemm(X.cuda(), *dev_t[:3], group_size=32)
    Y2 = w4.gemm(X.cuda(), *dev_t[:3], group_size=32)
    torch.cuda.synchronize()
    assert torch.equal(Y1.view(torch.int16), Y2.view(torch.int16))
    Y_ref, A = _expected(q, sc, z, 32, dtype, X)
    assert_close(to_f64(Y1), Y_ref, A, f"g=32 split tail sym={sym} {dtype}")


# ---------------------------------------------------------------- AWQ layout
@pytest.mark.parametrize("sym", [False, True])
@pytest.mark.parametrize("K,N,g", [(1024, 520, 128), (2048, 4104, 64)])
def test_awq_repack_matches_oracle_and_products(K, N, g, sym):
    # the same checkpoint in AWQ's layout (codes packed along N in AWQ's
    # column order) is repacked bit for bit into this library's layout, and
    # products through it equal the oracle's
    from oracle import awq
    W = gaussian_weights(K, N, 0.02, K + N)
    if sym:
        q, sc = int4.rtn_quantize_sym(W, g)
        z = int4.sym_zeros(*sc.shape)
        qa, za = awq.pack_awq(q), None
    else:
        qa, sc, za, q, z = awq.awq_checkpoint(W, g)
    qw, qz = w4.repack_awq(to_dev_u32(qa), None if za is None else to_dev_u32(za), group_size=g)
    assert np.array_equal(qw.cpu().numpy().view(np.uint32), int4.pack_along_k(q))
    if sym:
        assert qz is None
    else:
        assert np.array_equal(qz.cpu().numpy().view(np.uint32), int4.pack_zeros(z))
    for M in (3, 48):
        X = activations(M, K, "bf16", M)
        Y = w4.gemm(X.cuda(), qw, to_dev(sc), qz, group_size=g)
        torch.cuda.synchronize()
        Y_ref, A = _expected(q, sc, z, g, "bf16", X)
        assert_close(to_f64(Y), Y_ref, A, f"AWQ repack K={K} N={N} g={g} sym={sym} M={M}")


# ------------------------------------------------- fused SiLU(gate) * up
@pytest.mark.parametrize("M", [1, 4, 16, 40, 300])
@pytest.mark.parametrize("g,sym", [(128, False), (64, True)])
def test_gate_up_silu_mul(M, g, sym):
    # A = SiLU(X W_gate) * (X W_up) against the oracle's fp64 activation, on
    # both kernels; F = 776 leaves a ragged last block, K several groups
    K, F = 1536, 776
    dtype = "bf16" if M % 2 == 0 else "f16"
    W = gaussian_weights(K, 2 * F, 0.02, M + g)
    dev_t, (q, sc, z) = _quantize(W, g, sym)
    X = activations(M, K, dtype, M)
    A_ = w4.gemm_silu_mul(X.cuda(), *dev_t[:3], group_size=g)
    torch.cuda.synchronize()
    assert A_.shape == (M, F)
    w_hat = numerics.dtype_bits_to_f64(int4.dequant(q, sc, z, dtype, g), dtype)
    act, A_ref = product.silu_mul_reference(X.double().numpy(), w_hat)
    assert_close(to_f64(A_), act, A_ref, f"silu_mul M={M} g={g} sym={sym} {dtype}")
    # and the same as the unfused product followed by the activation, to
    # rounding: the two halves are the plain product's columns
    Y = w4.gemm(X.cuda(), *dev_t[:3], group_size=g).double().cpu()
    ref2 = (torch.nn.functional.silu(Y[:, :F]) * Y[:, F:]).numpy()
    assert np.allclose(to_f64(A_), ref2, rtol=3e-2, atol=3e-2 * (np.abs(ref2).max() + 1e-30))


def test_gate_up_silu_mul_full_size_decode():
    # the Qwen2.5-32B-shaped gate_up (5120 -> 2 x 27648) at M = 1, sampled outputs
    K, F = 5120, 27648
    W = gaussian_weights(K, 2 * F, 0.02, 11)
    X = activations(1, K, "bf16", 11)
    dev_t, _ = _quantize(W, 128, False)
    A_ = w4.gemm_silu_mul(X.cuda(), *dev_t[:3])
    torch.cuda.synchronize()
    cols = np.unique(np.concatenate([np.arange(8), np.arange(F - 8, F),
                                     np.random.default_rng(3).choice(F, 120, replace=False)]))
    _, (q, sc, z) = _quantize(W[:, np.concatenate([cols, F + cols])], 128, False)
    w_hat = numerics.dtype_bits_to_f64(int4.dequant(q, sc, z, "bf16", 128), "bf16")
    act, A_ref = product.silu_mul_reference(X.double().numpy(), w_hat)
    assert_close(to_f64(A_)[:, cols], act, A_ref, "silu_mul full size")
