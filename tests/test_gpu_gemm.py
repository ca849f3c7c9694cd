"""Prefill-shape products (M > 16) on the tcgen05 tensor-core kernel, through
the C ABI, against the oracle."""

import numpy as np
import pytest
import torch

import bit_weight_only_wise_b300 as w4
from oracle import int4, nf4, numerics, product
from synth import WORKLOADS, activations, gaussian_weights, student_t_weights, weights_for

from gpu_util import (TDT, assert_close, bits, dev, int4_expected, nf4_expected, sample_columns, to_dev, to_dev_u32,
                      to_f64)

pytestmark = pytest.mark.gpu


def _int4_dev(W, g_idx=None):
    qw, sc, qz, q, z = int4.quantize_packed(W, 128, g_idx)
    return (to_dev_u32(qw), to_dev(sc), to_dev_u32(qz), None if g_idx is None else to_dev(g_idx)), (q, sc, z)


def _status():
    return torch.zeros(1, dtype=torch.int32, device=dev())


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("M,K,N", [(17, 256, 128), (32, 256, 264), (64, 1024, 384), (100, 512, 136),
                                   (256, 1024, 256), (300, 768, 520)])
def test_gemm_small_all_outputs(dtype, M, K, N):
    W = gaussian_weights(K, N, 0.02, M + K)
    dev_t, _ = _int4_dev(W)
    X = activations(M, K, dtype, M)
    st = _status()
    Y = w4.gemm(X.cuda(), *dev_t[:3], dev_status=st)
    torch.cuda.synchronize()
    assert st.item() == 0
    Y_ref, A = int4_expected(W, X.double().numpy(), dtype)
    assert_close(to_f64(Y), Y_ref, A, f"gemm M={M} K={K} N={N} {dtype}")


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_gemm_one_hot_rows_are_exact(dtype):
    K, N = 1024, 264
    W = student_t_weights(K, N, 5, 0.01, 2)
    dev_t, (q, sc, z) = _int4_dev(W)
    rng = np.random.default_rng(0)
    rows = np.concatenate([[0, 1, 63, 64, 127, 128, 1023], rng.choice(K, 57, replace=False)])
    M = rows.size
    X = torch.zeros((M, K), dtype=TDT[dtype])
    X[torch.arange(M), torch.from_numpy(rows)] = 1.0
    Y = w4.gemm(X.cuda(), *dev_t[:3])
    w_hat = int4.dequant(q, sc, z, dtype)
    assert np.array_equal(bits(Y), w_hat[rows])


def test_gemm_zero_when_codes_equal_zero_points():
    K, N = 512, 256
    rng = np.random.default_rng(1)
    z = rng.integers(0, 16, size=(K // 128, N)).astype(np.uint8)
    q = z[np.arange(K) // 128]
    sc = numerics.to_f16(rng.uniform(1e-3, 0.1, size=(K // 128, N)))
    X = activations(64, K, "bf16", 1).cuda()
    Y = w4.gemm(X, to_dev_u32(int4.pack_along_k(q)), to_dev(sc), to_dev_u32(int4.pack_zeros(z)))
    assert torch.count_nonzero(Y.float()).item() == 0


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("M", [64, 300])
def test_nf4_gemm_small(dtype, M):
    K, N = 1024 + 64, 264
    W = gaussian_weights(K, N, 0.02, 9)
    cb = nf4.codebook()
    qw, am, _ = nf4.nf4_quantize_packed(W, cb)
    X = activations(M, K, dtype, 3)
    Y = w4.nf4_gemm(X.cuda(), to_dev_u32(qw), to_dev(am), to_dev(cb))
    Y_ref, A = nf4_expected(W, X.double().numpy(), cb, dtype)
    assert_close(to_f64(Y), Y_ref, A, f"nf4 gemm M={M} {dtype}")


def _sample_rows(M, n=64, seed=0):
    if M <= n:
        return np.arange(M)
    rng = np.random.default_rng(seed)
    return np.unique(np.concatenate([[0, M - 1], rng.choice(M, n - 2, replace=False)]))


def _full_cases():
    out = []
    wl = WORKLOADS["qwen32b"]
    for (K, N), lab in zip(wl.shapes, wl.labels):
        out.append(pytest.param("qwen32b", K, N, tuple(m for m in wl.Ms if m > 16), id=f"qwen32b-{lab}"))
    return out


@pytest.mark.parametrize("name,K,N,Ms", _full_cases())
def test_gemm_full_size_sampled(name, K, N, Ms):
    # the workload's full shapes and token counts, as the bench launches them;
    # the oracle recomputes 64 sampled rows x ~200 sampled columns
    wl = WORKLOADS[name]
    W = weights_for(wl, K, N, 0)
    qw, sc, qz = w4.quantize(to_dev(W))
    cols = sample_columns(N)
    for M in Ms:
        X = activations(M, K, wl.dtype, M)
        st = _status()
        Y = w4.gemm(X.cuda(), qw, sc, qz, dev_status=st)
        torch.cuda.synchronize()
        assert st.item() == 0
        rows = _sample_rows(M)
        Y_ref, A = int4_expected(W, X.double().numpy()[rows], wl.dtype, cols)
        assert_close(to_f64(Y)[np.ix_(rows, cols)], Y_ref, A, f"{name} {K}x{N} M={M}")


def test_nf4_gemm_full_size_sampled():
    wl = WORKLOADS["nf4"]
    K, N = wl.shapes[0]
    W = weights_for(wl, K, N, 0)
    cb = nf4.codebook()
    qw, am = w4.nf4_quantize(to_dev(W), to_dev(cb))
    cols = sample_columns(N)
    for M in (64, 1024):
        X = activations(M, K, "bf16", M)
        Y = w4.nf4_gemm(X.cuda(), qw, am, to_dev(cb))
        rows = _sample_rows(M)
        Y_ref, A = nf4_expected(W, X.double().numpy()[rows], cb, "bf16", cols)
        assert_close(to_f64(Y)[np.ix_(rows, cols)], Y_ref, A, f"nf4 full M={M}")


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("M,K,N", [(17, 512, 264), (64, 1024, 384), (200, 2048, 136)])
def test_gemm_act_order_small(dtype, M, K, N):
    from synth import act_order_g_idx

    W = student_t_weights(K, N, 5, 0.01, M)
    g_idx = act_order_g_idx(K, 128, M)
    dev_t, _ = _int4_dev(W, g_idx)
    X = activations(M, K, dtype, M)
    Y = w4.gemm(X.cuda(), *dev_t[:3], g_idx=dev_t[3])
    Y_ref, A = int4_expected(W, X.double().numpy(), dtype, None, g_idx)
    assert_close(to_f64(Y), Y_ref, A, f"act-order gemm M={M} {dtype}")


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_gemm_act_order_one_hot_exact(dtype):
    from synth import act_order_g_idx

    K, N = 1024, 264
    W = gaussian_weights(K, N, 0.02, 4)
    g_idx = act_order_g_idx(K, 128, 4)
    dev_t, (q, sc, z) = _int4_dev(W, g_idx)
    rows = np.arange(0, K, 13)[:48]
    X = torch.zeros((rows.size, K), dtype=TDT[dtype])
    X[torch.arange(rows.size), torch.from_numpy(rows)] = 1.0
    Y = w4.gemm(X.cuda(), *dev_t[:3], g_idx=dev_t[3])
    assert np.array_equal(bits(Y), int4.dequant(q, sc, z, dtype, 128, g_idx)[rows])


@pytest.mark.parametrize("K,N", WORKLOADS["act_order"].shapes)
def test_gemm_act_order_full_size_m64(K, N):
    from synth import act_order_g_idx

    wl = WORKLOADS["act_order"]
    W = weights_for(wl, K, N, 0)
    g_idx = act_order_g_idx(K, 128, 0)
    (qw, sc, qz, gi), _ = _int4_dev(W, g_idx)
    cols = sample_columns(N)
    X = activations(64, K, wl.dtype, 64)
    st = _status()
    Y = w4.gemm(X.cuda(), qw, sc, qz, g_idx=gi, dev_status=st)
    torch.cuda.synchronize()
    assert st.item() == 0
    Y_ref, A = int4_expected(W, X.double().numpy(), wl.dtype, cols, g_idx)
    assert_close(to_f64(Y)[:, cols], Y_ref, A, f"act-order {K}x{N} M=64")


def test_gemm_split_k_is_deterministic_and_matches():
    # 256 tokens over 5120 x 5120: 40 output tiles leave most SMs idle, so the
    # kernel splits K; the partial tiles are summed in a fixed order
    K, N, M = 5120, 5120, 256
    W = gaussian_weights(K, N, 0.02, 21)
    qw, sc, qz = w4.quantize(to_dev(W))
    assert w4.workspace_bytes(M, N, K) > 0  # the split plan needs partial tiles
    X = activations(M, K, "bf16", 21).cuda()
    Y1 = w4.gemm(X, qw, sc, qz)
    Y2 = w4.gemm(X, qw, sc, qz)
    torch.cuda.synchronize()
    assert torch.equal(Y1.view(torch.int16), Y2.view(torch.int16))
    rows = _sample_rows(M)
    cols = sample_columns(N)
    Y_ref, A = int4_expected(W, X.cpu().double().numpy()[rows], "bf16", cols)
    assert_close(to_f64(Y1)[np.ix_(rows, cols)], Y_ref, A, "split-K 5120x5120 M=256")


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("M,K,N", [(17, 1024, 150 * 128), (40, 2048, 150 * 128 + 72)])
def test_gemm_whole_waves_and_split_tail_all_outputs(dtype, M, K, N):
    # 150 output tiles of 128 columns: one full wave of 148 whole tiles, and
    # the 2 tiles left over cut along K (the split-tail schedule), every
    # output checked, run twice for determinism
    assert w4.workspace_bytes(M, N, K) > 0  # the leftover tiles need partial tiles
    W = gaussian_weights(K, N, 0.02, M + N)
    dev_t, _ = _int4_dev(W)
    X = activations(M, K, dtype, M).cuda()
    st = _status()
    Y1 = w4.gemm(X, *dev_t[:3], dev_status=st)
    Y2 = w4.gemm(X, *dev_t[:3], dev_status=st)
    torch.cuda.synchronize()
    assert st.item() == 0
    assert torch.equal(Y1.view(torch.int16), Y2.view(torch.int16))
    Y_ref, A = int4_expected(W, X.cpu().double().numpy(), dtype)
    assert_close(to_f64(Y1), Y_ref, A, f"split tail M={M} K={K} N={N} {dtype}")


def test_tickets_are_left_at_zero():
    # the split-K tickets wrap back to zero at each block's contributor count:
    # after decode calls (split column blocks on every shape below) and a
    # split-K prefill call through one workspace, the ticket area is all zero
    ticket_bytes = 4096 * 8 * 4  # one int per 32-column slice of up to 4096 column blocks
    shapes = [(1, 5120, 5120), (5, 27648, 1024), (16, 2048, 3072), (256, 5120, 1280), (17, 1024, 150 * 128)]
    need = max(w4.workspace_bytes(M, N, K) for M, K, N in shapes)
    ws = torch.zeros(need, dtype=torch.uint8, device=dev())
    st = _status()
    for M, K, N in shapes:
        W = gaussian_weights(K, N, 0.02, M + N)
        qw, sc, qz = w4.quantize(to_dev(W))
        X = activations(M, K, "bf16", M).cuda()
        for _ in range(3):
            w4.gemm(X, qw, sc, qz, ws=ws, dev_status=st)
        torch.cuda.synchronize()
        assert st.item() == 0
        assert torch.count_nonzero(ws[:ticket_bytes]).item() == 0, f"tickets left set after M={M} {K}x{N}"
    # the act-order decode kernel (g_idx as stored) takes the same tickets
    from synth import act_order_g_idx

    K, N = 4096, 1024
    g_idx = act_order_g_idx(K, 128, 3)
    W = student_t_weights(K, N, 5, 0.01, 3)
    (qw, sc, qz, gi), _ = _int4_dev(W, g_idx)
    for M in (1, 9):
        w4.gemm(activations(M, K, "f16", M).cuda(), qw, sc, qz, g_idx=gi, ws=ws, dev_status=st)
    torch.cuda.synchronize()
    assert st.item() == 0
    assert torch.count_nonzero(ws[:ticket_bytes]).item() == 0, "tickets left set after act-order decode"
