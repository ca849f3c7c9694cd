"""Act-order prepack (rows reordered by group once, X's columns gathered per
call) through the C ABI, against the oracle's act-order product."""

import numpy as np
import pytest
import torch

import bit_weight_only_wise_b300 as w4
from oracle import int4
from synth import WORKLOADS, act_order_g_idx, activations, student_t_weights, weights_for

from gpu_util import assert_close, int4_expected, sample_columns, to_dev, to_dev_u32, to_f64

pytestmark = pytest.mark.gpu


def _prepack(W, g_idx):
    qw, sc, qz, q, _ = int4.quantize_packed(W, 128, g_idx)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    q_sorted, perm = w4.act_order_prepack(to_dev_u32(qw), to_dev(g_idx), dev_status=st)
    torch.cuda.synchronize()
    assert st.item() == 0
    return q, q_sorted, perm, to_dev(sc), to_dev_u32(qz)


def test_prepack_layout():
    K, N = 1024, 264
    W = student_t_weights(K, N, 5, 0.01, 3)
    g_idx = act_order_g_idx(K, 128, 3)
    q, q_sorted, perm, _, _ = _prepack(W, g_idx)
    perm = perm.cpu().numpy()
    assert np.array_equal(np.sort(perm), np.arange(K))  # a permutation
    assert np.array_equal(g_idx[perm], np.arange(K) // 128)  # sorted row j sits in group j // 128
    for g in range(K // 128):  # rows of a group keep their original order
        assert np.all(np.diff(perm[g * 128:(g + 1) * 128]) > 0)
    rows = int4.unpack_along_k(q_sorted.cpu().numpy().view(np.uint32))
    assert np.array_equal(rows, q[perm])


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("M", [1, 5, 16, 64, 200])
def test_prepacked_product_small(dtype, M):
    K, N = 2048, 520
    W = student_t_weights(K, N, 5, 0.01, M)
    g_idx = act_order_g_idx(K, 128, M)
    _, q_sorted, perm, sc, qz = _prepack(W, g_idx)
    X = activations(M, K, dtype, M)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    Y = w4.gemm_prepacked(X.cuda(), q_sorted, sc, qz, perm, dev_status=st)
    torch.cuda.synchronize()
    assert st.item() == 0
    Y_ref, A = int4_expected(W, X.double().numpy(), dtype, None, g_idx)
    assert_close(to_f64(Y), Y_ref, A, f"prepacked act-order M={M} {dtype}")


@pytest.mark.parametrize("K,N", WORKLOADS["act_order"].shapes)
def test_prepacked_full_size_sampled(K, N):
    wl = WORKLOADS["act_order"]
    W = weights_for(wl, K, N, 0)
    g_idx = act_order_g_idx(K, 128, 0)
    _, q_sorted, perm, sc, qz = _prepack(W, g_idx)
    cols = sample_columns(N)
    for M in wl.Ms:
        X = activations(M, K, wl.dtype, M)
        Y = w4.gemm_prepacked(X.cuda(), q_sorted, sc, qz, perm)
        Y_ref, A = int4_expected(W, X.double().numpy(), wl.dtype, cols, g_idx)
        assert_close(to_f64(Y)[:, cols], Y_ref, A, f"prepacked act-order {K}x{N} M={M}")


def test_prepack_reports_groups_of_the_wrong_size():
    # group 0 gets 129 rows and group 1 127: no sorted layout with 128-row
    # groups exists, so the prepack reports UNSUPPORTED (its outputs are
    # unspecified but it reads nothing out of range)
    K, N = 512, 64
    g_idx = (np.arange(K) // 128).astype(np.int32)
    g_idx[200] = 0
    qw = np.zeros((K // 8, N), dtype=np.uint32)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    w4.act_order_prepack(to_dev_u32(qw), to_dev(g_idx), dev_status=st)
    torch.cuda.synchronize()
    assert st.item() == w4.ERR_UNSUPPORTED


def test_prepacked_large_m_keeps_the_shared_tickets():
    # a prepacked call with M > 16 (no split-K) followed by decode calls on
    # the same cached workspace: the gathered X must not land on the tickets
    from synth import gaussian_weights

    K, N = 2048, 1024
    W = student_t_weights(K, N, 5, 0.01, 7)
    g_idx = act_order_g_idx(K, 128, 7)
    _, q_sorted, perm, sc, qz = _prepack(W, g_idx)
    X64 = activations(64, K, "bf16", 1)
    w4.gemm_prepacked(X64.cuda(), q_sorted, sc, qz, perm)
    W2 = gaussian_weights(4096, 4096, 0.02, 8)
    qw2, sc2, qz2 = w4.quantize(to_dev(W2))
    for M in (1, 16):
        X = activations(M, 4096, "bf16", M)
        Y = w4.gemv(X.cuda(), qw2, sc2, qz2)
        Y_ref, A = int4_expected(W2, X.double().numpy(), "bf16")
        assert_close(to_f64(Y), Y_ref, A, f"decode after prepacked M=64, M={M}")
        Yp = w4.gemm_prepacked(X.cuda()[:, :K].contiguous(), q_sorted, sc, qz, perm)
        Yp_ref, Ap = int4_expected(W, X.double().numpy()[:, :K], "bf16", None, g_idx)
        assert_close(to_f64(Yp), Yp_ref, Ap, f"prepacked M={M} after the others")
