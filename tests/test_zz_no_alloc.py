"""The allocation-free decode entry point, through the C ABI.

w4a16_gemv_noalloc exists for callers that cannot allocate a workspace (they
run inside a memory pool they do not own, or on a path where cudaMalloc is not
allowed); it keeps its split-K scratch in a device array inside the library.
Its results must match the ordinary entry point's, call after call, since the
shared scratch keeps the previous call's contents.

This file is named to be collected last, so a run that stops at the first
failure has already run every other test; it also passes on its own in a fresh
process (the first call sets up the scratch address).
"""

import ctypes

import numpy as np
import pytest
import torch

import bit_weight_only_wise_b300 as w4
from oracle import int4
from synth import activations, gaussian_weights, student_t_weights, act_order_g_idx

from gpu_util import assert_close, int4_expected, to_dev, to_dev_u32, to_f64

pytestmark = pytest.mark.gpu


def _noalloc(X, qw, sc, qz, g_idx, Y, dtype_code, status=None):
    M, K = X.shape
    N = qw.shape[1]
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    p = lambda t: None if t is None else ctypes.c_void_p(t.data_ptr())  # noqa: E731
    return w4._lib.w4a16_gemv_noalloc(p(X), p(qw), p(sc), p(qz), p(g_idx), p(Y), M, N, K, 128, dtype_code,
                                      p(status), stream)


@pytest.mark.parametrize("dtype,code", [("f16", 0), ("bf16", 1)])
@pytest.mark.parametrize("M,K,N,act", [(1, 4096, 4096, False), (5, 1536, 776, False), (16, 2048, 3072, False),
                                       (3, 1024, 520, True)])
def test_noalloc_matches_workspace_entry_two_calls(dtype, code, M, K, N, act):
    W = student_t_weights(K, N, 5, 0.01, M) if act else gaussian_weights(K, N, 0.02, M + N)
    g_idx = act_order_g_idx(K, 128, 1) if act else None
    qw, sc, qz, _, _ = int4.quantize_packed(W, 128, g_idx)
    qw, sc, qz = to_dev_u32(qw), to_dev(sc), to_dev_u32(qz)
    gi = None if g_idx is None else to_dev(g_idx)
    X = activations(M, K, dtype, 3).cuda()
    ref = w4.gemv(X, qw, sc, qz, g_idx=gi)  # the ordinary entry point, with its own workspace
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    for _ in range(2):  # back to back: the shared scratch keeps the last call's contents
        Y = torch.empty_like(ref)
        assert _noalloc(X, qw, sc, qz, gi, Y, code, status) == w4.OK
        torch.cuda.synchronize()
        assert status.item() == 0
        Y_ref, A = int4_expected(W, X.double().cpu().numpy(), dtype, None, g_idx)
        assert_close(to_f64(Y), to_f64(ref), A, "noalloc vs workspace entry")
        assert_close(to_f64(Y), Y_ref, A, "noalloc vs oracle")


def test_noalloc_rejects_out_of_range_requests():
    X = torch.zeros((17, 256), dtype=torch.bfloat16, device="cuda")
    qw = torch.zeros((32, 64), dtype=torch.int32, device="cuda")
    sc = torch.zeros((2, 64), dtype=torch.float16, device="cuda")
    qz = torch.zeros((2, 8), dtype=torch.int32, device="cuda")
    Y = torch.empty((17, 64), dtype=torch.bfloat16, device="cuda")
    assert _noalloc(X, qw, sc, qz, None, Y, 1) == w4.ERR_INVALID_ARG  # M above the decode limit
    assert _noalloc(X[:4], qw, sc, qz, None, Y[:4], 7) == w4.ERR_INVALID_ARG  # bad dtype


def _case(M, K, N, dtype, act, seed):
    W = student_t_weights(K, N, 5, 0.01, seed) if act else gaussian_weights(K, N, 0.02, seed)
    g_idx = act_order_g_idx(K, 128, seed) if act else None
    qw, sc, qz, _, _ = int4.quantize_packed(W, 128, g_idx)
    X = activations(M, K, dtype, seed).cuda()
    gi = None if g_idx is None else to_dev(g_idx)
    return W, g_idx, X, (to_dev_u32(qw), to_dev(sc), to_dev_u32(qz), gi)


def test_noalloc_sequence_of_different_shapes():
    # One call leaves its split-K tickets and partial sums in the shared array;
    # the next call, of another shape, must not be disturbed by them: a wide
    # product with many contributors per column block, then a narrow one whose
    # blocks are split over other CTAs, then act-order, then the first again,
    # each checked against the oracle.
    cases = [(16, 8192, 8192, "bf16", False, 21), (1, 4096, 264, "f16", False, 22),
             (3, 2048, 1032, "bf16", True, 23), (16, 8192, 8192, "bf16", False, 21)]
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    for M, K, N, dtype, act, seed in cases:
        W, g_idx, X, (qw, sc, qz, gi) = _case(M, K, N, dtype, act, seed)
        cols = np.unique(np.concatenate([np.arange(8), np.arange(N - 8, N),
                                         np.random.default_rng(seed).choice(N, 96, replace=False)]))
        Y = torch.empty((M, N), dtype=X.dtype, device="cuda")
        assert _noalloc(X, qw, sc, qz, gi, Y, 1 if dtype == "bf16" else 0, status) == w4.OK
        torch.cuda.synchronize()
        assert status.item() == 0
        Y_ref, A = int4_expected(W, X.double().cpu().numpy(), dtype, cols, g_idx)
        assert_close(to_f64(Y)[:, cols], Y_ref, A, f"noalloc M={M} K={K} N={N} act={act}")


def test_noalloc_after_a_timed_out_wait():
    # a bounded wait that ran out elsewhere leaves the context usable, and the
    # allocation-free entry still gives the oracle's product afterwards
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    w4.selftest_wait_timeout(st, 2_000_000)
    torch.cuda.synchronize()
    assert st.item() == w4.ERR_TIMEOUT
    W, g_idx, X, (qw, sc, qz, gi) = _case(4, 4096, 2048, "bf16", False, 31)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    Y = torch.empty((4, 2048), dtype=X.dtype, device="cuda")
    assert _noalloc(X, qw, sc, qz, gi, Y, 1, status) == w4.OK
    torch.cuda.synchronize()
    assert status.item() == 0
    Y_ref, A = int4_expected(W, X.double().cpu().numpy(), "bf16")
    assert_close(to_f64(Y), Y_ref, A, "noalloc after a timeout")
