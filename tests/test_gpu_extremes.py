"""The largest shapes the ABI accepts, through the C ABI, against the oracle.

N = 4096 * 256 columns (the last column block the ticket area serves) and
K = 4095 * 128 rows (the largest group-aligned K whose word-rows fit a grid
dimension): at the largest N every column-block index is in use; at the
largest K a single column block is split over every CTA of the decode grid
(296 contributors to one sum) and over 74 K ranges of the tensor-core grid.
The codes, zero points and scales are drawn directly (uniform codes and zero
points, scales spread over two binades), so no quantizer pass over a
gigabyte-sized matrix is needed; the oracle dequantizes the sampled columns
and forms their product in fp64.
"""

import numpy as np
import pytest
import torch

import bit_weight_only_wise_b300 as w4
from oracle import int4, numerics, product
from synth import activations

from gpu_util import assert_close, to_dev, to_dev_u32, to_f64

pytestmark = pytest.mark.gpu

MAX_N = 4096 * 256
MAX_K = 4095 * 128
TICKET_BYTES = 4096 * 8 * 4


def _packed(K, N, seed):
    rng = np.random.default_rng(seed)
    qweight = rng.integers(0, 2**32, size=(K // 8, N), dtype=np.uint64).astype(np.uint32)
    qzeros = rng.integers(0, 2**32, size=(K // 128, N // 8), dtype=np.uint64).astype(np.uint32)
    scales = numerics.to_f16(rng.uniform(1e-3, 4e-3, size=(K // 128, N)))
    return qweight, scales, qzeros


def _expected(qweight, scales, qzeros, X, dtype, cols):
    q = int4.unpack_along_k(qweight[:, cols])
    z = int4.unpack_zeros(qzeros)[:, cols]
    w_hat = numerics.dtype_bits_to_f64(int4.dequant(q, scales[:, cols], z, dtype, 128), dtype)
    return product.reference(X.double().numpy(), w_hat)


def _columns(N, n, seed):
    rng = np.random.default_rng(seed)
    return np.unique(np.concatenate([np.arange(8), np.arange(N - 8, N), rng.choice(N, n, replace=False)]))


@pytest.mark.parametrize("M,dtype", [(1, "bf16"), (16, "f16"), (64, "bf16")])
def test_largest_n(M, dtype):
    K, N = 256, MAX_N
    qweight, scales, qzeros = _packed(K, N, 1)
    qw, sc, qz = to_dev_u32(qweight), to_dev(scales), to_dev_u32(qzeros)
    X = activations(M, K, dtype, M)
    ws = torch.zeros(w4.workspace_bytes(M, N, K) or 16, dtype=torch.uint8, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    Y = w4.gemm(X.cuda(), qw, sc, qz, ws=ws, dev_status=st)
    torch.cuda.synchronize()
    assert st.item() == 0
    cols = _columns(N, 256, M)
    Y_ref, A = _expected(qweight, scales, qzeros, X, dtype, cols)
    assert_close(to_f64(Y)[:, cols], Y_ref, A, f"N={N} M={M} {dtype}")
    assert torch.count_nonzero(ws[:TICKET_BYTES]).item() == 0


@pytest.mark.parametrize("M,dtype", [(1, "bf16"), (16, "f16"), (64, "bf16")])
def test_largest_k(M, dtype):
    K, N = MAX_K, 256
    qweight, scales, qzeros = _packed(K, N, 2)
    qw, sc, qz = to_dev_u32(qweight), to_dev(scales), to_dev_u32(qzeros)
    X = activations(M, K, dtype, M)
    ws = torch.zeros(w4.workspace_bytes(M, N, K) or 16, dtype=torch.uint8, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    Y1 = w4.gemm(X.cuda(), qw, sc, qz, ws=ws, dev_status=st)
    Y2 = w4.gemm(X.cuda(), qw, sc, qz, ws=ws, dev_status=st)
    torch.cuda.synchronize()
    assert st.item() == 0
    assert torch.equal(Y1.view(torch.int16), Y2.view(torch.int16))  # the split sums in a fixed order
    cols = _columns(N, 8, M)
    Y_ref, A = _expected(qweight, scales, qzeros, X, dtype, cols)
    assert_close(to_f64(Y1)[:, cols], Y_ref, A, f"K={K} M={M} {dtype}")
    assert torch.count_nonzero(ws[:TICKET_BYTES]).item() == 0


def test_shapes_past_the_limits_are_rejected():
    X = torch.zeros((1, 256), dtype=torch.bfloat16, device="cuda")
    qw = torch.zeros((32, 8), dtype=torch.int32, device="cuda")
    sc = torch.zeros((2, 8), dtype=torch.float16, device="cuda")
    qz = torch.zeros((2, 1), dtype=torch.int32, device="cuda")
    Y = torch.zeros((1, 8), dtype=torch.bfloat16, device="cuda")
    p = lambda t: t.data_ptr()  # noqa: E731
    stream = torch.cuda.current_stream().cuda_stream
    for M, N, K in ((1, MAX_N + 8, 256), (1, 256, MAX_K + 128)):
        st = w4._lib.w4a16_gemm(p(X), p(qw), p(sc), p(qz), None, p(Y), M, N, K, 128, 1, None, 0, None, stream)
        assert st == w4.ERR_INVALID_ARG, (N, K)
