"""Products launched back to back on one stream, each reading the previous
one's output, with no synchronisation in between.  Both kernels are launched
with programmatic stream serialization: a kernel may start while the one
before it finishes, and must not read X before that kernel's writes are
complete.  Each product is checked against the oracle on the output the GPU
actually produced before it."""

import numpy as np
import pytest
import torch

import bit_weight_only_wise_b300 as w4
from oracle import int4
from synth import activations, gaussian_weights

from gpu_util import assert_close, int4_expected, to_dev, to_dev_u32, to_f64

pytestmark = pytest.mark.gpu


def _dev_weights(K, N, seed):
    W = gaussian_weights(K, N, 0.02, seed)
    qw, sc, qz, _, _ = int4.quantize_packed(W, 128)
    return W, (to_dev_u32(qw), to_dev(sc), to_dev_u32(qz))


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_prefill_chain_reads_the_previous_output(dtype):
    # gemm -> gemm -> gemm, M = 300 (two token tiles), the middle one with a
    # split tail (150 column tiles), each consuming the previous Y
    M, dims = 300, [1024, 1024, 150 * 128, 512]
    mats = [_dev_weights(dims[i], dims[i + 1], 20 + i) for i in range(3)]
    X = activations(M, dims[0], dtype, 7).cuda()
    st = torch.zeros(1, dtype=torch.int32, device=X.device)
    outs, x = [], X
    for _, dev_t in mats:
        x = w4.gemm(x, *dev_t, dev_status=st)
        outs.append(x)
    torch.cuda.synchronize()
    assert st.item() == 0
    ins = [X] + outs[:-1]
    for i, (W, _) in enumerate(mats):
        Y_ref, A = int4_expected(W, ins[i].cpu().double().numpy(), dtype)
        assert_close(to_f64(outs[i]), Y_ref, A, f"chain step {i} {dtype}")


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_decode_chain_reads_the_previous_output(dtype):
    # gemv -> gemv -> gemm (M = 4 then the tensor-core kernel at M = 4 rows
    # repeated into 40), each consuming the previous Y
    M, dims = 4, [2048, 4096, 2048]
    mats = [_dev_weights(dims[i], dims[i + 1], 40 + i) for i in range(2)]
    X = activations(M, dims[0], dtype, 9).cuda()
    st = torch.zeros(1, dtype=torch.int32, device=X.device)
    Y1 = w4.gemv(X, *mats[0][1], dev_status=st)
    Y2 = w4.gemv(Y1, *mats[1][1], dev_status=st)
    W3, dev3 = _dev_weights(dims[2], 1024, 60)
    Y3 = w4.gemm(Y2.repeat(10, 1), *dev3, dev_status=st)
    torch.cuda.synchronize()
    assert st.item() == 0
    for W, x, y, tag in ((mats[0][0], X, Y1, "gemv 1"), (mats[1][0], Y1, Y2, "gemv 2"),
                         (W3, Y2.repeat(10, 1), Y3, "gemm")):
        Y_ref, A = int4_expected(W, x.cpu().double().numpy(), dtype)
        assert_close(to_f64(y), Y_ref, A, f"decode chain {tag} {dtype}")
