"""Failure detection on the GPU without a fault: a bounded wait that runs out
(on a barrier that nothing completes) ends its kernel with W4A16_ERR_TIMEOUT in
the caller's status word, and the context stays usable afterwards."""

import time

import pytest
import torch

import bit_weight_only_wise_b300 as w4
from synth import activations, gaussian_weights

from gpu_util import assert_close, int4_expected, to_dev, to_f64

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("limit_ms", [5, 50])
def test_wait_that_runs_out_reports_timeout(limit_ms):
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    w4.selftest_wait_timeout(st, limit_ms * 1_000_000)
    torch.cuda.synchronize()
    dt = time.perf_counter() - t0
    assert st.item() == w4.ERR_TIMEOUT
    assert dt >= limit_ms * 1e-3 * 0.9  # it waited for (about) the limit ...
    assert dt < 2.0                     # ... and no longer


def test_context_is_usable_after_a_timeout():
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    w4.selftest_wait_timeout(st, 2_000_000)
    torch.cuda.synchronize()
    assert st.item() == w4.ERR_TIMEOUT
    K, N = 1024, 512
    W = gaussian_weights(K, N, 0.02, 3)
    qw, sc, qz = w4.quantize(to_dev(W))
    X = activations(2, K, "bf16", 3)
    st2 = torch.zeros(1, dtype=torch.int32, device="cuda")
    Y = w4.gemv(X.cuda(), qw, sc, qz, dev_status=st2)
    torch.cuda.synchronize()
    assert st2.item() == 0
    Y_ref, A = int4_expected(W, X.double().numpy(), "bf16")
    assert_close(to_f64(Y), Y_ref, A, "decode after a timed-out wait")
