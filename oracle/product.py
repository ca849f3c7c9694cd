"""The reference product Y = X . W_hat in fp64, and the tolerance checks.

What the fused kernels compute is a plain matrix product with the
dequantized weights: "LLM量化技术深度对比:GPTQ vs AWQ vs bitsandbytes
2026基准全解析", key-data item 1, describes Marlin as fusing dequantization
into the matrix multiply so that 16-bit weights are never materialised --
the result is the same product, only the memory traffic changes.  The oracle
is therefore that product written out, with a library matmul (numpy, fp64)
as the step.

Reading (listed in the design notes): the tolerance is measured against
``W_hat`` rounded to the compute dtype (the values the kernels must produce
bit for bit), not against the exact (q - z) * s.

Tolerances: per output, |Y - Y_ref| / sum_k |x_mk| |w_hat_kn| <= 1e-2, and
over all checked outputs ||Y - Y_ref||_F / ||Y_ref||_F <= 2e-3.

Fused MLP activation.  A decoder layer's gate_up projection is followed by
SiLU(gate) * up before the down projection; per-token latency is the weight
bytes streamed per forward ("LLM量化技术深度对比" key-data items 1 and 3), so
the activation is applied as the product's epilogue instead of writing and
re-reading the 2F-wide projection.  Readings (the pages do not spell the
layer out): the gate_up weight is ``[K, 2F]`` with the gate in columns
``[0, F)`` and the up projection in ``[F, 2F)``; ``SiLU(t) = t / (1 + e^-t)``;
``act[m, j] = SiLU(y[m, j]) * y[m, F + j]`` with ``y = X . W_hat`` in fp64.
Its tolerance uses the same two bounds with the normaliser carried through
the activation to first order:
``A_act = |SiLU'(g)| |u| A_g + |SiLU(g)| A_u``.
"""

from __future__ import annotations

import numpy as np

MAX_REL = 1e-2
FRO_REL = 2e-3


def reference(X: np.ndarray, W_hat: np.ndarray):
    """``(Y_ref, A)`` in fp64: ``Y_ref = X @ W_hat``, ``A = |X| @ |W_hat|``."""
    X = np.asarray(X, dtype=np.float64)
    W_hat = np.asarray(W_hat, dtype=np.float64)
    return X @ W_hat, np.abs(X) @ np.abs(W_hat)


def errors(Y, Y_ref, A):
    """``(max_rel, fro_rel)`` of a candidate ``Y`` against ``Y_ref``.

    Outputs whose normaliser ``A`` is zero must match exactly; they count as
    infinite error otherwise.
    """
    Y = np.asarray(Y, dtype=np.float64)
    Y_ref = np.asarray(Y_ref, dtype=np.float64)
    A = np.asarray(A, dtype=np.float64)
    diff = np.abs(Y - Y_ref)
    with np.errstate(divide="ignore", invalid="ignore"):
        rel = np.where(A > 0, diff / np.where(A > 0, A, 1.0), np.where(diff > 0, np.inf, 0.0))
    max_rel = float(rel.max()) if rel.size else 0.0
    nref = float(np.linalg.norm(Y_ref))
    ndiff = float(np.linalg.norm(Y - Y_ref))
    fro = ndiff / nref if nref > 0 else (0.0 if ndiff == 0 else np.inf)
    return max_rel, fro


def within_tolerance(Y, Y_ref, A, max_rel: float = MAX_REL, fro_rel: float = FRO_REL):
    """``(ok, max_rel, fro_rel)``."""
    m, f = errors(Y, Y_ref, A)
    return (m <= max_rel and f <= fro_rel), m, f


def silu(t):
    """SiLU(t) = t / (1 + exp(-t)), fp64."""
    t = np.asarray(t, dtype=np.float64)
    with np.errstate(over="ignore"):
        return t / (1.0 + np.exp(-t))


def silu_grad(t):
    """d/dt SiLU(t) = sigma(t) (1 + t (1 - sigma(t))), fp64."""
    t = np.asarray(t, dtype=np.float64)
    with np.errstate(over="ignore"):
        sg = 1.0 / (1.0 + np.exp(-t))
    return sg * (1.0 + t * (1.0 - sg))


def silu_mul_reference(X: np.ndarray, W_hat: np.ndarray):
    """``(act_ref, A_act)`` for a gate_up weight ``W_hat[K, 2F]`` (gate first)."""
    Y, A = reference(X, W_hat)
    F = Y.shape[1] // 2
    g, u = Y[:, :F], Y[:, F:]
    Ag, Au = A[:, :F], A[:, F:]
    return silu(g) * u, np.abs(silu_grad(g)) * np.abs(u) * Ag + np.abs(silu(g)) * Au
