"""Helpers for the GPU parity tests: move oracle / synthetic data to the device
and compute the oracle's expected products on a subset of output columns."""

from __future__ import annotations

import numpy as np
import torch

from oracle import int4, nf4, numerics, product

TDT = {"f16": torch.float16, "bf16": torch.bfloat16}


def dev():
    return torch.device("cuda", 0)


def to_dev_u32(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int32)).to(dev())


def to_dev(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a)).to(dev())


def bits(t: torch.Tensor) -> np.ndarray:
    """uint16 bit patterns of a CUDA fp16/bf16 tensor."""
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


def to_f64(t: torch.Tensor) -> np.ndarray:
    return t.float().cpu().numpy().astype(np.float64)


def sample_columns(N: int, n: int = 192, seed: int = 0) -> np.ndarray:
    """Sorted column indices: the first and last 8 columns plus random ones."""
    rng = np.random.default_rng(seed)
    cols = set(range(min(8, N))) | set(range(max(0, N - 8), N))
    cols |= set(rng.choice(N, size=min(n, N), replace=False).tolist())
    return np.array(sorted(cols))


def int4_expected(W: np.ndarray, X_f64: np.ndarray, dtype: str, cols=None, g_idx=None):
    """Oracle (Y_ref, A) on the given columns (all if None), quantizing them itself."""
    Wc = W if cols is None else W[:, cols]
    q, s, z = int4.rtn_quantize(Wc, 128, g_idx)
    w_hat = numerics.dtype_bits_to_f64(int4.dequant(q, s, z, dtype, 128, g_idx), dtype)
    return product.reference(X_f64, w_hat)


def nf4_expected(W: np.ndarray, X_f64: np.ndarray, cb: np.ndarray, dtype: str, cols=None):
    Wc = W if cols is None else W[:, cols]
    codes, am = nf4.nf4_quantize(Wc, cb, 64)
    w_hat = numerics.dtype_bits_to_f64(nf4.nf4_dequant(codes, am, cb, dtype), dtype)
    return product.reference(X_f64, w_hat)


def assert_close(Y, Y_ref, A, what=""):
    ok, m, f = product.within_tolerance(Y, Y_ref, A)
    assert ok, f"{what}: max_rel={m:.3e} (<= {product.MAX_REL}) fro={f:.3e} (<= {product.FRO_REL})"
    return m, f
