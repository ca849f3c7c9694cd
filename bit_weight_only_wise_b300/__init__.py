"""Python binding of the W4A16 / NF4 C-ABI library (``libw4a16.so``).

Argument marshalling only: tensors are checked for dtype/shape/device, their
device pointers and the current CUDA stream are handed to the C entry points,
and every step of the computation runs in the library's CUDA kernels.  There
is no CPU fallback: if the library is missing, importing this package raises.

Tensor conventions (all CUDA, contiguous):
  X        [M, K]  torch.float16 / torch.bfloat16
  qweight  [K/8, N] torch.int32 (bit pattern of the packed uint32 words)
  scales   [K/g, N] torch.float16 (g = group_size: 32, 64, a multiple of 128, or K)
  qzeros   [K/g, N/8] torch.int32, or None for symmetric weights
  g_idx    [K] torch.int32 or None
  absmax   [K/64, N] torch.float32 (NF4)
  codebook [16] torch.float32 (NF4), or None for the library's built-in table
"""

from __future__ import annotations

import ctypes
import os

import torch

_LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libw4a16.so")

if not os.path.exists(_LIB_PATH):
    raise ImportError(
        f"{_LIB_PATH} is missing: build the CUDA library first "
        "(python -c 'import __graft_entry__ as g; g.build()')")

_lib = ctypes.CDLL(_LIB_PATH)

_vp = ctypes.c_void_p
_i = ctypes.c_int
_sz = ctypes.c_size_t

_SIGS = {
    "w4a16_gemm": [_vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _vp, _sz, _vp, _vp],
    "w4a16_gemv": [_vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _vp, _sz, _vp, _vp],
    "w4a16_gemv_noalloc": [_vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _vp, _vp],
    "nf4_gemm": [_vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _vp, _sz, _vp, _vp],
    "w4a16_dequant": [_vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _vp],
    "nf4_dequant": [_vp, _vp, _vp, _vp, _i, _i, _i, _i, _vp],
    "w4a16_quantize": [_vp, _i, _i, _i, _vp, _vp, _vp, _vp],
    "nf4_quantize": [_vp, _i, _i, _i, _vp, _vp, _vp, _vp],
    "w4a16_workspace_bytes": [_i, _i, _i],
    "w4a16_act_order_prepack": [_vp, _vp, _i, _i, _i, _vp, _vp, _vp, _vp],
    "w4a16_gemm_prepacked": [_vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _vp, _sz, _vp, _vp],
    "w4a16_prepacked_workspace_bytes": [_i, _i, _i],
    "w4a16_selftest_wait_timeout": [_vp, ctypes.c_ulonglong, _vp],
    "w4a16_status_string": [_i],
    "nf4_default_codebook": [_vp],
    "nf4dq_gemm": [_vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _vp, _sz, _vp, _vp],
    "nf4dq_dequant": [_vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _vp],
    "nf4_double_quantize": [_vp, _i, _i, _i, _vp, _vp, _vp],
    "w4a16_repack_awq": [_vp, _vp, _i, _i, _i, _vp, _vp, _vp],
    "w4a16_gemm_silu_mul": [_vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _vp, _sz, _vp, _vp],
    "w4a16_gemv_batch": [_vp, _i, _vp, _sz, _vp, _vp],
}
for _name, _args in _SIGS.items():
    _fn = getattr(_lib, _name)
    _fn.argtypes = _args
    _fn.restype = _i
_lib.w4a16_workspace_bytes.restype = _sz
_lib.w4a16_prepacked_workspace_bytes.restype = _sz
_lib.w4a16_status_string.restype = ctypes.c_char_p

OK, ERR_INVALID_ARG, ERR_UNSUPPORTED, ERR_CUDA, ERR_TIMEOUT = 0, 1, 2, 3, 4
GEMV_MAX_M = 16
GROUP_SIZE = 128
NF4_BLOCK = 64
_DTYPES = {torch.float16: 0, torch.bfloat16: 1}

EXPORTED = tuple(_SIGS)


class W4A16Error(RuntimeError):
    def __init__(self, status: int, fn: str):
        self.status = status
        super().__init__(f"{fn}: {_lib.w4a16_status_string(status).decode()} (status {status})")


def _check(status: int, fn: str):
    if status != OK:
        raise W4A16Error(status, fn)


def status_string(status: int) -> str:
    return _lib.w4a16_status_string(status).decode()


# Pointers and streams go to ctypes as plain ints (or None for NULL): the
# c_void_p argtypes convert them, which costs less per call than building
# c_void_p objects.
def _ptr(t):
    return None if t is None else t.data_ptr()


def _stream(device) -> int:
    return torch.cuda.current_stream(device).cuda_stream


def workspace_bytes(M: int, N: int, K: int) -> int:
    return int(_lib.w4a16_workspace_bytes(M, N, K))


_workspaces: dict = {}


def workspace(M: int, N: int, K: int, device=None, nbytes: int | None = None) -> torch.Tensor | None:
    """A zero-initialised workspace big enough for (M, N, K) (or ``nbytes``),
    cached per device and stream.

    Calls on one stream run in order, so sharing one buffer between them is
    safe; each stream gets its own.  Every layout starts with the split-K
    tickets, which the calls leave at zero, so one buffer serves them all.
    """
    n = workspace_bytes(M, N, K) if nbytes is None else nbytes
    if n == 0:
        return None
    device = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    key = (device.index, torch.cuda.current_stream(device).cuda_stream)
    ws = _workspaces.get(key)
    if ws is None or ws.numel() < n:
        ws = torch.zeros(max(n, 1 << 20), dtype=torch.uint8, device=device)
        _workspaces[key] = ws
    return ws


def _check_x(X, K):
    if X.dtype not in _DTYPES or not X.is_cuda or X.dim() != 2 or X.shape[1] != K or not X.is_contiguous():
        raise ValueError("X must be a contiguous CUDA [M, K] float16/bfloat16 tensor")


def _out(X, N, out):
    M = X.shape[0]
    if out is None:
        return torch.empty((M, N), dtype=X.dtype, device=X.device)
    if out.shape != (M, N) or out.dtype != X.dtype or not out.is_contiguous():
        raise ValueError("out must be a contiguous [M, N] tensor of X's dtype")
    return out


def _int4_call(fn, X, qweight, scales, qzeros, g_idx, out, group_size, ws, dev_status):
    K = qweight.shape[0] * 8
    N = qweight.shape[1]
    _check_x(X, K)
    M = X.shape[0]
    Y = _out(X, N, out)
    if ws is None:
        ws = workspace(M, N, K, X.device)
    nbytes = 0 if ws is None else ws.numel() * ws.element_size()
    st = getattr(_lib, fn)(_ptr(X), _ptr(qweight), _ptr(scales), _ptr(qzeros), _ptr(g_idx), _ptr(Y), M, N, K,
                           group_size, _DTYPES[X.dtype], _ptr(ws), nbytes, _ptr(dev_status), _stream(X.device))
    _check(st, fn)
    return Y


def gemm(X, qweight, scales, qzeros, g_idx=None, out=None, group_size=GROUP_SIZE, ws=None, dev_status=None):
    """Y = X . W_hat (INT4), any M."""
    return _int4_call("w4a16_gemm", X, qweight, scales, qzeros, g_idx, out, group_size, ws, dev_status)


def gemv(X, qweight, scales, qzeros, g_idx=None, out=None, group_size=GROUP_SIZE, ws=None, dev_status=None):
    """Y = X . W_hat (INT4), M <= 16 (the split-K decode kernel)."""
    return _int4_call("w4a16_gemv", X, qweight, scales, qzeros, g_idx, out, group_size, ws, dev_status)


class _GemvItem(ctypes.Structure):
    """The C struct w4a16_gemv_item."""
    _fields_ = [("X", _vp), ("qweight", _vp), ("scales", _vp), ("qzeros", _vp), ("g_idx", _vp), ("Y", _vp),
                ("M", _i), ("N", _i), ("K", _i), ("group_size", _i), ("dtype", _i)]


class GemvBatch:
    """A fixed list of decode products (each as ``gemv`` would compute it),
    launched in order by one library call (``w4a16_gemv_batch``) each time the
    object is called.

    ``items``: a sequence of ``(X, qweight, scales, qzeros, Y)`` tuples, or
    of dicts with those keys plus optional ``g_idx`` and ``group_size``.  The
    tensors are checked once, here, and kept alive by the object; a call
    re-reads their current contents (so X can be refilled between calls).
    """

    def __init__(self, items, ws=None, dev_status=None):
        rows, self._keep = [], []
        need, device = 0, None
        for it in items:
            d = dict(zip(("X", "qweight", "scales", "qzeros", "Y"), it)) if not isinstance(it, dict) else dict(it)
            X, qw, Y = d["X"], d["qweight"], d["Y"]
            K, N = qw.shape[0] * 8, qw.shape[1]
            _check_x(X, K)
            M = X.shape[0]
            _out(X, N, Y)
            g = d.get("group_size", GROUP_SIZE)
            rows.append(_GemvItem(_ptr(X), _ptr(qw), _ptr(d["scales"]), _ptr(d.get("qzeros")), _ptr(d.get("g_idx")),
                                  _ptr(Y), M, N, K, g, _DTYPES[X.dtype]))
            self._keep.append(d)
            need = max(need, workspace_bytes(M, N, K))
            device = X.device
        self._items = (_GemvItem * max(1, len(rows)))(*rows)
        self._count = len(rows)
        if ws is None and need and device is not None:
            ws = workspace(1, 1, 1, device, nbytes=need)
        self._ws = ws
        self._ws_bytes = 0 if ws is None else ws.numel() * ws.element_size()
        self._status = dev_status
        self._device = device

    def __call__(self):
        if self._count:
            st = _lib.w4a16_gemv_batch(ctypes.addressof(self._items), self._count, _ptr(self._ws), self._ws_bytes,
                                       _ptr(self._status), _stream(self._device))
            _check(st, "w4a16_gemv_batch")


def gemv_batch(items, ws=None, dev_status=None):
    """Run a list of decode products once (see ``GemvBatch``)."""
    GemvBatch(items, ws, dev_status)()


def gemm_silu_mul(X, qweight, scales, qzeros, out=None, group_size=GROUP_SIZE, ws=None, dev_status=None):
    """A = SiLU(X . W_hat[:, :F]) * (X . W_hat[:, F:]) for a gate_up weight of
    N = 2F columns (gate first), any M; returns A [M, F]."""
    K = qweight.shape[0] * 8
    N = qweight.shape[1]
    _check_x(X, K)
    M = X.shape[0]
    A = _out(X, N // 2, out)
    if ws is None:
        ws = workspace(M, N, K, X.device)
    nbytes = 0 if ws is None else ws.numel() * ws.element_size()
    st = _lib.w4a16_gemm_silu_mul(_ptr(X), _ptr(qweight), _ptr(scales), _ptr(qzeros), _ptr(A), M, N, K, group_size,
                                  _DTYPES[X.dtype], _ptr(ws), nbytes, _ptr(dev_status), _stream(X.device))
    _check(st, "w4a16_gemm_silu_mul")
    return A


def nf4_gemm(X, qweight, absmax, codebook=None, out=None, blocksize=NF4_BLOCK, ws=None, dev_status=None):
    """Y = X . W_hat (NF4), any M.  ``codebook`` None: the built-in table."""
    K = qweight.shape[0] * 8
    N = qweight.shape[1]
    _check_x(X, K)
    M = X.shape[0]
    Y = _out(X, N, out)
    if ws is None:
        ws = workspace(M, N, K, X.device)
    nbytes = 0 if ws is None else ws.numel() * ws.element_size()
    st = _lib.nf4_gemm(_ptr(X), _ptr(qweight), _ptr(absmax), _ptr(codebook), _ptr(Y), M, N, K, blocksize,
                       _DTYPES[X.dtype], _ptr(ws), nbytes, _ptr(dev_status), _stream(X.device))
    _check(st, "nf4_gemm")
    return Y


def act_order_prepack(qweight, g_idx, group_size=GROUP_SIZE, dev_status=None):
    """One-time reorder of an act-order checkpoint: (qweight_sorted, perm) with
    each group's rows contiguous; use with :func:`gemm_prepacked`.  A group
    that does not hold exactly ``group_size`` rows is reported as
    ERR_UNSUPPORTED through ``dev_status``."""
    K, N = qweight.shape[0] * 8, qweight.shape[1]
    if g_idx.dtype != torch.int32 or g_idx.numel() != K:
        raise ValueError("g_idx must be an int32 tensor of K entries")
    q_sorted = torch.empty_like(qweight)
    perm = torch.empty(K, dtype=torch.int32, device=qweight.device)
    st = _lib.w4a16_act_order_prepack(_ptr(qweight), _ptr(g_idx), K, N, group_size, _ptr(q_sorted), _ptr(perm),
                                      _ptr(dev_status), _stream(qweight.device))
    _check(st, "w4a16_act_order_prepack")
    return q_sorted, perm


def repack_awq(qweight_awq, qzeros_awq, group_size=GROUP_SIZE):
    """AWQ checkpoint (qweight int32 [K, N/8] and qzeros [K/g, N/8] packed
    along N in AWQ's column order) -> (qweight [K/8, N], qzeros [K/g, N/8]) in
    this library's layout; ``qzeros_awq`` None for symmetric weights."""
    K, C = qweight_awq.shape
    N = 8 * C
    qweight = torch.empty((K // 8, N), dtype=torch.int32, device=qweight_awq.device)
    qzeros = None if qzeros_awq is None else torch.empty_like(qzeros_awq)
    st = _lib.w4a16_repack_awq(_ptr(qweight_awq), _ptr(qzeros_awq), K, N, group_size, _ptr(qweight), _ptr(qzeros),
                               _stream(qweight_awq.device))
    _check(st, "w4a16_repack_awq")
    return qweight, qzeros


def prepacked_workspace_bytes(M: int, N: int, K: int) -> int:
    return int(_lib.w4a16_prepacked_workspace_bytes(M, N, K))


def gemm_prepacked(X, qweight_sorted, scales, qzeros, perm, out=None, group_size=GROUP_SIZE, ws=None,
                   dev_status=None):
    """Y = X . W_hat for act-order weights prepacked by :func:`act_order_prepack`."""
    K = qweight_sorted.shape[0] * 8
    N = qweight_sorted.shape[1]
    _check_x(X, K)
    M = X.shape[0]
    Y = _out(X, N, out)
    need = prepacked_workspace_bytes(M, N, K)
    if ws is None:
        ws = workspace(M, N, K, X.device, nbytes=need)
    nbytes = 0 if ws is None else ws.numel() * ws.element_size()
    st = _lib.w4a16_gemm_prepacked(_ptr(X), _ptr(qweight_sorted), _ptr(scales), _ptr(qzeros), _ptr(perm), _ptr(Y),
                                   M, N, K, group_size, _DTYPES[X.dtype], _ptr(ws), nbytes, _ptr(dev_status),
                                   _stream(X.device))
    _check(st, "w4a16_gemm_prepacked")
    return Y


def selftest_wait_timeout(dev_status, limit_ns: int = 20_000_000):
    """Run the bounded-wait self-test on ``dev_status``'s device: a wait on a
    barrier nothing completes must end after ``limit_ns`` with ERR_TIMEOUT
    written to ``dev_status``."""
    st = _lib.w4a16_selftest_wait_timeout(_ptr(dev_status), limit_ns, _stream(dev_status.device))
    _check(st, "w4a16_selftest_wait_timeout")


def dequant(qweight, scales, qzeros, g_idx=None, dtype=torch.bfloat16, group_size=GROUP_SIZE):
    """W_hat [K, N] in ``dtype`` (bit-exact dequantization)."""
    K, N = qweight.shape[0] * 8, qweight.shape[1]
    W = torch.empty((K, N), dtype=dtype, device=qweight.device)
    st = _lib.w4a16_dequant(_ptr(qweight), _ptr(scales), _ptr(qzeros), _ptr(g_idx), _ptr(W), K, N, group_size,
                            _DTYPES[dtype], _stream(qweight.device))
    _check(st, "w4a16_dequant")
    return W


def nf4_dequant(qweight, absmax, codebook=None, dtype=torch.bfloat16, blocksize=NF4_BLOCK):
    K, N = qweight.shape[0] * 8, qweight.shape[1]
    W = torch.empty((K, N), dtype=dtype, device=qweight.device)
    st = _lib.nf4_dequant(_ptr(qweight), _ptr(absmax), _ptr(codebook), _ptr(W), K, N, blocksize, _DTYPES[dtype],
                          _stream(qweight.device))
    _check(st, "nf4_dequant")
    return W


def quantize(W, group_size=GROUP_SIZE, symmetric=False):
    """RTN INT4 quantization of fp32 CUDA ``W[K, N]`` -> (qweight, scales, qzeros);
    ``symmetric``: no zero points (qzeros is None; every zero point is 8)."""
    if W.dtype != torch.float32 or not W.is_cuda or not W.is_contiguous():
        raise ValueError("W must be a contiguous CUDA float32 tensor")
    K, N = W.shape
    dev = W.device
    qweight = torch.empty((K // 8, N), dtype=torch.int32, device=dev)
    scales = torch.empty((K // group_size, N), dtype=torch.float16, device=dev)
    qzeros = None if symmetric else torch.empty((K // group_size, N // 8), dtype=torch.int32, device=dev)
    st = _lib.w4a16_quantize(_ptr(W), K, N, group_size, _ptr(qweight), _ptr(scales), _ptr(qzeros), _stream(dev))
    _check(st, "w4a16_quantize")
    return qweight, scales, qzeros


def nf4dq_gemm(X, qweight, absmax_q, absmax_s2, codebook=None, out=None, blocksize=NF4_BLOCK, ws=None,
               dev_status=None):
    """Y = X . W_hat (NF4 with double-quantized absmax), any M."""
    K = qweight.shape[0] * 8
    N = qweight.shape[1]
    _check_x(X, K)
    M = X.shape[0]
    Y = _out(X, N, out)
    if ws is None:
        ws = workspace(M, N, K, X.device)
    nbytes = 0 if ws is None else ws.numel() * ws.element_size()
    st = _lib.nf4dq_gemm(_ptr(X), _ptr(qweight), _ptr(absmax_q), _ptr(absmax_s2), _ptr(codebook), _ptr(Y), M, N, K,
                         blocksize, _DTYPES[X.dtype], _ptr(ws), nbytes, _ptr(dev_status), _stream(X.device))
    _check(st, "nf4dq_gemm")
    return Y


def nf4_double_quantize(absmax, blocksize=NF4_BLOCK):
    """Second-level quantization of an NF4 absmax [K/bs, N] -> (absmax_q uint8
    [K/bs, N], absmax_s2 float32 [K/bs, ceil(N/256)])."""
    B, N = absmax.shape
    q = torch.empty((B, N), dtype=torch.uint8, device=absmax.device)
    s2 = torch.empty((B, (N + 255) // 256), dtype=torch.float32, device=absmax.device)
    st = _lib.nf4_double_quantize(_ptr(absmax), B * blocksize, N, blocksize, _ptr(q), _ptr(s2),
                                  _stream(absmax.device))
    _check(st, "nf4_double_quantize")
    return q, s2


def nf4dq_dequant(qweight, absmax_q, absmax_s2, codebook=None, dtype=torch.bfloat16, blocksize=NF4_BLOCK):
    K, N = qweight.shape[0] * 8, qweight.shape[1]
    W = torch.empty((K, N), dtype=dtype, device=qweight.device)
    st = _lib.nf4dq_dequant(_ptr(qweight), _ptr(absmax_q), _ptr(absmax_s2), _ptr(codebook), _ptr(W), K, N, blocksize,
                            _DTYPES[dtype], _stream(qweight.device))
    _check(st, "nf4dq_dequant")
    return W


def nf4_quantize(W, codebook=None, blocksize=NF4_BLOCK):
    """NF4 quantization of fp32 CUDA ``W[K, N]`` -> (qweight, absmax)."""
    if W.dtype != torch.float32 or not W.is_cuda or not W.is_contiguous():
        raise ValueError("W must be a contiguous CUDA float32 tensor")
    K, N = W.shape
    dev = W.device
    qweight = torch.empty((K // 8, N), dtype=torch.int32, device=dev)
    absmax = torch.empty((K // blocksize, N), dtype=torch.float32, device=dev)
    st = _lib.nf4_quantize(_ptr(W), K, N, blocksize, _ptr(codebook), _ptr(qweight), _ptr(absmax), _stream(dev))
    _check(st, "nf4_quantize")
    return qweight, absmax


def nf4_codebook(device="cuda") -> torch.Tensor:
    """The library's built-in 16-entry NF4 table (``nf4_default_codebook``),
    as a float32 tensor on ``device``: the table a ``None`` codebook stands
    for in :func:`nf4_gemm`, :func:`nf4_dequant` and :func:`nf4_quantize`."""
    buf = (ctypes.c_float * 16)()
    _check(_lib.nf4_default_codebook(ctypes.addressof(buf)), "nf4_default_codebook")
    return torch.tensor(list(buf), dtype=torch.float32).to(device)
