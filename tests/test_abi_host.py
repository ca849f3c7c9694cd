"""Host-only checks of the C ABI: the library loads without a GPU, exports every
function include/w4a16.h declares, and rejects bad arguments before launching
anything (these calls fail validation, so they never reach the GPU)."""

import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "w4a16.h")


def _declared():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:w4a16_status|size_t|const char\*)\s+(\w+)\s*\(", src, flags=re.M)))


@pytest.fixture(scope="module")
def lib():
    import bit_weight_only_wise_b300 as w4

    return w4._lib


def test_header_declares_expected_entry_points():
    names = _declared()
    for n in ("w4a16_gemm", "w4a16_gemv", "nf4_gemm", "w4a16_dequant", "nf4_dequant", "w4a16_quantize",
              "nf4_quantize", "w4a16_workspace_bytes", "w4a16_status_string", "w4a16_act_order_prepack",
              "w4a16_gemm_prepacked", "w4a16_prepacked_workspace_bytes"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    import bit_weight_only_wise_b300 as w4

    for name in _declared():
        assert hasattr(lib, name), name
        assert name in w4.EXPORTED, name


def test_builtin_nf4_codebook_equals_the_oracles(lib):
    # the library's own table (host code, Newton's method on libm's erfc) and
    # the oracle's (scipy's normal quantile) are bit-identical fp32 tables
    import ctypes

    import numpy as np

    from oracle import nf4

    buf = (ctypes.c_float * 16)()
    assert lib.nf4_default_codebook(ctypes.addressof(buf)) == 0
    got = np.frombuffer(bytes(buf), dtype=np.float32)
    assert np.array_equal(got.view(np.uint32), nf4.codebook().view(np.uint32))
    assert lib.nf4_default_codebook(None) == 1  # NULL destination: invalid argument


def test_status_strings(lib):
    import bit_weight_only_wise_b300 as w4

    for s in range(5):
        assert len(w4.status_string(s)) >= 2
    assert "unknown" in w4.status_string(99)


def _gemm(lib, fn="w4a16_gemm", X=16, qw=16, sc=16, qz=16, gi=None, Y=16, M=4, N=64, K=256, g=128, dt=1,
          ws=None, wsb=0):
    return getattr(lib, fn)(X, qw, sc, qz, gi, Y, M, N, K, g, dt, ws, wsb, None, None)


def test_validation_rejects_without_launch(lib):
    import bit_weight_only_wise_b300 as w4

    INV, UNS = w4.ERR_INVALID_ARG, w4.ERR_UNSUPPORTED
    assert _gemm(lib, dt=7) == INV  # dtype
    assert _gemm(lib, N=60) == INV  # N % 8
    assert _gemm(lib, K=260) == INV  # K % 8
    assert _gemm(lib, K=192) == INV  # K % group
    assert _gemm(lib, K=384, g=48) == UNS  # group size other than 32, 64, a multiple of 128 or K
    assert _gemm(lib, K=256, g=16) == UNS
    assert _gemm(lib, K=0) == INV
    assert _gemm(lib, M=-1) == INV
    assert _gemm(lib, X=None) == INV  # null pointer
    assert _gemm(lib, qw=8) == INV  # misaligned (8 bytes)
    assert _gemm(lib, gi=4) == INV  # misaligned g_idx
    assert _gemm(lib, fn="w4a16_gemv", M=17) == INV  # decode kernel limit
    # empty problems are valid no-ops (nothing launched, pointers unused)
    assert _gemm(lib, M=0, X=None, Y=None) == w4.OK
    assert _gemm(lib, N=0, X=None, Y=None) == w4.OK
    # split-K workspace missing or too small
    need = lib.w4a16_workspace_bytes(4, 64, 256 * 32)
    if need:
        assert _gemm(lib, K=256 * 32, ws=None, wsb=0) == INV
        assert _gemm(lib, K=256 * 32, ws=16, wsb=need - 1) == INV
    # NF4
    # a codebook is optional (NULL: the built-in table) but must be aligned
    assert lib.nf4_gemm(16, 16, 16, 8, 16, 4, 64, 256, 64, 1, None, 0, None, None) == INV
    assert lib.nf4_gemm(16, 16, None, None, 16, 4, 64, 256, 64, 1, None, 0, None, None) == INV  # absmax
    assert lib.nf4_gemm(16, 16, 16, 16, 16, 4, 64, 256, 32, 1, None, 0, None, None) == UNS
    assert lib.nf4_gemm(16, 16, 16, 16, 16, 4, 64, 100, 64, 1, None, 0, None, None) == INV
    assert lib.w4a16_dequant(16, 16, 16, None, 16, 256, 60, 128, 0, None) == INV
    assert lib.nf4_dequant(16, 16, 8, 16, 256, 64, 64, 0, None) == INV
    assert lib.nf4_dequant(16, None, None, 16, 256, 64, 64, 0, None) == INV
    assert lib.w4a16_quantize(None, 256, 64, 128, 16, 16, 16, None) == INV
    assert lib.nf4_quantize(16, 256, 64, 64, 8, 16, 16, None) == INV
    assert lib.nf4_quantize(16, 256, 64, 64, None, 16, None, None) == INV
    # the wait self-test needs a status word and a limit in (0, 10 s]
    assert lib.w4a16_selftest_wait_timeout(None, 1000, None) == INV
    assert lib.w4a16_selftest_wait_timeout(16, 0, None) == INV
    assert lib.w4a16_selftest_wait_timeout(16, 20 * 10**9, None) == INV
    # act-order prepack: no in-place reorder, group size, g_idx required
    assert lib.w4a16_act_order_prepack(16, 16, 256, 64, 128, 16, 32, None, None) == INV  # aliasing
    assert lib.w4a16_act_order_prepack(16, 16, 384, 64, 48, 32, 48, None, None) == UNS
    assert lib.w4a16_act_order_prepack(16, None, 256, 64, 128, 32, 48, None, None) == INV
    need = lib.w4a16_prepacked_workspace_bytes(4, 64, 256)
    assert need >= 4 * 256 * 2
    assert lib.w4a16_gemm_prepacked(16, 16, 16, 16, 16, 16, 4, 64, 256, 128, 1, 32, need - 1, None, None) == INV
    assert lib.w4a16_gemm_prepacked(16, 16, 16, 16, None, 16, 4, 64, 256, 128, 1, 32, need, None, None) == INV


def test_workspace_sizes_are_pure_and_bounded(lib):
    assert lib.w4a16_workspace_bytes(0, 4096, 4096) == 0
    for M in (1, 4, 16):
        for K, N in ((4096, 4096), (5120, 55296), (27648, 5120), (28672, 8192)):
            b = lib.w4a16_workspace_bytes(M, N, K)
            assert b == lib.w4a16_workspace_bytes(M, N, K)
            assert b <= 64 * 1024 * 1024


def _prefill_plan_bytes(M, N, K, act):
    # the tensor-core kernel's schedule as w4a16.h documents it beside
    # w4a16_workspace_bytes: tiles of 128 columns x BT tokens run whole in full waves of
    # the 148 SMs; the tiles left over for a ragged last wave (all of them
    # below one wave) are cut along K into splits = min(148 // rest, K blocks
    # / 8) group-aligned parts, each with an fp32 partial tile
    cap = 128 if act else 256
    BT = cap if M >= cap else (M + 31) // 32 * 32
    tiles = -(-N // 128) * -(-M // BT)
    kb = -(-K // 64)
    rest = tiles % 148
    splits = max(1, min(148 // rest if rest else 1, kb // 8))
    per = -(-kb // splits)
    per += per & 1
    splits = -(-kb // per)
    if splits <= 1:
        return 0
    return 4096 * 8 * 4 + rest * splits * BT * 128 * 4


def test_prefill_schedule_workspace(lib):
    # the prefill workspace is the ticket area plus one fp32 partial tile per
    # part of each leftover tile, whichever of the plain and act-order plans
    # needs more
    for M, N, K in ((17, 150 * 128, 1024), (1024, 5120, 5120), (256, 5120, 5120), (1024, 5120, 27648),
                    (4096, 55296, 5120), (4096, 5120, 5120), (64, 8192, 8192), (300, 520, 768)):
        want = max(_prefill_plan_bytes(M, N, K, False), _prefill_plan_bytes(M, N, K, True))
        assert lib.w4a16_workspace_bytes(M, N, K) == want, (M, N, K)
    # one full wave and no leftover: no partial tiles
    assert lib.w4a16_workspace_bytes(256, 148 * 128, 4096) == _prefill_plan_bytes(256, 148 * 128, 4096, True)
    assert _prefill_plan_bytes(256, 148 * 128, 4096, False) == 0


def test_noalloc_scratch_fits_every_decode_call(lib):
    # the header promises that the allocation-free decode entry's fixed
    # scratch array serves every M <= 16 under the current split-K plan
    m = re.search(r"#define\s+W4A16_NOALLOC_SCRATCH_BYTES\s+\((\d+)u\s*<<\s*(\d+)\)", open(HEADER).read())
    assert m, "W4A16_NOALLOC_SCRATCH_BYTES not found"
    scratch = int(m.group(1)) << int(m.group(2))
    for M in range(1, 17):
        for K, N in ((128, 8), (4096, 4096), (5120, 55296), (4095 * 128, 256), (256, 4096 * 256)):
            assert lib.w4a16_workspace_bytes(M, N, K) <= scratch, (M, N, K)


def _header_int(name):
    m = re.search(rf"#define\s+{name}\s+(\d+)", open(HEADER).read())
    assert m, name
    return int(m.group(1))


def test_size_limits(lib):
    # sizes past the header's limits are rejected before anything is launched,
    # and the pure size functions do no arithmetic on them
    import bit_weight_only_wise_b300 as w4

    MAX_M, MAX_N, MAX_K = (_header_int(n) for n in ("W4A16_MAX_M", "W4A16_MAX_N", "W4A16_MAX_K"))
    assert (MAX_M, MAX_N, MAX_K) == (65535 * 128, 4096 * 256, 65535 * 8)
    INV = w4.ERR_INVALID_ARG
    assert _gemm(lib, M=MAX_M + 1) == INV
    assert _gemm(lib, M=2**31 - 1) == INV
    assert _gemm(lib, N=MAX_N + 8) == INV
    assert _gemm(lib, K=(MAX_K // 128 + 1) * 128) == INV
    assert lib.nf4_gemm(16, 16, 16, 16, 16, MAX_M + 1, 64, 256, 64, 1, None, 0, None, None) == INV
    assert lib.w4a16_gemv_noalloc(16, 16, 16, 16, None, 16, 1, 2**31 - 8, 256, 128, 1, None, None) == INV
    assert lib.w4a16_gemv_noalloc(16, 16, 16, 16, None, 16, 1, 64, 2**31 - 8, 128, 1, None, None) == INV
    big = 2**31 - 1
    for M, N, K in ((big, 64, 256), (4, big, 256), (4, 64, big), (big, big, big), (MAX_M + 1, MAX_N, MAX_K)):
        assert lib.w4a16_workspace_bytes(M, N, K) == 0, (M, N, K)
        assert lib.w4a16_prepacked_workspace_bytes(M, N, K) == 0, (M, N, K)
    # at the limits themselves the sizes are defined and bounded
    for M in (1, 16, 17, 4096, MAX_M):
        for N, K in ((MAX_N, 128), (256, MAX_K // 128 * 128), (MAX_N, MAX_K // 128 * 128)):
            assert 0 <= lib.w4a16_workspace_bytes(M, N, K) <= 1 << 36, (M, N, K)
