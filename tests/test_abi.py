"""The C-ABI library without a GPU: it loads, exports every symbol the header
declares, and its host-side validation rejects bad arguments before any CUDA
call (fake, never-dereferenced addresses are enough for that)."""
import os
import re

import pytest

import device_wide_prefix_gb300 as dwp
from device_wide_prefix_gb300 import build as dwp_build

HEADER = os.path.join(dwp_build.INCLUDE, "dwp.h")
A = 0x7F0000000000  # a 16-byte aligned fake device address

# Fake addresses must never reach a real GPU: every case below is rejected by
# host validation, but a wrong expectation would hand one to the CUDA runtime.
pytestmark = pytest.mark.skipif(
    __import__("torch").cuda.is_available(),
    reason="host-validation tests use fake device addresses; run them without a GPU")


@pytest.fixture(scope="module")
def lib():
    dwp_build.build()
    return dwp.load()


def declared_functions():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(dwp_\w+)\s*\(", text, re.M)))


def test_exports_every_declared_symbol(lib):
    names = declared_functions()
    assert names, "no declarations parsed"
    assert sorted(dwp.EXPORTS) == names
    for name in names:
        assert hasattr(lib, name), name


def test_version_and_status_strings(lib):
    assert dwp.dwp_version() >= 100
    for code in range(10):
        s = dwp.dwp_status_string(code)
        assert s.startswith("DWP_") and "UNKNOWN" not in s
    assert dwp.dwp_status_string(dwp.DWP_ERR_BOUNDS) == "DWP_ERR_BOUNDS"
    assert "UNKNOWN" in dwp.dwp_status_string(99)


def test_scan_size_query(lib):
    tile = None
    for n in (0, 1, 5, 1 << 20, (1 << 28), (1 << 32) - 1):
        for entry in (dwp.dwp_scan_exclusive, dwp.dwp_scan_inclusive):
            st, b = entry(dwp.DWP_U32_ADD, 0, 0, n, 0, 0, 0)
            assert st == dwp.DWP_SUCCESS
            assert b >= 128 and (b - 128) % 8 == 0
            tiles = (b - 128) // 8
            if n == 0:
                assert tiles == 0
            else:
                if tile is None:
                    tile = n if n > 1 else None
                assert tiles >= 1
    # scratch sized for a large n serves every smaller n: the size query
    # never decreases (the small-input kernel sizes its tile by n)
    prev = 0
    for n in sorted({1, 2, 3071, 3072, 3073, (1 << 18) - 1, 1 << 18, (1 << 18) + 1, 15360 * 20,
                     15360 * 86, 15360 * 86 + 1, (1 << 22) - 1, 1 << 22, (1 << 22) + 1,
                     (1 << 23) - 1, 1 << 23, (1 << 23) + 1, 1 << 24,
                     (1 << 28) + 5, (1 << 32) - 1}):
        b = dwp.dwp_scan_exclusive(dwp.DWP_U32_ADD, 0, 0, n, 0, 0, 0)[1]
        assert b >= prev, n
        prev = b
    # above 2^23 one descriptor per tile of the large-input kernel; its tile
    # size T follows from a large query
    big = 1 << 30
    tiles = (dwp.dwp_scan_exclusive(dwp.DWP_U32_ADD, 0, 0, big, 0, 0, 0)[1] - 128) // 8
    T = -(-big // tiles)
    assert -(-big // T) == tiles
    for k in (2000, 7777):
        assert k * T > 1 << 23
        assert dwp.dwp_scan_exclusive(dwp.DWP_U32_ADD, 0, 0, k * T, 0, 0, 0)[1] == 128 + 8 * k
        assert dwp.dwp_scan_exclusive(dwp.DWP_U32_ADD, 0, 0, k * T + 1, 0, 0, 0)[1] == 128 + 8 * (k + 1)


def test_scan_validation(lib):
    E = dwp.dwp_scan_exclusive
    n = 1000
    _, need = E(dwp.DWP_U32_ADD, 0, 0, n, 0, 0, 0)
    scratch = A + (1 << 30)
    # unknown op, n too large
    assert E(7, A, A + 8192, n, scratch, need, 0)[0] == dwp.DWP_ERR_INVALID_VALUE
    assert E(-1, A, A + 8192, n, scratch, need, 0)[0] == dwp.DWP_ERR_INVALID_VALUE
    assert E(dwp.DWP_U32_ADD, A, A + 8192, 1 << 32, scratch, need, 0)[0] == dwp.DWP_ERR_INVALID_VALUE
    # scratch too small
    assert E(dwp.DWP_U32_ADD, A, A + 8192, n, scratch, need - 1, 0)[0] == dwp.DWP_ERR_SCRATCH_TOO_SMALL
    # null data pointers with n > 0
    assert E(dwp.DWP_U32_ADD, 0, A, n, scratch, need, 0)[0] == dwp.DWP_ERR_INVALID_VALUE
    assert E(dwp.DWP_U32_ADD, A, 0, n, scratch, need, 0)[0] == dwp.DWP_ERR_INVALID_VALUE
    # misaligned pointers
    assert E(dwp.DWP_U32_ADD, A + 4, A + 8192, n, scratch, need, 0)[0] == dwp.DWP_ERR_MISALIGNED
    assert E(dwp.DWP_U32_ADD, A, A + 8200, n, scratch, need, 0)[0] == dwp.DWP_ERR_MISALIGNED
    assert E(dwp.DWP_U32_ADD, A, A + 8192, n, scratch + 8, need, 0)[0] == dwp.DWP_ERR_MISALIGNED
    # partial overlap of in and out; scratch overlapping data
    assert E(dwp.DWP_U32_ADD, A, A + 16, n, scratch, need, 0)[0] == dwp.DWP_ERR_ALIASING
    assert E(dwp.DWP_U32_ADD, A, A + 8192, n, A + 3008, need, 0)[0] == dwp.DWP_ERR_ALIASING
    assert E(dwp.DWP_U32_ADD, A, A + 8192, n, A + 8192 + 16, need, 0)[0] == dwp.DWP_ERR_ALIASING


def test_null_scratch_bytes_pointer(lib):
    import ctypes
    st = lib.dwp_scan_exclusive(0, None, None, 10, None, ctypes.POINTER(ctypes.c_size_t)(), None)
    assert st == dwp.DWP_ERR_INVALID_VALUE
    assert lib.dwp_read_status(None, None) == dwp.DWP_ERR_INVALID_VALUE
    v = ctypes.c_uint32(7)
    assert lib.dwp_read_fallbacks(None, None, ctypes.byref(v)) == dwp.DWP_ERR_INVALID_VALUE
    assert lib.dwp_read_fallbacks(ctypes.c_void_p(4096), None, None) == dwp.DWP_ERR_INVALID_VALUE
    assert v.value == 7


def test_recurrence_size_query_and_validation(lib):
    R = dwp.dwp_linear_recurrence_f32
    st, b0 = R(0, 0, 0, 0, dwp.DWP_INCLUSIVE, 0, 0, 0)
    assert st == dwp.DWP_SUCCESS and b0 == 128
    _, b1 = R(0, 0, 0, 1, dwp.DWP_INCLUSIVE, 0, 0, 0)
    assert b1 == 128 + 16  # two descriptor words per tile
    T = 1
    while R(0, 0, 0, 2 * T, dwp.DWP_INCLUSIVE, 0, 0, 0)[1] == b1:
        T *= 2
    lo, hi = T, 2 * T
    while hi - lo > 1:
        mid = (lo + hi) // 2
        if R(0, 0, 0, mid, dwp.DWP_INCLUSIVE, 0, 0, 0)[1] == b1:
            lo = mid
        else:
            hi = mid
    T = lo
    for k in (1, 9, 1000):
        assert R(0, 0, 0, k * T, dwp.DWP_EXCLUSIVE, 0, 0, 0)[1] == 128 + 16 * k
        assert R(0, 0, 0, k * T + 1, dwp.DWP_EXCLUSIVE, 0, 0, 0)[1] == 128 + 16 * (k + 1)
    n = 1000
    need = R(0, 0, 0, n, dwp.DWP_INCLUSIVE, 0, 0, 0)[1]
    a, b, h, s = A, A + 8192, A + 16384, A + (1 << 30)
    ok = dwp.DWP_INCLUSIVE
    assert R(a, b, h, n, 2, s, need, 0)[0] == dwp.DWP_ERR_INVALID_VALUE
    assert R(a, b, h, 1 << 32, ok, s, need, 0)[0] == dwp.DWP_ERR_INVALID_VALUE
    assert R(a, b, h, n, ok, s, need - 1, 0)[0] == dwp.DWP_ERR_SCRATCH_TOO_SMALL
    assert R(0, b, h, n, ok, s, need, 0)[0] == dwp.DWP_ERR_INVALID_VALUE
    assert R(a, 0, h, n, ok, s, need, 0)[0] == dwp.DWP_ERR_INVALID_VALUE
    assert R(a, b, 0, n, ok, s, need, 0)[0] == dwp.DWP_ERR_INVALID_VALUE
    assert R(a + 4, b, h, n, ok, s, need, 0)[0] == dwp.DWP_ERR_MISALIGNED
    assert R(a, b + 8, h, n, ok, s, need, 0)[0] == dwp.DWP_ERR_MISALIGNED
    assert R(a, b, h + 12, n, ok, s, need, 0)[0] == dwp.DWP_ERR_MISALIGNED
    assert R(a, b, h, n, ok, s + 8, need, 0)[0] == dwp.DWP_ERR_MISALIGNED
    assert R(a, b, b + 16, n, ok, s, need, 0)[0] == dwp.DWP_ERR_ALIASING   # h overlaps b partly
    assert R(a, b, a + 32, n, ok, s, need, 0)[0] == dwp.DWP_ERR_ALIASING   # h overlaps a partly
    assert R(a, b, h, n, ok, h + 16, need, 0)[0] == dwp.DWP_ERR_ALIASING   # scratch over h
    import ctypes
    assert lib.dwp_linear_recurrence_f32(None, None, None, 10, 1, None, None, None) == dwp.DWP_ERR_INVALID_VALUE


def test_segreduce_size_query_and_validation(lib):
    R = dwp.dwp_segmented_reduce_u32
    for n in (0, 1, 1 << 20, (1 << 32) - 1):
        st, b = R(0, 0, 0, 0, n, 0, 0, 0)
        assert st == dwp.DWP_SUCCESS and b == 128  # no per-tile state
    v, o, out, s = A, A + 8192, A + 16384, A + (1 << 30)
    n, nseg = 1000, 10
    assert R(v, o, nseg, out, 1 << 32, s, 128, 0)[0] == dwp.DWP_ERR_INVALID_VALUE
    assert R(v, o, (1 << 32) - 1, out, n, s, 128, 0)[0] == dwp.DWP_ERR_INVALID_VALUE
    assert R(v, o, nseg, out, n, s, 127, 0)[0] == dwp.DWP_ERR_SCRATCH_TOO_SMALL
    assert R(0, o, nseg, out, n, s, 128, 0)[0] == dwp.DWP_ERR_INVALID_VALUE
    assert R(v, 0, nseg, out, n, s, 128, 0)[0] == dwp.DWP_ERR_INVALID_VALUE
    assert R(v, o, nseg, 0, n, s, 128, 0)[0] == dwp.DWP_ERR_INVALID_VALUE
    assert R(v + 4, o, nseg, out, n, s, 128, 0)[0] == dwp.DWP_ERR_MISALIGNED
    assert R(v, o + 2, nseg, out, n, s, 128, 0)[0] == dwp.DWP_ERR_MISALIGNED
    assert R(v, o, nseg, out + 1, n, s, 128, 0)[0] == dwp.DWP_ERR_MISALIGNED
    assert R(v, o, nseg, out, n, s + 4, 128, 0)[0] == dwp.DWP_ERR_MISALIGNED
    assert R(v, o, nseg, v + 400, n, s, 128, 0)[0] == dwp.DWP_ERR_ALIASING    # out inside values
    assert R(v, o, nseg, o + 8, n, s, 128, 0)[0] == dwp.DWP_ERR_ALIASING      # out over offsets
    assert R(v, o, nseg, out, n, out + 16, 128, 0)[0] == dwp.DWP_ERR_ALIASING  # scratch over out


def test_two_level_size_query_and_validation(lib):
    R = dwp.dwp_scan_two_level
    assert R(dwp.DWP_U32_ADD, dwp.DWP_EXCLUSIVE, 0, 0, 0, 0, 0, 0) == (dwp.DWP_SUCCESS, 128)
    assert R(dwp.DWP_U32_ADD, dwp.DWP_EXCLUSIVE, 0, 0, 1, 0, 0, 0) == (dwp.DWP_SUCCESS, 132)
    assert R(dwp.DWP_U32_ADD, dwp.DWP_EXCLUSIVE, 0, 0, 4096 * 4, 0, 0, 0) == (dwp.DWP_SUCCESS, 144)
    assert R(dwp.DWP_U32_ADD, dwp.DWP_EXCLUSIVE, 0, 0, 4096 * 4 + 1, 0, 0, 0) == (dwp.DWP_SUCCESS, 148)
    # a 4-byte total per 4096-element block
    for n in (4096, 4097, 7168, 12000, 1 << 20, (1 << 26) - 1):
        assert R(0, 0, 0, 0, n, 0, 0, 0)[1] == 128 + 4 * (-(-n // 4096)), n
    assert R(dwp.DWP_U32_ADD, dwp.DWP_EXCLUSIVE, 0, 0, 1 << 26, 0, 0, 0) == (dwp.DWP_SUCCESS, 128 + 4 * 16384)
    assert R(dwp.DWP_U32_ADD, dwp.DWP_EXCLUSIVE, 0, 0, (1 << 26) + 1, 0, 0, 0)[0] == dwp.DWP_ERR_INVALID_VALUE
    n, need = 1000, 132
    s = A + (1 << 30)
    assert R(5, 0, A, A + 8192, n, s, need, 0)[0] == dwp.DWP_ERR_INVALID_VALUE
    assert R(0, 3, A, A + 8192, n, s, need, 0)[0] == dwp.DWP_ERR_INVALID_VALUE
    assert R(0, 0, A, A + 8192, n, s, need - 1, 0)[0] == dwp.DWP_ERR_SCRATCH_TOO_SMALL
    assert R(0, 0, 0, A + 8192, n, s, need, 0)[0] == dwp.DWP_ERR_INVALID_VALUE
    assert R(0, 0, A + 4, A + 8192, n, s, need, 0)[0] == dwp.DWP_ERR_MISALIGNED
    assert R(0, 0, A, A + 16, n, s, need, 0)[0] == dwp.DWP_ERR_ALIASING
    assert R(0, 0, A, A + 8192, n, A + 32, need, 0)[0] == dwp.DWP_ERR_ALIASING


def test_staged_compaction_size_query_and_validation(lib):
    R = dwp.dwp_compact_by_flags_staged
    scan = dwp.dwp_scan_exclusive
    for n in (0, 1, 17, 1000, (1 << 23) + 1, 1 << 26):
        st, need = R(0, 0, n, 0, 0, 0, 0, 0)
        assert st == dwp.DWP_SUCCESS
        scan_need = scan(dwp.DWP_U32_ADD, 0, 0, n, 0, 0, 0)[1]
        r16 = lambda b: (b + 15) // 16 * 16  # noqa: E731
        assert need == r16(scan_need) + 2 * r16(4 * n), n
    n = 1000
    _, need = R(0, 0, n, 0, 0, 0, 0, 0)
    rec, fl, out, cnt, s = A, A + (1 << 20), A + (2 << 20), A + (3 << 20), A + (4 << 20)
    assert R(rec, fl, n, out, cnt, s, need - 1, 0)[0] == dwp.DWP_ERR_SCRATCH_TOO_SMALL
    assert R(rec, fl, n, out, 0, s, need, 0)[0] == dwp.DWP_ERR_INVALID_VALUE     # no count
    assert R(0, fl, n, out, cnt, s, need, 0)[0] == dwp.DWP_ERR_INVALID_VALUE     # no records
    assert R(rec + 8, fl, n, out, cnt, s, need, 0)[0] == dwp.DWP_ERR_MISALIGNED
    assert R(rec, fl, n, out, cnt + 2, s, need, 0)[0] == dwp.DWP_ERR_MISALIGNED
    assert R(rec, fl, n, rec + 16, cnt, s, need, 0)[0] == dwp.DWP_ERR_ALIASING  # out over records
    assert R(rec, fl, n, out, out + 16, s, need, 0)[0] == dwp.DWP_ERR_ALIASING  # count inside out
    assert R(rec, fl, n, out, cnt, fl, need, 0)[0] == dwp.DWP_ERR_ALIASING      # scratch over flags
    assert R(rec, fl, 1 << 32, out, cnt, s, need, 0)[0] == dwp.DWP_ERR_INVALID_VALUE


def test_test_hooks_validate_their_arguments(lib):
    assert dwp.dwp_debug_set_delay(1, 1000001, 10) == dwp.DWP_ERR_INVALID_VALUE
    assert dwp.dwp_debug_set_delay(1, 10, 100001) == dwp.DWP_ERR_INVALID_VALUE
    assert dwp.dwp_debug_set_delay(0, 0, 0) == dwp.DWP_SUCCESS
    assert dwp.dwp_debug_warp_scan_trace(A, 0, A, 0) == dwp.DWP_ERR_INVALID_VALUE
    assert dwp.dwp_debug_warp_scan_trace(A, 33, A, 0) == dwp.DWP_ERR_INVALID_VALUE
    assert dwp.dwp_debug_warp_scan_trace(0, 8, A, 0) == dwp.DWP_ERR_INVALID_VALUE
    assert dwp.dwp_debug_warp_scan_trace(A, 8, 0, 0) == dwp.DWP_ERR_INVALID_VALUE
    assert dwp.dwp_read_lookback_stats(0, 0)[0] == dwp.DWP_ERR_INVALID_VALUE
    assert dwp.dwp_set_lookback_window(0) == dwp.DWP_SUCCESS


def test_static_scratch_rejects_before_any_cuda_call(lib):
    L = dwp.load()
    assert L.dwp_scan_static_scratch(dwp.DWP_U32_ADD, 7, None, None, 10, None) == dwp.DWP_ERR_INVALID_VALUE
    assert L.dwp_scan_static_scratch(9, dwp.DWP_EXCLUSIVE, None, None, 10, None) == dwp.DWP_ERR_INVALID_VALUE
    assert (L.dwp_scan_static_scratch(dwp.DWP_U32_ADD, dwp.DWP_EXCLUSIVE, None, None, (1 << 28) + 1, None)
            == dwp.DWP_ERR_SCRATCH_TOO_SMALL)
