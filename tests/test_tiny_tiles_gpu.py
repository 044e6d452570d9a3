"""Long look-back chains from tiny tiles: the library built with 4 elements
per thread (tiles of 8 * 32 * 4 = 1024 elements in the large plain scan and
the segmented scan, against 7168 by default), so that a call of 2^24
elements chains 16,388 tiles and every look-back crosses many 32-tile
windows.  Parity with the oracle, alone and under the schedule-perturbation
hook (seeded delays that shuffle the order in which tiles publish), with the
unbounded and a bounded look-back window."""
import ctypes
import os

import numpy as np
import pytest

import oracle
import synth

pytestmark = [pytest.mark.gpu, pytest.mark.slow]

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import device_wide_prefix_gb300 as dwp  # noqa: E402
from device_wide_prefix_gb300 import build as dwp_build  # noqa: E402

TINY_LIB = os.path.join(os.path.dirname(dwp.__file__), "libdwp_tiny.so")
SMALL_MAX = 1 << 23  # the large kernel (the one with tiny tiles) runs above this
OPS = {"u32_add": dwp.DWP_U32_ADD, "f32_add": dwp.DWP_F32_ADD, "u32_max": dwp.DWP_U32_MAX}
SENTINEL = 0xDEADBEEF


@pytest.fixture(scope="module")
def lib():
    dwp_build.build(extra=["-DDWP_SCAN_ITEMS=4", "-DDWP_SEG_ITEMS=4"], lib=TINY_LIB)
    return dwp.load(TINY_LIB)


@pytest.fixture(scope="module")
def ref():
    return oracle.Oracle()


def _stream():
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def scan(lib, x, op, inclusive):
    t = torch.from_numpy(x.view(np.float32 if op == "f32_add" else np.int32)).cuda()
    y = torch.empty_like(t)
    entry = lib.dwp_scan_inclusive if inclusive else lib.dwp_scan_exclusive
    sb = ctypes.c_size_t(0)
    assert entry(OPS[op], None, None, x.size, None, ctypes.byref(sb), None) == dwp.DWP_SUCCESS
    scratch = torch.empty(sb.value, dtype=torch.uint8, device="cuda")
    assert entry(OPS[op], ctypes.c_void_p(t.data_ptr()), ctypes.c_void_p(y.data_ptr()), x.size,
                 ctypes.c_void_p(scratch.data_ptr()), ctypes.byref(sb), _stream()) == dwp.DWP_SUCCESS
    status = lib.dwp_read_status(ctypes.c_void_p(scratch.data_ptr()), _stream())
    return y.cpu().numpy().view(x.dtype), status, sb.value


def check_scan(ref, x, op, inclusive, y):
    if op == "f32_add":
        yr, ab = ref.scan_f32_add(x, inclusive)
        assert (np.abs(y.astype(np.float64) - yr) <= 1e-4 * ab + 1e-6).all()
    else:
        assert np.array_equal(y, ref.scan(op, x, inclusive))


def values(n, op, seed):
    return synth.f32_values(n, seed) if op == "f32_add" else synth.u32_full_values(n, seed)


def test_the_build_has_tiny_tiles(lib):
    """The size query counts one descriptor per 1024-element tile."""
    n = (1 << 24) + 4097
    sb = ctypes.c_size_t(0)
    assert lib.dwp_scan_exclusive(0, None, None, n, None, ctypes.byref(sb), None) == dwp.DWP_SUCCESS
    assert sb.value == 128 + 8 * -(-n // 1024)


@pytest.mark.parametrize("op", sorted(OPS))
@pytest.mark.parametrize("inclusive", [False, True])
def test_plain_scan_long_chains(lib, ref, op, inclusive):
    for n in (SMALL_MAX + 1, (1 << 24) + 4097):
        x = values(n, op, 300 + n % 31)
        y, status, _ = scan(lib, x, op, inclusive)
        assert status == dwp.DWP_SUCCESS
        check_scan(ref, x, op, inclusive, y)


@pytest.mark.parametrize("window", [0, 32])
@pytest.mark.parametrize("seed", [0x71, 0x72])
def test_plain_scan_long_chains_under_perturbation(lib, ref, window, seed):
    n = (1 << 24) + 4097
    x = values(n, "u32_add", seed)
    try:
        assert lib.dwp_set_lookback_window(window) == dwp.DWP_SUCCESS
        assert lib.dwp_debug_set_delay(seed, 100000, 20000) == dwp.DWP_SUCCESS
        y, status, _ = scan(lib, x, "u32_add", False)
    finally:
        lib.dwp_debug_set_delay(0, 0, 0)
        lib.dwp_set_lookback_window(0)
    assert status == dwp.DWP_SUCCESS
    check_scan(ref, x, "u32_add", False, y)


def segscan(lib, values_, offsets, inclusive):
    n, nseg = values_.size, offsets.size - 1
    v = torch.from_numpy(values_.view(np.int32)).cuda()
    o = torch.from_numpy(np.ascontiguousarray(offsets, dtype=np.uint32).view(np.int32)).cuda()
    out = torch.full((n,), SENTINEL - (1 << 32), dtype=torch.int32, device="cuda")
    mode = dwp.DWP_INCLUSIVE if inclusive else dwp.DWP_EXCLUSIVE
    sb = ctypes.c_size_t(0)
    assert lib.dwp_segmented_scan_u32(None, None, nseg, None, n, mode, None, ctypes.byref(sb), None) == 0
    scratch = torch.empty(sb.value, dtype=torch.uint8, device="cuda")
    assert lib.dwp_segmented_scan_u32(ctypes.c_void_p(v.data_ptr()), ctypes.c_void_p(o.data_ptr()), nseg,
                                      ctypes.c_void_p(out.data_ptr()), n, mode,
                                      ctypes.c_void_p(scratch.data_ptr()), ctypes.byref(sb),
                                      _stream()) == dwp.DWP_SUCCESS
    status = lib.dwp_read_status(ctypes.c_void_p(scratch.data_ptr()), _stream())
    return out.cpu().numpy().view(np.uint32), status


@pytest.mark.parametrize("inclusive", [False, True])
@pytest.mark.parametrize("perturbed", [False, True])
def test_segmented_scan_long_chains(lib, ref, inclusive, perturbed):
    n = (1 << 22) + 5  # 4097 tiles of 1024 rows
    for offsets in (synth.segment_offsets(n, seed=0x73),
                    np.array([0, 3, 3, n - 2000, n], np.uint32)):  # two segments over thousands of tiles
        vals = synth.u32_byte_values(n, seed=0x74)
        try:
            if perturbed:
                assert lib.dwp_debug_set_delay(0x75, 100000, 20000) == dwp.DWP_SUCCESS
            got, status = segscan(lib, vals, offsets, inclusive)
        finally:
            lib.dwp_debug_set_delay(0, 0, 0)
        assert status == dwp.DWP_SUCCESS
        want = ref.segmented_scan_u32(vals, offsets, inclusive, out=np.full(n, SENTINEL, np.uint32))
        assert np.array_equal(got, want)
