"""The look-back kernels in the debug bounds build (-DDWP_DEBUG_BOUNDS=1):
the plain scan, the segmented scan, compaction, the linear recurrence and
the segmented reduction check every global access against its buffer
first, and an access that would leave it is skipped and reported as
DWP_ERR_BOUNDS instead of being made.  The checked build runs over the
sizes where index arithmetic is most likely to slip: tile and tier edges,
ragged tails, the switch between the two plain-scan kernels, in place, a
rescued tile and a bounded window; for the segmented scan and reduction the
global offset search and rows outside the segments; for compaction none,
some and all records kept.  It must report no bounds error and still match
the oracle."""
import ctypes
import os

import numpy as np
import pytest

import oracle
import synth

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import device_wide_prefix_gb300 as dwp  # noqa: E402
from device_wide_prefix_gb300 import build as dwp_build  # noqa: E402

BOUNDS_LIB = os.path.join(os.path.dirname(dwp.__file__), "libdwp_bounds.so")
LARGE_TILE = 7168
SMALL_MAX = 1 << 23
OPS = {"u32_add": dwp.DWP_U32_ADD, "f32_add": dwp.DWP_F32_ADD, "u32_max": dwp.DWP_U32_MAX}


@pytest.fixture(scope="module")
def lib():
    dwp_build.build(extra=["-DDWP_DEBUG_BOUNDS=1"], lib=BOUNDS_LIB)
    return dwp.load(BOUNDS_LIB)


@pytest.fixture(scope="module")
def ref():
    return oracle.Oracle()


def run(lib, x, op, inclusive, inplace=False):
    """One call of the checked library; returns (output, device status)."""
    t = torch.from_numpy(x.view(np.float32 if op == "f32_add" else np.int32)).cuda()
    y = t if inplace else torch.empty_like(t)
    sb = ctypes.c_size_t(0)
    entry = lib.dwp_scan_inclusive if inclusive else lib.dwp_scan_exclusive
    assert entry(OPS[op], None, None, x.size, None, ctypes.byref(sb), None) == dwp.DWP_SUCCESS
    scratch = torch.empty(max(sb.value, 16), dtype=torch.uint8, device="cuda")
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    st = entry(OPS[op], ctypes.c_void_p(t.data_ptr()), ctypes.c_void_p(y.data_ptr()), x.size,
               ctypes.c_void_p(scratch.data_ptr()), ctypes.byref(sb), stream)
    assert st == dwp.DWP_SUCCESS
    status = lib.dwp_read_status(ctypes.c_void_p(scratch.data_ptr()), stream)
    return y.cpu().numpy().view(x.dtype), status


def check(ref, x, op, inclusive, y):
    if op == "f32_add":
        yr, ab = ref.scan_f32_add(x, inclusive)
        assert (np.abs(y.astype(np.float64) - yr) <= 1e-4 * ab + 1e-6).all()
    else:
        assert np.array_equal(y, ref.scan(op, x, inclusive))


def values(n, op, seed):
    return synth.f32_values(n, seed) if op == "f32_add" else synth.u32_full_values(n, seed)


SIZES = (1, 3, 4, 5, 3071, 3072, 3073, (1 << 18) + 1, 7167, 7168 * 50 + 3, (1 << 20) + 1,
         15360 * 70 - 1, SMALL_MAX - 1, SMALL_MAX, SMALL_MAX + 1, LARGE_TILE * 1500 + 4097)


@pytest.mark.parametrize("op", sorted(OPS))
@pytest.mark.parametrize("inclusive", [False, True])
def test_no_bounds_error_at_tile_and_tier_edges(lib, ref, op, inclusive):
    for n in SIZES:
        x = values(n, op, 900 + n % 89)
        y, status = run(lib, x, op, inclusive)
        assert status == dwp.DWP_SUCCESS, (n, dwp.status_string(status))
        check(ref, x, op, inclusive, y)


@pytest.mark.parametrize("n", [7168 * 50 + 9, LARGE_TILE * 1500 + 9])
def test_no_bounds_error_in_place(lib, ref, n):
    x = values(n, "u32_add", 7)
    y, status = run(lib, x.copy(), "u32_add", False, inplace=True)
    assert status == dwp.DWP_SUCCESS
    check(ref, x, "u32_add", False, y)


@pytest.mark.parametrize("n", [15360 * 100 + 77, LARGE_TILE * 1500 + 77])
def test_no_bounds_error_with_a_rescued_tile_and_a_window(lib, ref, n):
    """The Decoupled Fallback reads a tile from the input, and a bounded
    window publishes intermediates: both paths under the checks."""
    x = values(n, "u32_add", 8)
    try:
        lib.dwp_debug_set_fault(7, 0, 64)
        y, status = run(lib, x, "u32_add", True)
        assert status == dwp.DWP_SUCCESS
        check(ref, x, "u32_add", True, y)
        assert lib.dwp_set_lookback_window(32) == dwp.DWP_SUCCESS
        y, status = run(lib, x, "u32_add", True)
        assert status == dwp.DWP_SUCCESS
        check(ref, x, "u32_add", True, y)
    finally:
        lib.dwp_set_lookback_window(0)
        lib.dwp_debug_set_fault(0xFFFFFFFF, 0, 0)


def test_the_default_library_is_not_the_checked_one(lib):
    assert os.path.abspath(dwp.LIB_PATH) != os.path.abspath(BOUNDS_LIB)


# ------------------------------------------------ segmented scan, compaction

SENTINEL = 0xDEADBEEF


def _stream():
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def seg_run(lib, values, offsets, inclusive):
    n, nseg = values.size, offsets.size - 1
    v = torch.from_numpy(values.view(np.int32)).cuda()
    o = torch.from_numpy(np.ascontiguousarray(offsets, dtype=np.uint32).view(np.int32)).cuda()
    out = torch.full((n,), SENTINEL - (1 << 32), dtype=torch.int32, device="cuda")
    sb = ctypes.c_size_t(0)
    mode = dwp.DWP_INCLUSIVE if inclusive else dwp.DWP_EXCLUSIVE
    assert lib.dwp_segmented_scan_u32(None, None, nseg, None, n, mode, None, ctypes.byref(sb), None) == 0
    scratch = torch.empty(max(sb.value, 16), dtype=torch.uint8, device="cuda")
    st = lib.dwp_segmented_scan_u32(ctypes.c_void_p(v.data_ptr()), ctypes.c_void_p(o.data_ptr()), nseg,
                                    ctypes.c_void_p(out.data_ptr()), n, mode,
                                    ctypes.c_void_p(scratch.data_ptr()), ctypes.byref(sb), _stream())
    assert st == dwp.DWP_SUCCESS
    status = lib.dwp_read_status(ctypes.c_void_p(scratch.data_ptr()), _stream())
    return out.cpu().numpy().view(np.uint32), status


def seg_cases():
    yield "skewed 1", np.array([0, 1], np.uint32), 1
    for n in (7167, 7168 * 3 + 5, (1 << 20) + 3):
        yield "skewed %d" % n, synth.segment_offsets(n, seed=40 + n % 7), n
    n = 7168 * 40 + 11  # more offsets than the per-block sample: the global search
    yield "every 100 rows", np.append(np.arange(0, n, 100, dtype=np.uint32), np.uint32(n)), n
    n = 7168 * 9 + 3  # rows outside the segments at both ends, empty segments
    yield "uncovered ends", np.array([5, 5, 5, 7168, 7169, 7169, 30000, n - 7], np.uint32), n


@pytest.mark.parametrize("inclusive", [False, True])
def test_segmented_scan_no_bounds_error(lib, ref, inclusive):
    for name, offsets, n in seg_cases():
        values = synth.u32_byte_values(n, seed=50 + n % 13)
        got, status = seg_run(lib, values, offsets, inclusive)
        assert status == dwp.DWP_SUCCESS, (name, dwp.status_string(status))
        want = ref.segmented_scan_u32(values, offsets, inclusive, out=np.full(n, SENTINEL, np.uint32))
        assert np.array_equal(got, want), name


def compact_run(lib, rec, flags):
    n = flags.size
    r = torch.from_numpy(rec.view(np.int32)).cuda()
    f = torch.from_numpy(flags).cuda()
    out = torch.full_like(r, SENTINEL - (1 << 32))
    cnt = torch.zeros(1, dtype=torch.int32, device="cuda")
    sb = ctypes.c_size_t(0)
    assert lib.dwp_compact_by_flags(None, None, n, None, None, None, ctypes.byref(sb), None) == 0
    scratch = torch.empty(max(sb.value, 16), dtype=torch.uint8, device="cuda")
    st = lib.dwp_compact_by_flags(ctypes.c_void_p(r.data_ptr()), ctypes.c_void_p(f.data_ptr()), n,
                                  ctypes.c_void_p(out.data_ptr()), ctypes.c_void_p(cnt.data_ptr()),
                                  ctypes.c_void_p(scratch.data_ptr()), ctypes.byref(sb), _stream())
    assert st == dwp.DWP_SUCCESS
    status = lib.dwp_read_status(ctypes.c_void_p(scratch.data_ptr()), _stream())
    return out.cpu().numpy().view(np.uint32), int(cnt.item()), status


@pytest.mark.parametrize("n", [1, 17, 2559, 2560, 2561, 2560 * 37 + 5, (1 << 20) + 3])
@pytest.mark.parametrize("p", [0.0, 0.3, 1.0])
def test_compaction_no_bounds_error(lib, ref, n, p):
    rec = synth.records(n, seed=60 + n % 11)
    flags = synth.keep_flags(n, p=p, seed=61 + n % 5)
    got, k, status = compact_run(lib, rec, flags)
    assert status == dwp.DWP_SUCCESS, dwp.status_string(status)
    want, kw = ref.compact(rec, flags)
    assert k == kw
    assert np.array_equal(got[:k], want[:k])
    assert (got[k:] == SENTINEL).all()


# ------------------------------------ linear recurrence, segmented reduction


def rec_run(lib, a, b, inclusive):
    n = a.size
    ta, tb = torch.from_numpy(a).cuda(), torch.from_numpy(b).cuda()
    h = torch.full_like(tb, 12345.0)
    sb = ctypes.c_size_t(0)
    mode = dwp.DWP_INCLUSIVE if inclusive else dwp.DWP_EXCLUSIVE
    assert lib.dwp_linear_recurrence_f32(None, None, None, n, mode, None, ctypes.byref(sb), None) == 0
    scratch = torch.empty(max(sb.value, 16), dtype=torch.uint8, device="cuda")
    st = lib.dwp_linear_recurrence_f32(ctypes.c_void_p(ta.data_ptr()), ctypes.c_void_p(tb.data_ptr()),
                                       ctypes.c_void_p(h.data_ptr()), n, mode,
                                       ctypes.c_void_p(scratch.data_ptr()), ctypes.byref(sb), _stream())
    assert st == dwp.DWP_SUCCESS
    status = lib.dwp_read_status(ctypes.c_void_p(scratch.data_ptr()), _stream())
    return h.cpu().numpy(), status


@pytest.mark.parametrize("inclusive", [False, True])
def test_recurrence_no_bounds_error(lib, ref, inclusive):
    for n in (1, 5, 4607, 4608, 4609, 4608 * 200 + 3, (1 << 22) + 1):
        a = synth.decay_values(n, seed=70 + n % 7)
        b = synth.f32_values(n, seed=71 + n % 5)
        got, status = rec_run(lib, a, b, inclusive)
        assert status == dwp.DWP_SUCCESS, (n, dwp.status_string(status))
        want, g = ref.linear_recurrence(a, b, inclusive)
        assert (np.abs(got.astype(np.float64) - want) <= 1e-4 * g + 1e-6).all(), n


def red_run(lib, values, offsets):
    n, nseg = values.size, offsets.size - 1
    v = torch.from_numpy(values.view(np.int32)).cuda()
    o = torch.from_numpy(np.ascontiguousarray(offsets, dtype=np.uint32).view(np.int32)).cuda()
    out = torch.full((max(nseg, 1),), SENTINEL - (1 << 32), dtype=torch.int32, device="cuda")
    sb = ctypes.c_size_t(0)
    assert lib.dwp_segmented_reduce_u32(None, None, nseg, None, n, None, ctypes.byref(sb), None) == 0
    scratch = torch.empty(max(sb.value, 16), dtype=torch.uint8, device="cuda")
    st = lib.dwp_segmented_reduce_u32(ctypes.c_void_p(v.data_ptr()), ctypes.c_void_p(o.data_ptr()), nseg,
                                      ctypes.c_void_p(out.data_ptr()), n,
                                      ctypes.c_void_p(scratch.data_ptr()), ctypes.byref(sb), _stream())
    assert st == dwp.DWP_SUCCESS
    status = lib.dwp_read_status(ctypes.c_void_p(scratch.data_ptr()), _stream())
    return out.cpu().numpy().view(np.uint32)[:nseg], status


def test_segmented_reduction_no_bounds_error(lib, ref):
    for name, offsets, n in seg_cases():
        values = synth.u32_byte_values(n, seed=80 + n % 13)
        got, status = red_run(lib, values, offsets)
        assert status == dwp.DWP_SUCCESS, (name, dwp.status_string(status))
        assert np.array_equal(got, ref.segmented_reduce_u32(values, offsets)), name


@pytest.mark.parametrize("n", [1, 2561, 2560 * 37 + 5, (1 << 20) + 3])
def test_staged_compaction_no_bounds_error(lib, ref, n):
    """The staged form's scatter writes to slots its own scan computed."""
    rec = synth.records(n, seed=90 + n % 11)
    flags = synth.keep_flags(n, seed=91 + n % 5)
    r = torch.from_numpy(rec.view(np.int32)).cuda()
    f = torch.from_numpy(flags).cuda()
    out = torch.full_like(r, SENTINEL - (1 << 32))
    cnt = torch.zeros(1, dtype=torch.int32, device="cuda")
    sb = ctypes.c_size_t(0)
    assert lib.dwp_compact_by_flags_staged(None, None, n, None, None, None, ctypes.byref(sb), None) == 0
    scratch = torch.empty(max(sb.value, 16), dtype=torch.uint8, device="cuda")
    st = lib.dwp_compact_by_flags_staged(ctypes.c_void_p(r.data_ptr()), ctypes.c_void_p(f.data_ptr()), n,
                                         ctypes.c_void_p(out.data_ptr()), ctypes.c_void_p(cnt.data_ptr()),
                                         ctypes.c_void_p(scratch.data_ptr()), ctypes.byref(sb), _stream())
    assert st == dwp.DWP_SUCCESS
    assert lib.dwp_read_status(ctypes.c_void_p(scratch.data_ptr()), _stream()) == dwp.DWP_SUCCESS
    want, k = ref.compact(rec, flags)
    got = out.cpu().numpy().view(np.uint32)
    assert int(cnt.item()) == k
    assert np.array_equal(got[:k], want[:k])
    assert (got[k:] == SENTINEL).all()
