"""The scan entry point with built-in scratch, for callers that cannot
allocate device memory (allocator hooks, memory-pool callbacks, plug-ins
whose host owns all device memory).

It is called through the C ABI twice in a row on the same data and each
result is compared with the regular, caller-scratch entry point: bit for bit
for the integer operators, within the f32 scan tolerance
(1e-4 * sum|x| + 1e-6 per prefix) for f32.  The file sorts last so that a
run stopping at the first failure has already run every other test; it also
passes on its own in a fresh process.
"""
import ctypes

import numpy as np
import pytest

import synth

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import device_wide_prefix_gb300 as dwp  # noqa: E402
from device_wide_prefix_gb300 import build as dwp_build  # noqa: E402

MAX_N = 268435456  # DWP_SCAN_STATIC_MAX_N


@pytest.fixture(scope="module", autouse=True)
def lib():
    dwp_build.build()
    return dwp.load()


def _regular(x, op, inclusive):
    return (dwp.scan_inclusive if inclusive else dwp.scan_exclusive)(x, op)


def _static(x, op, inclusive):
    y = torch.empty_like(x)
    stream = torch.cuda.current_stream().cuda_stream
    st = dwp.dwp_scan_static_scratch(dwp.OPS[op], dwp.DWP_INCLUSIVE if inclusive else dwp.DWP_EXCLUSIVE,
                                     x.data_ptr(), y.data_ptr(), x.numel(), stream)
    assert st == dwp.DWP_SUCCESS, dwp.status_string(st)
    return y


def _same(x, op, a, b, inclusive):
    if op == "f32_add":
        xa = np.abs(x.cpu().numpy().astype(np.float64))
        ab = np.cumsum(xa) if inclusive else np.concatenate([[0.0], np.cumsum(xa)[:-1]])
        d = np.abs(a.cpu().numpy().astype(np.float64) - b.cpu().numpy().astype(np.float64))
        assert (d <= 1e-4 * ab + 1e-6).all()
    else:
        assert torch.equal(a, b)


@pytest.mark.parametrize("op", ["u32_add", "u32_max", "f32_add"])
@pytest.mark.parametrize("inclusive", [False, True], ids=["excl", "incl"])
def test_static_scratch_matches_regular_entry_point(op, inclusive):
    n = 1000003
    x_np = synth.f32_values(n, 41) if op == "f32_add" else synth.u32_full_values(n, 41)
    x = torch.from_numpy(x_np.view(np.float32 if op == "f32_add" else np.int32)).cuda()
    want = _regular(x, op, inclusive)
    first = _static(x, op, inclusive)
    second = _static(x, op, inclusive)  # the array still holds the first call's contents
    torch.cuda.synchronize()
    _same(x, op, first, want, inclusive)
    _same(x, op, second, want, inclusive)


def test_static_scratch_at_its_maximum_size():
    x = torch.from_numpy(synth.u32_small_values(MAX_N, 43).view(np.int32)).cuda()
    want = _regular(x, "u32_add", False)
    for _ in range(2):
        assert torch.equal(_static(x, "u32_add", False), want)


def test_static_scratch_rejects_sizes_beyond_its_maximum():
    lib = dwp.load()
    st = lib.dwp_scan_static_scratch(dwp.DWP_U32_ADD, dwp.DWP_EXCLUSIVE, None, None, MAX_N + 1, None)
    assert st == dwp.DWP_ERR_SCRATCH_TOO_SMALL
    assert lib.dwp_scan_static_scratch(dwp.DWP_U32_ADD, 7, None, None, 10, None) == dwp.DWP_ERR_INVALID_VALUE
    assert lib.dwp_scan_static_scratch(9, dwp.DWP_EXCLUSIVE, None, None, 10, None) == dwp.DWP_ERR_INVALID_VALUE


def test_static_status_reports_a_device_timeout():
    """The built-in array's status word is readable: a tile that never
    publishes (fallback off, short spin) makes its successors record a
    look-back timeout, which dwp_read_static_status returns; the next healthy
    call clears it."""
    st, b = dwp.dwp_scan_exclusive(dwp.DWP_U32_ADD, 0, 0, 1 << 30, 0, 0, 0)
    tile = (1 << 30) // ((b - 128) // 8)
    x = torch.from_numpy(synth.u32_small_values(2000 * tile, 44).view(np.int32)).cuda()
    stream = torch.cuda.current_stream().cuda_stream
    try:
        dwp.dwp_debug_set_fault(5, 2000, 0xFFFFFFFF)
        _static(x, "u32_add", False)
        assert dwp.dwp_read_static_status(stream) == dwp.DWP_ERR_LOOKBACK_TIMEOUT
    finally:
        dwp.dwp_debug_set_fault(0xFFFFFFFF, 0, 0)
    y = _static(x, "u32_add", False)
    assert dwp.dwp_read_static_status(stream) == dwp.DWP_SUCCESS
    assert torch.equal(y, _regular(x, "u32_add", False))
