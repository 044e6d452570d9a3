"""Parity of the two-level (three-launch) scan with the sequential oracle:
integers bit for bit, f32 within 1e-4 * sum|x| + 1e-6."""
import numpy as np
import pytest

import golden_io
import oracle
import synth

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import device_wide_prefix_gb300 as dwp  # noqa: E402
from device_wide_prefix_gb300 import build as dwp_build  # noqa: E402


@pytest.fixture(scope="module", autouse=True)
def lib():
    dwp_build.build()
    return dwp.load()


@pytest.fixture(scope="module")
def ref():
    return oracle.Oracle()


def run(x, op, inclusive, inplace=False):
    t = torch.from_numpy(x.view(np.float32 if op == "f32_add" else np.int32)).cuda()
    y = dwp.scan_two_level(t, op, inclusive, out=t if inplace else None)
    return y.cpu().numpy().view(x.dtype)


def check(ref, x, op, inclusive, y):
    if op == "f32_add":
        yr, ab = ref.scan_f32_add(x, inclusive)
        assert (np.abs(y.astype(np.float64) - yr) <= 1e-4 * ab + 1e-6).all()
    else:
        assert (y == ref.scan(op, x, inclusive)).all()


@pytest.mark.parametrize("op", ["u32_add", "u32_max", "f32_add"])
@pytest.mark.parametrize("inclusive", [False, True])
def test_sizes(ref, op, inclusive):
    for n in (1, 5, 15, 16, 17, 4095, 4096, 4097, 3 * 4096 + 11, 1000003):
        x = synth.f32_values(n, 60 + n % 7) if op == "f32_add" else synth.u32_full_values(n, 60 + n % 7)
        check(ref, x, op, inclusive, run(x, op, inclusive))


def test_largest_size_and_in_place(ref):
    n = 1 << 26
    x = synth.u32_full_values(n, 71)
    check(ref, x, "u32_add", False, run(x, "u32_add", False, inplace=True))


def test_golden_example():
    x = np.array([3, 1, 4, 1], np.uint32)
    assert run(x, "u32_add", False).tolist() == [0, 3, 4, 8]
    assert run(x, "u32_add", True).tolist() == [3, 4, 8, 9]


def test_too_large_is_rejected():
    st, _ = dwp.dwp_scan_two_level(dwp.DWP_U32_ADD, dwp.DWP_EXCLUSIVE, None, None, (1 << 26) + 1,
                                   None, 0, None)
    assert st == dwp.DWP_ERR_INVALID_VALUE


def test_warp_hillis_steele_steps_match_the_printed_trace():
    """The page's 8-element Hillis-Steele trace, step by step, on the warp
    scan the two-level kernels run: after d = 1, 2, 4 the eight lanes hold
    the printed rows; the steps d = 8, 16 change nothing in them (they only
    pull from lanes 8 and up, which hold the identity)."""
    ex = golden_io.load()["hillis_steele_8"]
    x = torch.tensor(ex["x"], dtype=torch.int32, device="cuda")
    steps = torch.full((5 * 8,), -1, dtype=torch.int32, device="cuda")
    st = dwp.dwp_debug_warp_scan_trace(x.data_ptr(), 8, steps.data_ptr(),
                                       torch.cuda.current_stream().cuda_stream)
    assert st == dwp.DWP_SUCCESS
    rows = steps.view(5, 8).cpu().tolist()
    assert rows[0] == ex["step_d1"]
    assert rows[1] == ex["step_d2"]
    assert rows[2] == ex["step_d4"]
    assert rows[3] == ex["inclusive"] and rows[4] == ex["inclusive"]


def test_warp_scan_trace_rejects_bad_widths():
    x = torch.zeros(32, dtype=torch.int32, device="cuda")
    assert dwp.dwp_debug_warp_scan_trace(x.data_ptr(), 0, x.data_ptr(), 0) == dwp.DWP_ERR_INVALID_VALUE
    assert dwp.dwp_debug_warp_scan_trace(x.data_ptr(), 33, x.data_ptr(), 0) == dwp.DWP_ERR_INVALID_VALUE
