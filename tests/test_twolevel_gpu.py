"""Parity of the two-level (three-launch) scan with the sequential oracle:
integers bit for bit, f32 within 1e-4 * sum|x| + 1e-6."""
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
