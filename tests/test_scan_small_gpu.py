"""Parity of the small-input plain scan (one block per tile of 3072 elements
up to n = 2^18, 7168 up to 2^20, 15360 up to n = 2^23) with the sequential
oracle, through the C ABI, and the same failure paths as the large-input
kernel: Decoupled Fallback, timeout reporting, bounded look-back window,
schedule perturbation.  Integers bit for bit; f32 within
1e-4 * sum|x| + 1e-6."""
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

SMALL_MAX = 1 << 23
T = 3072        # elements per tile up to 2^18
TM = 7168       # elements per tile above 2^18, up to 2^20
T2 = 15360      # elements per tile above 2^20, up to 2^23


def descriptors(n):
    """The size query's descriptor count: the tile count, never fewer than
    the largest count of a lower tier."""
    if n <= 1 << 18:
        return -(-n // T)
    if n <= 1 << 20:
        return max(-(-n // TM), 86)
    return max(-(-n // T2), 147)


@pytest.fixture(scope="module", autouse=True)
def lib():
    dwp_build.build()
    return dwp.load()


@pytest.fixture(scope="module")
def ref():
    return oracle.Oracle()


def values(n, op, seed):
    return synth.f32_values(n, seed) if op == "f32_add" else synth.u32_full_values(n, seed)


def run(x, op, inclusive, scratch=None, inplace=False):
    t = torch.from_numpy(x.view(np.float32 if op == "f32_add" else np.int32)).cuda()
    if scratch is None:
        scratch = dwp.alloc_scratch(dwp.scan_scratch_bytes(x.size, op), t.device)
    y = (dwp.scan_inclusive if inclusive else dwp.scan_exclusive)(t, op, out=t if inplace else None,
                                                                  scratch=scratch)
    return y.cpu().numpy().view(x.dtype), scratch


def check(ref, x, op, inclusive, y):
    if op == "f32_add":
        yr, ab = ref.scan_f32_add(x, inclusive)
        assert (np.abs(y.astype(np.float64) - yr) <= 1e-4 * ab + 1e-6).all()
    else:
        assert np.array_equal(y, ref.scan(op, x, inclusive))


def test_small_kernel_tiles_in_the_size_query():
    """One descriptor per tile of the tier n falls in, never fewer than the
    largest count of a lower tier (the size query does not shrink)."""
    for n, tiles in ((1, 1), (T, 1), (T + 1, 2), (1 << 18, 86), ((1 << 18) + 1, 86),
                     (87 * TM, 87), (1 << 20, 147), ((1 << 20) + 1, 147), (148 * T2, 148),
                     (1 << 22, 274), (SMALL_MAX, 547)):
        assert descriptors(n) == tiles, n
        assert dwp.scan_scratch_bytes(n) == 128 + 8 * tiles, n


@pytest.mark.parametrize("op", ["u32_add", "u32_max", "f32_add"])
@pytest.mark.parametrize("inclusive", [False, True])
def test_sizes_around_tiles_and_the_switch(ref, op, inclusive):
    for n in (1, 3, 15, 16, 17, T - 1, T, T + 1, 3 * T + 5, 100003, 1 << 18, (1 << 18) + 1,
              TM * 50 - 1, TM * 50 + 3, (1 << 20) + 1, T2 * 70 - 1, T2 * 70 + 3, SMALL_MAX - 1,
              SMALL_MAX, SMALL_MAX + 1):
        x = values(n, op, 700 + n % 97)
        y, scratch = run(x, op, inclusive)
        assert dwp.read_status(scratch) == dwp.DWP_SUCCESS
        check(ref, x, op, inclusive, y)


@pytest.mark.parametrize("n", [50 * T + 9, 100 * TM + 9, 200 * T2 + 9])
def test_in_place(ref, n):
    x = values(n, "u32_add", 5)
    y, _ = run(x.copy(), "u32_add", False, inplace=True)
    check(ref, x, "u32_add", False, y)


@pytest.mark.parametrize("tile,tiles", [(T, 60), (TM, 120), (T2, 250)])
@pytest.mark.parametrize("silent", ["first", "inner", "last"])
@pytest.mark.parametrize("op,inclusive", [("u32_add", False), ("f32_add", True)])
def test_fallback_rescues_a_silent_tile(ref, tile, tiles, silent, op, inclusive):
    n = (tiles - 1) * tile + 77  # the last tile ragged
    s_tile = {"first": 0, "inner": 5, "last": tiles - 1}[silent]
    x = values(n, op, 31)
    try:
        dwp.dwp_debug_set_fault(s_tile, 0, 64)
        y, scratch = run(x, op, inclusive)
        st = dwp.read_status(scratch)
        stats = dwp.read_lookback_stats(scratch)
    finally:
        dwp.dwp_debug_set_fault(0xFFFFFFFF, 0, 0)
    assert st == dwp.DWP_SUCCESS
    if silent != "last":  # the last tile has no successor to rescue it
        assert stats["fallbacks"] >= 1
    check(ref, x, op, inclusive, y)


@pytest.mark.parametrize("n", [60 * T, 120 * TM, 250 * T2])
def test_timeout_is_reported_not_hung(ref, n):
    x = values(n, "u32_add", 32)
    try:
        dwp.dwp_debug_set_fault(5, 2000, 0xFFFFFFFF)
        _, scratch = run(x, "u32_add", False)
        assert dwp.read_status(scratch) == dwp.DWP_ERR_LOOKBACK_TIMEOUT
    finally:
        dwp.dwp_debug_set_fault(0xFFFFFFFF, 0, 0)
    y, scratch = run(x, "u32_add", False, scratch=scratch)
    assert dwp.read_status(scratch) == dwp.DWP_SUCCESS
    check(ref, x, "u32_add", False, y)


@pytest.mark.parametrize("window", [1, 32])
def test_bounded_window(ref, window):
    n = SMALL_MAX - 3
    x = values(n, "u32_add", 33)
    try:
        dwp.dwp_set_lookback_window(window)
        for silent in (0xFFFFFFFF, 100):
            dwp.dwp_debug_set_fault(silent, 0, 64)
            y, scratch = run(x, "u32_add", True)
            assert dwp.read_status(scratch) == dwp.DWP_SUCCESS
            check(ref, x, "u32_add", True, y)
    finally:
        dwp.dwp_set_lookback_window(0)
        dwp.dwp_debug_set_fault(0xFFFFFFFF, 0, 0)


@pytest.mark.parametrize("seed", [0x61, 0x62])
@pytest.mark.parametrize("n", [(1 << 18) - 5, (1 << 20) - 77, SMALL_MAX - 1234])
@pytest.mark.parametrize("op,inclusive", [("u32_add", False), ("u32_max", True), ("f32_add", True)])
def test_under_perturbation(ref, seed, n, op, inclusive):
    x = values(n, op, seed)
    try:
        assert dwp.dwp_debug_set_delay(seed, 150000, 20000) == dwp.DWP_SUCCESS
        y, scratch = run(x, op, inclusive)
        assert dwp.read_status(scratch) == dwp.DWP_SUCCESS
    finally:
        dwp.dwp_debug_set_delay(0, 0, 0)
    check(ref, x, op, inclusive, y)
