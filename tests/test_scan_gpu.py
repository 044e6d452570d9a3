"""Parity of the CUDA scans (through the C ABI) with the sequential oracle.

Integers must match bit for bit; f32 must satisfy
|y_gpu[i] - y_ref[i]| <= 1e-4 * sum_{j in range(i)} |x_j| + 1e-6
against the double-accumulating oracle, the bound the f32 workload states.
"""
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

F32_REL, F32_ABS = 1e-4, 1e-6


@pytest.fixture(scope="module", autouse=True)
def lib():
    dwp_build.build()
    return dwp.load()


@pytest.fixture(scope="module")
def ref():
    return oracle.Oracle()


def tile():
    st, b = dwp.dwp_scan_exclusive(dwp.DWP_U32_ADD, 0, 0, 1 << 30, 0, 0, 0)
    return (1 << 30) // ((b - 128) // 8)


def gpu_scan(x: np.ndarray, op: str, inclusive: bool, inplace: bool = False) -> np.ndarray:
    t = torch.from_numpy(x.view(np.float32 if op == "f32_add" else np.int32)).cuda()
    out = t if inplace else None
    scratch = dwp.alloc_scratch(dwp.scan_scratch_bytes(x.size, op), t.device)
    y = (dwp.scan_inclusive if inclusive else dwp.scan_exclusive)(t, op, out=out, scratch=scratch)
    assert dwp.read_status(scratch) == dwp.DWP_SUCCESS
    return y.cpu().numpy().view(x.dtype)


def check(ref, x, op, inclusive, y):
    if op == "f32_add":
        yr, ab = ref.scan_f32_add(x, inclusive)
        err = np.abs(y.astype(np.float64) - yr)
        bound = F32_REL * ab + F32_ABS
        bad = np.nonzero(err > bound)[0]
        assert bad.size == 0, "f32 out of tolerance at %s: err %s bound %s" % (
            bad[:5], err[bad[:5]], bound[bad[:5]])
    else:
        yr = ref.scan(op, x, inclusive)
        bad = np.nonzero(y != yr)[0]
        assert bad.size == 0, "mismatch at %s: got %s want %s" % (bad[:5], y[bad[:5]], yr[bad[:5]])


def values(op, n, seed):
    return synth.f32_values(n, seed) if op == "f32_add" else synth.u32_full_values(n, seed)


def test_golden_examples_on_gpu():
    for name, ex in golden_io.load().items():
        if ex.get("op") != "u32_add":
            continue
        x = np.array(ex["x"], np.uint32)
        if "exclusive" in ex:
            assert gpu_scan(x, "u32_add", False).tolist() == ex["exclusive"], name
        if "inclusive" in ex:
            assert gpu_scan(x, "u32_add", True).tolist() == ex["inclusive"], name


@pytest.mark.parametrize("op", ["u32_add", "u32_max", "f32_add"])
@pytest.mark.parametrize("inclusive", [False, True], ids=["excl", "incl"])
def test_edge_sizes(ref, op, inclusive):
    T = tile()
    sizes = [1, 2, 3, 4, 5, 31, 32, 33, 1023, 1024, 1025, T - 1, T, T + 1, 2 * T - 1, 2 * T + 3,
             32 * T - 1, 32 * T, 32 * T + 1, 33 * T + 7, 65 * T + 2, 1000003]
    for k, n in enumerate(sizes):
        x = values(op, n, 100 + k)
        check(ref, x, op, inclusive, gpu_scan(x, op, inclusive))


def test_empty_input():
    x = np.zeros(0, np.uint32)
    assert gpu_scan(x, "u32_add", False).size == 0


@pytest.mark.parametrize("op", ["u32_add", "u32_max", "f32_add"])
def test_inplace(ref, op):
    n = 3 * tile() + 17
    x = values(op, n, 7)
    check(ref, x, op, True, gpu_scan(x.copy(), op, True, inplace=True))
    check(ref, x, op, False, gpu_scan(x.copy(), op, False, inplace=True))


def test_small_workload_u32_values_0_15(ref):
    """2^20 elements uniform in [0, 15], exclusive u32 add."""
    x = synth.u32_small_values(1 << 20)
    check(ref, x, "u32_add", False, gpu_scan(x, "u32_add", False))
    check(ref, x, "u32_add", True, gpu_scan(x, "u32_add", True))


def test_closed_forms_on_gpu():
    n = 5 * tile() + 3
    i = np.arange(n, dtype=np.uint64)
    assert (gpu_scan(np.ones(n, np.uint32), "u32_add", False) == i.astype(np.uint32)).all()
    y = gpu_scan(np.full(n, 0xFFFFFFFF, np.uint32), "u32_add", False)
    assert (y == ((2**32 - i) % 2**32).astype(np.uint32)).all()
    asc = np.sort(synth.u32_full_values(n, 9))
    assert (gpu_scan(asc, "u32_max", True) == asc).all()
    desc = asc[::-1].copy()
    ye = gpu_scan(desc, "u32_max", False)
    assert ye[0] == 0 and (ye[1:] == desc[0]).all()


def test_repeat_calls_same_scratch_bit_identical():
    n = 200 * tile() + 5
    x = torch.from_numpy(synth.u32_full_values(n, 11).view(np.int32)).cuda()
    scratch = dwp.alloc_scratch(dwp.scan_scratch_bytes(n), x.device)
    first = dwp.scan_exclusive(x, "u32_add", scratch=scratch).clone()
    for _ in range(5):
        y = dwp.scan_exclusive(x, "u32_add", scratch=scratch)
        assert torch.equal(y, first)
    assert dwp.read_status(scratch) == dwp.DWP_SUCCESS


def test_stream_ordering_on_side_stream(ref):
    n = 50 * tile() + 1
    x_np = synth.u32_full_values(n, 12)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        x = torch.from_numpy(x_np.view(np.int32)).cuda(non_blocking=False)
        y = dwp.scan_inclusive(x, "u32_add")
    s.synchronize()
    check(ref, x_np, "u32_add", True, y.cpu().numpy().view(np.uint32))


# ---------------------------------------------------------------- full sizes

_full = {}


def full_u32():
    if "u32" not in _full:
        _full["u32"] = synth.u32_full_values(1 << 28)
    return _full["u32"]


@pytest.mark.slow
@pytest.mark.parametrize("op,inclusive", [("u32_add", False), ("u32_add", True),
                                          ("u32_max", False), ("u32_max", True)])
def test_full_u32_2p28(ref, op, inclusive):
    """2^28 full-range u32: exclusive/inclusive add (wrapping) and max, every element."""
    x = full_u32()
    check(ref, x, op, inclusive, gpu_scan(x, op, inclusive))


@pytest.mark.slow
def test_full_f32_inclusive_2p28(ref):
    """2^28 f32 uniform in [-1, 1), inclusive add, every element within the bound."""
    x = synth.f32_values(1 << 28)
    check(ref, x, "f32_add", True, gpu_scan(x, "f32_add", True))


# ---------------------------------------------------------------- failure path

def test_lookback_timeout_is_reported_not_hung(ref):
    """A tile that never publishes, with the Decoupled Fallback off: its
    successors give up after a short spin, record DWP_ERR_LOOKBACK_TIMEOUT
    and exit; the context stays usable."""
    n = 2000 * tile()
    x = torch.from_numpy(synth.u32_small_values(n, 13).view(np.int32)).cuda()
    scratch = dwp.alloc_scratch(dwp.scan_scratch_bytes(n), x.device)
    try:
        dwp.dwp_debug_set_fault(5, 2000, 0xFFFFFFFF)
        dwp.scan_exclusive(x, "u32_add", scratch=scratch)
        assert dwp.read_status(scratch) == dwp.DWP_ERR_LOOKBACK_TIMEOUT
    finally:
        dwp.dwp_debug_set_fault(0xFFFFFFFF, 0, 0)
    y = dwp.scan_exclusive(x, "u32_add", scratch=scratch)
    assert dwp.read_status(scratch) == dwp.DWP_SUCCESS
    check(ref, x.cpu().numpy().view(np.uint32), "u32_add", False, y.cpu().numpy().view(np.uint32))


# ------------------------------------------------------- Decoupled Fallback

FALLBACK_POLLS = 64  # far below the default: the silent tile is rescued in microseconds


@pytest.mark.parametrize("op,inclusive,silent", [
    ("u32_add", False, 5), ("u32_add", True, 0), ("u32_max", False, 777),
    ("f32_add", True, 1999)])
def test_fallback_rescues_a_silent_tile(ref, op, inclusive, silent):
    """Decoupled Fallback: a tile that never publishes is reduced by the
    successors that wait for it; the call succeeds with the oracle's output
    and reports at least one fallback.  Tile 0 is rescued as a prefix, the
    last tile (1999, ragged) from its partial extent."""
    n = 1999 * tile() + 1234
    x = synth.f32_values(n, 21) if op == "f32_add" else synth.u32_full_values(n, 21)
    t = torch.from_numpy(x.view(np.float32 if op == "f32_add" else np.int32)).cuda()
    scratch = dwp.alloc_scratch(dwp.scan_scratch_bytes(n, op), t.device)
    try:
        dwp.dwp_debug_set_fault(silent, 0, FALLBACK_POLLS)
        y = (dwp.scan_inclusive if inclusive else dwp.scan_exclusive)(t, op, scratch=scratch)
        st = dwp.read_status(scratch)
        fb = dwp.read_fallbacks(scratch)
    finally:
        dwp.dwp_debug_set_fault(0xFFFFFFFF, 0, 0)
    assert st == dwp.DWP_SUCCESS
    if silent < 1999:  # the last tile has no successor to rescue it
        assert fb >= 1
    check(ref, x, op, inclusive, y.cpu().numpy().view(x.dtype))


def test_fallback_off_in_place(ref):
    """In place the input of a silent tile may already be output, so the
    fallback stays off and the timeout path reports the silent tile."""
    n = 2000 * tile()
    x = torch.from_numpy(synth.u32_small_values(n, 14).view(np.int32)).cuda()
    scratch = dwp.alloc_scratch(dwp.scan_scratch_bytes(n), x.device)
    try:
        dwp.dwp_debug_set_fault(5, 2000, FALLBACK_POLLS)
        dwp.scan_exclusive(x, "u32_add", out=x, scratch=scratch)
        assert dwp.read_status(scratch) == dwp.DWP_ERR_LOOKBACK_TIMEOUT
        assert dwp.read_fallbacks(scratch) == 0
    finally:
        dwp.dwp_debug_set_fault(0xFFFFFFFF, 0, 0)


def test_no_fallback_in_a_healthy_run(ref):
    """At the default threshold a healthy full-size run never falls back."""
    n = 1 << 28
    x = torch.from_numpy(synth.u32_full_values(n).view(np.int32)).cuda()
    scratch = dwp.alloc_scratch(dwp.scan_scratch_bytes(n), x.device)
    for _ in range(3):
        dwp.scan_exclusive(x, "u32_add", scratch=scratch)
        assert dwp.read_status(scratch) == dwp.DWP_SUCCESS
        assert dwp.read_fallbacks(scratch) == 0


# ------------------------------------------------ bounded look-back window

@pytest.mark.parametrize("window", [1, 32, 100])
@pytest.mark.parametrize("op,inclusive", [("u32_add", False), ("u32_max", True), ("f32_add", True)])
def test_bounded_window_same_result(ref, window, op, inclusive):
    """A bounded look-back window publishes intermediates and jumps over them;
    the output is the oracle's either way.  A silent tile rescued after 64
    polls makes every tile behind it fold a long chain of aggregates, so the
    intermediates are really published and followed: the scratch header's
    counters must show both."""
    n = 3000 * tile() + 77
    x = synth.f32_values(n, 31) if op == "f32_add" else synth.u32_full_values(n, 31)
    t = torch.from_numpy(x.view(np.float32 if op == "f32_add" else np.int32)).cuda()
    scratch = dwp.alloc_scratch(dwp.scan_scratch_bytes(n, op), t.device)
    try:
        dwp.dwp_set_lookback_window(window)
        for silent in (0xFFFFFFFF, 1234):
            dwp.dwp_debug_set_fault(silent, 0, 64)
            y = (dwp.scan_inclusive if inclusive else dwp.scan_exclusive)(t, op, scratch=scratch)
            assert dwp.read_status(scratch) == dwp.DWP_SUCCESS
            stats = dwp.read_lookback_stats(scratch)
            check(ref, x, op, inclusive, y.cpu().numpy().view(x.dtype))
            if silent != 0xFFFFFFFF:
                # the tiles queued behind the silent one fold long chains:
                # they publish intermediates, and later look-backs jump them
                assert stats["intermediates"] > 0 and stats["jumps"] > 0, stats
    finally:
        dwp.dwp_set_lookback_window(0)
        dwp.dwp_debug_set_fault(0xFFFFFFFF, 0, 0)
