"""Schedule perturbation: the look-back kernels under shuffled publication
orders must still match the oracle.

A missing ordering or synchronisation step in a chained scan fails only under
rare interleavings ("Parallel Prefix Sum (Scan), in depth", section "Failure
modes"; "Single-Pass Prefix Scan with Decoupled Look-Back", section "Where the
algorithm meets the hardware").  dwp_debug_set_delay makes a seeded subset of
tiles sleep (bounded) after drawing their index, before publishing their
aggregate, before their look-back, before publishing their prefix, and
between the two words of the recurrence's descriptor.  Each case runs
thousands of tiles under several seeds, with the unbounded and a bounded
look-back window, and with a Decoupled Fallback threshold low enough that
rescuers race live owners.  Integers must match bit for bit, f32 within the
scan (or recurrence) bound.  All waits stay bounded, so nothing can hang.
"""
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

SEEDS = [0x51, 0x52, 0x53]
FRACTION_PPM = 150000  # 15% of (tile, point) pairs sleep
MAX_NS = 20000         # up to 20 us each


@pytest.fixture(scope="module", autouse=True)
def lib():
    dwp_build.build()
    return dwp.load()


@pytest.fixture(scope="module")
def ref():
    return oracle.Oracle()


class perturbed:
    """Delay hook, look-back window and fallback threshold for one block."""

    def __init__(self, seed, window=0, fallback_polls=0):
        self.seed, self.window, self.fallback_polls = seed, window, fallback_polls

    def __enter__(self):
        assert dwp.dwp_debug_set_delay(self.seed, FRACTION_PPM, MAX_NS) == dwp.DWP_SUCCESS
        dwp.dwp_set_lookback_window(self.window)
        dwp.dwp_debug_set_fault(0xFFFFFFFF, 0, self.fallback_polls)
        return self

    def __exit__(self, *exc):
        dwp.dwp_debug_set_delay(0, 0, 0)
        dwp.dwp_set_lookback_window(0)
        dwp.dwp_debug_set_fault(0xFFFFFFFF, 0, 0)
        return False


def test_delay_hook_validates_arguments():
    assert dwp.dwp_debug_set_delay(1, 1000001, 10) == dwp.DWP_ERR_INVALID_VALUE
    assert dwp.dwp_debug_set_delay(1, 10, 100001) == dwp.DWP_ERR_INVALID_VALUE
    assert dwp.dwp_debug_set_delay(0, 0, 0) == dwp.DWP_SUCCESS


def _check_scan(ref, x, op, inclusive, y):
    if op == "f32_add":
        yr, ab = ref.scan_f32_add(x, inclusive)
        assert (np.abs(y.astype(np.float64) - yr) <= 1e-4 * ab + 1e-6).all()
    else:
        assert np.array_equal(y, ref.scan(op, x, inclusive))


SCAN_TILES = 3000


@pytest.mark.parametrize("seed", SEEDS)
@pytest.mark.parametrize("window", [0, 32])
@pytest.mark.parametrize("op,inclusive", [("u32_add", False), ("u32_max", True), ("f32_add", True)])
def test_scan_under_perturbation(ref, seed, window, op, inclusive):
    st, b = dwp.dwp_scan_exclusive(dwp.DWP_U32_ADD, 0, 0, 1 << 30, 0, 0, 0)
    tile = (1 << 30) // ((b - 128) // 8)
    n = SCAN_TILES * tile + 333
    x = synth.f32_values(n, seed) if op == "f32_add" else synth.u32_full_values(n, seed)
    t = torch.from_numpy(x.view(np.float32 if op == "f32_add" else np.int32)).cuda()
    scratch = dwp.alloc_scratch(dwp.scan_scratch_bytes(n, op), t.device)
    with perturbed(seed, window):
        y = (dwp.scan_inclusive if inclusive else dwp.scan_exclusive)(t, op, scratch=scratch)
        assert dwp.read_status(scratch) == dwp.DWP_SUCCESS
        stats = dwp.read_lookback_stats(scratch)
    assert stats["fallbacks"] == 0  # sleeps are far below the default threshold
    _check_scan(ref, x, op, inclusive, y.cpu().numpy().view(x.dtype))


@pytest.mark.parametrize("seed", SEEDS[:2])
@pytest.mark.parametrize("op", ["u32_add", "f32_add"])
def test_scan_fallback_races_live_owners(ref, seed, op):
    """With the fallback after 8 polls, sleeping tiles are rescued while
    their owners are still running: both publish, the compare-and-swap
    decides which descriptor successors see first, and the owner's later
    store rewrites it with the same value (another grouping for f32)."""
    st, b = dwp.dwp_scan_exclusive(dwp.DWP_U32_ADD, 0, 0, 1 << 30, 0, 0, 0)
    tile = (1 << 30) // ((b - 128) // 8)
    n = SCAN_TILES * tile + 5
    x = synth.f32_values(n, seed) if op == "f32_add" else synth.u32_full_values(n, seed)
    t = torch.from_numpy(x.view(np.float32 if op == "f32_add" else np.int32)).cuda()
    scratch = dwp.alloc_scratch(dwp.scan_scratch_bytes(n, op), t.device)
    with perturbed(seed, 0, fallback_polls=8):
        y = dwp.scan_inclusive(t, op, scratch=scratch)
        assert dwp.read_status(scratch) == dwp.DWP_SUCCESS
        stats = dwp.read_lookback_stats(scratch)
    assert stats["fallbacks"] > 0
    _check_scan(ref, x, op, True, y.cpu().numpy().view(x.dtype))


@pytest.mark.parametrize("seed", SEEDS[:2])
@pytest.mark.parametrize("window", [0, 32])
@pytest.mark.parametrize("inclusive", [False, True])
def test_segscan_under_perturbation(ref, seed, window, inclusive):
    n = 1 << 24
    values = synth.u32_byte_values(n, seed)
    offsets = synth.segment_offsets(n, seed)
    v = torch.from_numpy(values.view(np.int32)).cuda()
    o = torch.from_numpy(offsets.view(np.int32)).cuda()
    out = torch.empty_like(v)
    scratch = dwp.alloc_scratch(dwp.segmented_scan_scratch_bytes(n), v.device)
    with perturbed(seed, window):
        dwp.segmented_scan(v, o, inclusive, out=out, scratch=scratch)
        assert dwp.read_status(scratch) == dwp.DWP_SUCCESS
    want = ref.segmented_scan_u32(values, offsets, inclusive)
    assert np.array_equal(out.cpu().numpy().view(np.uint32), want)


@pytest.mark.parametrize("seed", SEEDS[:2])
@pytest.mark.parametrize("window,fallback_polls", [(0, 0), (64, 0), (0, 8)])
def test_compact_under_perturbation(ref, seed, window, fallback_polls):
    n = (1 << 23) + 9
    rec = synth.records(n, seed)
    flags = synth.keep_flags(n, 0.3, seed)
    r = torch.from_numpy(rec.view(np.int32)).cuda()
    f = torch.from_numpy(flags).cuda()
    scratch = dwp.alloc_scratch(dwp.compact_scratch_bytes(n), r.device)
    with perturbed(seed, window, fallback_polls):
        out, cnt = dwp.compact_by_flags(r, f, scratch=scratch)
        assert dwp.read_status(scratch) == dwp.DWP_SUCCESS
    want, k = ref.compact(rec, flags)
    assert int(cnt.item()) == k
    assert np.array_equal(out.cpu().numpy().view(np.uint32).reshape(-1)[: 4 * k],
                          want.view(np.uint32).reshape(-1)[: 4 * k])


@pytest.mark.parametrize("seed", SEEDS[:2])
@pytest.mark.parametrize("inclusive,fallback_polls", [(True, 0), (False, 0), (True, 8)])
def test_recurrence_under_perturbation(ref, seed, inclusive, fallback_polls):
    n = (1 << 23) + 3
    a = synth.decay_values(n, seed)
    b = synth.f32_values(n, seed + 1)
    ta, tb = torch.from_numpy(a).cuda(), torch.from_numpy(b).cuda()
    scratch = dwp.alloc_scratch(dwp.linear_recurrence_scratch_bytes(n), ta.device)
    with perturbed(seed, 0, fallback_polls):
        h = dwp.linear_recurrence(ta, tb, inclusive, scratch=scratch)
        assert dwp.read_status(scratch) == dwp.DWP_SUCCESS
    want, g = ref.linear_recurrence(a, b, inclusive)
    err = np.abs(h.cpu().numpy().astype(np.float64) - want)
    assert (err <= 1e-4 * g + 1e-6).all()
