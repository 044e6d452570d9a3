"""Parity of the CUDA segmented u32 scan (through the C ABI) with the oracle:
bit-exact on every row, rows outside [offsets[0], offsets[N]) untouched."""
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

SENTINEL = 0xDEADBEEF


@pytest.fixture(scope="module", autouse=True)
def lib():
    dwp_build.build()
    return dwp.load()


@pytest.fixture(scope="module")
def ref():
    return oracle.Oracle()


def tile():
    b1 = dwp.segmented_scan_scratch_bytes(1)
    T = 1
    while dwp.segmented_scan_scratch_bytes(2 * T) == b1:
        T *= 2
    lo, hi = T, 2 * T
    while hi - lo > 1:
        mid = (lo + hi) // 2
        if dwp.segmented_scan_scratch_bytes(mid) == b1:
            lo = mid
        else:
            hi = mid
    return lo


def gpu_seg(values, offsets, inclusive):
    v = torch.from_numpy(values.view(np.int32)).cuda()
    o = torch.from_numpy(np.ascontiguousarray(offsets, dtype=np.uint32).view(np.int32)).cuda()
    out = torch.full((values.size,), SENTINEL - (1 << 32), dtype=torch.int32, device="cuda")
    scratch = dwp.alloc_scratch(dwp.segmented_scan_scratch_bytes(values.size), v.device)
    dwp.segmented_scan(v, o, inclusive, out=out, scratch=scratch)
    assert dwp.read_status(scratch) == dwp.DWP_SUCCESS
    return out.cpu().numpy().view(np.uint32)


def check(ref, values, offsets, inclusive):
    want = ref.segmented_scan_u32(values, offsets, inclusive,
                                  out=np.full(values.size, SENTINEL, np.uint32))
    got = gpu_seg(values, offsets, inclusive)
    bad = np.nonzero(got != want)[0]
    assert bad.size == 0, "mismatch at %s: got %s want %s" % (bad[:5], got[bad[:5]], want[bad[:5]])


def test_golden_example():
    ex = golden_io.load()["segmented_luma"]
    v = np.array(ex["values"], np.uint32)
    off = np.array(ex["offsets"], np.uint32)
    assert gpu_seg(v, off, False).tolist() == ex["exclusive"]
    assert gpu_seg(v, off, True).tolist() == ex["inclusive"]


@pytest.mark.parametrize("inclusive", [False, True], ids=["excl", "incl"])
def test_segment_shapes(ref, inclusive):
    T = tile()
    n = 5 * T + 77
    v = synth.u32_full_values(n, 501)
    shapes = {
        "one_segment": [0, n],
        "all_length_one": list(range(n + 1)),
        "leading_trailing_consecutive_empties": [0, 0, 0, 5, 5, 100, 100, 100, T, 2 * T - 1, n, n, n],
        "partial_cover": [7, 7, 40, T + 3, 3 * T + 11],
        "heads_on_tile_edges": [0, T, 2 * T, 3 * T, 4 * T, 5 * T, n],
        "heads_next_to_tile_edges": [0, T - 1, T + 1, 2 * T - 1, 3 * T + 1, n],
        "many_empties_at_one_row": [0] + [T + 5] * 3000 + [n],
        "one_segment_many_tiles_then_short": [0, 4 * T + 9, 4 * T + 10, n],
        "first_row_not_covered": [1, n],
        "last_row_not_covered": [0, n - 1],
    }
    for name, offs in shapes.items():
        check(ref, v, np.array(offs, np.uint32), inclusive)


@pytest.mark.parametrize("inclusive", [False, True], ids=["excl", "incl"])
def test_many_segments_global_search(ref, inclusive):
    """More offsets than the per-block sample holds: the head search falls back
    to the warp-wide search in global memory."""
    n = 1 << 20
    v = synth.u32_byte_values(n, 502)
    u = synth.u64(503, 0, n)
    lens = (u % np.uint64(100)).astype(np.int64)  # 0 .. 99, with empties
    cum = np.cumsum(lens)
    cum = cum[cum < n]
    off = np.concatenate([[0], cum, [n]]).astype(np.uint32)
    assert off.size > 5000
    check(ref, v, off, inclusive)
    check(ref, v[: 300001].copy(), np.arange(300002, dtype=np.uint32), inclusive)


@pytest.mark.parametrize("inclusive", [False, True], ids=["excl", "incl"])
def test_zipf_lengths_small(ref, inclusive):
    n = 1 << 21
    off = synth.segment_offsets(n, seed=504, cap=1 << 16)
    check(ref, synth.u32_byte_values(n, 505), off, inclusive)


def test_degenerate_sizes(ref):
    T = tile()
    for n in (1, 2, 3, 4, 5, 31, 33, T - 1, T, T + 1):
        v = synth.u32_full_values(n, 506)
        for offs in ([0, n], [0, n // 2, n], [0] * 3 + [n]):
            for inc in (False, True):
                check(ref, v, np.array(offs, np.uint32), inc)
    # no segments: nothing is written
    v = synth.u32_full_values(1000, 507)
    assert (gpu_seg(v, np.array([0], np.uint32), False) == SENTINEL).all()
    # no rows
    assert gpu_seg(np.zeros(0, np.uint32), np.array([0, 0], np.uint32), True).size == 0


@pytest.mark.slow
@pytest.mark.parametrize("inclusive", [False, True], ids=["excl", "incl"])
def test_full_skewed_2p27(ref, inclusive):
    """n = 2^27 values in [0, 255]; Zipf(1.2) lengths capped at 2^22, 5% empty."""
    n = 1 << 27
    off = synth.segment_offsets(n)
    check(ref, synth.u32_byte_values(n), off, inclusive)


# ------------------------------------------------------- Decoupled Fallback

def test_fallback_rescues_silent_tiles(ref):
    """Decoupled Fallback on the segmented scan: a silent tile with heads (its
    rescue publishes the sum after its last head as a prefix) and one without
    (the rescue publishes its row sum as an aggregate); output bit-exact."""
    T = tile()
    n = 600 * T + 77
    values = synth.u32_byte_values(n, seed=41)
    offsets = synth.segment_offsets(n, seed=42)
    starts = np.arange(0, n, T, dtype=np.int64)
    heads = np.searchsorted(offsets, starts + T) - np.searchsorted(offsets, starts)
    with_head = [int(i) for i in np.nonzero(heads > 0)[0] if 0 < i < starts.size - 1]
    without = [int(i) for i in np.nonzero(heads == 0)[0] if 0 < i < starts.size - 1]
    assert with_head and without
    for silent in (with_head[len(with_head) // 2], without[len(without) // 2], 0):
        want = ref.segmented_scan_u32(values, offsets, False, out=np.full(n, SENTINEL, np.uint32))
        v = torch.from_numpy(values.view(np.int32)).cuda()
        o = torch.from_numpy(offsets.astype(np.uint32).view(np.int32)).cuda()
        out = torch.full((n,), SENTINEL - (1 << 32), dtype=torch.int32, device="cuda")
        scratch = dwp.alloc_scratch(dwp.segmented_scan_scratch_bytes(n), v.device)
        try:
            dwp.dwp_debug_set_fault(silent, 0, 64)
            dwp.segmented_scan(v, o, False, out=out, scratch=scratch)
            st = dwp.read_status(scratch)
            fb = dwp.read_fallbacks(scratch)
        finally:
            dwp.dwp_debug_set_fault(0xFFFFFFFF, 0, 0)
        assert st == dwp.DWP_SUCCESS
        got = out.cpu().numpy().view(np.uint32)
        bad = np.nonzero(got != want)[0]
        assert bad.size == 0, "silent %d: mismatch at %s" % (silent, bad[:5])
        # the next tile looks back at the silent one unless its first row is
        # a head (then no tile needs the silent tile's descriptor)
        if not np.isin(starts[silent + 1], offsets):
            assert fb >= 1


def test_bounded_window_same_result(ref):
    """Bounded look-back window on the segmented scan (tiles that hold a head
    never publish an intermediate over their prefix); bit-exact, with and
    without a silent tile."""
    T = tile()
    n = 1500 * T + 19
    values = synth.u32_byte_values(n, seed=43)
    offsets = synth.segment_offsets(n, seed=44)
    want = ref.segmented_scan_u32(values, offsets, True, out=np.full(n, SENTINEL, np.uint32))
    try:
        dwp.dwp_set_lookback_window(32)
        for silent in (0xFFFFFFFF, 700):
            dwp.dwp_debug_set_fault(silent, 0, 64)
            got = gpu_seg(values, offsets, True)
            bad = np.nonzero(got != want)[0]
            assert bad.size == 0, "silent %d: mismatch at %s" % (silent, bad[:5])
    finally:
        dwp.dwp_set_lookback_window(0)
        dwp.dwp_debug_set_fault(0xFFFFFFFF, 0, 0)
