"""Parity of the CUDA segmented u32 reduction (through the C ABI) with the
oracle: one wrapping sum per segment, bit for bit; empty segments 0."""
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


T = None


def tile():
    """Rows per tile: the largest tile size is not visible in the scratch size
    (no per-tile state), so the tests use sizes around several candidates."""
    return 3072


def gpu_reduce(values, offsets):
    v = torch.from_numpy(values.view(np.int32)).cuda() if values.size else \
        torch.zeros(0, dtype=torch.int32, device="cuda")
    o = torch.from_numpy(np.ascontiguousarray(offsets, dtype=np.uint32).view(np.int32)).cuda()
    nseg = max(offsets.size - 1, 0)
    out = torch.full((max(nseg, 1),), 0x5A5A5A5A, dtype=torch.int32, device="cuda")[:nseg]
    scratch = dwp.alloc_scratch(dwp.segmented_reduce_scratch_bytes(values.size), o.device)
    dwp.segmented_reduce(v, o, out=out, scratch=scratch)
    assert dwp.read_status(scratch) == dwp.DWP_SUCCESS
    return out.cpu().numpy().view(np.uint32)


def check(ref, values, offsets):
    want = ref.segmented_reduce_u32(values, offsets)
    got = gpu_reduce(values, offsets)
    bad = np.nonzero(got != want)[0]
    assert bad.size == 0, "mismatch at segments %s: got %s want %s" % (bad[:5], got[bad[:5]], want[bad[:5]])


def test_golden_example():
    ex = golden_io.load()["segmented_luma"]
    v = np.array(ex["values"], np.uint32)
    off = np.array(ex["offsets"], np.uint32)
    assert gpu_reduce(v, off).tolist() == [5, 15, 7]


def test_shapes(ref):
    for n in (1, 5, 3071, 3072, 3073, 7 * 3072 + 5, 1000003):
        v = synth.u32_full_values(n, seed=1100 + n % 97)
        shapes = {
            "one": [0, n],
            "all_len1": list(range(n + 1)) if n <= 100000 else [0, n],
            "empties": sorted({0, 0, 0, n // 7, n // 7, n // 3, n, n} | {n // 2}) + [n, n],
            "partial": [min(7, n), min(7, n), n // 2, max(n - 3, n // 2)],
            "tile_aligned": sorted(set([0] + list(range(0, n, 3072)) + [n])),
            "inside_and_across": sorted(set([0, 1, 2, 3070, 3071, 3072, 3073, 6144, 6200, n]) & set(range(n + 1))) + [n],
        }
        for name, offs in shapes.items():
            off = np.array(offs, np.uint32)
            off = np.maximum.accumulate(off)
            check(ref, v, off)


def test_many_segments(ref):
    """100,000 random cuts of 2^22 rows (many segments per tile, some empty)."""
    n = 1 << 22
    v = synth.u32_full_values(n, seed=1201)
    cuts = np.sort((synth.u64(1202, 0, 100000) % np.uint64(n + 1)).astype(np.uint32))
    off = np.concatenate([[0], cuts, [n]]).astype(np.uint32)
    check(ref, v, off)


def test_zipf_small(ref):
    n = 1 << 22
    check(ref, synth.u32_byte_values(n, seed=1203), synth.segment_offsets(n, seed=1204, cap=1 << 16))


def test_degenerate():
    # no rows: every segment is empty, all zeros
    off = np.zeros(6, np.uint32)
    assert (gpu_reduce(np.zeros(0, np.uint32), off) == 0).all()
    # no segments: nothing to write
    assert gpu_reduce(synth.u32_full_values(100, seed=1), np.zeros(1, np.uint32)).size == 0


def test_repeat_calls_identical(ref):
    n = 1 << 21
    v = synth.u32_full_values(n, seed=1205)
    off = synth.segment_offsets(n, seed=1206, cap=1 << 15)
    a = gpu_reduce(v, off)
    b = gpu_reduce(v, off)
    assert (a == b).all()


@pytest.mark.slow
def test_full_2p27_skewed(ref):
    """The skewed workload of the segmented scan: n = 2^27, Zipf(1.2) lengths."""
    n = 1 << 27
    check(ref, synth.u32_byte_values(n), synth.segment_offsets(n))
