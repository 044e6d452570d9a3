"""Parity of the CUDA stable compaction (through the C ABI) with the oracle:
the count and every kept 16-byte record bit for bit, in input order; rows of
the output past the count untouched."""
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

SENTINEL = 0x5EED5EED


@pytest.fixture(scope="module", autouse=True)
def lib():
    dwp_build.build()
    return dwp.load()


@pytest.fixture(scope="module")
def ref():
    return oracle.Oracle()


def tile():
    b1 = dwp.compact_scratch_bytes(1)
    T = 1
    while dwp.compact_scratch_bytes(2 * T) == b1:
        T *= 2
    lo, hi = T, 2 * T
    while hi - lo > 1:
        mid = (lo + hi) // 2
        if dwp.compact_scratch_bytes(mid) == b1:
            lo = mid
        else:
            hi = mid
    return lo


def gpu_compact(rec: np.ndarray, flags: np.ndarray):
    r = torch.from_numpy(rec.view(np.int32)).cuda()
    f = torch.from_numpy(flags).cuda()
    out = torch.full_like(r, SENTINEL)
    scratch = dwp.alloc_scratch(dwp.compact_scratch_bytes(flags.size), r.device)
    out, cnt = dwp.compact_by_flags(r, f, out=out, scratch=scratch)
    assert dwp.read_status(scratch) == dwp.DWP_SUCCESS
    return out.cpu().numpy().view(np.uint32), int(cnt.item())


def check(ref, rec, flags):
    want, k = ref.compact(rec, flags)
    got, kg = gpu_compact(rec, flags)
    assert kg == k
    bad = np.nonzero((got[:k] != want[:k]).any(axis=1))[0]
    assert bad.size == 0, "mismatch at rows %s" % bad[:5]
    assert (got[k:] == SENTINEL).all()


def test_golden_example():
    ex = golden_io.load()["compaction_positives"]
    vals = np.array(ex["values"], np.int32)
    rec = np.zeros((vals.size, 4), np.uint32)
    rec[:, 0] = vals.view(np.uint32)
    flags = (vals > 0).astype(np.uint8)
    got, k = gpu_compact(rec, flags)
    assert k == ex["count"] and got[:k, 0].view(np.int32).tolist() == ex["out"]


@pytest.mark.parametrize("kind", ["none", "all", "clustered", "random"])
def test_edge_lengths_and_predicates(ref, kind):
    T = tile()
    for n in (1, 31, 32, 33, 1024, T - 1, T, T + 1, 3 * T + 17, 1000003):
        rec = synth.records(n, seed=600 + n)
        check(ref, rec, synth.flags_pattern(n, kind, seed=700 + n))


def test_empty_input():
    count = torch.full((1,), 77, dtype=torch.int32, device="cuda")
    r = torch.zeros((0, 4), dtype=torch.int32, device="cuda")
    f = torch.zeros(0, dtype=torch.uint8, device="cuda")
    _, cnt = dwp.compact_by_flags(r, f, count=count)
    assert int(cnt.item()) == 0


def test_nonzero_bytes_mean_keep(ref):
    n = 5 * tile() + 3
    rec = synth.records(n, seed=801)
    flags = (synth.u64(802, 0, n) & np.uint64(3)).astype(np.uint8) * np.uint8(85)  # 0, 85, 170, 255
    check(ref, rec, flags)


def test_repeat_calls_bit_identical(ref):
    n = 1 << 20
    rec = synth.records(n, seed=803)
    flags = synth.keep_flags(n, 0.3, seed=804)
    a, ka = gpu_compact(rec, flags)
    b, kb = gpu_compact(rec, flags)
    assert ka == kb and (a == b).all()


@pytest.mark.slow
def test_full_2p26_records_p03(ref):
    """2^26 records {id = i, 3 x N(0,1)}, keep flag Bernoulli(0.3)."""
    n = 1 << 26
    rec = synth.records(n)
    flags = synth.keep_flags(n)
    want, k = ref.compact(rec, flags)
    got, kg = gpu_compact(rec, flags)
    assert kg == k
    assert (got[:k] == want[:k]).all()
    ids = got[:k, 0].astype(np.int64)
    assert (np.diff(ids) > 0).all()  # stable: ids = input index, strictly increasing


# ------------------------------------------------------- Decoupled Fallback

@pytest.mark.parametrize("silent", [0, 7, 399])
def test_fallback_rescues_a_silent_tile(ref, silent):
    """Decoupled Fallback on compaction: a silent tile's kept count is
    counted from its flags by a waiting successor; count and records exact."""
    n = 400 * tile() - 9
    rec = synth.records(n, seed=901)
    flags = synth.keep_flags(n, 0.3, seed=902)
    want, k = ref.compact(rec, flags)
    r = torch.from_numpy(rec.view(np.int32)).cuda()
    f = torch.from_numpy(flags).cuda()
    out = torch.full_like(r, SENTINEL)
    scratch = dwp.alloc_scratch(dwp.compact_scratch_bytes(n), r.device)
    try:
        dwp.dwp_debug_set_fault(silent, 0, 64)
        out, cnt = dwp.compact_by_flags(r, f, out=out, scratch=scratch)
        st = dwp.read_status(scratch)
        fb = dwp.read_fallbacks(scratch)
    finally:
        dwp.dwp_debug_set_fault(0xFFFFFFFF, 0, 0)
    assert st == dwp.DWP_SUCCESS
    if silent < 399:
        assert fb >= 1
    got = out.cpu().numpy().view(np.uint32)
    assert int(cnt.item()) == k
    assert (got[:k] == want[:k]).all() and (got[k:] == SENTINEL).all()


def test_bounded_window_same_result(ref):
    n = 1500 * tile() + 5
    rec = synth.records(n, seed=903)
    flags = synth.keep_flags(n, 0.3, seed=904)
    try:
        dwp.dwp_set_lookback_window(64)
        for silent in (0xFFFFFFFF, 600):
            dwp.dwp_debug_set_fault(silent, 0, 64)
            check(ref, rec, flags)
    finally:
        dwp.dwp_set_lookback_window(0)
        dwp.dwp_debug_set_fault(0xFFFFFFFF, 0, 0)
