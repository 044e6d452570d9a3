"""Parity of the staged compaction (flags and offsets written to scratch,
three launches) with the oracle, and with the fused kernel it is compared to
("Prefix scans and compaction", section "Worked example: Stable stream
compaction"): the count and every kept record bit for bit, in input order,
output rows past the count untouched."""
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


def gpu_staged(rec: np.ndarray, flags: np.ndarray):
    r = torch.from_numpy(rec.view(np.int32)).cuda()
    f = torch.from_numpy(flags).cuda()
    out = torch.full_like(r, SENTINEL)
    scratch = dwp.alloc_scratch(dwp.compact_staged_scratch_bytes(flags.size), r.device)
    out, cnt = dwp.compact_by_flags_staged(r, f, out=out, scratch=scratch)
    assert dwp.read_status(scratch) == dwp.DWP_SUCCESS
    return out.cpu().numpy().view(np.uint32), int(cnt.item())


def check(ref, rec, flags):
    want, k = ref.compact(rec, flags)
    got, kg = gpu_staged(rec, flags)
    assert kg == k
    bad = np.nonzero((got[:k] != want[:k]).any(axis=1))[0]
    assert bad.size == 0, "mismatch at rows %s" % bad[:5]
    assert (got[k:] == SENTINEL).all()


def test_golden_example():
    ex = golden_io.load()["compaction_positives"]
    vals = np.array(ex["values"], np.int32)
    rec = np.zeros((vals.size, 4), np.uint32)
    rec[:, 0] = vals.view(np.uint32)
    got, k = gpu_staged(rec, (vals > 0).astype(np.uint8))
    assert k == ex["count"] and got[:k, 0].view(np.int32).tolist() == ex["out"]


@pytest.mark.parametrize("kind", ["none", "all", "clustered", "random"])
def test_edge_lengths_and_predicates(ref, kind):
    for n in (1, 3, 4, 5, 15, 16, 17, 31, 1024, 7167, 7168, 7169, 3 * 7168 + 17, 1000003):
        check(ref, synth.records(n, seed=610 + n), synth.flags_pattern(n, kind, seed=710 + n))


def test_empty_input():
    count = torch.full((1,), 77, dtype=torch.int32, device="cuda")
    r = torch.zeros((0, 4), dtype=torch.int32, device="cuda")
    f = torch.zeros(0, dtype=torch.uint8, device="cuda")
    _, cnt = dwp.compact_by_flags_staged(r, f, count=count)
    assert int(cnt.item()) == 0


def test_nonzero_bytes_mean_keep(ref):
    n = 40003
    rec = synth.records(n, seed=811)
    flags = (synth.u64(812, 0, n) & np.uint64(3)).astype(np.uint8) * np.uint8(85)  # 0, 85, 170, 255
    check(ref, rec, flags)


def test_same_output_as_fused(ref):
    """Staged and fused give the same bytes for the same input."""
    n = (1 << 22) + 11
    rec = synth.records(n, seed=813)
    flags = synth.keep_flags(n, 0.3, seed=814)
    got, k = gpu_staged(rec, flags)
    r = torch.from_numpy(rec.view(np.int32)).cuda()
    out = torch.full_like(r, SENTINEL)
    out, cnt = dwp.compact_by_flags(r, torch.from_numpy(flags).cuda(), out=out)
    assert int(cnt.item()) == k
    assert (out.cpu().numpy().view(np.uint32) == got).all()


def test_argument_errors():
    r = torch.zeros((16, 4), dtype=torch.int32, device="cuda")
    f = torch.ones(16, dtype=torch.uint8, device="cuda")
    cnt = torch.zeros(1, dtype=torch.int32, device="cuda")
    need = dwp.compact_staged_scratch_bytes(16)
    scratch = dwp.alloc_scratch(need, r.device)
    st, _ = dwp.dwp_compact_by_flags_staged(r.data_ptr(), f.data_ptr(), 16, r.data_ptr(),
                                            cnt.data_ptr(), scratch.data_ptr(), need, 0)
    assert st == dwp.DWP_ERR_ALIASING
    st, _ = dwp.dwp_compact_by_flags_staged(r.data_ptr(), f.data_ptr(), 16, r.data_ptr() + 4,
                                            cnt.data_ptr(), scratch.data_ptr(), need, 0)
    assert st == dwp.DWP_ERR_MISALIGNED
    st, _ = dwp.dwp_compact_by_flags_staged(r.data_ptr(), f.data_ptr(), 16, 0, cnt.data_ptr(),
                                            scratch.data_ptr(), need - 1, 0)
    assert st == dwp.DWP_ERR_SCRATCH_TOO_SMALL


@pytest.mark.slow
def test_full_2p26_records_p03(ref):
    """The compaction workload: 2^26 records {id = i, 3 x N(0,1)}, keep
    flag Bernoulli(0.3); ids of the output strictly increasing (stable)."""
    n = 1 << 26
    rec = synth.records(n)
    flags = synth.keep_flags(n)
    want, k = ref.compact(rec, flags)
    got, kg = gpu_staged(rec, flags)
    assert kg == k
    assert (got[:k] == want[:k]).all()
    assert (np.diff(got[:k, 0].astype(np.int64)) > 0).all()
