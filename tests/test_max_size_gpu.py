"""The largest sizes the C ABI accepts (n < 2^32 rows; 2^31 + 5 records for
compaction, 32 GiB of records), where a 32-bit product of a tile index and a
tile size would overflow.  The inputs have closed-form results, so the check
runs on the device chunk by chunk instead of through the oracle:
  * all ones: the exclusive u32 scan is y[i] = i mod 2^32, the inclusive one
    i + 1 (the closed form the oracle's pins also use);
  * all ones over hand-placed segments: a segment's exclusive scan counts up
    from 0 at its first row, its sum is its length;
  * every third record kept: out[j] is record 3j, the count ceil(n / 3).
Every row of every output is compared."""
import pytest

pytestmark = [pytest.mark.gpu, pytest.mark.slow]

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import device_wide_prefix_gb300 as dwp  # noqa: E402
from device_wide_prefix_gb300 import build as dwp_build  # noqa: E402

N_MAX = (1 << 32) - 1
CHUNK = 1 << 28


@pytest.fixture(scope="module", autouse=True)
def lib():
    dwp_build.build()
    return dwp.load()


def as_i32(v: torch.Tensor) -> torch.Tensor:
    """int64 values to their low 32 bits, as int32 (the u32 bit pattern)."""
    return (v & 0xFFFFFFFF).to(torch.int64).sub((v & 0x80000000) << 1).to(torch.int32)


def check_counting(y: torch.Tensor, first_value: int, lo: int, hi: int):
    """y[lo:hi] == first_value + (i - lo) modulo 2^32, chunk by chunk."""
    for c0 in range(lo, hi, CHUNK):
        c1 = min(hi, c0 + CHUNK)
        want = as_i32(torch.arange(first_value + (c0 - lo), first_value + (c1 - lo), dtype=torch.int64,
                                   device=y.device))
        assert torch.equal(y[c0:c1], want), (c0, c1)


@pytest.mark.parametrize("inclusive", [False, True])
def test_plain_scan_at_2p32_minus_1(inclusive):
    x = torch.ones(N_MAX, dtype=torch.int32, device="cuda")
    scratch = dwp.alloc_scratch(dwp.scan_scratch_bytes(N_MAX), x.device)
    y = (dwp.scan_inclusive if inclusive else dwp.scan_exclusive)(x, "u32_add", scratch=scratch)
    assert dwp.read_status(scratch) == dwp.DWP_SUCCESS
    del x
    check_counting(y, 1 if inclusive else 0, 0, N_MAX)


def test_segmented_scan_and_reduce_at_2p32_minus_1():
    cuts = [0, 5, 5, 1 << 31, N_MAX - 7, N_MAX]  # an empty segment, and one of 7 rows at the end
    v = torch.ones(N_MAX, dtype=torch.int32, device="cuda")
    off = as_i32(torch.tensor(cuts, dtype=torch.int64)).cuda()
    y = torch.empty_like(v)
    scratch = dwp.alloc_scratch(dwp.segmented_scan_scratch_bytes(N_MAX), v.device)
    dwp.segmented_scan(v, off, False, out=y, scratch=scratch)
    assert dwp.read_status(scratch) == dwp.DWP_SUCCESS
    sums = dwp.segmented_reduce(v, off)
    del v
    for a, b in zip(cuts[:-1], cuts[1:]):
        if b > a:
            check_counting(y, 0, a, b)
    want = [(b - a) & 0xFFFFFFFF for a, b in zip(cuts[:-1], cuts[1:])]
    assert (sums.cpu().to(torch.int64) & 0xFFFFFFFF).tolist() == want


def test_compaction_of_2p31_plus_5_records():
    n = (1 << 31) + 5
    rec = torch.zeros((n, 4), dtype=torch.int32, device="cuda")
    flags = torch.empty(n, dtype=torch.uint8, device="cuda")
    for c0 in range(0, n, CHUNK):
        c1 = min(n, c0 + CHUNK)
        i = torch.arange(c0, c1, dtype=torch.int64, device="cuda")
        rec[c0:c1, 0] = as_i32(i)
        rec[c0:c1, 1] = as_i32(i * 7 + 1)
        flags[c0:c1] = (i % 3 == 0).to(torch.uint8)
    out = torch.empty_like(rec)
    scratch = dwp.alloc_scratch(dwp.compact_scratch_bytes(n), rec.device)
    out, cnt = dwp.compact_by_flags(rec, flags, out=out, scratch=scratch)
    assert dwp.read_status(scratch) == dwp.DWP_SUCCESS
    k = (n + 2) // 3
    assert int(cnt.item()) & 0xFFFFFFFF == k
    del rec, flags
    for c0 in range(0, k, CHUNK):
        c1 = min(k, c0 + CHUNK)
        src = 3 * torch.arange(c0, c1, dtype=torch.int64, device="cuda")
        assert torch.equal(out[c0:c1, 0], as_i32(src)), c0
        assert torch.equal(out[c0:c1, 1], as_i32(src * 7 + 1)), c0
        assert not out[c0:c1, 2:].any()
