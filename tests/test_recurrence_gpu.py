"""Parity of the CUDA linear recurrence h[t] = a[t] h[t-1] + b[t] (through the
C ABI) with the sequential oracle.

The bar is |h_gpu[t] - h_ref[t]| <= 1e-4 * g[t] + 1e-6, where g is the
magnitude recurrence g[t] = |a[t]| g[t-1] + |b[t]| the oracle returns beside
h.  It is the f32 scan's bound with the running sum of |x| replaced by g (for
a = 1 the two coincide): every f32 rounding in the pair scan, whatever its
grouping, is at most 2^-24 of a term the magnitude recurrence bounds, and
the longest chain of roundings between an input and an output (one thread's
items, the block fold, the look-back fold) is a few hundred steps.
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

REL, ABS = 1e-4, 1e-6
SENTINEL = np.float32(-12345.0)


@pytest.fixture(scope="module", autouse=True)
def lib():
    dwp_build.build()
    return dwp.load()


@pytest.fixture(scope="module")
def ref():
    return oracle.Oracle()


def tile():
    b1 = dwp.linear_recurrence_scratch_bytes(1)
    T = 1
    while dwp.linear_recurrence_scratch_bytes(2 * T) == b1:
        T *= 2
    lo, hi = T, 2 * T
    while hi - lo > 1:
        mid = (lo + hi) // 2
        if dwp.linear_recurrence_scratch_bytes(mid) == b1:
            lo = mid
        else:
            hi = mid
    return lo


def gpu_rec(a, b, inclusive, inplace=None):
    ta, tb = torch.from_numpy(a).cuda(), torch.from_numpy(b).cuda()
    out = {"a": ta, "b": tb}.get(inplace) if inplace else torch.full_like(tb, float(SENTINEL))
    scratch = dwp.alloc_scratch(dwp.linear_recurrence_scratch_bytes(a.size), ta.device)
    dwp.linear_recurrence(ta, tb, inclusive, out=out, scratch=scratch)
    assert dwp.read_status(scratch) == dwp.DWP_SUCCESS
    return out.cpu().numpy()


def check(ref, a, b, inclusive, got):
    want, g = ref.linear_recurrence(a, b, inclusive)
    err = np.abs(got.astype(np.float64) - want)
    bound = REL * g + ABS
    bad = np.nonzero(~(err <= bound))[0]
    assert bad.size == 0, "out of tolerance at %s: got %s want %s bound %s" % (
        bad[:5], got[bad[:5]], want[bad[:5]], bound[bad[:5]])


def test_golden_example(ref):
    ex = golden_io.load()["linear_recurrence"]
    a, b = np.array(ex["a"], np.float32), np.array(ex["b"], np.float32)
    got = gpu_rec(a, b, True)
    assert np.allclose(got, ex["h"], rtol=1e-6, atol=0)
    check(ref, a, b, True, got)
    check(ref, a, b, False, gpu_rec(a, b, False))


@pytest.mark.parametrize("inclusive", [False, True])
def test_edge_sizes(ref, inclusive):
    T = tile()
    for n in (1, 3, 4, 5, 31, 32, 33, T - 1, T, T + 1, 3 * T + 17, 1000003):
        a = synth.decay_values(n, seed=300 + n)
        b = synth.f32_values(n, seed=400 + n)
        check(ref, a, b, inclusive, gpu_rec(a, b, inclusive))


def test_signed_and_unit_coefficients(ref):
    """a in [-1, -0.5) (the state alternates in sign), and a = 1 exactly (the
    recurrence is then the f32 running sum of b)."""
    n = 777 * tile() + 5
    b = synth.f32_values(n, seed=501)
    for a in (synth.decay_values(n, seed=502, lo=-1.0), np.ones(n, np.float32)):
        for inc in (False, True):
            check(ref, a, b, inc, gpu_rec(a, b, inc))


def test_zero_coefficients_are_exact(ref):
    """a = 0 cuts every step off from the last: h = b exactly (one fused
    multiply-add of 0 * h + b), exclusive = b shifted by one."""
    n = 50 * tile() + 3
    a = np.zeros(n, np.float32)
    b = synth.f32_values(n, seed=503)
    assert (gpu_rec(a, b, True) == b).all()
    ye = gpu_rec(a, b, False)
    assert ye[0] == 0.0 and (ye[1:] == b[:-1]).all()


@pytest.mark.parametrize("which", ["a", "b"])
def test_in_place(ref, which):
    n = 40 * tile() + 9
    a = synth.decay_values(n, seed=504)
    b = synth.f32_values(n, seed=505)
    check(ref, a, b, True, gpu_rec(a, b, True, inplace=which))


def test_empty(ref):
    ta = torch.zeros(0, dtype=torch.float32, device="cuda")
    out = dwp.linear_recurrence(ta, ta.clone(), True)
    assert out.numel() == 0


def test_rows_past_n_untouched(ref):
    """The output buffer is longer than n: nothing past n is written."""
    n = 5 * tile() + 11
    a = synth.decay_values(n, seed=506)
    b = synth.f32_values(n, seed=507)
    ta, tb = torch.from_numpy(a).cuda(), torch.from_numpy(b).cuda()
    big = torch.full((n + 64,), float(SENTINEL), dtype=torch.float32, device="cuda")
    dwp.linear_recurrence(ta, tb, True, out=big[:n])
    got = big.cpu().numpy()
    check(ref, a, b, True, got[:n])
    assert (got[n:] == SENTINEL).all()


@pytest.mark.slow
@pytest.mark.parametrize("inclusive", [True, False])
def test_full_2p28_decay(ref, inclusive):
    """n = 2^28, a uniform in [0.5, 1), b uniform in [-1, 1): every element."""
    n = 1 << 28
    a = synth.decay_values(n)
    b = synth.f32_values(n, seed=synth.SEED_RECURRENCE_B)
    check(ref, a, b, inclusive, gpu_rec(a, b, inclusive))


# ------------------------------------------------------- Decoupled Fallback

@pytest.mark.parametrize("silent", [0, 6, 999])
def test_fallback_rescues_a_silent_tile(ref, silent):
    """A tile that never publishes is composed by a waiting successor from a
    and b (lane runs folded in order); the call succeeds within the bound."""
    n = 999 * tile() + 321
    a = synth.decay_values(n, seed=508)
    b = synth.f32_values(n, seed=509)
    ta, tb = torch.from_numpy(a).cuda(), torch.from_numpy(b).cuda()
    scratch = dwp.alloc_scratch(dwp.linear_recurrence_scratch_bytes(n), ta.device)
    try:
        dwp.dwp_debug_set_fault(silent, 0, 64)
        out = dwp.linear_recurrence(ta, tb, True, scratch=scratch)
        st = dwp.read_status(scratch)
        fb = dwp.read_fallbacks(scratch)
    finally:
        dwp.dwp_debug_set_fault(0xFFFFFFFF, 0, 0)
    assert st == dwp.DWP_SUCCESS
    if silent < 999:
        assert fb >= 1
    check(ref, a, b, True, out.cpu().numpy())


def test_timeout_without_fallback(ref):
    n = 1000 * tile()
    a = torch.from_numpy(synth.decay_values(n, seed=510)).cuda()
    b = torch.from_numpy(synth.f32_values(n, seed=511)).cuda()
    scratch = dwp.alloc_scratch(dwp.linear_recurrence_scratch_bytes(n), a.device)
    try:
        dwp.dwp_debug_set_fault(5, 2000, 0xFFFFFFFF)
        dwp.linear_recurrence(a, b, True, scratch=scratch)
        assert dwp.read_status(scratch) == dwp.DWP_ERR_LOOKBACK_TIMEOUT
    finally:
        dwp.dwp_debug_set_fault(0xFFFFFFFF, 0, 0)
    dwp.linear_recurrence(a, b, True, scratch=scratch)
    assert dwp.read_status(scratch) == dwp.DWP_SUCCESS
