"""Pins for the oracle: checks against what the pages print and what the
mathematics fixes, none of which re-types the oracle's own loop.

Each pin is a function taking an `oracle.Oracle` and raising AssertionError
on a mismatch.  test_oracle.py runs every pin on the real oracle;
test_oracle_mutants.py runs them all on copies of the oracle with a planted
mistake and requires that some pin fails for every mistake.

Independent references used here:
  * the worked examples printed on the pages (tests/golden/worked_examples.ini);
  * a brute-force O(n^2) definition, each output reduced on its own from its
    index range ("Parallel Prefix Sum (Scan), in depth", "Inclusive, exclusive
    and associative");
  * a Hillis-Steele step simulation and a Blelloch up/down-sweep written from
    the descriptions in "Parallel Prefix Sum (Scan), in depth";
  * closed forms and invariants, and numpy library routines (cumsum, boolean
    indexing, nonzero) that the oracle does not use;
  * for the linear recurrence, its closed-form expansion and a tree scan of
    the (a, b) pairs under the page's pair combination, both in exact
    rational arithmetic (fractions.Fraction) on the f32 inputs.
"""
from __future__ import annotations

import math

import numpy as np

import golden_io
import synth

M32 = 0xFFFFFFFF
GOLD = golden_io.load()


# ----------------------------------------------------------------------------
# independent reference algorithms


def brute_scan(x, op: str, inclusive: bool):
    """y[i] = reduction of x over [0, i] or [0, i), each i reduced from scratch."""
    out = []
    for i in range(len(x)):
        hi = i + 1 if inclusive else i
        if op == "u32_add":
            acc = 0
            for j in range(hi):
                acc = (acc + int(x[j])) & M32
        elif op == "u32_max":
            acc = 0
            for j in range(hi):
                acc = max(acc, int(x[j]))
        elif op == "f32_add":
            acc = math.fsum(float(x[j]) for j in range(hi))
        else:
            raise ValueError(op)
        out.append(acc)
    return out


def hillis_steele_steps(x):
    """All intermediate arrays of the Hillis-Steele scan: in the step with
    distance d every element i >= d adds the value d places to its left, all
    reading the previous step's array (double buffering)."""
    cur = [int(v) for v in x]
    steps = []
    d = 1
    while d < len(cur):
        nxt = [cur[i] + (cur[i - d] if i >= d else 0) for i in range(len(cur))]
        steps.append(nxt)
        cur = nxt
        d *= 2
    return steps


def blelloch(x):
    """Work-efficient exclusive scan on a power-of-two length: an up-sweep that
    builds subtree totals, the root cleared to the identity, then a down-sweep
    where a left child takes its parent's prefix and a right child takes the
    parent's prefix plus the old left-subtree total.  Returns (scan, total)."""
    a = [int(v) for v in x]
    n = len(a)
    assert n & (n - 1) == 0
    span = 2
    while span <= n:
        for right in range(span - 1, n, span):
            a[right] += a[right - span // 2]
        span *= 2
    total = a[n - 1]
    a[n - 1] = 0
    span = n
    while span >= 2:
        half = span // 2
        for right in range(span - 1, n, span):
            left = right - half
            a[left], a[right] = a[right], a[right] + a[left]
        span //= 2
    return a, total


# ----------------------------------------------------------------------------
# pins: scans


def pin_golden_scans(o):
    """Every printed scan example, exclusive and inclusive where printed."""
    for name, ex in GOLD.items():
        if ex.get("op") != "u32_add":
            continue
        x = np.array(ex["x"], dtype=np.uint32)
        if "exclusive" in ex:
            assert o.scan_u32_add(x, False).tolist() == ex["exclusive"], name
        if "inclusive" in ex:
            assert o.scan_u32_add(x, True).tolist() == ex["inclusive"], name
        if "total" in ex:
            assert int(o.scan_u32_add(x, True)[-1]) == ex["total"], name


def pin_hillis_steele_trace(o):
    """The printed 8-element Hillis-Steele trace ends in the oracle's inclusive scan."""
    ex = GOLD["hillis_steele_8"]
    steps = hillis_steele_steps(ex["x"])
    assert steps == [ex["step_d1"], ex["step_d2"], ex["step_d4"]]
    assert o.scan_u32_add(np.array(ex["x"], np.uint32), True).tolist() == steps[-1]


def pin_blelloch(o):
    """The printed Blelloch example, and Blelloch == oracle exclusive on random
    power-of-two inputs (values small enough that no sum wraps)."""
    ex = GOLD["blelloch_8"]
    scan, total = blelloch(ex["x"])
    assert scan == ex["exclusive"] and total == ex["total"]
    for k, n in enumerate((1, 2, 16, 256, 4096)):
        x = synth.u32_small_values(n, seed=1000 + k)
        ref, tot = blelloch(x.tolist())
        y = o.scan_u32_add(x, False)
        assert y.tolist() == ref
        assert int(o.scan_u32_add(x, True)[-1]) == tot


def pin_brute_force(o):
    """O(n^2) definition, every op and mode, n = 0 .. 64, full-range values."""
    for n in list(range(0, 17)) + [31, 32, 33, 63, 64]:
        xu = synth.u32_full_values(n, seed=2000 + n)
        xf = synth.f32_values(n, seed=3000 + n)
        for inc in (False, True):
            assert o.scan_u32_add(xu, inc).tolist() == brute_scan(xu, "u32_add", inc), (n, inc)
            assert o.scan_u32_max(xu, inc).tolist() == brute_scan(xu, "u32_max", inc), (n, inc)
            # f32 inputs on the 2^-23 grid in [-1, 1): every partial sum of <= 64
            # of them is exact in double, so the oracle must equal fsum exactly.
            y, a = o.scan_f32_add(xf, inc)
            assert y.tolist() == brute_scan(xf, "f32_add", inc), (n, inc)
            assert a.tolist() == brute_scan(np.abs(xf), "f32_add", inc), (n, inc)


def pin_closed_forms(o):
    n = 5000
    i = np.arange(n, dtype=np.uint64)
    ones = np.ones(n, np.uint32)
    assert (o.scan_u32_add(ones, False) == i.astype(np.uint32)).all()
    assert (o.scan_u32_add(ones, True) == (i + 1).astype(np.uint32)).all()
    c = 0x9E3779B9
    y = o.scan_u32_add(np.full(n, c, np.uint32), False)
    assert (y == ((i * c) % 2**32).astype(np.uint32)).all()
    y = o.scan_u32_add(np.full(n, M32, np.uint32), False)
    assert (y == ((2**32 - i) % 2**32).astype(np.uint32)).all()  # -i mod 2^32
    asc = np.sort(synth.u32_full_values(n, seed=4000))
    assert (o.scan_u32_max(asc, True) == asc).all()
    desc = asc[::-1].copy()
    assert (o.scan_u32_max(desc, True) == desc[0]).all()
    assert o.scan_u32_max(desc, False)[0] == 0 and (o.scan_u32_max(desc, False)[1:] == desc[0]).all()
    assert o.scan_u32_add(np.zeros(0, np.uint32), False).size == 0


def pin_invariants(o):
    for k, n in enumerate((1, 2, 1000, 100003)):
        x = synth.u32_full_values(n, seed=5000 + k)
        ex, inc = o.scan_u32_add(x, False), o.scan_u32_add(x, True)
        assert ((inc - ex) == x).all()                      # wraps: uint32 arithmetic
        assert ex[0] == 0
        assert (ex[1:] == inc[:-1]).all()
        assert int(inc[-1]) == int(np.sum(x, dtype=np.uint64)) % 2**32
        mx, mi = o.scan_u32_max(x, False), o.scan_u32_max(x, True)
        assert (mi == np.maximum(mx, x)).all()
        assert mx[0] == 0 and (mx[1:] == mi[:-1]).all()
        assert (np.diff(mi.astype(np.int64)) >= 0).all()
        assert (mi == np.maximum.accumulate(x)).all()
        assert int(mi[-1]) == int(x.max())


def pin_f32(o):
    """4096 copies of 0.1f: the exact total is 4096 * 0.1f = 409.600006103515625
    ("Parallel Prefix Sum (Scan), in depth", "Numerics and determinism"; the
    page's printed f32 result is a rounded figure, the exact sum is used); and
    the double prefix equals numpy's sequential double cumsum bit for bit."""
    x = np.full(4096, 0.1, np.float32)
    y, a = o.scan_f32_add(x, True)
    assert y[-1] == 409.600006103515625 and a[-1] == 409.600006103515625
    assert (y == np.arange(1, 4097) * float(np.float32(0.1))).all()
    ye, _ = o.scan_f32_add(x, False)
    assert ye[0] == 0.0 and (ye[1:] == y[:-1]).all()
    xf = synth.f32_values(200001, seed=6000)
    y, a = o.scan_f32_add(xf, True)
    assert (y == np.cumsum(xf.astype(np.float64))).all()
    assert (a == np.cumsum(np.abs(xf.astype(np.float64)))).all()
    ye, ae = o.scan_f32_add(xf, False)
    assert ye[0] == 0.0 and (ye[1:] == y[:-1]).all() and (ae[1:] == a[:-1]).all()


# ----------------------------------------------------------------------------
# pins: segmented scan


def _segmented_ref(values, offsets, inclusive, fill):
    """Per segment, numpy cumsum in uint64 then reduced mod 2^32."""
    out = np.array(fill, dtype=np.uint32, copy=True)
    for s in range(len(offsets) - 1):
        lo, hi = int(offsets[s]), int(offsets[s + 1])
        if hi <= lo:
            continue
        c = np.cumsum(values[lo:hi].astype(np.uint64)) % 2**32
        if inclusive:
            out[lo:hi] = c
        else:
            out[lo] = 0
            out[lo + 1:hi] = c[:-1]
    return out


def pin_segmented_golden(o):
    ex = GOLD["segmented_luma"]
    v = np.array(ex["values"], np.uint32)
    off = np.array(ex["offsets"], np.uint32)
    assert o.segmented_scan_u32(v, off, False).tolist() == ex["exclusive"]
    assert o.segmented_scan_u32(v, off, True).tolist() == ex["inclusive"]


def pin_segmented_shapes(o):
    """Empty segments (leading, trailing, consecutive), one segment, all length 1,
    rows outside [offsets[0], offsets[N]) untouched, heads reset to 0."""
    n = 3000
    v = synth.u32_full_values(n, seed=7000)
    sentinel = np.full(n, 0xDEADBEEF, np.uint32)
    shapes = {
        "one": [0, n],
        "all_len1": list(range(n + 1)),
        "empties": [0, 0, 0, 5, 5, 100, 100, 100, 1500, 2999, n, n, n],
        "partial_cover": [7, 7, 40, 1000, 2500],
    }
    for name, offs in shapes.items():
        off = np.array(offs, np.uint32)
        for inc in (False, True):
            y = o.segmented_scan_u32(v, off, inc, out=sentinel)
            assert (y == _segmented_ref(v, off, inc, sentinel)).all(), (name, inc)
        ye = o.segmented_scan_u32(v, off, False, out=sentinel)
        yi = o.segmented_scan_u32(v, off, True, out=sentinel)
        lo, hi = int(off[0]), int(off[-1])
        assert (ye[:lo] == 0xDEADBEEF).all() and (ye[hi:] == 0xDEADBEEF).all(), name
        assert ((yi[lo:hi] - ye[lo:hi]) == v[lo:hi]).all(), name
        heads = sorted({int(p) for p in off[:-1] if int(p) < hi})
        for h in heads:
            assert ye[h] == 0 and yi[h] == v[h], (name, h)
    one = np.array([0, n], np.uint32)
    for inc in (False, True):
        assert (o.segmented_scan_u32(v, one, inc) == o.scan_u32_add(v, inc)).all()


def pin_segmented_zipf(o):
    """The skewed-length generator's offsets on a smaller n, checked per segment."""
    n = 1 << 18
    off = synth.segment_offsets(n, seed=7100, cap=1 << 14)
    v = synth.u32_byte_values(n, seed=7101)
    for inc in (False, True):
        assert (o.segmented_scan_u32(v, off, inc) == _segmented_ref(v, off, inc, np.zeros(n, np.uint32))).all()


# ----------------------------------------------------------------------------
# pins: segmented reduction


def _reduce_ref(values, offsets):
    """numpy: uint64 reduceat per non-empty segment, then mod 2^32; 0 for empty."""
    nseg = len(offsets) - 1
    out = np.zeros(nseg, np.uint64)
    v64 = values.astype(np.uint64)
    lo = offsets[:-1].astype(np.int64)
    hi = offsets[1:].astype(np.int64)
    nonempty = np.nonzero(hi > lo)[0]
    if nonempty.size:
        sums = np.add.reduceat(v64, lo[nonempty])
        # reduceat sums up to the next listed start; the next start of a
        # non-empty segment is the end of it (empties are skipped), except
        # after the last one, which runs to the end of the array
        if hi[nonempty[-1]] < values.size:
            sums[-1] -= np.sum(v64[hi[nonempty[-1]]:], dtype=np.uint64)
        out[nonempty] = sums
    return (out % 2**32).astype(np.uint32)


def pin_segmented_reduce(o):
    """The printed segmented example's segment totals (the last inclusive value
    of each segment: [5, 15, 7]); numpy reduceat on the shapes of the
    segmented pins and on the skewed generator; brute force on tiny inputs;
    empty segments give 0; one segment gives the wrapping total; all length
    1 gives the values; the totals add up to the covered rows' sum."""
    ex = GOLD["segmented_luma"]
    v = np.array(ex["values"], np.uint32)
    off = np.array(ex["offsets"], np.uint32)
    incl = ex["inclusive"]
    ends = [int(off[s + 1]) - 1 for s in range(len(off) - 1)]
    assert o.segmented_reduce_u32(v, off).tolist() == [incl[e] for e in ends] == [5, 15, 7]
    n = 3000
    v = synth.u32_full_values(n, seed=7200)
    shapes = [[0, n], list(range(n + 1)), [0, 0, 0, 5, 5, 100, 100, 100, 1500, 2999, n, n, n],
              [7, 7, 40, 1000, 2500]]
    for offs in shapes:
        off = np.array(offs, np.uint32)
        got = o.segmented_reduce_u32(v, off)
        assert (got == _reduce_ref(v, off)).all(), offs[:4]
        assert int(np.sum(got, dtype=np.uint64)) % 2**32 == \
            int(np.sum(v[off[0]:off[-1]], dtype=np.uint64)) % 2**32
        empty = np.nonzero(off[1:] == off[:-1])[0]
        assert (got[empty] == 0).all()
    assert (o.segmented_reduce_u32(v, np.arange(n + 1, dtype=np.uint32)) == v).all()
    assert int(o.segmented_reduce_u32(v, np.array([0, n], np.uint32))[0]) == \
        int(np.sum(v, dtype=np.uint64)) % 2**32
    for k in range(20):
        m = k + 1
        vv = synth.u32_full_values(m, seed=7300 + k)
        cuts = np.sort(synth.u32_small_values(k % 5 + 1, seed=7400 + k) % (m + 1))
        off = np.concatenate([[0], cuts, [m]]).astype(np.uint32)
        want = [sum(int(vv[j]) for j in range(int(off[s]), int(off[s + 1]))) % 2**32
                for s in range(off.size - 1)]
        assert o.segmented_reduce_u32(vv, off).tolist() == want
    nz = 1 << 18
    off = synth.segment_offsets(nz, seed=7500, cap=1 << 14)
    vz = synth.u32_byte_values(nz, seed=7501)
    assert (o.segmented_reduce_u32(vz, off) == _reduce_ref(vz, off)).all()


# ----------------------------------------------------------------------------
# pins: compaction


def pin_compaction_golden(o):
    ex = GOLD["compaction_positives"]
    vals = np.array(ex["values"], np.int32).reshape(-1, 1)
    flags = (vals[:, 0] > 0).astype(np.uint8)
    assert flags.tolist() == ex["flags"]
    # the printed offsets are the exclusive scan of the flags
    assert o.scan_u32_add(flags.astype(np.uint32), False).tolist() == ex["offsets"]
    out, k = o.compact(vals, flags)
    assert k == ex["count"] and out[:k, 0].tolist() == ex["out"]
    # "Expose every array in stable stream compaction": keep values >= 5, checked
    # against a stable Python filter (the page gives the task, not the answer)
    arr = [7, 2, 9, 4, 5, 8, 1, 6]
    vals = np.array(arr, np.int32).reshape(-1, 1)
    fl = (vals[:, 0] >= 5).astype(np.uint8)
    out, k = o.compact(vals, fl)
    kept = [v for v in arr if v >= 5]
    assert k == len(kept) and out[:k, 0].tolist() == kept


def pin_compaction_properties(o):
    """Lengths 0, 1, 31, 32, 33, 1024, 1,000,003 x predicates none/all/clustered/random:
    count = popcount, ids strictly increasing and exactly the kept indices, bytes
    equal to numpy boolean indexing, rows past count untouched (zero)."""
    for n in (0, 1, 31, 32, 33, 1024, 1000003):
        rec = synth.records(n, seed=8000 + n)
        for kind in ("none", "all", "clustered", "random"):
            fl = synth.flags_pattern(n, kind, seed=8100 + n)
            out, k = o.compact(rec, fl)
            assert k == int(np.count_nonzero(fl)), (n, kind)
            ids = out[:k, 0].astype(np.int64)
            assert (np.diff(ids) > 0).all(), (n, kind)
            assert (ids == np.nonzero(fl)[0]).all(), (n, kind)
            assert (out[:k] == rec[fl != 0]).all(), (n, kind)
            assert (out[k:] == 0).all(), (n, kind)


# ----------------------------------------------------------------------------
# pins: linear recurrence h[t] = a[t] h[t-1] + b[t], h[-1] = 0


def _exact(v):
    from fractions import Fraction
    return [Fraction(float(x)) for x in v]


def recurrence_expansion(a, b, inclusive):
    """Each output written out on its own: the state after step s is
    sum_{j <= s} b[j] * prod_{j < k <= s} a[k]; inclusive reports s = t,
    exclusive s = t - 1 (the empty sum, 0, for t = 0).  Exact rationals,
    rounded once to double."""
    from fractions import Fraction
    A, B = _exact(a), _exact(b)
    out = []
    for t in range(len(A)):
        s = t if inclusive else t - 1
        acc = Fraction(0)
        for j in range(s + 1):
            p = B[j]
            for k in range(j + 1, s + 1):
                p *= A[k]
            acc += p
        out.append(float(acc))
    return out


def pair_tree_scan(a, b):
    """Inclusive scan of the pairs under the page's combination, (a1, b1) then
    (a2, b2) = (a1 a2, a2 b1 + b2), evaluated as a Hillis-Steele tree (in step
    d every element combines with the one d places to its left, reading the
    previous step), exact rationals.  The b part of pair t is h[t]."""
    cur = list(zip(_exact(a), _exact(b)))
    d = 1
    while d < len(cur):
        nxt = list(cur)
        for i in range(d, len(cur)):
            (a1, b1), (a2, b2) = cur[i - d], cur[i]
            nxt[i] = (a1 * a2, a2 * b1 + b2)
        cur = nxt
        d *= 2
    return [float(y) for _, y in cur]


def pin_recurrence_golden(o):
    """The printed example: a = [0.5, 0.9, 0.1, 1.0], b = [1, 2, 3, 4] gives
    [1.0, 2.9, 3.29, 7.29] by the loop and by the pair scan.  The inputs are
    f32 (0.9 and 0.1 are not exact), so agreement is to f32 input rounding."""
    ex = GOLD["linear_recurrence"]
    a, b = np.array(ex["a"], np.float32), np.array(ex["b"], np.float32)
    want = np.array(ex["h"], np.float64)
    y, g = o.linear_recurrence(a, b, True)
    assert (np.abs(y - want) <= 1e-6 * g).all(), y
    assert (np.abs(np.array(pair_tree_scan(a, b)) - want) <= 1e-6 * g).all()
    ye, _ = o.linear_recurrence(a, b, False)
    assert ye[0] == 0.0 and (np.abs(ye[1:] - want[:-1]) <= 1e-6 * g[:-1]).all()


def pin_recurrence_expansion(o):
    """n = 0 .. 12, 31, 32, 33, 40 with signed a in [-1.5, 1.5) and b in [-1, 1):
    the oracle equals the closed-form expansion and the pair tree scan to
    double rounding, in both modes; its magnitude output equals the expansion
    on |a| and |b|."""
    for n in list(range(0, 13)) + [31, 32, 33, 40]:
        a = (synth.f32_values(n, seed=9000 + n) * np.float32(1.5)).astype(np.float32)
        b = synth.f32_values(n, seed=9100 + n)
        for inc in (False, True):
            y, g = o.linear_recurrence(a, b, inc)
            ref = np.array(recurrence_expansion(a, b, inc))
            mag = np.array(recurrence_expansion(np.abs(a), np.abs(b), inc))
            assert (np.abs(y - ref) <= 1e-12 * (mag + 1.0)).all(), (n, inc)
            assert (np.abs(g - mag) <= 1e-12 * (mag + 1.0)).all(), (n, inc)
        tree = np.array(pair_tree_scan(a, b))
        assert (tree == np.array(recurrence_expansion(a, b, True))).all(), n


def pin_recurrence_special_cases(o):
    """a = 1: the running sum of b (numpy's sequential double cumsum, bit for
    bit); a = 0: h = b; b = 0: h = 0; a = c, b = 1: the geometric series
    (1 - c^(t+1)) / (1 - c); a, b >= 0: magnitude = h; exclusive = inclusive
    shifted by one, starting at 0; empty input."""
    n = 20000
    b = synth.f32_values(n, seed=9200)
    ones, zeros = np.ones(n, np.float32), np.zeros(n, np.float32)
    y, g = o.linear_recurrence(ones, b, True)
    assert (y == np.cumsum(b.astype(np.float64))).all()
    assert (g == np.cumsum(np.abs(b.astype(np.float64)))).all()
    assert (o.linear_recurrence(zeros, b, True)[0] == b.astype(np.float64)).all()
    assert (o.linear_recurrence(synth.decay_values(n, seed=9201), zeros, True)[0] == 0.0).all()
    c = 0.75
    y, _ = o.linear_recurrence(np.full(n, c, np.float32), ones, True)
    t = np.arange(n, dtype=np.float64)
    assert np.allclose(y, (1.0 - c ** (t + 1.0)) / (1.0 - c), rtol=1e-12, atol=0.0)
    a = synth.decay_values(n, seed=9202)
    bp = np.abs(b)
    y, g = o.linear_recurrence(a, bp, True)
    assert (y == g).all()
    a = (synth.f32_values(n, seed=9203) * np.float32(1.1)).astype(np.float32)
    for arr_b in (b, bp):
        yi, gi = o.linear_recurrence(a, arr_b, True)
        ye, ge = o.linear_recurrence(a, arr_b, False)
        assert ye[0] == 0.0 and ge[0] == 0.0
        assert (ye[1:] == yi[:-1]).all() and (ge[1:] == gi[:-1]).all()
    y, g = o.linear_recurrence(np.zeros(0, np.float32), np.zeros(0, np.float32), True)
    assert y.size == 0 and g.size == 0


ALL_PINS = [
    pin_golden_scans,
    pin_hillis_steele_trace,
    pin_blelloch,
    pin_brute_force,
    pin_closed_forms,
    pin_invariants,
    pin_f32,
    pin_segmented_golden,
    pin_segmented_shapes,
    pin_segmented_zipf,
    pin_segmented_reduce,
    pin_compaction_golden,
    pin_compaction_properties,
    pin_recurrence_golden,
    pin_recurrence_expansion,
    pin_recurrence_special_cases,
]
