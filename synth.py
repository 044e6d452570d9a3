"""Seeded synthetic inputs shared by the tests, the oracle checks and bench.py.

This module holds random-number generation and workload shapes only: no scan,
no look-back, no compaction arithmetic.  Every array is a pure function of
(seed, index) through the counter-based SplitMix64 generator, so the same
inputs come out on x86 and on Arm, in any chunking.

SplitMix64 (Steele, Lea and Flood, "Fast splittable pseudorandom number
generators", OOPSLA 2014): the i-th output of stream `seed` is
mix(seed + (i + 1) * 0x9E3779B97F4A7C15) with the published mix
z ^= z >> 30; z *= 0xBF58476D1CE4E5B9; z ^= z >> 27; z *= 0x94D049BB133111EB;
z ^= z >> 31.

Workloads (one seed per workload):
  u32 small      n=2^20, x = u & 15                      seed 0xD3B00001
  u32 full       n=2^28, x = u >> 32                     seed 0xD3B00002
  f32            n=2^28, x = (u >> 40) * 2^-23 - 1       seed 0xD3B00003
  records        n=2^26, id=i, 3 x N(0,1) (Box-Muller),  seed 0xD3B00004
                 keep flag = (u < 0.3 * 2^64)
  segmented      n=2^27, x = u & 255, segment lengths     seed 0xD3B00005
                 empty with p=0.05 else Zipf(1.2) clamped to 2^22
  recurrence     n=2^28, a = 0.5 + (u >> 41) * 2^-24      seed 0xD3B00006
                 (uniform in [0.5, 1)), b as f32 above     seed 0xD3B00007
"""
from __future__ import annotations

import functools
import math

import numpy as np

GAMMA = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)

SEED_U32_SMALL = 0xD3B00001
SEED_U32_FULL = 0xD3B00002
SEED_F32 = 0xD3B00003
SEED_RECORDS = 0xD3B00004
SEED_SEGMENTED = 0xD3B00005
SEED_RECURRENCE_A = 0xD3B00006
SEED_RECURRENCE_B = 0xD3B00007

_CHUNK = 1 << 22


def _mix(z: np.ndarray, t: np.ndarray) -> np.ndarray:
    """SplitMix64 output function, in place on a uint64 array (t: same-size scratch)."""
    np.bitwise_xor(z, np.right_shift(z, np.uint64(30), out=t), out=z)
    np.multiply(z, _M1, out=z)
    np.bitwise_xor(z, np.right_shift(z, np.uint64(27), out=t), out=z)
    np.multiply(z, _M2, out=z)
    np.bitwise_xor(z, np.right_shift(z, np.uint64(31), out=t), out=z)
    return z


@functools.lru_cache(maxsize=1)
def _iota() -> np.ndarray:
    return np.arange(1, _CHUNK + 1, dtype=np.int64).view(np.uint64)


def mix64(v: int) -> int:
    """Scalar SplitMix64 output function (used to derive sub-stream seeds)."""
    with np.errstate(over="ignore"):
        z = np.array([v & (2**64 - 1)], dtype=np.uint64)
        return int(_mix(z, np.empty_like(z))[0])


def substream(seed: int, k: int) -> int:
    """Seed of the k-th independent sub-stream of `seed`."""
    return mix64((seed + k * 0x632BE59BD9B4E019) & (2**64 - 1))


def u64(seed: int, start: int, count: int, out: np.ndarray | None = None) -> np.ndarray:
    """Outputs start .. start+count-1 of SplitMix64 stream `seed` (uint64)."""
    if out is None:
        out = np.empty(count, dtype=np.uint64)
    iota = _iota()
    z = np.empty(min(count, _CHUNK), dtype=np.uint64)
    t = np.empty_like(z)
    with np.errstate(over="ignore"):
        for c0 in range(0, count, _CHUNK):
            m = min(count, c0 + _CHUNK) - c0
            # state = seed + (start + c0 + j + 1) * gamma, j = 0 .. m-1
            base = np.uint64((seed + (start + c0) * 0x9E3779B97F4A7C15) & (2**64 - 1))
            np.multiply(iota[:m], GAMMA, out=z[:m])
            np.add(z[:m], base, out=z[:m])
            out[c0:c0 + m] = _mix(z[:m], t[:m])
    return out


def _u32_from(seed: int, n: int, fn) -> np.ndarray:
    out = np.empty(n, dtype=np.uint32)
    for c0 in range(0, n, _CHUNK):
        c1 = min(n, c0 + _CHUNK)
        out[c0:c1] = fn(u64(seed, c0, c1 - c0))
    return out


def u32_small_values(n: int, seed: int = SEED_U32_SMALL) -> np.ndarray:
    """Integers uniform in [0, 15]: the low 4 bits of each draw."""
    return _u32_from(seed, n, lambda u: (u & np.uint64(15)).astype(np.uint32))


def u32_full_values(n: int, seed: int = SEED_U32_FULL) -> np.ndarray:
    """Integers uniform in [0, 2^32): the high 32 bits of each draw."""
    return _u32_from(seed, n, lambda u: (u >> np.uint64(32)).astype(np.uint32))


def u32_byte_values(n: int, seed: int = SEED_SEGMENTED) -> np.ndarray:
    """Integers uniform in [0, 255]: the low 8 bits of each draw."""
    return _u32_from(seed, n, lambda u: (u & np.uint64(255)).astype(np.uint32))


def f32_values(n: int, seed: int = SEED_F32) -> np.ndarray:
    """Floats uniform on the 2^-23 grid of [-1, 1): exactly representable in f32."""
    out = np.empty(n, dtype=np.float32)
    for c0 in range(0, n, _CHUNK):
        c1 = min(n, c0 + _CHUNK)
        k = (u64(seed, c0, c1 - c0) >> np.uint64(40)).astype(np.float64)
        out[c0:c1] = (k * 2.0**-23 - 1.0).astype(np.float32)
    return out


def decay_values(n: int, seed: int = SEED_RECURRENCE_A, lo: float = 0.5) -> np.ndarray:
    """Floats uniform on the 2^-24 grid of [lo, lo + 0.5) (lo = 0.5: [0.5, 1)),
    exactly representable in f32 for lo in {-1, -0.5, 0.5}."""
    out = np.empty(n, dtype=np.float32)
    for c0 in range(0, n, _CHUNK):
        c1 = min(n, c0 + _CHUNK)
        k = (u64(seed, c0, c1 - c0) >> np.uint64(41)).astype(np.float64)
        out[c0:c1] = (lo + k * 2.0**-24).astype(np.float32)
    return out


def keep_flags(n: int, p: float = 0.3, seed: int = SEED_RECORDS) -> np.ndarray:
    """u8 keep flags, 1 with probability p: (u < p * 2^64)."""
    thr = np.uint64(min(int(p * 2.0**64), 2**64 - 1))
    s = substream(seed, 1)
    out = np.empty(n, dtype=np.uint8)
    for c0 in range(0, n, _CHUNK):
        c1 = min(n, c0 + _CHUNK)
        out[c0:c1] = (u64(s, c0, c1 - c0) < thr).astype(np.uint8)
    return out


def flags_pattern(n: int, kind: str, seed: int = SEED_RECORDS) -> np.ndarray:
    """Predicate shapes: 'none', 'all', 'random' (p=0.3), 'clustered' (runs)."""
    if kind == "none":
        return np.zeros(n, dtype=np.uint8)
    if kind == "all":
        return np.ones(n, dtype=np.uint8)
    if kind == "random":
        return keep_flags(n, 0.3, seed)
    if kind == "clustered":
        # runs of kept / dropped rows whose lengths are drawn from [1, 4096]
        u = u64(substream(seed, 7), 0, max(1, n // 64 + 2))
        out = np.zeros(n, dtype=np.uint8)
        pos, k, keep = 0, 0, 1
        while pos < n:
            run = int(u[k % len(u)] % np.uint64(4096)) + 1
            out[pos:pos + run] = keep
            pos += run
            k += 1
            keep ^= 1
        return out
    raise ValueError(kind)


def _unit_open(u: np.ndarray) -> np.ndarray:
    """(0, 1] doubles from the top 53 bits."""
    return ((u >> np.uint64(11)).astype(np.float64) + 1.0) * 2.0**-53


def records(n: int, seed: int = SEED_RECORDS) -> np.ndarray:
    """n 16-byte records {u32 id = index; f32 a, b, c ~ N(0, 1)} as a (n, 4) uint32 view.

    Normals come from the Box-Muller transform of pairs of uniforms of a
    sub-stream: record i uses pairs 2i and 2i+1 (four normals, three kept).
    """
    rec = np.empty((n, 4), dtype=np.uint32)
    rec[:, 0] = np.arange(n, dtype=np.uint32)
    s = substream(seed, 2)
    chunk = _CHUNK // 4
    for c0 in range(0, n, chunk):
        c1 = min(n, c0 + chunk)
        m = c1 - c0
        u = u64(s, 4 * c0, 4 * m).reshape(m, 4)
        r0 = np.sqrt(-2.0 * np.log(_unit_open(u[:, 0])))
        r1 = np.sqrt(-2.0 * np.log(_unit_open(u[:, 2])))
        t0 = 2.0 * math.pi * _unit_open(u[:, 1])
        t1 = 2.0 * math.pi * _unit_open(u[:, 3])
        f = np.empty((m, 3), dtype=np.float32)
        f[:, 0] = r0 * np.cos(t0)
        f[:, 1] = r0 * np.sin(t0)
        f[:, 2] = r1 * np.cos(t1)
        rec[c0:c1, 1:] = f.view(np.uint32)
    return rec


def _zeta(s: float, m: int = 1 << 16) -> float:
    """Riemann zeta(s), s > 1: direct sum to m-1 plus the Euler-Maclaurin tail."""
    k = np.arange(1, m, dtype=np.float64)
    head = float(np.sum(k ** -s))
    mm = float(m)
    tail = mm ** (1 - s) / (s - 1) + 0.5 * mm ** -s + s * mm ** (-s - 1) / 12.0 \
        - s * (s + 1) * (s + 2) * mm ** (-s - 3) / 720.0
    return head + tail


@functools.lru_cache(maxsize=4)
def _zipf_cdf(alpha: float, cap: int) -> np.ndarray:
    """P(L <= k) for k = 1 .. cap-1."""
    k = np.arange(1, cap, dtype=np.float64)
    return np.cumsum(k ** -alpha) / _zeta(alpha)


def zipf_lengths(count: int, alpha: float, cap: int, seed: int, start: int = 0) -> np.ndarray:
    """Draws start .. start+count-1 of min(L, cap), L ~ Zipf(alpha) on {1, 2, ...},
    by inverse CDF of one uniform per draw."""
    u = (u64(seed, start, count) >> np.uint64(11)).astype(np.float64) * 2.0**-53
    idx = np.searchsorted(_zipf_cdf(alpha, cap), u, side="right")
    return np.minimum(idx + 1, cap).astype(np.int64)


def segment_offsets(n: int, seed: int = SEED_SEGMENTED, alpha: float = 1.2,
                    cap: int = 1 << 22, p_empty: float = 0.05) -> np.ndarray:
    """CSR offsets (u32, N+1 entries, offsets[0]=0, offsets[N]=n).

    Segment s is empty with probability p_empty, else its length is
    Zipf(alpha) clamped to `cap`; segments are drawn until they cover n
    rows and the last one is trimmed so the lengths sum to n.
    """
    lens: list[int] = []
    total, batch, drawn = 0, 4096, 0
    se, sz = substream(seed, 3), substream(seed, 4)
    thr = np.uint64(int(p_empty * 2.0**64))
    while total < n:
        ue = u64(se, drawn, batch)
        lz = zipf_lengths(batch, alpha, cap, sz, drawn)
        for i in range(batch):
            ln = 0 if ue[i] < thr else int(lz[i])
            if total + ln >= n:
                lens.append(n - total)
                total = n
                break
            lens.append(ln)
            total += ln
        drawn += batch
    if n == 0:
        lens = []
    off = np.zeros(len(lens) + 1, dtype=np.uint32)
    off[1:] = np.cumsum(np.asarray(lens, dtype=np.int64)).astype(np.uint32)
    return off

