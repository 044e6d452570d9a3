"""bench.py's selective-read bound for compaction, on the CPU: the bytes of
the unit-sized pieces of the record array (16-byte records) that hold at
least one kept record, checked against brute force and closed forms."""
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def brute(flags, unit):
    per = unit // 16
    return sum(unit for i in range(0, len(flags), per) if any(flags[i:i + per]))


def test_matches_brute_force():
    rng = np.random.default_rng(5)
    for n in (1, 2, 3, 7, 8, 9, 100, 1001):
        flags = (rng.random(n) < 0.3).astype(np.uint8)
        for unit in (32, 64, 128):
            assert bench.kept_sector_bytes(flags, unit) == brute(flags, unit), (n, unit)


def test_closed_forms():
    n = 4096
    assert bench.kept_sector_bytes(np.zeros(n, np.uint8), 32) == 0
    assert bench.kept_sector_bytes(np.ones(n, np.uint8), 32) == 16 * n
    assert bench.kept_sector_bytes(np.ones(n, np.uint8), 128) == 16 * n
    every_8th = (np.arange(n) % 8 == 0).astype(np.uint8)
    assert bench.kept_sector_bytes(every_8th, 32) == n // 8 * 32
    assert bench.kept_sector_bytes(every_8th, 128) == 16 * n  # one per 128-byte piece


def test_expected_fraction_at_p_03():
    # a piece of m records holds a kept one with probability 1 - 0.7^m
    flags = (np.random.default_rng(6).random(1 << 20) < 0.3).astype(np.uint8)
    for unit, m in ((32, 2), (128, 8)):
        frac = bench.kept_sector_bytes(flags, unit) / (16 * flags.size)
        assert abs(frac - (1 - 0.7 ** m)) < 0.005, unit
