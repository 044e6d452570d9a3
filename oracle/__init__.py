"""Sequential CPU oracle (ctypes binding of oracle.c).

TEST INFRASTRUCTURE ONLY.  Only tests/, __graft_entry__.smoke() and the CPU
baseline leg of bench.py may import this package.  The product path (the
CUDA library and its Python binding) never imports, links or runs it, and it
shares no code with the product path: the only code both sides use is the
seeded input generator in synth.py, which holds no scan arithmetic.

Each wrapper below calls the plain sequential definition in oracle.c; see
that file for the passages each function follows.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lib = None

_u32p = np.ctypeslib.ndpointer(dtype=np.uint32, flags="C_CONTIGUOUS")
_f32p = np.ctypeslib.ndpointer(dtype=np.float32, flags="C_CONTIGUOUS")
_f64p = np.ctypeslib.ndpointer(dtype=np.float64, flags="C_CONTIGUOUS")
_u8p = np.ctypeslib.ndpointer(dtype=np.uint8, flags="C_CONTIGUOUS")


def build(src: str = _SRC, out: str = _LIB, force: bool = False) -> str:
    """Compile oracle.c into a shared library (plain C11, -O2, no fast-math)."""
    if force or not os.path.exists(out) or os.path.getmtime(out) < os.path.getmtime(src):
        tmp = out + ".tmp%d" % os.getpid()
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared",
                               "-fno-fast-math", "-o", tmp, src])
        os.replace(tmp, out)
    return out


def load(path: str | None = None) -> ctypes.CDLL:
    """Load (building first if needed) and declare the oracle's functions."""
    global _lib
    if path is None and _lib is not None:
        return _lib
    lib = ctypes.CDLL(path or build())
    c = ctypes
    lib.oracle_scan_u32_add.argtypes = [_u32p, c.c_uint64, c.c_int, _u32p]
    lib.oracle_scan_u32_add.restype = None
    lib.oracle_scan_u32_max.argtypes = [_u32p, c.c_uint64, c.c_int, _u32p]
    lib.oracle_scan_u32_max.restype = None
    lib.oracle_scan_f32_add.argtypes = [_f32p, c.c_uint64, c.c_int, _f64p, _f64p]
    lib.oracle_scan_f32_add.restype = None
    lib.oracle_segmented_scan_u32.argtypes = [_u32p, _u32p, c.c_uint64, c.c_uint64,
                                              c.c_int, _u32p]
    lib.oracle_segmented_scan_u32.restype = None
    lib.oracle_compact.argtypes = [c.c_void_p, _u8p, c.c_uint64, c.c_uint64, c.c_void_p]
    lib.oracle_compact.restype = c.c_uint64
    lib.oracle_linear_recurrence_f32.argtypes = [_f32p, _f32p, c.c_uint64, c.c_int, _f64p, _f64p]
    lib.oracle_linear_recurrence_f32.restype = None
    lib.oracle_segmented_reduce_u32.argtypes = [_u32p, _u32p, c.c_uint64, c.c_uint64, _u32p]
    lib.oracle_segmented_reduce_u32.restype = None
    if path is None:
        _lib = lib
    return lib


class Oracle:
    """Thin numpy front end over one loaded copy of the oracle library."""

    def __init__(self, lib: ctypes.CDLL | None = None):
        self.lib = lib if lib is not None else load()

    def scan_u32_add(self, x: np.ndarray, inclusive: bool) -> np.ndarray:
        x = np.ascontiguousarray(x, dtype=np.uint32)
        y = np.empty_like(x)
        self.lib.oracle_scan_u32_add(x, x.size, int(inclusive), y)
        return y

    def scan_u32_max(self, x: np.ndarray, inclusive: bool) -> np.ndarray:
        x = np.ascontiguousarray(x, dtype=np.uint32)
        y = np.empty_like(x)
        self.lib.oracle_scan_u32_max(x, x.size, int(inclusive), y)
        return y

    def scan_f32_add(self, x: np.ndarray, inclusive: bool):
        """Returns (double prefix, double prefix of |x|) over the same ranges."""
        x = np.ascontiguousarray(x, dtype=np.float32)
        y = np.empty(x.size, dtype=np.float64)
        a = np.empty(x.size, dtype=np.float64)
        self.lib.oracle_scan_f32_add(x, x.size, int(inclusive), y, a)
        return y, a

    def scan(self, op: str, x: np.ndarray, inclusive: bool):
        if op == "u32_add":
            return self.scan_u32_add(x, inclusive)
        if op == "u32_max":
            return self.scan_u32_max(x, inclusive)
        if op == "f32_add":
            return self.scan_f32_add(x, inclusive)
        raise ValueError(op)

    def segmented_scan_u32(self, values: np.ndarray, offsets: np.ndarray, inclusive: bool,
                           out: np.ndarray | None = None) -> np.ndarray:
        """Rows outside every segment keep the contents of `out` (zeros if None)."""
        values = np.ascontiguousarray(values, dtype=np.uint32)
        offsets = np.ascontiguousarray(offsets, dtype=np.uint32)
        out = np.zeros_like(values) if out is None else np.array(out, dtype=np.uint32, copy=True)
        nseg = max(offsets.size - 1, 0)
        if nseg:
            self.lib.oracle_segmented_scan_u32(values, offsets, nseg, values.size,
                                               int(inclusive), out)
        return out

    def segmented_reduce_u32(self, values: np.ndarray, offsets: np.ndarray) -> np.ndarray:
        """One wrapping u32 sum per segment of the CSR offsets (0 if empty)."""
        values = np.ascontiguousarray(values, dtype=np.uint32)
        offsets = np.ascontiguousarray(offsets, dtype=np.uint32)
        nseg = max(offsets.size - 1, 0)
        out = np.empty(nseg, dtype=np.uint32)
        if nseg:
            self.lib.oracle_segmented_reduce_u32(values, offsets, nseg, values.size, out)
        return out

    def linear_recurrence(self, a: np.ndarray, b: np.ndarray, inclusive: bool):
        """h[t] = a[t] h[t-1] + b[t] from h[-1] = 0.  Returns (double h, or the
        state before each step if exclusive; double magnitude recurrence
        g[t] = |a[t]| g[t-1] + |b[t]| over the same range)."""
        a = np.ascontiguousarray(a, dtype=np.float32)
        b = np.ascontiguousarray(b, dtype=np.float32)
        assert a.size == b.size
        y = np.empty(a.size, dtype=np.float64)
        g = np.empty(a.size, dtype=np.float64)
        self.lib.oracle_linear_recurrence_f32(a, b, a.size, int(inclusive), y, g)
        return y, g

    def compact(self, records: np.ndarray, flags: np.ndarray):
        """records: (n, w) array of any dtype, one row per record.  Returns (out, count)
        with out the same shape as records, rows past count zero."""
        records = np.ascontiguousarray(records)
        flags = np.ascontiguousarray(flags, dtype=np.uint8)
        n = records.shape[0]
        assert flags.size == n
        rb = records.itemsize * (records.size // max(n, 1)) if n else 0
        out = np.zeros_like(records)
        k = self.lib.oracle_compact(records.ctypes.data_as(ctypes.c_void_p), flags, n, rb,
                                    out.ctypes.data_as(ctypes.c_void_p))
        return out, int(k)


_default: Oracle | None = None


def default() -> Oracle:
    global _default
    if _default is None:
        _default = Oracle()
    return _default
