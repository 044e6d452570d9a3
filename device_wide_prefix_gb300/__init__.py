"""device_wide_prefix_gb300: Python binding of libdwp.so (include/dwp.h).

The binding only marshals arguments: every step of every operation runs in
the library's CUDA kernels.  PyTorch supplies device memory and streams.
There is no CPU fallback: if libdwp.so is missing or cannot be loaded, every
call raises.

Two layers:
  * the C entry points under their C names (dwp_scan_exclusive, ...), taking
    integer device addresses and returning the integer dwp_status;
  * tensor helpers (scan_exclusive, scan_inclusive, ...) that size and
    allocate the scratch with torch, call the C entry point on the current
    stream of the tensors' device and raise DwpError on a non-zero status.
"""
from __future__ import annotations

import ctypes
import os

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "libdwp.so")

DWP_SUCCESS = 0
DWP_ERR_INVALID_VALUE = 1
DWP_ERR_MISALIGNED = 2
DWP_ERR_ALIASING = 3
DWP_ERR_SCRATCH_TOO_SMALL = 4
DWP_ERR_CUDA = 5
DWP_ERR_LOOKBACK_TIMEOUT = 6
DWP_ERR_PIPELINE_TIMEOUT = 7
DWP_ERR_NO_DEVICE = 8
DWP_ERR_BOUNDS = 9

DWP_U32_ADD = 0
DWP_F32_ADD = 1
DWP_U32_MAX = 2
OPS = {"u32_add": DWP_U32_ADD, "f32_add": DWP_F32_ADD, "u32_max": DWP_U32_MAX}

DWP_EXCLUSIVE = 0
DWP_INCLUSIVE = 1

# Names the C header declares (checked by the tests against include/dwp.h).
EXPORTS = [
    "dwp_scan_exclusive",
    "dwp_scan_inclusive",
    "dwp_segmented_scan_u32",
    "dwp_compact_by_flags",
    "dwp_linear_recurrence_f32",
    "dwp_segmented_reduce_u32",
    "dwp_read_status",
    "dwp_read_fallbacks",
    "dwp_status_string",
    "dwp_version",
    "dwp_debug_set_fault",
    "dwp_set_lookback_window",
    "dwp_scan_static_scratch",
    "dwp_read_static_status",
    "dwp_scan_two_level",
    "dwp_compact_by_flags_staged",
    "dwp_read_lookback_stats",
    "dwp_debug_set_delay",
    "dwp_debug_warp_scan_trace",
]

_lib = None


class DwpError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__("%s failed: %s" % (what, status_string(status)))


def load(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load libdwp.so and declare its entry points.  Raises if it is missing."""
    global _lib
    if _lib is not None and path == LIB_PATH:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(
            "libdwp.so is not built (%s); run `python -c \"import __graft_entry__ as g; g.build()\"`"
            % path)
    lib = ctypes.CDLL(path)
    c = ctypes
    P, S, Z = c.c_void_p, c.c_size_t, c.POINTER(c.c_size_t)
    for name in ("dwp_scan_exclusive", "dwp_scan_inclusive"):
        f = getattr(lib, name)
        f.argtypes = [c.c_int, P, P, S, P, Z, P]
        f.restype = c.c_int
    lib.dwp_segmented_scan_u32.argtypes = [P, P, S, P, S, c.c_int, P, Z, P]
    lib.dwp_segmented_scan_u32.restype = c.c_int
    for name in ("dwp_compact_by_flags", "dwp_compact_by_flags_staged"):
        getattr(lib, name).argtypes = [P, P, S, P, P, P, Z, P]
        getattr(lib, name).restype = c.c_int
    lib.dwp_linear_recurrence_f32.argtypes = [P, P, P, S, c.c_int, P, Z, P]
    lib.dwp_linear_recurrence_f32.restype = c.c_int
    lib.dwp_segmented_reduce_u32.argtypes = [P, P, S, P, S, P, Z, P]
    lib.dwp_segmented_reduce_u32.restype = c.c_int
    lib.dwp_read_status.argtypes = [P, P]
    lib.dwp_read_status.restype = c.c_int
    lib.dwp_read_fallbacks.argtypes = [P, P, c.POINTER(c.c_uint32)]
    lib.dwp_read_fallbacks.restype = c.c_int
    U = c.POINTER(c.c_uint32)
    lib.dwp_read_lookback_stats.argtypes = [P, P, U, U, U]
    lib.dwp_read_lookback_stats.restype = c.c_int
    lib.dwp_read_static_status.argtypes = [P]
    lib.dwp_read_static_status.restype = c.c_int
    lib.dwp_debug_set_delay.argtypes = [c.c_uint32, c.c_uint32, c.c_uint32]
    lib.dwp_debug_set_delay.restype = c.c_int
    lib.dwp_debug_warp_scan_trace.argtypes = [P, S, P, P]
    lib.dwp_debug_warp_scan_trace.restype = c.c_int
    lib.dwp_status_string.argtypes = [c.c_int]
    lib.dwp_status_string.restype = c.c_char_p
    lib.dwp_version.argtypes = []
    lib.dwp_version.restype = c.c_int
    lib.dwp_debug_set_fault.argtypes = [c.c_uint32, c.c_uint32, c.c_uint32]
    lib.dwp_debug_set_fault.restype = c.c_int
    lib.dwp_set_lookback_window.argtypes = [c.c_uint32]
    lib.dwp_set_lookback_window.restype = c.c_int
    lib.dwp_scan_static_scratch.argtypes = [c.c_int, c.c_int, P, P, S, P]
    lib.dwp_scan_static_scratch.restype = c.c_int
    lib.dwp_scan_two_level.argtypes = [c.c_int, c.c_int, P, P, S, P, Z, P]
    lib.dwp_scan_two_level.restype = c.c_int
    if path == LIB_PATH:
        _lib = lib
    return lib


# ---------------------------------------------------------------------------
# C entry points under their C names (integer addresses in, status out)


def _scan_entry(name, op, d_in, d_out, n, d_scratch, scratch_bytes, stream):
    sb = ctypes.c_size_t(scratch_bytes)
    st = getattr(load(), name)(int(op), d_in or None, d_out or None, n, d_scratch or None,
                               ctypes.byref(sb), stream or None)
    return st, sb.value


def dwp_scan_exclusive(op, d_in, d_out, n, d_scratch, scratch_bytes, stream):
    """dwp.h dwp_scan_exclusive; returns (status, scratch_bytes after the call)."""
    return _scan_entry("dwp_scan_exclusive", op, d_in, d_out, n, d_scratch, scratch_bytes, stream)


def dwp_scan_inclusive(op, d_in, d_out, n, d_scratch, scratch_bytes, stream):
    """dwp.h dwp_scan_inclusive; returns (status, scratch_bytes after the call)."""
    return _scan_entry("dwp_scan_inclusive", op, d_in, d_out, n, d_scratch, scratch_bytes, stream)


def dwp_scan_two_level(op, mode, d_in, d_out, n, d_scratch, scratch_bytes, stream):
    """dwp.h dwp_scan_two_level; returns (status, scratch_bytes after the call)."""
    sb = ctypes.c_size_t(scratch_bytes)
    st = load().dwp_scan_two_level(int(op), int(mode), d_in or None, d_out or None, n,
                                   d_scratch or None, ctypes.byref(sb), stream or None)
    return st, sb.value


def dwp_segmented_scan_u32(d_values, d_offsets, num_segments, d_out, n, mode, d_scratch,
                           scratch_bytes, stream):
    """dwp.h dwp_segmented_scan_u32; returns (status, scratch_bytes after the call)."""
    sb = ctypes.c_size_t(scratch_bytes)
    st = load().dwp_segmented_scan_u32(d_values or None, d_offsets or None, num_segments,
                                       d_out or None, n, int(mode), d_scratch or None,
                                       ctypes.byref(sb), stream or None)
    return st, sb.value


def dwp_segmented_reduce_u32(d_values, d_offsets, num_segments, d_out, n, d_scratch,
                             scratch_bytes, stream):
    """dwp.h dwp_segmented_reduce_u32; returns (status, scratch_bytes after the call)."""
    sb = ctypes.c_size_t(scratch_bytes)
    st = load().dwp_segmented_reduce_u32(d_values or None, d_offsets or None, num_segments,
                                         d_out or None, n, d_scratch or None, ctypes.byref(sb),
                                         stream or None)
    return st, sb.value


def dwp_linear_recurrence_f32(d_a, d_b, d_h, n, mode, d_scratch, scratch_bytes, stream):
    """dwp.h dwp_linear_recurrence_f32; returns (status, scratch_bytes after the call)."""
    sb = ctypes.c_size_t(scratch_bytes)
    st = load().dwp_linear_recurrence_f32(d_a or None, d_b or None, d_h or None, n, int(mode),
                                          d_scratch or None, ctypes.byref(sb), stream or None)
    return st, sb.value


def dwp_compact_by_flags(d_records, d_flags, n, d_out, d_count, d_scratch, scratch_bytes, stream):
    """dwp.h dwp_compact_by_flags; returns (status, scratch_bytes after the call)."""
    sb = ctypes.c_size_t(scratch_bytes)
    st = load().dwp_compact_by_flags(d_records or None, d_flags or None, n, d_out or None,
                                     d_count or None, d_scratch or None, ctypes.byref(sb),
                                     stream or None)
    return st, sb.value


def dwp_scan_static_scratch(op, mode, d_in, d_out, n, stream) -> int:
    """dwp.h dwp_scan_static_scratch: the scan with the library's built-in
    scratch, for callers that cannot allocate device memory; returns the status."""
    return load().dwp_scan_static_scratch(int(op), int(mode), d_in or None, d_out or None, n,
                                          stream or None)


def dwp_read_static_status(stream) -> int:
    """dwp.h dwp_read_static_status: device status of the last
    dwp_scan_static_scratch call on the current device (synchronises)."""
    return load().dwp_read_static_status(stream or None)


def dwp_compact_by_flags_staged(d_records, d_flags, n, d_out, d_count, d_scratch, scratch_bytes,
                                stream):
    """dwp.h dwp_compact_by_flags_staged; returns (status, scratch_bytes after the call)."""
    sb = ctypes.c_size_t(scratch_bytes)
    st = load().dwp_compact_by_flags_staged(d_records or None, d_flags or None, n, d_out or None,
                                            d_count or None, d_scratch or None, ctypes.byref(sb),
                                            stream or None)
    return st, sb.value


def dwp_read_status(d_scratch, stream) -> int:
    return load().dwp_read_status(d_scratch or None, stream or None)


def dwp_read_lookback_stats(d_scratch, stream):
    """(status, fallbacks, intermediates, jumps) of the last call on d_scratch."""
    a, b, c_ = ctypes.c_uint32(0), ctypes.c_uint32(0), ctypes.c_uint32(0)
    st = load().dwp_read_lookback_stats(d_scratch or None, stream or None, ctypes.byref(a),
                                        ctypes.byref(b), ctypes.byref(c_))
    return st, a.value, b.value, c_.value


def dwp_debug_warp_scan_trace(d_x, width, d_steps, stream) -> int:
    """dwp.h dwp_debug_warp_scan_trace (test hook): the warp Hillis-Steele
    scan's value per lane after each of its five steps."""
    return load().dwp_debug_warp_scan_trace(d_x or None, width, d_steps or None, stream or None)


def dwp_debug_set_delay(seed: int, fraction_ppm: int, max_ns: int) -> int:
    """dwp.h dwp_debug_set_delay (test hook): seeded sleeps at publication points."""
    return load().dwp_debug_set_delay(seed & 0xFFFFFFFF, fraction_ppm, max_ns)


def dwp_read_fallbacks(d_scratch, stream):
    """(status, count of Decoupled Fallbacks the last call on d_scratch made)."""
    v = ctypes.c_uint32(0)
    st = load().dwp_read_fallbacks(d_scratch or None, stream or None, ctypes.byref(v))
    return st, v.value


def dwp_status_string(status: int) -> str:
    return load().dwp_status_string(int(status)).decode()


def dwp_version() -> int:
    return load().dwp_version()


def dwp_debug_set_fault(never_publish_tile: int, spin_limit: int, fallback_polls: int = 0) -> int:
    return load().dwp_debug_set_fault(never_publish_tile & 0xFFFFFFFF, spin_limit,
                                      fallback_polls & 0xFFFFFFFF)


def dwp_set_lookback_window(tiles: int) -> int:
    """dwp.h dwp_set_lookback_window: 0 unbounded (default), else the window in tiles."""
    return load().dwp_set_lookback_window(int(tiles) & 0xFFFFFFFF)


def status_string(status: int) -> str:
    try:
        return dwp_status_string(status)
    except Exception:  # library not loadable: still give a readable message
        return "status %d" % status


def _check(st: int, what: str) -> None:
    if st != DWP_SUCCESS:
        raise DwpError(st, what)


# ---------------------------------------------------------------------------
# tensor helpers (torch is the memory and stream provider only)


def _torch():
    import torch
    return torch


def _stream_of(t, stream=None) -> int:
    torch = _torch()
    if stream is None:
        stream = torch.cuda.current_stream(t.device)
    return int(stream.cuda_stream)


def _scan_dtype(op: str):
    torch = _torch()
    return torch.float32 if op == "f32_add" else torch.int32


def scan_scratch_bytes(n: int, op: str = "u32_add") -> int:
    st, b = dwp_scan_exclusive(OPS[op], None, None, n, None, 0, None)
    _check(st, "scratch size query")
    return b


def alloc_scratch(nbytes: int, device):
    """A scratch buffer from torch's caching allocator (16-byte aligned)."""
    torch = _torch()
    return torch.empty(max(int(nbytes), 16), dtype=torch.uint8, device=device)


def _scan(inclusive: bool, x, op: str, out=None, scratch=None, stream=None):
    torch = _torch()
    if op not in OPS:
        raise ValueError("unknown op %r" % op)
    if not x.is_cuda or not x.is_contiguous() or x.element_size() != 4:
        raise ValueError("x must be a contiguous CUDA tensor of 4-byte elements")
    n = x.numel()
    if out is None:
        out = torch.empty_like(x)
    need = scan_scratch_bytes(n, op)
    if scratch is None:
        scratch = alloc_scratch(need, x.device)
    entry = dwp_scan_inclusive if inclusive else dwp_scan_exclusive
    with torch.cuda.device(x.device):
        st, _ = entry(OPS[op], x.data_ptr(), out.data_ptr(), n, scratch.data_ptr(),
                      scratch.numel(), _stream_of(x, stream))
    _check(st, "dwp_scan_inclusive" if inclusive else "dwp_scan_exclusive")
    return out


def scan_exclusive(x, op: str = "u32_add", out=None, scratch=None, stream=None):
    """Exclusive scan of a contiguous CUDA tensor (int32/uint32 bits or float32)."""
    return _scan(False, x, op, out, scratch, stream)


def scan_inclusive(x, op: str = "u32_add", out=None, scratch=None, stream=None):
    """Inclusive scan of a contiguous CUDA tensor (int32/uint32 bits or float32)."""
    return _scan(True, x, op, out, scratch, stream)


def two_level_scratch_bytes(n: int) -> int:
    st, b = dwp_scan_two_level(DWP_U32_ADD, DWP_EXCLUSIVE, None, None, n, None, 0, None)
    _check(st, "two-level scan scratch size query")
    return b


def scan_two_level(x, op: str = "u32_add", inclusive: bool = False, out=None, scratch=None,
                   stream=None):
    """The plain scan by the two-level, three-launch form (n <= 2^26)."""
    torch = _torch()
    if op not in OPS:
        raise ValueError("unknown op %r" % op)
    if not x.is_cuda or not x.is_contiguous() or x.element_size() != 4:
        raise ValueError("x must be a contiguous CUDA tensor of 4-byte elements")
    n = x.numel()
    if out is None:
        out = torch.empty_like(x)
    if scratch is None:
        scratch = alloc_scratch(two_level_scratch_bytes(n), x.device)
    with torch.cuda.device(x.device):
        st, _ = dwp_scan_two_level(OPS[op], DWP_INCLUSIVE if inclusive else DWP_EXCLUSIVE,
                                   x.data_ptr(), out.data_ptr(), n, scratch.data_ptr(),
                                   scratch.numel(), _stream_of(x, stream))
    _check(st, "dwp_scan_two_level")
    return out


def segmented_scan_scratch_bytes(n: int) -> int:
    st, b = dwp_segmented_scan_u32(None, None, 0, None, n, DWP_EXCLUSIVE, None, 0, None)
    _check(st, "segmented scan scratch size query")
    return b


def segmented_scan(values, offsets, inclusive: bool = False, out=None, scratch=None,
                   stream=None):
    """Segmented u32 scan of `values` (CUDA int32/uint32 bits) over CSR `offsets`
    (CUDA, N+1 entries).  Rows outside [offsets[0], offsets[N]) keep the
    contents of `out` (uninitialised when `out` is None)."""
    torch = _torch()
    if not (values.is_cuda and offsets.is_cuda and values.is_contiguous() and offsets.is_contiguous()):
        raise ValueError("values and offsets must be contiguous CUDA tensors")
    if values.element_size() != 4 or offsets.element_size() != 4:
        raise ValueError("values and offsets must have 4-byte elements")
    n = values.numel()
    nseg = max(offsets.numel() - 1, 0)
    if out is None:
        out = torch.empty_like(values)
    need = segmented_scan_scratch_bytes(n)
    if scratch is None:
        scratch = alloc_scratch(need, values.device)
    with torch.cuda.device(values.device):
        st, _ = dwp_segmented_scan_u32(values.data_ptr(), offsets.data_ptr() if offsets.numel() else 0,
                                       nseg, out.data_ptr(), n,
                                       DWP_INCLUSIVE if inclusive else DWP_EXCLUSIVE,
                                       scratch.data_ptr(), scratch.numel(), _stream_of(values, stream))
    _check(st, "dwp_segmented_scan_u32")
    return out


def segmented_reduce_scratch_bytes(n: int) -> int:
    st, b = dwp_segmented_reduce_u32(None, None, 0, None, n, None, 0, None)
    _check(st, "segmented reduction scratch size query")
    return b


def segmented_reduce(values, offsets, out=None, scratch=None, stream=None):
    """One wrapping u32 sum per segment of CSR `offsets` (CUDA, N+1 entries)
    over `values` (CUDA int32/uint32 bits); 0 for an empty segment.  Returns
    `out` (N int32 entries, the u32 bits)."""
    torch = _torch()
    if not (values.is_cuda and offsets.is_cuda and values.is_contiguous() and offsets.is_contiguous()):
        raise ValueError("values and offsets must be contiguous CUDA tensors")
    if values.element_size() != 4 or offsets.element_size() != 4:
        raise ValueError("values and offsets must have 4-byte elements")
    n = values.numel()
    nseg = max(offsets.numel() - 1, 0)
    if out is None:
        out = torch.empty(nseg, dtype=torch.int32, device=values.device)
    need = segmented_reduce_scratch_bytes(n)
    if scratch is None:
        scratch = alloc_scratch(need, values.device)
    with torch.cuda.device(values.device):
        st, _ = dwp_segmented_reduce_u32(values.data_ptr() if n else 0,
                                         offsets.data_ptr() if offsets.numel() else 0, nseg,
                                         out.data_ptr() if nseg else 0, n, scratch.data_ptr(),
                                         scratch.numel(), _stream_of(values, stream))
    _check(st, "dwp_segmented_reduce_u32")
    return out


def linear_recurrence_scratch_bytes(n: int) -> int:
    st, b = dwp_linear_recurrence_f32(None, None, None, n, DWP_INCLUSIVE, None, 0, None)
    _check(st, "linear recurrence scratch size query")
    return b


def linear_recurrence(a, b, inclusive: bool = True, out=None, scratch=None, stream=None):
    """h[t] = a[t] h[t-1] + b[t] from h[-1] = 0 over contiguous CUDA float32
    tensors `a` and `b` of equal length.  Inclusive returns h; exclusive the
    state before each step.  `out` may be `a` or `b` itself (in place)."""
    torch = _torch()
    if not (a.is_cuda and b.is_cuda and a.is_contiguous() and b.is_contiguous()):
        raise ValueError("a and b must be contiguous CUDA tensors")
    if a.dtype != torch.float32 or b.dtype != torch.float32 or a.numel() != b.numel():
        raise ValueError("a and b must be float32 tensors of the same length")
    n = a.numel()
    if out is None:
        out = torch.empty_like(b)
    need = linear_recurrence_scratch_bytes(n)
    if scratch is None:
        scratch = alloc_scratch(need, a.device)
    with torch.cuda.device(a.device):
        st, _ = dwp_linear_recurrence_f32(a.data_ptr(), b.data_ptr(), out.data_ptr(), n,
                                          DWP_INCLUSIVE if inclusive else DWP_EXCLUSIVE,
                                          scratch.data_ptr(), scratch.numel(), _stream_of(a, stream))
    _check(st, "dwp_linear_recurrence_f32")
    return out


def compact_scratch_bytes(n: int) -> int:
    st, b = dwp_compact_by_flags(None, None, n, None, None, None, 0, None)
    _check(st, "compaction scratch size query")
    return b


def compact_by_flags(records, flags, out=None, count=None, scratch=None, stream=None):
    """Stable compaction of `records` (CUDA tensor, 16 bytes per row, e.g.
    shape (n, 4) int32) by `flags` (CUDA uint8, n).  Returns (out, count) with
    count a 1-element CUDA int32 tensor; rows of `out` past the count are
    untouched."""
    torch = _torch()
    n = flags.numel()
    if not (records.is_cuda and flags.is_cuda and records.is_contiguous() and flags.is_contiguous()):
        raise ValueError("records and flags must be contiguous CUDA tensors")
    if records.numel() * records.element_size() != 16 * n or flags.element_size() != 1:
        raise ValueError("records must hold 16 bytes per flag byte")
    if out is None:
        out = torch.empty_like(records)
    if count is None:
        count = torch.empty(1, dtype=torch.int32, device=records.device)
    need = compact_scratch_bytes(n)
    if scratch is None:
        scratch = alloc_scratch(need, records.device)
    with torch.cuda.device(records.device):
        st, _ = dwp_compact_by_flags(records.data_ptr(), flags.data_ptr(), n, out.data_ptr(),
                                     count.data_ptr(), scratch.data_ptr(), scratch.numel(),
                                     _stream_of(records, stream))
    _check(st, "dwp_compact_by_flags")
    return out, count


def compact_staged_scratch_bytes(n: int) -> int:
    st, b = dwp_compact_by_flags_staged(None, None, n, None, None, None, 0, None)
    _check(st, "staged compaction scratch size query")
    return b


def compact_by_flags_staged(records, flags, out=None, count=None, scratch=None, stream=None):
    """compact_by_flags by the staged three-launch form (flags and offsets
    written to scratch): the comparison point for the fused kernel."""
    torch = _torch()
    n = flags.numel()
    if not (records.is_cuda and flags.is_cuda and records.is_contiguous() and flags.is_contiguous()):
        raise ValueError("records and flags must be contiguous CUDA tensors")
    if records.numel() * records.element_size() != 16 * n or flags.element_size() != 1:
        raise ValueError("records must hold 16 bytes per flag byte")
    if out is None:
        out = torch.empty_like(records)
    if count is None:
        count = torch.empty(1, dtype=torch.int32, device=records.device)
    if scratch is None:
        scratch = alloc_scratch(compact_staged_scratch_bytes(n), records.device)
    with torch.cuda.device(records.device):
        st, _ = dwp_compact_by_flags_staged(records.data_ptr(), flags.data_ptr(), n, out.data_ptr(),
                                            count.data_ptr(), scratch.data_ptr(), scratch.numel(),
                                            _stream_of(records, stream))
    _check(st, "dwp_compact_by_flags_staged")
    return out, count


def read_lookback_stats(scratch, stream=None) -> dict:
    """Fallbacks, intermediates published and jumps over them in the last
    call that used `scratch` (synchronises)."""
    st, fb, im, jp = dwp_read_lookback_stats(scratch.data_ptr(), _stream_of(scratch, stream))
    _check(st, "dwp_read_lookback_stats")
    return {"fallbacks": fb, "intermediates": im, "jumps": jp}


def read_status(scratch, stream=None) -> int:
    """Device-side status of the last call that used `scratch` (synchronises)."""
    return dwp_read_status(scratch.data_ptr(), _stream_of(scratch, stream))


def read_fallbacks(scratch, stream=None) -> int:
    """Tiles whose aggregate a waiting successor computed itself (Decoupled
    Fallback) in the last call that used `scratch` (synchronises)."""
    st, v = dwp_read_fallbacks(scratch.data_ptr(), _stream_of(scratch, stream))
    _check(st, "dwp_read_fallbacks")
    return v
