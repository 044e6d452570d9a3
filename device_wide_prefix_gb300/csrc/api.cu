// C entry points: argument validation, the scratch size query, the scratch
// clear and the launch.  Validation happens before any CUDA call, so an
// argument error never enqueues work.  The scratch is cleared by a small
// kernel of the library rather than cudaMemsetAsync, so that the kernel
// after it can be launched programmatically (launch_pdl) and overlap its
// launch with the clear.
#include <cuda_runtime.h>

#include <cstddef>
#include <cstdint>

#include "launch.h"

namespace {

using namespace dwp;

constexpr uint64_t kMaxN = 0xffffffffull;  // n < 2^32

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Do [a, a+an) and [b, b+bn) share a byte?
bool overlap(const void *a, uint64_t an, const void *b, uint64_t bn) {
    if (!a || !b || an == 0 || bn == 0) return false;
    const uintptr_t pa = reinterpret_cast<uintptr_t>(a), pb = reinterpret_cast<uintptr_t>(b);
    return pa < pb + bn && pb < pa + an;
}

uint64_t ceil_div(uint64_t a, uint64_t b) { return (a + b - 1) / b; }

dwp_status scan_common(bool inclusive, dwp_op op, const void *in, void *out, size_t n,
                       void *scratch, size_t *scratch_bytes, dwp_stream stream) {
    if (!scratch_bytes) return DWP_ERR_INVALID_VALUE;
    const int iop = static_cast<int>(op);
    if (iop != DWP_U32_ADD && iop != DWP_F32_ADD && iop != DWP_U32_MAX) return DWP_ERR_INVALID_VALUE;
    if (uint64_t(n) > kMaxN) return DWP_ERR_INVALID_VALUE;
    const size_t need = scratch_bytes_for_tiles(scan_tiles(n));
    if (!scratch) {
        *scratch_bytes = need;
        return DWP_SUCCESS;
    }
    if (*scratch_bytes < need) return DWP_ERR_SCRATCH_TOO_SMALL;
    if (n > 0 && (!in || !out)) return DWP_ERR_INVALID_VALUE;
    if (!aligned16(scratch) || (n > 0 && (!aligned16(in) || !aligned16(out))))
        return DWP_ERR_MISALIGNED;
    const uint64_t bytes = uint64_t(n) * 4u;
    if (in != out && overlap(in, bytes, out, bytes)) return DWP_ERR_ALIASING;
    if (overlap(scratch, need, in, bytes) || overlap(scratch, need, out, bytes))
        return DWP_ERR_ALIASING;

    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (launch_clear(scratch, need, nullptr, 0, s) != cudaSuccess) {
        cudaGetLastError();
        return DWP_ERR_CUDA;
    }
    if (n == 0) return DWP_SUCCESS;
    if (launch_scan(op, inclusive, in, out, n, scratch, s) != cudaSuccess) {
        cudaGetLastError();
        return DWP_ERR_CUDA;
    }
    return DWP_SUCCESS;
}

dwp_status two_level_common(dwp_op op, dwp_mode mode, const void *in, void *out, size_t n,
                            void *scratch, size_t *scratch_bytes, dwp_stream stream) {
    if (!scratch_bytes) return DWP_ERR_INVALID_VALUE;
    const int iop = static_cast<int>(op), m = static_cast<int>(mode);
    if (iop != DWP_U32_ADD && iop != DWP_F32_ADD && iop != DWP_U32_MAX) return DWP_ERR_INVALID_VALUE;
    if (m != DWP_EXCLUSIVE && m != DWP_INCLUSIVE) return DWP_ERR_INVALID_VALUE;
    if (uint64_t(n) > two_level_max_n()) return DWP_ERR_INVALID_VALUE;
    const uint64_t blocks = ceil_div(n, two_level_chunk());
    const size_t need = kHeaderBytes + size_t(4u * blocks);  // one u32 total per block
    if (!scratch) {
        *scratch_bytes = need;
        return DWP_SUCCESS;
    }
    if (*scratch_bytes < need) return DWP_ERR_SCRATCH_TOO_SMALL;
    if (n > 0 && (!in || !out)) return DWP_ERR_INVALID_VALUE;
    if (!aligned16(scratch) || (n > 0 && (!aligned16(in) || !aligned16(out))))
        return DWP_ERR_MISALIGNED;
    const uint64_t bytes = uint64_t(n) * 4u;
    if (in != out && overlap(in, bytes, out, bytes)) return DWP_ERR_ALIASING;
    if (overlap(scratch, need, in, bytes) || overlap(scratch, need, out, bytes))
        return DWP_ERR_ALIASING;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    // only the status word needs clearing: the totals are written before use
    if (launch_clear(scratch, kHeaderBytes, nullptr, 0, s) != cudaSuccess) {
        cudaGetLastError();
        return DWP_ERR_CUDA;
    }
    if (n == 0) return DWP_SUCCESS;
    if (launch_two_level(op, m == DWP_INCLUSIVE, in, out, n, scratch, s) != cudaSuccess) {
        cudaGetLastError();
        return DWP_ERR_CUDA;
    }
    return DWP_SUCCESS;
}

bool aligned4(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }

dwp_status segscan_common(const uint32_t *values, const uint32_t *offsets, size_t nseg,
                          uint32_t *out, size_t n, dwp_mode mode, void *scratch,
                          size_t *scratch_bytes, dwp_stream stream) {
    if (!scratch_bytes) return DWP_ERR_INVALID_VALUE;
    const int m = static_cast<int>(mode);
    if (m != DWP_EXCLUSIVE && m != DWP_INCLUSIVE) return DWP_ERR_INVALID_VALUE;
    if (uint64_t(n) > kMaxN || uint64_t(nseg) >= kMaxN) return DWP_ERR_INVALID_VALUE;
    const uint64_t tiles = ceil_div(n, segscan_tile_elems());
    const size_t need = scratch_bytes_for_tiles(tiles);
    if (!scratch) {
        *scratch_bytes = need;
        return DWP_SUCCESS;
    }
    if (*scratch_bytes < need) return DWP_ERR_SCRATCH_TOO_SMALL;
    if (n > 0 && (!values || !out)) return DWP_ERR_INVALID_VALUE;
    if (!offsets && (nseg > 0 || n > 0)) return DWP_ERR_INVALID_VALUE;
    if (!aligned16(scratch) || (n > 0 && (!aligned16(values) || !aligned16(out))) ||
        (offsets && !aligned4(offsets)))
        return DWP_ERR_MISALIGNED;
    const uint64_t bytes = uint64_t(n) * 4u, obytes = (uint64_t(nseg) + 1u) * 4u;
    if (overlap(out, bytes, values, bytes) || overlap(out, bytes, offsets, obytes) ||
        overlap(scratch, need, values, bytes) || overlap(scratch, need, offsets, obytes) ||
        overlap(scratch, need, out, bytes))
        return DWP_ERR_ALIASING;

    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (launch_clear(scratch, need, nullptr, 0, s) != cudaSuccess) {
        cudaGetLastError();
        return DWP_ERR_CUDA;
    }
    if (n == 0 || nseg == 0) return DWP_SUCCESS;  // no row lies in a segment
    if (launch_segscan(values, offsets, uint32_t(nseg), out, n, m == DWP_INCLUSIVE, scratch, s) !=
        cudaSuccess) {
        cudaGetLastError();
        return DWP_ERR_CUDA;
    }
    return DWP_SUCCESS;
}

dwp_status compact_common(const void *records, const uint8_t *flags, size_t n, void *out,
                          uint32_t *count, void *scratch, size_t *scratch_bytes,
                          dwp_stream stream) {
    if (!scratch_bytes) return DWP_ERR_INVALID_VALUE;
    if (uint64_t(n) > kMaxN) return DWP_ERR_INVALID_VALUE;
    const uint64_t tiles = ceil_div(n, compact_tile_records());
    const size_t need = scratch_bytes_for_tiles(tiles);
    if (!scratch) {
        *scratch_bytes = need;
        return DWP_SUCCESS;
    }
    if (*scratch_bytes < need) return DWP_ERR_SCRATCH_TOO_SMALL;
    if (!count || (n > 0 && (!records || !flags || !out))) return DWP_ERR_INVALID_VALUE;
    if (!aligned16(scratch) || !aligned4(count) ||
        (n > 0 && (!aligned16(records) || !aligned16(flags) || !aligned16(out))))
        return DWP_ERR_MISALIGNED;
    const uint64_t rbytes = uint64_t(n) * 16u, fbytes = uint64_t(n);
    if (overlap(out, rbytes, records, rbytes) || overlap(out, rbytes, flags, fbytes) ||
        overlap(out, rbytes, count, 4) || overlap(out, rbytes, scratch, need) ||
        overlap(count, 4, records, rbytes) || overlap(count, 4, flags, fbytes) ||
        overlap(count, 4, scratch, need) || overlap(scratch, need, records, rbytes) ||
        overlap(scratch, need, flags, fbytes))
        return DWP_ERR_ALIASING;

    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    // n == 0: the count is cleared with the scratch, and nothing else runs
    if (launch_clear(scratch, need, n == 0 ? count : nullptr, sizeof(uint32_t), s) != cudaSuccess) {
        cudaGetLastError();
        return DWP_ERR_CUDA;
    }
    if (n == 0) return DWP_SUCCESS;
    if (launch_compact(records, flags, n, out, count, scratch, s) != cudaSuccess) {
        cudaGetLastError();
        return DWP_ERR_CUDA;
    }
    return DWP_SUCCESS;
}

dwp_status segreduce_common(const uint32_t *values, const uint32_t *offsets, size_t nseg,
                            uint32_t *out, size_t n, void *scratch, size_t *scratch_bytes,
                            dwp_stream stream) {
    if (!scratch_bytes) return DWP_ERR_INVALID_VALUE;
    if (uint64_t(n) > kMaxN || uint64_t(nseg) >= kMaxN) return DWP_ERR_INVALID_VALUE;
    const size_t need = kHeaderBytes;  // tile counter and status only: no descriptors
    if (!scratch) {
        *scratch_bytes = need;
        return DWP_SUCCESS;
    }
    if (*scratch_bytes < need) return DWP_ERR_SCRATCH_TOO_SMALL;
    if (n > 0 && !values) return DWP_ERR_INVALID_VALUE;
    if (nseg > 0 && (!offsets || !out)) return DWP_ERR_INVALID_VALUE;
    if (!aligned16(scratch) || (n > 0 && !aligned16(values)) || (offsets && !aligned4(offsets)) ||
        (out && !aligned4(out)))
        return DWP_ERR_MISALIGNED;
    const uint64_t vbytes = uint64_t(n) * 4u, obytes = (uint64_t(nseg) + 1u) * 4u,
                   rbytes = uint64_t(nseg) * 4u;
    if (overlap(out, rbytes, values, vbytes) || overlap(out, rbytes, offsets, obytes) ||
        overlap(out, rbytes, scratch, need) || overlap(scratch, need, values, vbytes) ||
        overlap(scratch, need, offsets, obytes))
        return DWP_ERR_ALIASING;

    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (launch_clear(scratch, need, nseg > 0 ? out : nullptr, rbytes, s) != cudaSuccess) {
        cudaGetLastError();
        return DWP_ERR_CUDA;
    }
    if (n == 0 || nseg == 0) return DWP_SUCCESS;  // every segment empty: all zeros
    if (launch_segreduce(values, offsets, uint32_t(nseg), out, n, scratch, s) != cudaSuccess) {
        cudaGetLastError();
        return DWP_ERR_CUDA;
    }
    return DWP_SUCCESS;
}

dwp_status recurrence_common(const float *a, const float *b, float *h, size_t n, dwp_mode mode,
                             void *scratch, size_t *scratch_bytes, dwp_stream stream) {
    if (!scratch_bytes) return DWP_ERR_INVALID_VALUE;
    const int m = static_cast<int>(mode);
    if (m != DWP_EXCLUSIVE && m != DWP_INCLUSIVE) return DWP_ERR_INVALID_VALUE;
    if (uint64_t(n) > kMaxN) return DWP_ERR_INVALID_VALUE;
    const uint64_t tiles = ceil_div(n, recurrence_tile_elems());
    const size_t need = kHeaderBytes + 16u * tiles;  // two descriptor words per tile
    if (!scratch) {
        *scratch_bytes = need;
        return DWP_SUCCESS;
    }
    if (*scratch_bytes < need) return DWP_ERR_SCRATCH_TOO_SMALL;
    if (n > 0 && (!a || !b || !h)) return DWP_ERR_INVALID_VALUE;
    if (!aligned16(scratch) || (n > 0 && (!aligned16(a) || !aligned16(b) || !aligned16(h))))
        return DWP_ERR_MISALIGNED;
    const uint64_t bytes = uint64_t(n) * 4u;
    // h may be a or b exactly (in place); a partial overlap is rejected
    if ((h != a && overlap(h, bytes, a, bytes)) || (h != b && overlap(h, bytes, b, bytes)))
        return DWP_ERR_ALIASING;
    if (overlap(scratch, need, a, bytes) || overlap(scratch, need, b, bytes) ||
        overlap(scratch, need, h, bytes))
        return DWP_ERR_ALIASING;

    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (launch_clear(scratch, need, nullptr, 0, s) != cudaSuccess) {
        cudaGetLastError();
        return DWP_ERR_CUDA;
    }
    if (n == 0) return DWP_SUCCESS;
    if (launch_recurrence(a, b, h, n, m == DWP_INCLUSIVE, scratch, s) != cudaSuccess) {
        cudaGetLastError();
        return DWP_ERR_CUDA;
    }
    return DWP_SUCCESS;
}

}  // namespace

extern "C" {

dwp_status dwp_compact_by_flags(const void *d_records, const uint8_t *d_flags, size_t n,
                                void *d_out, uint32_t *d_count, void *d_scratch,
                                size_t *scratch_bytes, dwp_stream stream) {
    return compact_common(d_records, d_flags, n, d_out, d_count, d_scratch, scratch_bytes, stream);
}

dwp_status dwp_segmented_scan_u32(const uint32_t *d_values, const uint32_t *d_offsets,
                                  size_t num_segments, uint32_t *d_out, size_t n, dwp_mode mode,
                                  void *d_scratch, size_t *scratch_bytes, dwp_stream stream) {
    return segscan_common(d_values, d_offsets, num_segments, d_out, n, mode, d_scratch,
                          scratch_bytes, stream);
}

dwp_status dwp_scan_exclusive(dwp_op op, const void *d_in, void *d_out, size_t n,
                              void *d_scratch, size_t *scratch_bytes, dwp_stream stream) {
    return scan_common(false, op, d_in, d_out, n, d_scratch, scratch_bytes, stream);
}

dwp_status dwp_scan_inclusive(dwp_op op, const void *d_in, void *d_out, size_t n,
                              void *d_scratch, size_t *scratch_bytes, dwp_stream stream) {
    return scan_common(true, op, d_in, d_out, n, d_scratch, scratch_bytes, stream);
}

dwp_status dwp_segmented_reduce_u32(const uint32_t *d_values, const uint32_t *d_offsets,
                                    size_t num_segments, uint32_t *d_out, size_t n,
                                    void *d_scratch, size_t *scratch_bytes, dwp_stream stream) {
    return segreduce_common(d_values, d_offsets, num_segments, d_out, n, d_scratch, scratch_bytes,
                            stream);
}

dwp_status dwp_linear_recurrence_f32(const float *d_a, const float *d_b, float *d_h, size_t n,
                                     dwp_mode mode, void *d_scratch, size_t *scratch_bytes,
                                     dwp_stream stream) {
    return recurrence_common(d_a, d_b, d_h, n, mode, d_scratch, scratch_bytes, stream);
}

dwp_status dwp_scan_two_level(dwp_op op, dwp_mode mode, const void *d_in, void *d_out, size_t n,
                              void *d_scratch, size_t *scratch_bytes, dwp_stream stream) {
    return two_level_common(op, mode, d_in, d_out, n, d_scratch, scratch_bytes, stream);
}

dwp_status dwp_read_status(const void *d_scratch, dwp_stream stream) {
    if (!d_scratch) return DWP_ERR_INVALID_VALUE;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    uint32_t st = 0;
    const auto *hdr = reinterpret_cast<const ScratchHeader *>(d_scratch);
    if (cudaMemcpyAsync(&st, &hdr->status, sizeof(st), cudaMemcpyDeviceToHost, s) != cudaSuccess ||
        cudaStreamSynchronize(s) != cudaSuccess) {
        cudaGetLastError();
        return DWP_ERR_CUDA;
    }
    return static_cast<dwp_status>(st);
}

const char *dwp_status_string(dwp_status status) {
    switch (status) {
        case DWP_SUCCESS: return "DWP_SUCCESS";
        case DWP_ERR_INVALID_VALUE: return "DWP_ERR_INVALID_VALUE";
        case DWP_ERR_MISALIGNED: return "DWP_ERR_MISALIGNED";
        case DWP_ERR_ALIASING: return "DWP_ERR_ALIASING";
        case DWP_ERR_SCRATCH_TOO_SMALL: return "DWP_ERR_SCRATCH_TOO_SMALL";
        case DWP_ERR_CUDA: return "DWP_ERR_CUDA";
        case DWP_ERR_LOOKBACK_TIMEOUT: return "DWP_ERR_LOOKBACK_TIMEOUT";
        case DWP_ERR_PIPELINE_TIMEOUT: return "DWP_ERR_PIPELINE_TIMEOUT";
        case DWP_ERR_NO_DEVICE: return "DWP_ERR_NO_DEVICE";
        case DWP_ERR_BOUNDS: return "DWP_ERR_BOUNDS";
    }
    return "DWP_UNKNOWN_STATUS";
}

int dwp_version(void) { return 100; }

dwp_status dwp_set_lookback_window(uint32_t tiles) {
    set_lookback_window(tiles);
    return DWP_SUCCESS;
}

dwp_status dwp_read_fallbacks(const void *d_scratch, dwp_stream stream, uint32_t *count) {
    if (!d_scratch || !count) return DWP_ERR_INVALID_VALUE;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    uint32_t v = 0;
    const auto *hdr = reinterpret_cast<const ScratchHeader *>(d_scratch);
    if (cudaMemcpyAsync(&v, &hdr->fallbacks, sizeof(v), cudaMemcpyDeviceToHost, s) != cudaSuccess ||
        cudaStreamSynchronize(s) != cudaSuccess) {
        cudaGetLastError();
        return DWP_ERR_CUDA;
    }
    *count = v;
    return DWP_SUCCESS;
}

dwp_status dwp_debug_set_fault(uint32_t never_publish_tile, uint32_t spin_limit,
                               uint32_t fallback_polls) {
    set_fault_config(never_publish_tile, spin_limit, fallback_polls);
    return DWP_SUCCESS;
}

dwp_status dwp_debug_set_delay(uint32_t seed, uint32_t fraction_ppm, uint32_t max_ns) {
    if (fraction_ppm > 1000000u || max_ns > kMaxDelayNs) return DWP_ERR_INVALID_VALUE;
    // a tile sleeps at a point when a 32-bit hash falls below the threshold
    const uint64_t thr = (uint64_t(fraction_ppm) << 32) / 1000000u;
    set_delay_config(seed, thr > 0xffffffffull ? 0xffffffffu : uint32_t(thr), max_ns);
    return DWP_SUCCESS;
}

dwp_status dwp_read_lookback_stats(const void *d_scratch, dwp_stream stream, uint32_t *fallbacks,
                                   uint32_t *intermediates, uint32_t *jumps) {
    if (!d_scratch) return DWP_ERR_INVALID_VALUE;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    uint32_t v[3] = {0u, 0u, 0u};
    const auto *hdr = reinterpret_cast<const ScratchHeader *>(d_scratch);
    static_assert(offsetof(ScratchHeader, jumps) == offsetof(ScratchHeader, fallbacks) + 8,
                  "the three counters are adjacent");
    if (cudaMemcpyAsync(v, &hdr->fallbacks, sizeof(v), cudaMemcpyDeviceToHost, s) != cudaSuccess ||
        cudaStreamSynchronize(s) != cudaSuccess) {
        cudaGetLastError();
        return DWP_ERR_CUDA;
    }
    if (fallbacks) *fallbacks = v[0];
    if (intermediates) *intermediates = v[1];
    if (jumps) *jumps = v[2];
    return DWP_SUCCESS;
}

}  // extern "C"
