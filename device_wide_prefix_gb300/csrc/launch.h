// Host-side launch helpers and the kernel launchers behind the C entry points.
#pragma once

#include <cuda_runtime.h>

#include "common.h"

namespace dwp {

// Launch `kernel` with programmatic stream serialisation: it may begin while
// the previous kernel on `stream` finishes, and waits for it (pdl_wait)
// before it touches global memory.  Hides most of one launch latency per
// kernel boundary.
template <class... KArgs, class... Args>
inline cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                              cudaStream_t stream, Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, args...);
}

// Zero [a, a + a_bytes) and [b, b + b_bytes) with one kernel on `stream`
// (launched like every other kernel here, so the kernel after it can start
// early).  Both pointers 4-byte aligned and both sizes multiples of 4 bytes;
// a null pointer or a zero size skips that range.
cudaError_t launch_clear(void *a, size_t a_bytes, void *b, size_t b_bytes, cudaStream_t stream);

// Resident blocks of `kernel` on the current device (SM count x blocks per
// SM at this block size and dynamic shared memory).  Also raises the
// kernel's dynamic shared-memory limit to `smem_bytes`.  Cached per device
// and kernel.  Returns 0 if the kernel cannot be resident at all.
int device_blocks(const void *kernel, int threads, size_t smem_bytes);

// Inputs of at most this many elements take the small-input plain scan
// (scan_small.cu: one block per tile); larger ones the persistent pipelined
// kernel (scan.cu).  Measured on GB300: at 2^23 the small-input kernel takes
// 19.3 us and the pipelined one 22.8; at 2^24, 43.3 against 34.4.
#ifndef DWP_SCAN_SMALL_LOG2
#define DWP_SCAN_SMALL_LOG2 23
#endif
constexpr uint64_t kScanSmallMax = uint64_t(1) << DWP_SCAN_SMALL_LOG2;
// Elements per tile of the large-input plain scan kernel.
uint32_t scan_tile_elems();
// Descriptors the small-input kernel needs for n <= kScanSmallMax: at least
// its tile count, and never fewer than for any smaller n (it sizes its tile
// by n, so its tile count alone is not monotone in n).
uint64_t scan_small_descriptors(uint64_t n);
// Descriptors the plain scan's size query asks for: non-decreasing in n, so
// scratch sized for the largest n serves every smaller one.
inline uint64_t scan_tiles(uint64_t n) {
    return n <= kScanSmallMax ? scan_small_descriptors(n)
                              : (n + scan_tile_elems() - 1) / scan_tile_elems();
}
// One launch of the plain scan (the scratch has already been cleared); picks
// the kernel by n as above.
cudaError_t launch_scan(dwp_op op, bool inclusive, const void *in, void *out, uint64_t n,
                        void *scratch, cudaStream_t stream);
cudaError_t launch_scan_small(dwp_op op, bool inclusive, const void *in, void *out, uint64_t n,
                              void *scratch, cudaStream_t stream, const LaunchKnobs &fault);

// Elements per tile of the segmented scan kernel.
uint32_t segscan_tile_elems();
// One launch of the segmented u32 scan (scratch already cleared; nseg >= 1).
cudaError_t launch_segscan(const uint32_t *values, const uint32_t *offsets, uint32_t nseg,
                           uint32_t *out, uint64_t n, bool inclusive, void *scratch,
                           cudaStream_t stream);

// Records per tile of the compaction kernel.
uint32_t compact_tile_records();
// One launch of the stable compaction (scratch already cleared; n >= 1).
cudaError_t launch_compact(const void *records, const uint8_t *flags, uint64_t n, void *out,
                           uint32_t *count, void *scratch, cudaStream_t stream);

// Largest n and elements per block of the two-level (three-launch) scan.
uint64_t two_level_max_n();
uint32_t two_level_chunk();
// The three launches of the two-level scan; the scratch holds the 128-byte
// header and then one u32 total per block.
cudaError_t launch_two_level(dwp_op op, bool inclusive, const void *in, void *out, uint64_t n,
                             void *scratch, cudaStream_t stream);

// Rows per tile of the segmented reduction kernel.
uint32_t segreduce_tile_elems();
// One launch of the segmented u32 reduction (out already cleared, scratch
// header cleared; nseg >= 1, n >= 1).
cudaError_t launch_segreduce(const uint32_t *values, const uint32_t *offsets, uint32_t nseg,
                             uint32_t *out, uint64_t n, void *scratch, cudaStream_t stream);

// Elements per tile of the linear-recurrence kernel.
uint32_t recurrence_tile_elems();
// One launch of the f32 linear recurrence h[t] = a[t] h[t-1] + b[t]
// (scratch already cleared: header + 16 bytes per tile; n >= 1).
cudaError_t launch_recurrence(const float *a, const float *b, float *h, uint64_t n, bool inclusive,
                              void *scratch, cudaStream_t stream);

}  // namespace dwp
