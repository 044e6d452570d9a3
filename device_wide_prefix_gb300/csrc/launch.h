// Host-side launch helpers and the kernel launchers behind the C entry points.
#pragma once

#include <cuda_runtime.h>

#include "common.h"

namespace dwp {

// Resident blocks of `kernel` on the current device (SM count x blocks per
// SM at this block size and dynamic shared memory).  Also raises the
// kernel's dynamic shared-memory limit to `smem_bytes`.  Cached per device
// and kernel.  Returns 0 if the kernel cannot be resident at all.
int device_blocks(const void *kernel, int threads, size_t smem_bytes);

// Elements per tile of the plain scan kernel.
uint32_t scan_tile_elems();
// One launch of the plain scan (the scratch has already been cleared).
cudaError_t launch_scan(dwp_op op, bool inclusive, const void *in, void *out, uint64_t n,
                        void *scratch, cudaStream_t stream);

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
