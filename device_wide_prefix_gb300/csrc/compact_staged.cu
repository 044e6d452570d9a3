// Staged stream compaction, the comparison point for the fused kernel.
//
// "Prefix scans and compaction", section "Worked example: Stable stream
// compaction", asks to compare an implementation that writes the keep flags
// and their prefixes to memory as separate arrays with a fused one, and to
// put the difference down to the extra passes over full arrays; section
// "Common errors" lists the cost of materialising predicates and prefixes
// among the usual mistakes.  This file is that staged implementation, built
// from the same pieces a library user would chain:
//   1. predicate   u8 flags -> u32 flags f[i] = (flags[i] != 0)   (reads n B, writes 4n B)
//   2. scan        exclusive u32-add scan of f into off[], by the
//                  library's own single-pass scan                (reads 4n B, writes 4n B)
//   3. scatter     record i -> out[off[i]] when f[i] != 0, and the
//                  count off[n-1] + f[n-1]                       (reads 8n B + the kept
//                                                                 records, writes 16 B each)
// Step 3 reads a record only when it is kept, so its record reads are the
// 32-byte sectors that hold a kept record.  The fused kernel (compact.cu)
// reads every record once and writes nothing but the output.
#include <cuda_runtime.h>

#include "device.cuh"
#include "launch.h"

namespace dwp {

namespace {

constexpr int kStagedThreads = 256;

// f[i] = flags[i] != 0; 16 flags per thread and step (one 16-byte load,
// four 16-byte stores), the last n % 16 flags one by one.
__global__ void __launch_bounds__(kStagedThreads)
    predicate_kernel(const uint8_t *flags, uint32_t *f, uint64_t n) {
    pdl_wait();
    pdl_trigger();
    const uint64_t nvec = n / 16;
    const uint64_t stride = uint64_t(gridDim.x) * blockDim.x;
    for (uint64_t q = uint64_t(blockIdx.x) * blockDim.x + threadIdx.x; q < nvec; q += stride) {
        const uint4 v = reinterpret_cast<const uint4 *>(flags)[q];
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
        uint4 *dst = reinterpret_cast<uint4 *>(f + 16 * q);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const uint32_t b = w[j];
            dst[j] = make_uint4((b & 0xffu) != 0u, (b & 0xff00u) != 0u, (b & 0xff0000u) != 0u,
                                (b & 0xff000000u) != 0u);
        }
    }
    const uint64_t i = 16 * nvec + uint64_t(blockIdx.x) * blockDim.x + threadIdx.x;
    if (i < n && i < 16 * nvec + 16) f[i] = flags[i] != 0 ? 1u : 0u;
}

// out[off[i]] = rec[i] for kept records; 4 records per thread and step (one
// 16-byte load each of f and off), the last n % 4 one by one.  The thread
// that handles record n - 1 writes the count.  The output slot comes from
// the scan, so the debug bounds build checks it (against n, in the scan's
// status word).
__global__ void __launch_bounds__(kStagedThreads)
    scatter_kernel(const uint4 *rec, const uint32_t *f, const uint32_t *off, uint64_t n, uint4 *out,
                   uint32_t *count, ScratchHeader *hdr) {
    pdl_wait();
    pdl_trigger();
    const uint64_t nvec = n / 4;
    const uint64_t stride = uint64_t(gridDim.x) * blockDim.x;
    for (uint64_t q = uint64_t(blockIdx.x) * blockDim.x + threadIdx.x; q < nvec; q += stride) {
        const uint4 fv = reinterpret_cast<const uint4 *>(f)[q];
        const uint4 ov = reinterpret_cast<const uint4 *>(off)[q];
        const uint32_t fk[4] = {fv.x, fv.y, fv.z, fv.w};
        const uint32_t ok[4] = {ov.x, ov.y, ov.z, ov.w};
#pragma unroll
        for (int j = 0; j < 4; ++j)
            if (fk[j] && in_bounds(hdr, ok[j], 1, n)) out[ok[j]] = rec[4 * q + j];
        if (4 * q + 4 == n) *count = ok[3] + fk[3];
    }
    const uint64_t i = 4 * nvec + uint64_t(blockIdx.x) * blockDim.x + threadIdx.x;
    if (i < n && i < 4 * nvec + 4) {
        if (f[i] && in_bounds(hdr, off[i], 1, n)) out[off[i]] = rec[i];
        if (i == n - 1) *count = off[i] + f[i];
    }
}

uint64_t round16(uint64_t b) { return (b + 15u) & ~uint64_t(15u); }

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool overlap(const void *a, uint64_t an, const void *b, uint64_t bn) {
    if (!a || !b || an == 0 || bn == 0) return false;
    const uintptr_t pa = reinterpret_cast<uintptr_t>(a), pb = reinterpret_cast<uintptr_t>(b);
    return pa < pb + bn && pb < pa + an;
}

// Blocks of a grid-stride launch: every SM filled at this block size.
uint32_t staged_grid(const void *kernel, uint64_t work_items) {
    const int dev_blocks = device_blocks(kernel, kStagedThreads, 0);
    if (dev_blocks <= 0) return 0;
    const uint64_t want = (work_items + kStagedThreads - 1) / kStagedThreads;
    return uint32_t(want < uint64_t(dev_blocks) ? (want ? want : 1) : uint64_t(dev_blocks));
}

}  // namespace

}  // namespace dwp

extern "C" dwp_status dwp_compact_by_flags_staged(const void *d_records, const uint8_t *d_flags,
                                                  size_t n, void *d_out, uint32_t *d_count,
                                                  void *d_scratch, size_t *scratch_bytes,
                                                  dwp_stream stream) {
    using namespace dwp;
    if (!scratch_bytes) return DWP_ERR_INVALID_VALUE;
    if (uint64_t(n) > 0xffffffffull) return DWP_ERR_INVALID_VALUE;
    // scratch: the scan's own scratch first (so dwp_read_status on d_scratch
    // reads the scan's status word), then f[] and off[]
    size_t scan_need = 0;
    dwp_status st = dwp_scan_exclusive(DWP_U32_ADD, nullptr, nullptr, n, nullptr, &scan_need, stream);
    if (st != DWP_SUCCESS) return st;
    const uint64_t scan_part = round16(scan_need), arr = round16(uint64_t(n) * 4u);
    const size_t need = size_t(scan_part + 2 * arr);
    if (!d_scratch) {
        *scratch_bytes = need;
        return DWP_SUCCESS;
    }
    if (*scratch_bytes < need) return DWP_ERR_SCRATCH_TOO_SMALL;
    if (!d_count || (n > 0 && (!d_records || !d_flags || !d_out))) return DWP_ERR_INVALID_VALUE;
    if (!aligned16(d_scratch) || (reinterpret_cast<uintptr_t>(d_count) & 3u) ||
        (n > 0 && (!aligned16(d_records) || !aligned16(d_flags) || !aligned16(d_out))))
        return DWP_ERR_MISALIGNED;
    const uint64_t rbytes = uint64_t(n) * 16u, fbytes = uint64_t(n);
    if (overlap(d_out, rbytes, d_records, rbytes) || overlap(d_out, rbytes, d_flags, fbytes) ||
        overlap(d_out, rbytes, d_count, 4) || overlap(d_out, rbytes, d_scratch, need) ||
        overlap(d_count, 4, d_records, rbytes) || overlap(d_count, 4, d_flags, fbytes) ||
        overlap(d_count, 4, d_scratch, need) || overlap(d_scratch, need, d_records, rbytes) ||
        overlap(d_scratch, need, d_flags, fbytes))
        return DWP_ERR_ALIASING;

    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    unsigned char *base = static_cast<unsigned char *>(d_scratch);
    uint32_t *f = reinterpret_cast<uint32_t *>(base + scan_part);
    uint32_t *off = reinterpret_cast<uint32_t *>(base + scan_part + arr);
    if (n == 0) {
        // still clear the scan's status word, as every call does
        size_t sb = scan_need;
        st = dwp_scan_exclusive(DWP_U32_ADD, nullptr, nullptr, 0, d_scratch, &sb, stream);
        if (st != DWP_SUCCESS) return st;
        if (launch_clear(d_count, sizeof(uint32_t), nullptr, 0, s) != cudaSuccess) {
            cudaGetLastError();
            return DWP_ERR_CUDA;
        }
        return DWP_SUCCESS;
    }
    const uint32_t g1 = staged_grid(reinterpret_cast<const void *>(predicate_kernel), (n + 15) / 16);
    const uint32_t g3 = staged_grid(reinterpret_cast<const void *>(scatter_kernel), (n + 3) / 4);
    if (g1 == 0 || g3 == 0) return DWP_ERR_CUDA;
    if (launch_pdl(predicate_kernel, dim3(g1), dim3(kStagedThreads), 0, s, d_flags, f, uint64_t(n)) !=
        cudaSuccess) {
        cudaGetLastError();
        return DWP_ERR_CUDA;
    }
    size_t sb = scan_need;
    st = dwp_scan_exclusive(DWP_U32_ADD, f, off, n, d_scratch, &sb, stream);
    if (st != DWP_SUCCESS) return st;
    if (launch_pdl(scatter_kernel, dim3(g3), dim3(kStagedThreads), 0, s,
                   static_cast<const uint4 *>(d_records), static_cast<const uint32_t *>(f),
                   static_cast<const uint32_t *>(off), uint64_t(n), static_cast<uint4 *>(d_out),
                   d_count, static_cast<ScratchHeader *>(d_scratch)) != cudaSuccess) {
        cudaGetLastError();
        return DWP_ERR_CUDA;
    }
    return DWP_SUCCESS;
}
