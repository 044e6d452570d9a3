// Scan entry point that needs no scratch buffer from the caller.
//
// Some callers cannot call cudaMalloc at the moment they need a scan: code
// running inside another framework's allocator hooks or memory-pool
// callbacks, where an allocation would re-enter that allocator, and plug-ins
// whose host application owns all device memory and forbids allocations
// after start-up.  For them this file keeps the scan's scratch (tile
// counter, status word, one descriptor per tile) in a fixed array that is
// part of the library's device image: every GPU that loads the library holds
// it until the process exits, and no call allocates or frees anything.
#include <cuda_runtime.h>

#include "launch.h"

namespace {

using namespace dwp;

// Room for DWP_SCAN_STATIC_MAX_N elements at any tile size of 4096 elements
// or more: the 128-byte header plus 65,536 descriptors (about 512 KiB).
constexpr uint64_t kStaticMaxN = DWP_SCAN_STATIC_MAX_N;
constexpr size_t kStaticScratchBytes = kHeaderBytes + 8u * 65536u;

static __device__ __align__(256) unsigned char g_static_scratch[kStaticScratchBytes];

// In host code `g_static_scratch` names a host-side stand-in, not device
// memory, so the kernels get the address that cudaGetSymbolAddress returns
// for the current device.  It is looked up on every call rather than cached:
// after cudaDeviceReset (or any reset of the primary context) the module is
// loaded again and the array may sit at another address, and a cached
// address would then point at memory this library no longer owns.  The
// lookup is a host-side table query, small next to a scan.
dwp_status static_scratch_address(void **out) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) {
        cudaGetLastError();
        return DWP_ERR_NO_DEVICE;
    }
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_static_scratch) != cudaSuccess || !p) {
        cudaGetLastError();
        return DWP_ERR_CUDA;
    }
    *out = p;
    return DWP_SUCCESS;
}

}  // namespace

extern "C" dwp_status dwp_scan_static_scratch(dwp_op op, dwp_mode mode, const void *d_in,
                                              void *d_out, size_t n, dwp_stream stream) {
    const int m = static_cast<int>(mode);
    if (m != DWP_EXCLUSIVE && m != DWP_INCLUSIVE) return DWP_ERR_INVALID_VALUE;
    if (uint64_t(n) > kStaticMaxN) return DWP_ERR_SCRATCH_TOO_SMALL;
    size_t need = 0;  // the size query also rejects an unknown op
    dwp_status st = dwp_scan_exclusive(op, nullptr, nullptr, n, nullptr, &need, stream);
    if (st != DWP_SUCCESS) return st;
    if (need > kStaticScratchBytes) return DWP_ERR_SCRATCH_TOO_SMALL;
    void *scratch = nullptr;
    st = static_scratch_address(&scratch);
    if (st != DWP_SUCCESS) return st;
    // The regular entry point validates the data pointers, clears the part
    // of the array this call uses on `stream` and launches the scan.
    size_t bytes = kStaticScratchBytes;
    return m == DWP_INCLUSIVE ? dwp_scan_inclusive(op, d_in, d_out, n, scratch, &bytes, stream)
                              : dwp_scan_exclusive(op, d_in, d_out, n, scratch, &bytes, stream);
}

extern "C" dwp_status dwp_read_static_status(dwp_stream stream) {
    void *scratch = nullptr;
    const dwp_status st = static_scratch_address(&scratch);
    if (st != DWP_SUCCESS) return st;
    return dwp_read_status(scratch, stream);
}
