// Host-side helpers: per-device occupancy cache and the test fault settings.
#include <cuda_runtime.h>

#include <atomic>
#include <map>
#include <mutex>
#include <utility>

#include "device.cuh"
#include "launch.h"

namespace dwp {

namespace {

struct ClearRange {
    uint32_t *p;
    uint64_t words;
};

// Words up to the first 16-byte boundary one by one, then 16-byte stores,
// then the last 0-3 words; grid-stride over the 16-byte part.
__device__ __forceinline__ void clear_range(const ClearRange &r, uint64_t tid, uint64_t nthr) {
    if (r.words == 0) return;
    const uint64_t mis = (reinterpret_cast<uintptr_t>(r.p) >> 2) & 3u;
    const uint64_t head = min(r.words, (4u - mis) & 3u);
    const uint64_t vec = (r.words - head) / 4u;
    const uint64_t tail0 = head + 4u * vec;
    if (tid < head) r.p[tid] = 0u;
    uint4 *v = reinterpret_cast<uint4 *>(r.p + head);
    for (uint64_t i = tid; i < vec; i += nthr) v[i] = make_uint4(0u, 0u, 0u, 0u);
    if (tid < r.words - tail0) r.p[tail0 + tid] = 0u;
}

constexpr int kClearThreads = 256;

__global__ void __launch_bounds__(kClearThreads) clear_kernel(ClearRange r0, ClearRange r1) {
    pdl_trigger();
    pdl_wait();  // the previous kernel may still use these bytes
    const uint64_t tid = uint64_t(blockIdx.x) * blockDim.x + threadIdx.x;
    const uint64_t nthr = uint64_t(gridDim.x) * blockDim.x;
    clear_range(r0, tid, nthr);
    clear_range(r1, tid, nthr);
}

}  // namespace

cudaError_t launch_clear(void *a, size_t a_bytes, void *b, size_t b_bytes, cudaStream_t stream) {
    const ClearRange r0{static_cast<uint32_t *>(a), a ? uint64_t(a_bytes) / 4u : 0u};
    const ClearRange r1{static_cast<uint32_t *>(b), b ? uint64_t(b_bytes) / 4u : 0u};
    if (r0.words == 0 && r1.words == 0) return cudaSuccess;
    const uint64_t vec = (r0.words > r1.words ? r0.words : r1.words) / 4u + 1u;
    uint64_t blocks = (vec + kClearThreads - 1) / kClearThreads;
    if (blocks > 1024u) blocks = 1024u;
    return launch_pdl(clear_kernel, dim3(uint32_t(blocks)), dim3(kClearThreads), 0, stream, r0, r1);
}

namespace {
std::mutex g_mu;
std::map<std::pair<int, const void *>, int> g_blocks;
std::atomic<uint32_t> g_never_publish{0xffffffffu};
std::atomic<uint32_t> g_spin_limit{0u};
std::atomic<uint32_t> g_fallback_polls{0u};
std::atomic<uint32_t> g_lookback_window{0u};
std::atomic<uint32_t> g_delay_seed{0u};
std::atomic<uint32_t> g_delay_threshold{0u};
std::atomic<uint32_t> g_delay_max_ns{0u};
}  // namespace

int device_blocks(const void *kernel, int threads, size_t smem_bytes) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    std::lock_guard<std::mutex> lock(g_mu);
    auto key = std::make_pair(dev, kernel);
    auto it = g_blocks.find(key);
    if (it != g_blocks.end()) return it->second;
    int sms = 0, per_sm = 0;
    if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             int(smem_bytes)) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, threads, smem_bytes) !=
            cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    const int blocks = sms * per_sm;
    g_blocks[key] = blocks;
    return blocks;
}

LaunchKnobs current_launch_knobs() {
    LaunchKnobs f;
    f.never_publish_tile = g_never_publish.load();
    const uint32_t lim = g_spin_limit.load();
    f.spin_limit = lim ? lim : kDefaultSpinLimit;
    const uint32_t fb = g_fallback_polls.load();
    f.fallback_polls = fb == 0u ? kDefaultFallbackPolls : (fb == 0xffffffffu ? 0u : fb);
    f.lookback_window = g_lookback_window.load();
    f.delay_seed = g_delay_seed.load();
    f.delay_threshold = g_delay_threshold.load();
    f.delay_max_ns = g_delay_max_ns.load();
    return f;
}

void set_delay_config(uint32_t seed, uint32_t threshold, uint32_t max_ns) {
    g_delay_seed.store(seed);
    g_delay_max_ns.store(max_ns);
    g_delay_threshold.store(threshold);
}

void set_lookback_window(uint32_t tiles) { g_lookback_window.store(tiles); }

void set_fault_config(uint32_t never_publish_tile, uint32_t spin_limit, uint32_t fallback_polls) {
    g_never_publish.store(never_publish_tile);
    g_spin_limit.store(spin_limit);
    g_fallback_polls.store(fallback_polls);
}

}  // namespace dwp
