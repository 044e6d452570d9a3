// Host-side helpers: per-device occupancy cache and the test fault settings.
#include <cuda_runtime.h>

#include <atomic>
#include <map>
#include <mutex>
#include <utility>

#include "launch.h"

namespace dwp {

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
