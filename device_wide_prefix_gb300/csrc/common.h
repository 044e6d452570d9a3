// Definitions shared by the host launchers and the kernels: scratch layout,
// tile geometry and the limits of every device-side wait.
#pragma once

#include <cstddef>
#include <cstdint>

#include "dwp.h"

namespace dwp {

// Scratch layout: a 128-byte header, then one 8-byte descriptor per tile.
struct ScratchHeader {
    uint32_t tile_counter;  // next tile index to hand out (atomicAdd)
    uint32_t status;        // 0, or the first device-side dwp_status recorded
    uint32_t fallbacks;     // tiles whose aggregate a successor computed and published
    uint32_t intermediates; // intermediate descriptors published by bounded-window look-backs
    uint32_t jumps;         // look-back steps that jumped over an intermediate
    uint32_t reserved[27];
};
static_assert(sizeof(ScratchHeader) == 128, "scratch header is 128 bytes");

constexpr size_t kHeaderBytes = sizeof(ScratchHeader);

inline size_t scratch_bytes_for_tiles(uint64_t tiles) { return kHeaderBytes + 8u * tiles; }

// Bounds of every device-side wait; a wait that reaches its bound records an
// error and the kernel exits instead of hanging.
constexpr uint32_t kDefaultSpinLimit = 1u << 20;  // look-back polls (~1 s with backoff)
constexpr uint32_t kPipeWaitLimit = 1u << 24;     // mbarrier polls (>1 s with backoff)
// Look-back polls on a window with an unpublished predecessor before the
// waiting tile reduces that predecessor itself (several ms with backoff:
// far above any wait of a healthy run).
constexpr uint32_t kDefaultFallbackPolls = 1u << 12;

// Settings carried into every launch: the test hooks of dwp_debug_set_fault
// and the look-back window of dwp_set_lookback_window.
struct LaunchKnobs {
    uint32_t never_publish_tile;  // UINT32_MAX: none
    uint32_t spin_limit;          // look-back polls before giving up
    uint32_t fallback_polls;      // polls before a Decoupled Fallback; 0: never
    uint32_t lookback_window;     // tiles folded between intermediate publications; 0: unbounded
    // schedule perturbation (dwp_debug_set_delay): a tile sleeps at a
    // publication point when a hash of (seed, tile, point) is below
    // delay_threshold (0: never), for up to delay_max_ns nanoseconds
    uint32_t delay_seed;
    uint32_t delay_threshold;
    uint32_t delay_max_ns;
};

// Longest sleep dwp_debug_set_delay accepts, in nanoseconds.
constexpr uint32_t kMaxDelayNs = 100000u;

LaunchKnobs current_launch_knobs();
void set_fault_config(uint32_t never_publish_tile, uint32_t spin_limit, uint32_t fallback_polls);
void set_lookback_window(uint32_t tiles);
void set_delay_config(uint32_t seed, uint32_t threshold, uint32_t max_ns);

}  // namespace dwp
