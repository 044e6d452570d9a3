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
    uint32_t reserved[30];
};
static_assert(sizeof(ScratchHeader) == 128, "scratch header is 128 bytes");

constexpr size_t kHeaderBytes = sizeof(ScratchHeader);

inline size_t scratch_bytes_for_tiles(uint64_t tiles) { return kHeaderBytes + 8u * tiles; }

// Bounds of every device-side wait; a wait that reaches its bound records an
// error and the kernel exits instead of hanging.
constexpr uint32_t kDefaultSpinLimit = 1u << 20;  // look-back polls (~1 s with backoff)
constexpr uint32_t kPipeWaitLimit = 1u << 24;     // mbarrier polls (>1 s with backoff)

// Test hooks carried into every launch (see dwp_debug_set_fault).
struct FaultConfig {
    uint32_t never_publish_tile;  // UINT32_MAX: none
    uint32_t spin_limit;          // look-back polls before giving up
};

FaultConfig current_fault_config();
void set_fault_config(uint32_t never_publish_tile, uint32_t spin_limit);

}  // namespace dwp
