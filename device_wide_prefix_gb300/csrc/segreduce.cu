// Segmented u32 addition reduction over CSR offsets, one pass, for sm_103a.
//
// "GPUSegmentedScan" (luma.gl), section "Composition", names a segmented
// reduction beside the segmented scan as the rest of the segmented algebra;
// read on the same contract ("Contract": segment s is rows
// [offsets[s], offsets[s+1])): out[s] is the wrapping u32 sum of segment s,
// and 0 for an empty segment.
//
// u32 addition wraps modulo 2^32, so it is exact in any order, and the sum
// of rows [lo, hi) of a tile is P(hi - 1) - P(lo - 1) for the tile's
// inclusive prefix P, also exactly.  So no tile waits for another: there is
// no look-back and no descriptor.  Per tile:
//   * the segments that overlap it come from two warp-wide searches of the
//     offsets (done while the tile's bulk copy is in flight);
//   * one pass over the tile gives the totals of its chunks (ITEMS contiguous
//     rows each) and their exclusive prefix;
//   * for each overlapping segment the tile's piece is P(hi-1) - P(lo-1),
//     P read from a chunk prefix plus at most ITEMS-1 rows of the tile;
//   * a segment that lies inside the tile is stored; a piece of a segment
//     that crosses a tile edge is added with one atomicAdd into out, which
//     the host cleared first.  Empty segments keep that 0.
// Each worker warp owns two stages and double-buffers its own tiles: it
// takes the next tile index and starts its bulk load before it reduces the
// current one.  Tile indices come from an atomic counter.
// Offsets are trusted (non-decreasing, offsets[N] <= n); every access stays
// inside offsets[0..N] and values[0..n) regardless.
#include <cuda_runtime.h>

#include "device.cuh"
#include "launch.h"

namespace dwp {

namespace {

template <int WARPS_, int CPL_, int ITEMS_>
struct RedConfig {
    static constexpr int kWarps = WARPS_;    // worker warps, two stages each
    static constexpr int kChunks = 32 * CPL_;  // chunks per tile (CPL per lane)
    static constexpr int kItems = ITEMS_;    // rows per chunk
    static constexpr int kTile = kChunks * ITEMS_;
    static constexpr int kThreads = WARPS_ * 32;
    static_assert(ITEMS_ % 4 == 0 && (ITEMS_ / 4) % 2 == 1, "ITEMS must be an odd multiple of 4");
    static constexpr size_t kStageBytes = size_t(kTile) * 4;
    static constexpr int kPrefixWords = kChunks + kChunks / 8;
    // per warp: 2 stages; 2 mbarriers; chunk prefixes; 33 lane totals
    static constexpr size_t kWarpBytes = 2 * kStageBytes + 16 + 4 * size_t(kPrefixWords + 33 + 3);
    static constexpr size_t kSmemBytes = kWarpBytes * WARPS_;
    static_assert(kWarpBytes % 16 == 0, "stages must stay 16-byte aligned");
    static_assert(kSmemBytes <= 232448, "more than 227 KiB of shared memory per block");
};

#ifndef DWP_RED_WARPS
#define DWP_RED_WARPS 8
#endif
#ifndef DWP_RED_CPL
#define DWP_RED_CPL 8
#endif
#ifndef DWP_RED_ITEMS
#define DWP_RED_ITEMS 12
#endif
using RedCfg = RedConfig<DWP_RED_WARPS, DWP_RED_CPL, DWP_RED_ITEMS>;

template <class C>
struct RedSmem {
    unsigned char *w;  // this warp's region
    __device__ RedSmem(unsigned char *base, uint32_t warp) : w(base + size_t(warp) * C::kWarpBytes) {}
    __device__ uint32_t *stage(int j) const {
        return reinterpret_cast<uint32_t *>(w + size_t(j) * C::kStageBytes);
    }
    __device__ uint64_t *full(int j) const {
        return reinterpret_cast<uint64_t *>(w + 2 * C::kStageBytes) + j;
    }
    __device__ uint32_t *pre() const {
        return reinterpret_cast<uint32_t *>(w + 2 * C::kStageBytes + 16);
    }
    __device__ uint32_t *lane_tot() const { return pre() + C::kPrefixWords; }
};

template <class C>
__global__ void __launch_bounds__(C::kThreads, 1)
    segreduce_kernel(const uint32_t *in, const uint32_t *off, uint32_t nseg, uint32_t *out,
                     uint64_t n, uint32_t num_tiles, ScratchHeader *hdr) {
    constexpr int TILE = C::kTile, ITEMS = C::kItems, CPL = C::kChunks / 32;
    extern __shared__ __align__(128) unsigned char smem_raw[];
    const uint32_t warp = threadIdx.x >> 5, lane = threadIdx.x & 31u;
    const RedSmem<C> sm(smem_raw, warp);
    if (lane == 0) {
        mbar_init(sm.full(0), 1);
        mbar_init(sm.full(1), 1);
        fence_mbar_init();
    }
    __syncwarp();
    // shared memory only so far; the kernel before may still be running.
    // No early trigger: the next kernel launches as the blocks exit (an
    // early one measured slower for this persistent kernel)
    pdl_wait();

    // take a tile index and start its bulk copy into stage j (lane 0 only)
    auto start = [&](int j) -> uint32_t {
        uint32_t t = atomicAdd(&hdr->tile_counter, 1u);
        if (t >= num_tiles) return kNoTile;
        const uint64_t rem = n - uint64_t(t) * TILE;
        const uint32_t valid = rem < uint64_t(TILE) ? uint32_t(rem) : uint32_t(TILE);
        const uint32_t bulk = valid == uint32_t(TILE) ? valid : (valid & ~3u);
        if (bulk && in_bounds(hdr, uint64_t(t) * TILE, bulk, n) && in_bounds(hdr, 0, bulk, TILE)) {
            mbar_arrive_expect_tx(sm.full(j), bulk * 4u);
            bulk_load_hint(sm.stage(j), in + uint64_t(t) * TILE, bulk * 4u, sm.full(j),
                           l2_policy_evict_first());
        } else {
            mbar_arrive(sm.full(j));
        }
        return t;
    };

    uint32_t next = lane == 0 ? start(0) : 0u;
    next = __shfl_sync(0xffffffffu, next, 0);
    for (uint32_t it = 0; next != kNoTile; ++it) {
        const int j = int(it & 1u);
        const uint32_t t = next;
        // the other stage was read completely by the previous iteration
        fence_proxy_async_smem();
        __syncwarp();
        next = lane == 0 ? start(j ^ 1) : 0u;
        next = __shfl_sync(0xffffffffu, next, 0);

        const uint64_t b = uint64_t(t) * TILE;
        const uint64_t rem = n - b;
        const uint32_t valid = rem < uint64_t(TILE) ? uint32_t(rem) : uint32_t(TILE);
        const uint32_t bulk = valid == uint32_t(TILE) ? valid : (valid & ~3u);
        const uint64_t e = b + valid;
        // segments overlapping [b, e): from the one holding row b (the last
        // offset <= b) to the last one starting before e
        const uint32_t k1 = warp_lower_bound(off, 0u, nseg + 1u, uint32_t(b + 1), lane);
        const uint32_t k2 = warp_lower_bound(off, k1, nseg + 1u, uint32_t(e), lane);
        const uint32_t s_lo = k1 > 0u ? k1 - 1u : 0u;
        const uint32_t s_hi = min(k2, nseg);  // exclusive

        if (!__all_sync(0xffffffffu, mbar_wait(sm.full(j), (it >> 1) & 1u, kPipeWaitLimit))) {
            if (lane == 0) record_error(hdr, DWP_ERR_PIPELINE_TIMEOUT);
            // Drain before the block retires: this copy and the one already
            // started into the other stage may still be writing shared
            // memory.  Each wait is bounded; after that the warp leaves.
            mbar_wait(sm.full(j), (it >> 1) & 1u, kPipeWaitLimit);
            if (next != kNoTile) mbar_wait(sm.full(j ^ 1), ((it + 1) >> 1) & 1u, kPipeWaitLimit);
            return;
        }
        const uint32_t *buf = sm.stage(j);
        auto row = [&](uint32_t q) -> uint32_t {  // row b + q of the tile
            if (q < bulk) return buf[q];
            if (q < valid && in_bounds(hdr, b + q, 1, n)) return in[b + q];
            return 0u;
        };
        uint32_t *pre = sm.pre();
        uint32_t *lt = sm.lane_tot();
        // chunk totals: lane handles chunks lane + 32*w2
#pragma unroll
        for (int w2 = 0; w2 < CPL; ++w2) {
            const uint32_t c = lane + 32u * w2;
            uint32_t acc = 0;
            if (valid == uint32_t(TILE)) {
                const uint4 *v4 = reinterpret_cast<const uint4 *>(buf) + c * (ITEMS / 4);
#pragma unroll
                for (int v = 0; v < ITEMS / 4; ++v) {
                    const uint4 q = v4[v];
                    acc += (q.x + q.y) + (q.z + q.w);
                }
            } else {
                for (int i = 0; i < ITEMS; ++i) acc += row(c * ITEMS + i);
            }
            pre[prefix_slot(c)] = acc;
        }
        __syncwarp();
        // exclusive prefix of the chunk totals: lane l takes CPL consecutive
        // chunks, then the 32 lane totals are folded through shared memory
        uint32_t mine[CPL], run = 0;
#pragma unroll
        for (int q = 0; q < CPL; ++q) {
            mine[q] = run;
            run += pre[prefix_slot(lane * CPL + q)];
        }
        lt[lane] = run;
        __syncwarp();
        uint32_t lane_excl = 0;
#pragma unroll
        for (int l = 0; l < 32; ++l)
            if (uint32_t(l) < lane) lane_excl += lt[l];
#pragma unroll
        for (int q = 0; q < CPL; ++q) pre[prefix_slot(lane * CPL + q)] = lane_excl + mine[q];
        __syncwarp();
        // inclusive prefix of the tile at row b + q
        auto prefix = [&](uint32_t q) -> uint32_t {
            const uint32_t c = q / ITEMS, r = q - c * ITEMS;
            uint32_t p = pre[prefix_slot(c)];
            for (uint32_t i = 0; i <= r; ++i) p += row(c * ITEMS + i);
            return p;
        };
        for (uint32_t s0 = s_lo; s0 < s_hi; s0 += 32u) {
            const uint32_t s = s0 + lane;
            if (s < s_hi && in_bounds(hdr, s, 2, uint64_t(nseg) + 1)) {
                const uint64_t o0 = __ldg(off + s), o1 = __ldg(off + s + 1);
                const uint64_t lo = o0 > b ? o0 : b;
                const uint64_t hi = o1 < e ? o1 : e;
                if (hi > lo && in_bounds(hdr, s, 1, nseg)) {
                    uint32_t sum = prefix(uint32_t(hi - 1 - b));
                    if (lo > b) sum -= prefix(uint32_t(lo - 1 - b));
                    if (o0 >= b && o1 <= e)
                        out[s] = sum;  // the whole segment lies in this tile
                    else
                        atomicAdd(out + s, sum);
                }
            }
        }
        __syncwarp();
    }
    // no bulk copy of this warp may still be writing shared memory: the last
    // start() returned no tile, so every started copy was waited for above
}

}  // namespace

uint32_t segreduce_tile_elems() { return RedCfg::kTile; }

cudaError_t launch_segreduce(const uint32_t *values, const uint32_t *offsets, uint32_t nseg,
                             uint32_t *out, uint64_t n, void *scratch, cudaStream_t stream) {
    using C = RedCfg;
    auto kern = segreduce_kernel<C>;
    const int dev_blocks = device_blocks(reinterpret_cast<const void *>(kern), C::kThreads,
                                         C::kSmemBytes);
    if (dev_blocks <= 0) return cudaErrorInvalidConfiguration;
    const uint64_t tiles = (n + C::kTile - 1) / C::kTile;
    const uint64_t warps_needed = (tiles + 1) / 2;
    const uint64_t blocks_needed = (warps_needed + C::kWarps - 1) / C::kWarps;
    const uint32_t grid = uint32_t(blocks_needed < uint64_t(dev_blocks) ? blocks_needed
                                                                         : uint64_t(dev_blocks));
    auto *hdr = reinterpret_cast<ScratchHeader *>(scratch);
    return launch_pdl(kern, dim3(grid), dim3(C::kThreads), C::kSmemBytes, stream, values, offsets,
                      nseg, out, n, uint32_t(tiles), hdr);
}

}  // namespace dwp
