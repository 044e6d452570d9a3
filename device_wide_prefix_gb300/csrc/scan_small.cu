// Single-pass chained scan with decoupled look-back for small inputs, sm_103a.
//
// The same method as scan.cu ("Single-Pass Prefix Scan with Decoupled
// Look-Back"; "Parallel Prefix Sum (Scan), in depth", sections "A CUDA scan:
// warp, block, grid" and "Scanning a whole array: three grid strategies"),
// with the same descriptors, look-back, Decoupled Fallback, bounded window
// and test hooks, shaped for latency instead of bandwidth.  Up to a few
// million elements the input sits in the 129 MB L2 and a call is a chain of
// latencies: the persistent kernel's hand-offs between its producer,
// reducer, look-back, reloader and consumer warps add up to more than the
// data takes to move.  Here one block owns one tile from load to store:
//   1. thread 0 takes the tile index from the atomic counter (tiles start in
//      index order, so a tile only waits for tiles running blocks hold) and
//      starts one bulk (TMA) copy of the tile into shared memory;
//   2. each of the 256 threads reads its ITEMS contiguous elements from
//      shared memory as 16-byte vectors into registers and reduces them
//      serially (thread layer).  ITEMS is an odd multiple of 4, so the
//      vectors of a quarter warp fall in 8 distinct bank groups;
//   3. a shuffle Hillis-Steele scan over the warp's 32 thread totals (warp
//      layer) and the 8 warp totals through shared memory (block layer) give
//      every thread its exclusive prefix in the tile and the tile aggregate;
//   4. the aggregate is published (tile 0: its inclusive prefix); warp 0
//      looks back and publishes the inclusive prefix;
//   5. every thread scans its registers from carry + its prefix into the
//      stage, and thread 0 writes the tile back with one bulk store.
// One block per tile, so the grid is the tile count.  A per-tile
// %globaltimer trace on GB300 chose the shape: thread-contiguous loads
// straight from global memory took 2.4 us for 64 elements a thread (every
// 16-byte load of a warp touches 32 lines), the bulk copy moves the tile in
// one request; and the look-back's wait after the last aggregate appears
// grew with the number of tiles polling at once (about 1 us with 64 tiles,
// 2.5 us with 256, 9 us with 1024), so tiles grow with n to keep their
// count low.
#include <cuda_runtime.h>

#include "device.cuh"
#include "launch.h"

namespace dwp {

namespace {

constexpr int kSmallThreads = 256;
constexpr int kSmallWarps = kSmallThreads / 32;

// Look-back sub-windows of 32 per poll.  Every tile of a small input starts
// at about the same time, so most look-backs fold aggregates back to tile 0
// rather than stop at a recent prefix: a poll covers 32 K predecessors.
__host__ __device__ constexpr int small_look_k(int items) { return items <= 12 ? 4 : 8; }
static_assert(kSmallThreads == 256, "tile sizes below assume 256 threads");

// Dynamic shared memory: the tile stage, then the mbarrier.
template <int ITEMS>
struct SmallSmem {
    static constexpr uint32_t kTile = uint32_t(kSmallThreads) * ITEMS;
    static constexpr size_t kStageBytes = size_t(kTile) * 4;
    static constexpr size_t kBytes = kStageBytes + 16;
};

template <class Op, bool INCL, int ITEMS>
__global__ void __launch_bounds__(kSmallThreads, 2)
    scan_small_kernel(const typename Op::T *in, typename Op::T *out, uint64_t n,
                      uint32_t num_tiles, ScratchHeader *hdr, uint64_t *desc, LaunchKnobs fault) {
    using T = typename Op::T;
    static_assert(ITEMS % 4 == 0 && (ITEMS / 4) % 2 == 1, "ITEMS must be an odd multiple of 4");
    constexpr uint32_t TILE = SmallSmem<ITEMS>::kTile;
    extern __shared__ __align__(128) unsigned char smem_raw[];
    uint32_t *stage = reinterpret_cast<uint32_t *>(smem_raw);
    uint64_t *full = reinterpret_cast<uint64_t *>(smem_raw + SmallSmem<ITEMS>::kStageBytes);
    __shared__ uint32_t s_tile, s_ok, s_carry, s_rc;
    __shared__ uint32_t s_wtot[kSmallWarps];
    const uint32_t warp = threadIdx.x >> 5, lane = threadIdx.x & 31u;
    if (threadIdx.x == 0) {
        mbar_init(full, 1);
        fence_mbar_init();
    }
    pdl_wait();  // the kernel before (the scratch clear) may still be running

    uint32_t valid = 0, bulk = 0;
    if (threadIdx.x == 0) {
        const uint32_t t = atomicAdd(&hdr->tile_counter, 1u);
        s_tile = t;
        if (t < num_tiles) {
            perturb(fault, t, kSiteDraw);
            const uint64_t rem = n - uint64_t(t) * TILE;
            valid = rem < uint64_t(TILE) ? uint32_t(rem) : TILE;
            bulk = valid & ~3u;  // the bulk copy moves whole 16-byte vectors
            if (bulk && in_bounds(hdr, uint64_t(t) * TILE, bulk, n) && in_bounds(hdr, 0, bulk, TILE)) {
                mbar_arrive_expect_tx(full, bulk * 4u);
                bulk_load(stage, in + uint64_t(t) * TILE, bulk * 4u, full);
            } else {
                mbar_arrive(full);
            }
            // wait here, bounded; on a timeout wait once more (the copy may
            // still be writing shared memory) and give the tile up
            bool ok = mbar_wait(full, 0, kPipeWaitLimit);
            if (!ok) {
                mbar_wait(full, 0, kPipeWaitLimit);
                if (in_bounds(hdr, t, 1, num_tiles)) st_relaxed_gpu(desc + t, make_desc(kPoison, 0u));
                record_error(hdr, DWP_ERR_PIPELINE_TIMEOUT);
            }
            s_ok = ok ? 1u : 0u;
        }
    }
    __syncthreads();
    const uint32_t t = s_tile;
    if (t >= num_tiles || s_ok == 0u) return;  // the first is not reached: grid = tile count
    {
        const uint64_t rem = n - uint64_t(t) * TILE;
        valid = rem < uint64_t(TILE) ? uint32_t(rem) : TILE;
        bulk = valid & ~3u;
    }
    const uint64_t base = uint64_t(t) * TILE;

    // -- thread layer: ITEMS contiguous elements into registers -----------
    const uint32_t p0 = threadIdx.x * ITEMS;
    const uint4 *sv = reinterpret_cast<const uint4 *>(stage + p0);
    T v[ITEMS];
#pragma unroll
    for (int q = 0; q < ITEMS / 4; ++q) {
        const uint32_t pos = p0 + 4u * q;
        uint4 w;
        if (pos < bulk) {
            w = sv[q];
        } else {  // the 1-3 elements past the bulk part, and the identity past the end
            uint32_t e[4];
#pragma unroll
            for (int j = 0; j < 4; ++j)
                e[j] = pos + j < valid && in_bounds(hdr, base + pos + j, 1, n) ? Op::to_bits(in[base + pos + j])
                                                                                 : Op::to_bits(Op::identity());
            w = make_uint4(e[0], e[1], e[2], e[3]);
        }
        v[4 * q + 0] = Op::from_bits(w.x);
        v[4 * q + 1] = Op::from_bits(w.y);
        v[4 * q + 2] = Op::from_bits(w.z);
        v[4 * q + 3] = Op::from_bits(w.w);
    }
    T tot = Op::identity();
#pragma unroll
    for (int j = 0; j < ITEMS; ++j) tot = Op::combine(tot, v[j]);

    // -- warp layer: inclusive Hillis-Steele over the 32 thread totals ----
    T incl = tot;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        const T u = __shfl_up_sync(0xffffffffu, incl, d);
        if (lane >= uint32_t(d)) incl = Op::combine(u, incl);
    }
    const T up = __shfl_up_sync(0xffffffffu, incl, 1);
    const T excl_in_warp = lane > 0 ? up : Op::identity();
    if (lane == 31) s_wtot[warp] = Op::to_bits(incl);
    __syncthreads();

    // -- block layer: the 8 warp totals (broadcast reads) ----------------
    T wpre = Op::identity(), agg = Op::identity();
#pragma unroll
    for (int w = 0; w < kSmallWarps; ++w) {
        const T x = Op::from_bits(s_wtot[w]);
        if (uint32_t(w) < warp) wpre = Op::combine(wpre, x);
        agg = Op::combine(agg, x);
    }

    // -- publish the aggregate, look back, publish the prefix -------------
    if (warp == 0) {
        perturb(fault, t, kSiteAggregate);
        if (lane == 0 && t != fault.never_publish_tile && in_bounds(hdr, t, 1, num_tiles))
            st_relaxed_gpu(desc + t, make_desc(t == 0 ? kPrefix : kAggregate, Op::to_bits(agg)));
        perturb(fault, t, kSiteLookback);
        T carry = Op::identity();
        int rc = 0;
        if (t != 0)
            rc = lookback<Op, small_look_k(ITEMS)>(desc, t, lane, fault.spin_limit,
                                                   fault.fallback_polls,
                                                   ScanRescue<Op, int(TILE)>{in, n}, hdr,
                                                   fault.lookback_window, Op::to_bits(agg),
                                                   t != fault.never_publish_tile, &carry);
        if (rc == 0) perturb(fault, t, kSitePrefix);
        if (lane == 0) {
            if (!in_bounds(hdr, t, 1, num_tiles)) {
                // debug bounds build only: no descriptor to publish
            } else if (rc == 0) {
                if (t != 0 && t != fault.never_publish_tile)
                    st_relaxed_gpu(desc + t, make_desc(kPrefix, Op::to_bits(Op::combine(carry, agg))));
            } else {
                // give up on this tile: poison it so no successor waits
                st_relaxed_gpu(desc + t, make_desc(kPoison, 0u));
                if (rc == 2) record_error(hdr, DWP_ERR_LOOKBACK_TIMEOUT);
            }
            s_carry = Op::to_bits(carry);
            s_rc = uint32_t(rc);
        }
    }
    __syncthreads();
    if (s_rc != 0u) return;  // the output of an abandoned tile is not written

    // -- scan the registers from carry + prefix into the stage; one bulk
    //    store (per-warp stores measured no faster)
    T run = Op::combine(Op::combine(Op::from_bits(s_carry), wpre), excl_in_warp);
    uint4 *dv = reinterpret_cast<uint4 *>(stage + p0);
#pragma unroll
    for (int q = 0; q < ITEMS / 4; ++q) {
        uint32_t y[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            if (INCL) {
                run = Op::combine(run, v[4 * q + j]);
                y[j] = Op::to_bits(run);
            } else {
                y[j] = Op::to_bits(run);
                run = Op::combine(run, v[4 * q + j]);
            }
        }
        const uint32_t pos = p0 + 4u * q;
        if (pos < bulk) {
            dv[q] = make_uint4(y[0], y[1], y[2], y[3]);
        } else {
#pragma unroll
            for (int j = 0; j < 4; ++j)
                if (pos + j < valid && in_bounds(hdr, base + pos + j, 1, n))
                    out[base + pos + j] = Op::from_bits(y[j]);
        }
    }
    fence_proxy_async_smem();  // the bulk store reads the stage through the async proxy
    __syncthreads();
    if (threadIdx.x == 0 && bulk && in_bounds(hdr, base, bulk, n)) {
        bulk_store(out + base, stage, bulk * 4u);
        bulk_commit();
        bulk_wait_all<0>();
    }
}

template <class Op, bool INCL, int ITEMS>
cudaError_t launch_small_items(const void *in, void *out, uint64_t n, void *scratch,
                               cudaStream_t stream, const LaunchKnobs &fault) {
    using S = SmallSmem<ITEMS>;
    auto kern = scan_small_kernel<Op, INCL, ITEMS>;
    if (device_blocks(reinterpret_cast<const void *>(kern), kSmallThreads, S::kBytes) <= 0)
        return cudaErrorInvalidConfiguration;  // also raises the kernel's shared-memory limit
    const uint64_t tiles = (n + S::kTile - 1) / S::kTile;
    auto *hdr = reinterpret_cast<ScratchHeader *>(scratch);
    auto *desc = reinterpret_cast<uint64_t *>(static_cast<unsigned char *>(scratch) + kHeaderBytes);
    return launch_pdl(kern, dim3(uint32_t(tiles)), dim3(kSmallThreads), S::kBytes, stream,
                      reinterpret_cast<const typename Op::T *>(in),
                      reinterpret_cast<typename Op::T *>(out), n, uint32_t(tiles), hdr, desc, fault);
}

// Tile sizes grow with n in three tiers, so the number of tiles polling the
// descriptors at once stays low: 256 * 12 = 3072 elements up to 2^18 (at
// most 86 tiles), 256 * 28 = 7168 up to 2^20 (at most 147), 256 * 60 = 15360
// above (at most 547 up to 2^23).
#ifndef DWP_SMALL_TIER1_LOG2
#define DWP_SMALL_TIER1_LOG2 18
#endif
#ifndef DWP_SMALL_TIER2_LOG2
#define DWP_SMALL_TIER2_LOG2 20
#endif
constexpr uint64_t kSmallTier1 = uint64_t(1) << DWP_SMALL_TIER1_LOG2;
constexpr uint64_t kSmallTier2 = uint64_t(1) << DWP_SMALL_TIER2_LOG2;

template <class Op, bool INCL>
cudaError_t launch_small(const void *in, void *out, uint64_t n, void *scratch, cudaStream_t stream,
                         const LaunchKnobs &fault) {
    if (n <= kSmallTier1) return launch_small_items<Op, INCL, 12>(in, out, n, scratch, stream, fault);
    if (n <= kSmallTier2) return launch_small_items<Op, INCL, 28>(in, out, n, scratch, stream, fault);
    return launch_small_items<Op, INCL, 60>(in, out, n, scratch, stream, fault);
}

}  // namespace

uint64_t scan_small_descriptors(uint64_t n) {
    // at least the tile count, and never fewer than the largest count of a
    // lower tier, so the size query does not shrink as n grows
    constexpr uint64_t t1 = SmallSmem<12>::kTile, t2 = SmallSmem<28>::kTile, t3 = SmallSmem<60>::kTile;
    constexpr uint64_t max1 = (kSmallTier1 + t1 - 1) / t1;
    constexpr uint64_t max2 = (kSmallTier2 + t2 - 1) / t2 > max1 ? (kSmallTier2 + t2 - 1) / t2 : max1;
    if (n <= kSmallTier1) return (n + t1 - 1) / t1;
    if (n <= kSmallTier2) {
        const uint64_t tiles = (n + t2 - 1) / t2;
        return tiles > max1 ? tiles : max1;
    }
    const uint64_t tiles = (n + t3 - 1) / t3;
    return tiles > max2 ? tiles : max2;
}

cudaError_t launch_scan_small(dwp_op op, bool inclusive, const void *in, void *out, uint64_t n,
                              void *scratch, cudaStream_t stream, const LaunchKnobs &fault) {
    switch (op) {
        case DWP_U32_ADD:
            return inclusive ? launch_small<OpU32Add, true>(in, out, n, scratch, stream, fault)
                             : launch_small<OpU32Add, false>(in, out, n, scratch, stream, fault);
        case DWP_F32_ADD:
            return inclusive ? launch_small<OpF32Add, true>(in, out, n, scratch, stream, fault)
                             : launch_small<OpF32Add, false>(in, out, n, scratch, stream, fault);
        case DWP_U32_MAX:
            return inclusive ? launch_small<OpU32Max, true>(in, out, n, scratch, stream, fault)
                             : launch_small<OpU32Max, false>(in, out, n, scratch, stream, fault);
    }
    return cudaErrorInvalidValue;
}

}  // namespace dwp
