// Single-pass chained scan with decoupled look-back for sm_103a.
//
// One persistent, warp-specialised launch ("Single-Pass Prefix Scan with
// Decoupled Look-Back"; "Parallel Prefix Sum (Scan), in depth", sections "A
// CUDA scan: warp, block, grid" and "Scanning a whole array: three grid
// strategies").  Per block:
//
//   producer warp    takes tile indices from the atomic counter in the order
//                    tiles start, AHEAD iterations before their load, and asks
//                    L2 to prefetch each tile when it takes it; when an input
//                    stage frees up it streams the tile global -> shared with
//                    one bulk (TMA) copy into a ring of SIN input stages;
//   reducer warps    one per input stage.  For its tile: every consumer
//                    thread's total and their exclusive prefix (block
//                    layer), written to a slot of the tile-info ring; the
//                    aggregate published at once; the input stage freed;
//   look-back warps  LW of them, iteration k taken by warp k % LW: the
//                    look-back, the inclusive prefix published, the carry
//                    written to the tile's info slot;
//   reloader warp    once a tile's carry is known, brings the tile back with
//                    one bulk copy into a ring of SOUT output stages.  The
//                    tile was read from HBM some microseconds earlier and
//                    still sits in the L2 (129 MB), so this copy costs L2
//                    bandwidth, not HBM bandwidth.  For that the first load
//                    marks the tile's lines evict-last, the reload and the
//                    output stores evict-first (without the hints about 60%
//                    of the reloads missed L2 and went back to HBM);
//   consumer warps   warp w owns chunk w of every tile; each thread scans its
//                    ITEMS contiguous elements serially from carry + its
//                    in-tile prefix, writes them back in place, and the warp
//                    streams its chunk shared -> global with one bulk store.
//
// Why the reload: a tile cannot finish before every earlier tile has
// published its aggregate, and tiles land from HBM out of order by several
// microseconds, so the look-back of a tile waits a few microseconds.  Held
// in shared memory for that wait, the tiles in flight per SM exceeded shared
// memory at full bandwidth; held in L2 they do not.  Shared memory now holds
// a tile only while it is reduced and while it is scanned and stored.
//
// Why the prefetch: with the reload in place the producer spent over 90% of
// its waiting time on a free input stage, because a bulk load straight from
// HBM held its stage for about 3 us.  Prefetched into L2 two iterations
// early, the load finds most of the tile there and the stage turns over
// faster, so two input stages do the work of three and more.  The lead is
// short on purpose: a tile whose index is taken early publishes its
// aggregate later, and every later tile's look-back waits for it (leads of
// 4 to 10 iterations were slower than no lead at all).
//
// ITEMS is an odd multiple of 4, so the 16-byte shared-memory accesses of a
// quarter warp (thread stride 16*odd bytes) fall in 8 distinct bank groups.
// No block-wide barrier is used after set-up: warps meet only at mbarriers,
// and every wait is bounded.
#include <cuda_runtime.h>

#include "device.cuh"
#include "launch.h"

namespace dwp {

template <int NW_, int ITEMS_, int SIN_, int SOUT_, int RING_, int LW_, int LOOKK_, int AHEAD_>
struct ScanConfig {
    static constexpr int kWarps = NW_;       // consumer warps (one chunk of the tile each)
    static constexpr int kItems = ITEMS_;    // contiguous elements per consumer thread
    static constexpr int kIn = SIN_;         // input stages = reducer warps
    static constexpr int kOut = SOUT_;       // output stages
    static constexpr int kRing = RING_;      // tile-info slots
    static constexpr int kLookers = LW_;     // look-back warps
    static constexpr int kLookK = LOOKK_;    // look-back sub-windows of 32 per poll
    static constexpr int kAhead = AHEAD_;    // iterations a tile index is drawn before its load
    static constexpr int kThreads = (2 + SIN_ + LW_ + NW_) * 32;
    static constexpr int kConsumers = NW_ * 32;
    static constexpr int kWarpElems = 32 * ITEMS_;
    static constexpr int kTile = NW_ * 32 * ITEMS_;
    static_assert(ITEMS_ % 4 == 0 && (ITEMS_ / 4) % 2 == 1, "ITEMS must be an odd multiple of 4");
    static_assert(NW_ >= 1 && NW_ <= 32, "one 32-slot row of thread totals per consumer warp");
    static_assert(RING_ % LW_ == 0, "a look-back warp must own every use of its info slots");
    static_assert(SOUT_ >= 2, "the reloader waits for the output stage of iteration k - SOUT");
    static_assert(RING_ >= SIN_ + SOUT_ + 2 + AHEAD_, "info ring shorter than the work in flight");
    static constexpr size_t kStageBytes = size_t(kTile) * 4;
    static constexpr int kPrefixWords = kConsumers + kConsumers / 8;
    // info slot: 4 mbarriers (32 B); tile id, aggregate, carry,
    // look-back result (16 B); thread prefixes
    static constexpr size_t kInfoBytes = 48 + 4 * kPrefixWords;
    // per-reducer scratch after the barriers: 33 lane totals
    static constexpr size_t kWarpScratchBytes = 4 * 33 * SIN_;
    // stage barriers: per input stage full + empty, per output stage ready + empty
    static constexpr size_t kBarBytes = 16 * (SIN_ + SOUT_);
    static constexpr size_t kSmemBytes =
        kStageBytes * (SIN_ + SOUT_) + kInfoBytes * RING_ + kBarBytes + 16 + kWarpScratchBytes;
    static_assert(kThreads <= 1024, "more than 1024 threads per block");
    static_assert(kSmemBytes <= 232448, "more than 227 KiB of shared memory per block");
};

#ifndef DWP_SCAN_WARPS
#define DWP_SCAN_WARPS 8
#endif
#ifndef DWP_SCAN_ITEMS
#define DWP_SCAN_ITEMS 28
#endif
#ifndef DWP_SCAN_IN
#define DWP_SCAN_IN 2
#endif
#ifndef DWP_SCAN_OUT
#define DWP_SCAN_OUT 4
#endif
#ifndef DWP_SCAN_RING
#define DWP_SCAN_RING 16
#endif
#ifndef DWP_SCAN_LOOKERS
#define DWP_SCAN_LOOKERS 16
#endif
#ifndef DWP_SCAN_LOOKK
#define DWP_SCAN_LOOKK 1
#endif
#ifndef DWP_SCAN_AHEAD
#define DWP_SCAN_AHEAD 2
#endif
// look-back back-off: sleep DWP_SCAN_LB_NS before every poll after the
// first DWP_SCAN_LB_AFTER.  A look-back here starts when its tile is drawn
// and polls while the tile loads; polling less often measured 7% faster at
// 2^24 and 3.5% at 2^26 than the default (8 polls, then 64 ns)
#ifndef DWP_SCAN_LB_AFTER
#define DWP_SCAN_LB_AFTER 0
#endif
#ifndef DWP_SCAN_LB_NS
#define DWP_SCAN_LB_NS 128
#endif
using ScanCfg = ScanConfig<DWP_SCAN_WARPS, DWP_SCAN_ITEMS, DWP_SCAN_IN, DWP_SCAN_OUT,
                           DWP_SCAN_RING, DWP_SCAN_LOOKERS, DWP_SCAN_LOOKK, DWP_SCAN_AHEAD>;

// Shared-memory layout of one block.
template <class C>
struct ScanSmem {
    unsigned char *base;
    __device__ explicit ScanSmem(unsigned char *p) : base(p) {}
    __device__ uint32_t *in_data(int s) const {
        return reinterpret_cast<uint32_t *>(base + size_t(s) * C::kStageBytes);
    }
    __device__ uint32_t *out_data(int o) const {
        return reinterpret_cast<uint32_t *>(base + size_t(C::kIn + o) * C::kStageBytes);
    }
    __device__ unsigned char *info(int i) const {
        return base + C::kStageBytes * (C::kIn + C::kOut) + size_t(i) * C::kInfoBytes;
    }
    __device__ uint64_t *info_ready(int i) const { return reinterpret_cast<uint64_t *>(info(i)); }
    __device__ uint64_t *carry_ready(int i) const { return info_ready(i) + 1; }
    __device__ uint64_t *info_free(int i) const { return info_ready(i) + 2; }
    // the producer has written tile_id(i) (the tile is drawn)
    __device__ uint64_t *id_ready(int i) const { return info_ready(i) + 3; }
    __device__ uint32_t *tile_id(int i) const { return reinterpret_cast<uint32_t *>(info(i) + 32); }
    __device__ uint32_t *agg(int i) const { return tile_id(i) + 1; }
    __device__ uint32_t *carry(int i) const { return tile_id(i) + 2; }
    __device__ uint32_t *lbres(int i) const { return tile_id(i) + 3; }
    __device__ uint32_t *prefix(int i) const { return tile_id(i) + 4; }

    __device__ uint64_t *bars() const {
        return reinterpret_cast<uint64_t *>(base + C::kStageBytes * (C::kIn + C::kOut) +
                                            C::kInfoBytes * C::kRing);
    }
    __device__ uint64_t *in_full(int s) const { return bars() + s; }
    __device__ uint64_t *in_empty(int s) const { return bars() + C::kIn + s; }
    __device__ uint64_t *out_full(int o) const { return bars() + 2 * C::kIn + o; }
    __device__ uint64_t *out_empty(int o) const { return bars() + 2 * C::kIn + C::kOut + o; }
    __device__ uint32_t *abort_flag() const {
        return reinterpret_cast<uint32_t *>(bars() + 2 * (C::kIn + C::kOut));
    }
    // first ring iteration that holds no tile (set once by the producer)
    __device__ uint32_t *end_iter() const { return abort_flag() + 1; }
    // reducer r's 33 lane totals
    __device__ uint32_t *lane_tot(int r) const { return abort_flag() + 4 + 33 * r; }
};

// Elements pos .. pos+3 of a tile as one vector when they lie past the
// bulk-copied part: from global memory below `valid`, the identity (bit
// pattern 0 for every operator here) past it.  Only the 1-3 elements after
// a ragged tile's bulk part come this way.
template <class Op>
__device__ __forceinline__ uint4 tail_vec(const typename Op::T *in, uint64_t base, uint32_t pos,
                                          uint32_t valid, ScratchHeader *hdr, uint64_t n) {
    uint32_t w[4];
#pragma unroll
    for (int e = 0; e < 4; ++e)
        w[e] = pos + e < valid && in_bounds(hdr, base + pos + e, 1, n) ? Op::to_bits(in[base + pos + e])
                                                                      : Op::to_bits(Op::identity());
    return make_uint4(w[0], w[1], w[2], w[3]);
}

template <class Op, bool INCL, class C>
__global__ void __launch_bounds__(C::kThreads, 1)
    scan_kernel(const typename Op::T *in, typename Op::T *out, uint64_t n, uint32_t num_tiles,
                ScratchHeader *hdr, uint64_t *desc, LaunchKnobs fault) {
    using T = typename Op::T;
    constexpr int NW = C::kWarps, ITEMS = C::kItems, TILE = C::kTile;
    constexpr int SIN = C::kIn, SOUT = C::kOut, RING = C::kRing, LW = C::kLookers;
    constexpr int WE = C::kWarpElems;
    constexpr int AHEAD = C::kAhead;
    constexpr uint32_t NCONS = C::kConsumers;
    constexpr uint32_t kReducer0 = 1, kLooker0 = 1 + SIN, kReloader = 1 + SIN + LW,
                       kConsumer0 = 2 + SIN + LW;

    extern __shared__ __align__(128) unsigned char smem_raw[];
    const ScanSmem<C> sm(smem_raw);
    const uint32_t warp = threadIdx.x >> 5, lane = threadIdx.x & 31u;
    if (threadIdx.x == 0) {
        for (int s = 0; s < SIN; ++s) {
            mbar_init(sm.in_full(s), 1);
            mbar_init(sm.in_empty(s), 1);
        }
        for (int o = 0; o < SOUT; ++o) {
            mbar_init(sm.out_full(o), 1);
            mbar_init(sm.out_empty(o), NW);
        }
        for (int i = 0; i < RING; ++i) {
            mbar_init(sm.info_ready(i), 1);
            mbar_init(sm.carry_ready(i), 1);
            mbar_init(sm.info_free(i), NW);
            mbar_init(sm.id_ready(i), 1);
        }
        *sm.abort_flag() = 0;
        *sm.end_iter() = kNoTile;
        fence_mbar_init();
    }
    __syncthreads();
    // shared memory only so far; the kernel before may still be running.
    // No early trigger: the next kernel launches as the blocks exit (an
    // early one measured slower for this persistent kernel)
    pdl_wait();

    auto tile_extent = [&](uint32_t t, uint32_t &valid, uint32_t &bulk) {
        const uint64_t rem = n - uint64_t(t) * TILE;
        valid = rem < uint64_t(TILE) ? uint32_t(rem) : uint32_t(TILE);
        bulk = valid == uint32_t(TILE) ? valid : (valid & ~3u);
    };
    auto stop_at = [&](uint32_t k) {  // no ring iteration from k on holds a tile
        *reinterpret_cast<volatile uint32_t *>(sm.end_iter()) = k;
    };

    if (warp == 0) {
        // ------------------------------------------------------- producer
        // Tile indices come from the atomic counter in the order tiles start
        // ("Scanning a whole array: three grid strategies"), so a tile only
        // ever waits for tiles that some running block already holds. The
        // tile of iteration k is taken AHEAD iterations before its input
        // stage frees up and L2 is asked to fetch it meanwhile: the bulk load
        // then finds it there, and a stage is held for a shorter time.
        if (lane != 0) return;
        const uint64_t keep = l2_policy_evict_last();
        uint32_t taken = 0;  // iterations whose tile index has been drawn
        bool drawn_all = false;
        for (uint32_t k = 0;; ++k) {
            const int s = int(k % SIN), i = int(k % RING);
            bool ok = true;
            while (ok && !drawn_all && taken <= k + uint32_t(AHEAD)) {
                const uint32_t g = taken;
                const int gi = int(g % RING);
                if (g >= uint32_t(RING) &&
                    !mbar_wait(sm.info_free(gi), ((g / RING) - 1) & 1u, kPipeWaitLimit)) {
                    ok = false;
                    break;
                }
                uint32_t t = kNoTile;
                if (ld_volatile_smem(sm.abort_flag()) == 0) {
                    t = atomicAdd(&hdr->tile_counter, 1u);
                    if (t >= num_tiles) t = kNoTile;
                    else perturb(fault, t, kSiteDraw);
                }
                *reinterpret_cast<volatile uint32_t *>(sm.tile_id(gi)) = t;
                mbar_arrive(sm.id_ready(gi));  // the look-back may start now
                ++taken;
                if (t == kNoTile) {
                    // iteration g carries the sentinel down the pipeline;
                    // warps waiting for later iterations see end_iter < their k
                    drawn_all = true;
                    stop_at(g);
                } else if (AHEAD > 0) {
                    uint32_t valid, bulk;
                    tile_extent(t, valid, bulk);
                    if (bulk && in_bounds(hdr, uint64_t(t) * TILE, bulk, n))
                        bulk_prefetch_l2(in + uint64_t(t) * TILE, bulk * 4u, keep);
                }
            }
            if (ok && k >= uint32_t(SIN))
                ok = mbar_wait(sm.in_empty(s), ((k / SIN) - 1) & 1u, kPipeWaitLimit);
            if (!ok) {
                record_error(hdr, DWP_ERR_PIPELINE_TIMEOUT);
                // tiles drawn but never loaded: poison them so no successor waits
                for (uint32_t g = k; g < taken; ++g) {
                    const uint32_t t = ld_volatile_smem(sm.tile_id(int(g % RING)));
                    if (t != kNoTile && in_bounds(hdr, t, 1, num_tiles))
                        st_relaxed_gpu(desc + t, make_desc(kPoison, 0u));
                }
                stop_at(k - 1);  // buffers still in use: leave them alone
                return;
            }
            const uint32_t t = ld_volatile_smem(sm.tile_id(i));
            if (t == kNoTile) {
                mbar_arrive(sm.in_full(s));
                return;
            }
            uint32_t valid, bulk;
            tile_extent(t, valid, bulk);
            if (bulk && in_bounds(hdr, uint64_t(t) * TILE, bulk, n) && in_bounds(hdr, 0, bulk, TILE)) {
                mbar_arrive_expect_tx(sm.in_full(s), bulk * 4u);
                bulk_load_hint(sm.in_data(s), in + uint64_t(t) * TILE, bulk * 4u, sm.in_full(s), keep);
            } else {
                mbar_arrive(sm.in_full(s));
            }
        }
    }

    if (warp >= kReducer0 && warp < kLooker0) {
        // -------------------------------------------------------- reducers
        const int s = int(warp - kReducer0);
        for (uint32_t use = 0;; ++use) {
            const uint32_t k = use * SIN + uint32_t(s);
            const int i = int(k % RING);
            const int w = warp_wait_or_end(sm.in_full(s), use & 1u, k, sm.end_iter());
            if (w != 2) {
                if (w == 0 && lane == 0) record_error(hdr, DWP_ERR_PIPELINE_TIMEOUT);
                return;
            }
            const uint32_t t = ld_volatile_smem(sm.tile_id(i));
            if (t == kNoTile) {
                if (lane == 0) mbar_arrive(sm.info_ready(i));
                return;
            }
            if (ld_volatile_smem(sm.abort_flag()) != 0) {
                // an earlier tile of this block gave up: poison this one
                if (lane == 0) {
                    if (in_bounds(hdr, t, 1, num_tiles)) st_relaxed_gpu(desc + t, make_desc(kPoison, 0u));
                    *sm.lbres(i) = 1u;
                    mbar_arrive(sm.in_empty(s));
                    mbar_arrive(sm.info_ready(i));
                }
                __syncwarp();
                continue;
            }
            uint32_t valid, bulk;
            tile_extent(t, valid, bulk);
            const uint64_t base = uint64_t(t) * TILE;
            const uint32_t *buf = sm.in_data(s);
            uint32_t *pre = sm.prefix(i);
            uint32_t *lt = sm.lane_tot(s);
            // totals of consumer threads c = lane + 32*w, whose ITEMS
            // contiguous elements start at c*ITEMS, read as 16-byte vectors
            // from the stage (the bulk part is a multiple of 4 elements, so
            // a vector lies wholly inside it or wholly past it).  In a
            // ragged last tile the 1-3 elements past the bulk part come from
            // global memory, and threads wholly past the end add nothing.
            T tot[NW];
            const uint4 *v4 = reinterpret_cast<const uint4 *>(buf);
            if (valid == uint32_t(TILE)) {  // every tile but a ragged last one
#pragma unroll
                for (int w2 = 0; w2 < NW; ++w2) {
                    const uint32_t c = lane + 32u * w2;
                    T acc = Op::identity();
#pragma unroll
                    for (int v = 0; v < ITEMS / 4; ++v) {
                        const uint4 q = v4[c * (ITEMS / 4) + v];
                        acc = Op::combine(acc, Op::combine(Op::combine(Op::from_bits(q.x), Op::from_bits(q.y)),
                                                           Op::combine(Op::from_bits(q.z), Op::from_bits(q.w))));
                    }
                    tot[w2] = acc;
                }
            } else {
#pragma unroll
            for (int w2 = 0; w2 < NW; ++w2) {
                const uint32_t c = lane + 32u * w2;
                const uint32_t p0 = c * ITEMS;
                T acc = Op::identity();
                if (p0 < valid) {
#pragma unroll
                    for (int v = 0; v < ITEMS / 4; ++v) {
                        const uint32_t pos = p0 + 4u * v;
                        const uint4 q = pos < bulk ? v4[c * (ITEMS / 4) + v] : tail_vec<Op>(in, base, pos, valid, hdr, n);
                        acc = Op::combine(acc, Op::combine(Op::combine(Op::from_bits(q.x), Op::from_bits(q.y)),
                                                           Op::combine(Op::from_bits(q.z), Op::from_bits(q.w))));
                    }
                }
                tot[w2] = acc;
            }
            }
            // the input stage is no longer needed
            __syncwarp();
            if (lane == 0) mbar_arrive(sm.in_empty(s));
#pragma unroll
            for (int w2 = 0; w2 < NW; ++w2) pre[prefix_slot(lane + 32u * w2)] = Op::to_bits(tot[w2]);
            __syncwarp();
            // lane l scans the PER consecutive thread totals PER*l .. (padded
            // slots; for PER = 8 words 9l+j, banks all distinct) ...
            constexpr int PER = NCONS / 32;
            T mine[PER];
            T run = Op::identity();
#pragma unroll
            for (int j = 0; j < PER; ++j) {
                mine[j] = run;
                run = Op::combine(run, Op::from_bits(pre[prefix_slot(lane * PER + j)]));
            }
            lt[lane] = Op::to_bits(run);
            __syncwarp();
            // ... and the 32 lane totals are scanned through shared memory
            // (all lanes read the same word at each step: a broadcast)
            T lane_excl = Op::identity(), agg = Op::identity();
#pragma unroll
            for (int l = 0; l < 32; ++l) {
                const T v = Op::from_bits(lt[l]);
                if (uint32_t(l) < lane) lane_excl = Op::combine(lane_excl, v);
                agg = Op::combine(agg, v);
            }
#pragma unroll
            for (int j = 0; j < PER; ++j)
                pre[prefix_slot(lane * PER + j)] = Op::to_bits(Op::combine(lane_excl, mine[j]));
            // publish the aggregate at once (tile 0: its inclusive prefix)
            perturb(fault, t, kSiteAggregate);
            if (lane == 0) {
                if (t != fault.never_publish_tile && in_bounds(hdr, t, 1, num_tiles))
                    st_relaxed_gpu(desc + t, make_desc(t == 0 ? kPrefix : kAggregate, Op::to_bits(agg)));
                *sm.agg(i) = Op::to_bits(agg);
                *sm.lbres(i) = 0u;
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(sm.info_ready(i));
        }
    }

    if (warp >= kLooker0 && warp < kReloader) {
        // --------------------------------------------------- look-back warps
        // The look-back reads only predecessors' descriptors, so it starts
        // as soon as the tile is drawn and runs while the tile loads and is
        // reduced; the prefix goes out once the reducer has published the
        // aggregate.  (With a bounded window an intermediate carries the
        // tile's own aggregate, so there the look-back waits for the reduce
        // first.)  Without the overlap the look-back's wait sat on every
        // tile's path and cost 13% at 2^28.
        const uint32_t j = warp - kLooker0;
        bool draining = false;
        for (uint32_t k = j;; k += LW) {
            const int i = int(k % RING);
            int w = warp_wait_or_end(sm.id_ready(i), (k / RING) & 1u, k, sm.end_iter());
            if (w != 2) {
                if (w == 0 && lane == 0) record_error(hdr, DWP_ERR_PIPELINE_TIMEOUT);
                return;
            }
            const uint32_t t = ld_volatile_smem(sm.tile_id(i));
            if (t == kNoTile) {
                if (lane == 0) mbar_arrive(sm.carry_ready(i));
                return;
            }
            if (!draining && ld_volatile_smem(sm.abort_flag()) != 0) draining = true;
            const bool early = fault.lookback_window == 0u;
            T carry = Op::identity();
            int rc = draining ? 1 : 0;
            if (early && rc == 0 && t != 0) {
                perturb(fault, t, kSiteLookback);
                rc = lookback<Op, C::kLookK>(desc, t, lane, fault.spin_limit, fault.fallback_polls,
                                             ScanRescue<Op, TILE>{in, n}, hdr, 0u, 0u, false, &carry,
                                             Backoff{DWP_SCAN_LB_AFTER, DWP_SCAN_LB_NS});
            }
            // the tile's aggregate (or the reducer's verdict on it)
            w = warp_wait_or_end(sm.info_ready(i), (k / RING) & 1u, k, sm.end_iter());
            if (w != 2) {
                if (w == 0 && lane == 0) record_error(hdr, DWP_ERR_PIPELINE_TIMEOUT);
                return;
            }
            if (ld_volatile_smem(sm.lbres(i)) != 0u) rc = 1;  // the reducer gave the tile up
            if (!early && rc == 0 && t != 0) {
                perturb(fault, t, kSiteLookback);
                rc = lookback<Op, C::kLookK>(desc, t, lane, fault.spin_limit, fault.fallback_polls,
                                             ScanRescue<Op, TILE>{in, n}, hdr,
                                             fault.lookback_window, *sm.agg(i),
                                             t != fault.never_publish_tile, &carry,
                                             Backoff{DWP_SCAN_LB_AFTER, DWP_SCAN_LB_NS});
            }
            if (rc == 0) perturb(fault, t, kSitePrefix);
            if (lane == 0) {
                if (!in_bounds(hdr, t, 1, num_tiles)) {
                    // debug bounds build only: no descriptor to publish
                } else if (rc == 0) {
                    if (t != 0 && t != fault.never_publish_tile)
                        st_relaxed_gpu(desc + t, make_desc(kPrefix, Op::to_bits(Op::combine(carry, Op::from_bits(*sm.agg(i))))));
                } else {
                    // give up on this tile: poison it so no successor waits
                    st_relaxed_gpu(desc + t, make_desc(kPoison, 0u));
                    if (rc == 2) record_error(hdr, DWP_ERR_LOOKBACK_TIMEOUT);
                    *reinterpret_cast<volatile uint32_t *>(sm.abort_flag()) = 1u;
                }
                *sm.carry(i) = Op::to_bits(carry);
                *sm.lbres(i) = uint32_t(rc);
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(sm.carry_ready(i));
            if (rc != 0) draining = true;
        }
    }

    if (warp == kReloader) {
        // ---------------------------------------------------------- reloader
        if (lane != 0) return;
        for (uint32_t k = 0;; ++k) {
            const int i = int(k % RING), o = int(k % SOUT);
            // carry_ready(k) is a single-lane wait here; end_iter as above
            int w = 0;
            for (uint32_t p = 0; p < kPipeWaitLimit; ++p) {
                if (mbar_try_wait(sm.carry_ready(i), (k / RING) & 1u)) { w = 2; break; }
                if (ld_volatile_smem(sm.end_iter()) < k) { w = 1; break; }
                if (p >= 8) __nanosleep(64);
            }
            if (w == 2 && k >= uint32_t(SOUT) &&
                !mbar_wait(sm.out_empty(o), ((k / SOUT) - 1) & 1u, kPipeWaitLimit))
                w = 0;
            if (w != 2) {
                if (w == 0) record_error(hdr, DWP_ERR_PIPELINE_TIMEOUT);
                return;
            }
            const uint32_t t = ld_volatile_smem(sm.tile_id(i));
            if (t == kNoTile || ld_volatile_smem(sm.lbres(i)) != 0u) {
                mbar_arrive(sm.out_full(o));
                if (t == kNoTile) return;
                continue;
            }
            uint32_t valid, bulk;
            tile_extent(t, valid, bulk);
            if (bulk && in_bounds(hdr, uint64_t(t) * TILE, bulk, n) && in_bounds(hdr, 0, bulk, TILE)) {
                mbar_arrive_expect_tx(sm.out_full(o), bulk * 4u);
                bulk_load_hint(sm.out_data(o), in + uint64_t(t) * TILE, bulk * 4u, sm.out_full(o),
                               l2_policy_evict_first());
            } else {
                mbar_arrive(sm.out_full(o));
            }
        }
    }

    if (warp < kConsumer0) return;
    // ---------------------------------------------------------- consumers
    // Consumer warp w owns chunk w of every tile; thread c = 32w + lane owns
    // ITEMS contiguous elements and needs no cross-thread step: its in-tile
    // exclusive prefix comes from the reducer, the carry from the look-back.
    const uint32_t cw = warp - kConsumer0;
    const uint32_t c = cw * 32 + lane;
    int pending = -1;  // lane 0: output stage whose bulk store may still read smem
    for (uint32_t k = 0;; ++k) {
        const int i = int(k % RING), o = int(k % SOUT);
        const int w = warp_wait_or_end(sm.out_full(o), (k / SOUT) & 1u, k, sm.end_iter());
        if (w != 2) {
            if (w == 0 && lane == 0) record_error(hdr, DWP_ERR_PIPELINE_TIMEOUT);
            break;
        }
        const uint32_t t = ld_volatile_smem(sm.tile_id(i));
        if (t == kNoTile) break;
        if (ld_volatile_smem(sm.lbres(i)) != 0u) {
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(sm.info_free(i));
                bulk_wait_read<0>();
                if (pending >= 0) mbar_arrive(sm.out_empty(pending));
                mbar_arrive(sm.out_empty(o));
                pending = -1;
            }
            __syncwarp();
            continue;
        }
        uint32_t valid, bulk;
        tile_extent(t, valid, bulk);
        const uint64_t base = uint64_t(t) * TILE;
        uint32_t *buf = sm.out_data(o);
        const uint32_t p0 = c * ITEMS;  // this thread's first element
        T acc = Op::combine(Op::from_bits(*sm.carry(i)), Op::from_bits(sm.prefix(i)[prefix_slot(c)]));
        __syncwarp();
        if (lane == 0) mbar_arrive(sm.info_free(i));  // the info slot has been read
        if (valid == uint32_t(TILE)) {  // every tile but a ragged last one
            uint4 *v4 = reinterpret_cast<uint4 *>(buf + p0);
#pragma unroll
            for (int v = 0; v < ITEMS / 4; ++v) {
                const uint4 q = v4[v];
                const uint32_t qq[4] = {q.x, q.y, q.z, q.w};
                uint32_t r[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const T xv = Op::from_bits(qq[e]);
                    if (INCL) {
                        acc = Op::combine(acc, xv);
                        r[e] = Op::to_bits(acc);
                    } else {
                        r[e] = Op::to_bits(acc);
                        acc = Op::combine(acc, xv);
                    }
                }
                v4[v] = make_uint4(r[0], r[1], r[2], r[3]);
            }
        } else if (p0 < valid) {
            // as in the reduce: 16-byte vectors in the stage, written back
            // in place; the 1-3 elements past the bulk part are read from
            // and written to global memory; nothing past the end
            uint4 *v4 = reinterpret_cast<uint4 *>(buf + p0);
#pragma unroll
            for (int v = 0; v < ITEMS / 4; ++v) {
                const uint32_t pos = p0 + 4u * v;
                const bool staged = pos < bulk;
                const uint4 q = staged ? v4[v] : tail_vec<Op>(in, base, pos, valid, hdr, n);
                const uint32_t qq[4] = {q.x, q.y, q.z, q.w};
                uint32_t r[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const T xv = Op::from_bits(qq[e]);
                    if (INCL) {
                        acc = Op::combine(acc, xv);
                        r[e] = Op::to_bits(acc);
                    } else {
                        r[e] = Op::to_bits(acc);
                        acc = Op::combine(acc, xv);
                    }
                }
                if (staged) {
                    v4[v] = make_uint4(r[0], r[1], r[2], r[3]);
                } else {
#pragma unroll
                    for (int e = 0; e < 4; ++e)
                        if (pos + e < valid && in_bounds(hdr, base + pos + e, 1, n))
                            out[base + pos + e] = Op::from_bits(r[e]);
                }
            }
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
            const uint32_t w0 = cw * WE;
            const uint32_t w1 = min(w0 + uint32_t(WE), bulk);
            if (w1 > w0 && in_bounds(hdr, base + w0, w1 - w0, n)) {
                bulk_store_hint(out + base + w0, buf + w0, (w1 - w0) * 4u, l2_policy_evict_first());
                bulk_commit();
                bulk_wait_read<1>();
                if (pending >= 0) mbar_arrive(sm.out_empty(pending));
                pending = o;
            } else {
                bulk_wait_read<0>();
                if (pending >= 0) mbar_arrive(sm.out_empty(pending));
                mbar_arrive(sm.out_empty(o));
                pending = -1;
            }
        }
        __syncwarp();
    }
    if (lane == 0) bulk_wait_all<0>();
}

// ------------------------------------------------------------------ host

namespace {

template <class Op, bool INCL>
cudaError_t launch_one(const void *in, void *out, uint64_t n, void *scratch, cudaStream_t stream,
                       const LaunchKnobs &fault) {
    using C = ScanCfg;
    auto kern = scan_kernel<Op, INCL, C>;
    const int dev_blocks = device_blocks(reinterpret_cast<const void *>(kern), C::kThreads,
                                         C::kSmemBytes);
    if (dev_blocks <= 0) return cudaErrorInvalidConfiguration;
    const uint64_t tiles = (n + C::kTile - 1) / C::kTile;
    const uint32_t grid = uint32_t(tiles < uint64_t(dev_blocks) ? tiles : uint64_t(dev_blocks));
    auto *hdr = reinterpret_cast<ScratchHeader *>(scratch);
    auto *desc = reinterpret_cast<uint64_t *>(static_cast<unsigned char *>(scratch) + kHeaderBytes);
    return launch_pdl(kern, dim3(grid), dim3(C::kThreads), C::kSmemBytes, stream,
                      reinterpret_cast<const typename Op::T *>(in),
                      reinterpret_cast<typename Op::T *>(out), n, uint32_t(tiles), hdr, desc, fault);
}

}  // namespace

uint32_t scan_tile_elems() { return ScanCfg::kTile; }

cudaError_t launch_scan(dwp_op op, bool inclusive, const void *in, void *out, uint64_t n,
                        void *scratch, cudaStream_t stream) {
    LaunchKnobs fault = current_launch_knobs();
    // in place, the input of a stalled tile may already be output: no fallback
    if (in == out) fault.fallback_polls = 0u;
    if (n <= kScanSmallMax) return launch_scan_small(op, inclusive, in, out, n, scratch, stream, fault);
    switch (op) {
        case DWP_U32_ADD:
            return inclusive ? launch_one<OpU32Add, true>(in, out, n, scratch, stream, fault)
                             : launch_one<OpU32Add, false>(in, out, n, scratch, stream, fault);
        case DWP_F32_ADD:
            return inclusive ? launch_one<OpF32Add, true>(in, out, n, scratch, stream, fault)
                             : launch_one<OpF32Add, false>(in, out, n, scratch, stream, fault);
        case DWP_U32_MAX:
            return inclusive ? launch_one<OpU32Max, true>(in, out, n, scratch, stream, fault)
                             : launch_one<OpU32Max, false>(in, out, n, scratch, stream, fault);
    }
    return cudaErrorInvalidValue;
}

}  // namespace dwp
