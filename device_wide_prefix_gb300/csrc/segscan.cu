// Segmented u32 addition scan over CSR offsets, single pass with decoupled
// look-back, for sm_103a.
//
// "GPUSegmentedScan" (luma.gl), sections "Prefix scans and segmented scans"
// and "Contract": segment s is rows [offsets[s], offsets[s+1]); the running
// total restarts at every segment; empty segments write nothing.  "Parallel
// Prefix Sum (Scan), in depth", section "What scan builds": a segmented scan
// carries a flag with each value, i.e. it scans (head, value) pairs with
//     (h1, v1) (+) (h2, v2) = (h1 | h2, h2 ? v2 : v1 + v2),
// an associative, non-commutative operator.
//
// The pipeline is the plain scan's (scan.cu): producer warp that draws tile
// indices AHEAD iterations early, prefetches those tiles into L2, and bulk
// loads them into SIN input stages; reducer warps that free their input stage as soon
// as the tile is reduced; a pool of look-back warps; a reloader warp that
// brings a tile back from L2 once its carry is known; consumer warps with
// per-warp bulk stores.  What differs:
//   * the reducer first marks the heads of its tile (every offset value in
//     [tile start, tile end)) in a bitmap kept in the tile's info slot.  It
//     finds the first offset at or after the tile start in a per-block
//     sample of the offsets held in shared memory (exact when N + 1 <=
//     kSample, the skewed-length workload's case), else by a warp-wide
//     32-ary search of global memory inside the sampled interval; then it
//     walks the offsets of the tile;
//   * per-thread totals and their exclusive prefix are (head, value) pairs;
//   * a tile holding a head publishes its inclusive prefix at once (its value
//     after its last head is final); the look-back is a plain u32-add
//     look-back that stops at the nearest prefix.  It starts when the tile
//     is drawn, before its heads are known, and its carry is dropped if the
//     tile's first row is a head (with a bounded window it waits for the
//     reduce and runs only when the first row is not a head);
//   * rows outside [offsets[0], min(offsets[N], n)) are not written.
// Offsets are trusted (no readback, "Limitations"): unordered offsets give
// unspecified values but every access stays inside offsets[0..N].
#include <cuda_runtime.h>

#include "device.cuh"
#include "launch.h"

namespace dwp {

namespace {

constexpr int kSample = 2048;  // offsets sampled into shared memory per block

template <int NW_, int ITEMS_, int SIN_, int SOUT_, int RING_, int LW_, int LOOKK_, int AHEAD_>
struct SegConfig {
    static constexpr int kWarps = NW_;
    static constexpr int kItems = ITEMS_;
    static constexpr int kIn = SIN_;
    static constexpr int kOut = SOUT_;
    static constexpr int kRing = RING_;
    static constexpr int kLookers = LW_;
    static constexpr int kLookK = LOOKK_;
    static constexpr int kAhead = AHEAD_;  // iterations a tile index is drawn before its load
    static constexpr int kThreads = (2 + SIN_ + LW_ + NW_) * 32;
    static constexpr int kConsumers = NW_ * 32;
    static constexpr int kWarpElems = 32 * ITEMS_;
    static constexpr int kTile = NW_ * 32 * ITEMS_;
    static_assert(ITEMS_ % 4 == 0 && (ITEMS_ / 4) % 2 == 1, "ITEMS must be an odd multiple of 4");
    static_assert(ITEMS_ <= 32, "a thread's head bits span at most two bitmap words");
    static_assert(NW_ >= 1 && NW_ <= 32, "");
    static_assert(RING_ % LW_ == 0, "a look-back warp must own every use of its info slots");
    static_assert(SOUT_ >= 2, "the reloader waits for the output stage of iteration k - SOUT");
    static_assert(RING_ >= SIN_ + SOUT_ + 2 + AHEAD_, "info ring shorter than the work in flight");
    static constexpr size_t kStageBytes = size_t(kTile) * 4;
    static constexpr int kPrefixWords = kConsumers + kConsumers / 8;
    static constexpr int kPHeadWords = kConsumers / 4;  // one head byte per consumer thread
    static constexpr int kHeadWords = kTile / 32 + 1;   // tile head bitmap (+1 spill word)
    // info slot: 4 mbarriers (32 B); tile id, aggregate, carry,
    // look-back result, aggregate head, first-row head, pad x2 (32 B);
    // prefix values; prefix head bytes; head bitmap; lane totals 33; lane
    // heads 33 (+ pad to 16 B)
    static constexpr size_t kInfoBytes =
        (64 + 4 * (kPrefixWords + kPHeadWords + kHeadWords + 33 + 33) + 15) / 16 * 16;
    static_assert(kInfoBytes % 8 == 0, "info slots hold mbarriers");
    static constexpr size_t kBarBytes = 16 * (SIN_ + SOUT_) + 8 * SIN_;
    // + abort, end, cover lo, cover hi, then the offset sample
    static constexpr size_t kSmemBytes = kStageBytes * (SIN_ + SOUT_) + kInfoBytes * RING_ +
                                         kBarBytes + 16 + 4 * kSample;
    static_assert(kThreads <= 1024, "more than 1024 threads per block");
    static_assert(kSmemBytes <= 232448, "more than 227 KiB of shared memory per block");
};

#ifndef DWP_SEG_WARPS
#define DWP_SEG_WARPS 8
#endif
#ifndef DWP_SEG_ITEMS
#define DWP_SEG_ITEMS 28
#endif
#ifndef DWP_SEG_IN
#define DWP_SEG_IN 3
#endif
#ifndef DWP_SEG_OUT
#define DWP_SEG_OUT 3
#endif
#ifndef DWP_SEG_RING
#define DWP_SEG_RING 12
#endif
#ifndef DWP_SEG_LOOKERS
#define DWP_SEG_LOOKERS 12
#endif
#ifndef DWP_SEG_LOOKK
#define DWP_SEG_LOOKK 1
#endif
#ifndef DWP_SEG_AHEAD
#define DWP_SEG_AHEAD 1
#endif
// look-back back-off: sleep DWP_SEG_LB_NS before every poll after the first
// DWP_SEG_LB_AFTER (as in the plain scan: the look-back starts at the draw
// and polls while the tile loads)
#ifndef DWP_SEG_LB_AFTER
#define DWP_SEG_LB_AFTER 0
#endif
#ifndef DWP_SEG_LB_NS
#define DWP_SEG_LB_NS 128
#endif
using SegCfg = SegConfig<DWP_SEG_WARPS, DWP_SEG_ITEMS, DWP_SEG_IN, DWP_SEG_OUT, DWP_SEG_RING,
                         DWP_SEG_LOOKERS, DWP_SEG_LOOKK, DWP_SEG_AHEAD>;

template <class C>
struct SegSmem {
    unsigned char *base;
    __device__ explicit SegSmem(unsigned char *p) : base(p) {}
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
    __device__ uint64_t *drawn(int i) const { return info_ready(i) + 3; }
    __device__ uint32_t *tile_id(int i) const { return reinterpret_cast<uint32_t *>(info(i) + 32); }
    __device__ uint32_t *agg(int i) const { return tile_id(i) + 1; }
    __device__ uint32_t *carry(int i) const { return tile_id(i) + 2; }
    __device__ uint32_t *lbres(int i) const { return tile_id(i) + 3; }
    __device__ uint32_t *agg_head(int i) const { return tile_id(i) + 4; }
    __device__ uint32_t *first_head(int i) const { return tile_id(i) + 5; }
    // tile holds at least one head; bitmap holds bits from an earlier use
    __device__ uint32_t *has_heads(int i) const { return tile_id(i) + 6; }
    __device__ uint32_t *heads_dirty(int i) const { return tile_id(i) + 7; }
    __device__ uint32_t *prefix(int i) const { return tile_id(i) + 8; }
    __device__ unsigned char *phead(int i) const {
        return reinterpret_cast<unsigned char *>(prefix(i) + C::kPrefixWords);
    }
    __device__ uint32_t *heads(int i) const { return prefix(i) + C::kPrefixWords + C::kPHeadWords; }
    __device__ uint32_t *lane_tot(int i) const { return heads(i) + C::kHeadWords; }
    __device__ uint32_t *lane_head(int i) const { return lane_tot(i) + 33; }
    __device__ uint64_t *bars() const {
        return reinterpret_cast<uint64_t *>(base + C::kStageBytes * (C::kIn + C::kOut) +
                                            C::kInfoBytes * C::kRing);
    }
    __device__ uint64_t *in_full(int s) const { return bars() + s; }
    __device__ uint64_t *in_empty(int s) const { return bars() + C::kIn + s; }
    __device__ uint64_t *out_full(int o) const { return bars() + 2 * C::kIn + o; }
    __device__ uint64_t *out_empty(int o) const { return bars() + 2 * C::kIn + C::kOut + o; }
    // the producer has written the tile id of input stage s (before its load)
    __device__ uint64_t *id_ready(int s) const { return bars() + 2 * (C::kIn + C::kOut) + s; }
    __device__ uint32_t *words() const {
        return reinterpret_cast<uint32_t *>(bars() + 2 * (C::kIn + C::kOut) + C::kIn);
    }
    __device__ uint32_t *abort_flag() const { return words(); }
    __device__ uint32_t *end_iter() const { return words() + 1; }
    __device__ uint32_t *cover_lo() const { return words() + 2; }
    __device__ uint32_t *cover_hi() const { return words() + 3; }
    __device__ uint32_t *sample() const { return words() + 4; }
};

__device__ __forceinline__ uint32_t seg_elem(const uint32_t *buf, const uint32_t *in, uint64_t base,
                                             uint32_t pos, uint32_t bulk, uint32_t valid,
                                             ScratchHeader *hdr, uint64_t n) {
    if (pos < bulk) return buf[pos];
    if (pos < valid && in_bounds(hdr, base + pos, 1, n)) return in[base + pos];
    return 0u;
}

// Head bits [pos, pos + cnt) of a tile bitmap, cnt <= 32, as the low bits.
__device__ __forceinline__ uint32_t head_bits(const uint32_t *heads, uint32_t pos, uint32_t cnt) {
    const uint32_t w = pos >> 5, b = pos & 31u;
    uint64_t v = (uint64_t(heads[w + 1]) << 32) | heads[w];
    v >>= b;
    return cnt >= 32 ? uint32_t(v) : uint32_t(v) & ((1u << cnt) - 1u);
}

// Decoupled Fallback for the segmented scan: the descriptor tile p would
// publish, from the values and the offsets.  The heads of a tile are the
// offset values inside it; offsets are nondecreasing, so its last head is the
// last offset below the tile end, if that offset is not below the tile
// start.  A tile with a head publishes its prefix, the sum from its last head
// to its end; a tile without one publishes the sum of its rows as its
// aggregate; tile 0 always publishes a prefix.
struct SegRescue {
    const uint32_t *in;
    const uint32_t *off;
    uint32_t nseg;
    uint64_t n;
    uint32_t tile;
    __device__ uint64_t operator()(uint32_t p, uint32_t lane) const {
        const uint64_t b = uint64_t(p) * tile;
        const uint64_t e = min(n, b + uint64_t(tile));  // e <= n < 2^32
        const uint32_t k = warp_lower_bound(off, 0u, nseg + 1u, uint32_t(e), lane);
        uint64_t from = b;
        bool head = false;
        if (k > 0u) {
            const uint32_t h = __ldg(off + k - 1u);
            if (uint64_t(h) >= b) {
                head = true;
                from = h;
            }
        }
        uint32_t acc = 0;
        for (uint64_t q = from + lane; q < e; q += 32u) acc += __ldg(in + q);
        acc = __reduce_add_sync(0xffffffffu, acc);
        return make_desc((p == 0 || head) ? kPrefix : kAggregate, acc);
    }
};

// PERTURB compiles in the schedule-perturbation points of the test hook
// dwp_debug_set_delay.  Launches pick the variant without them unless the
// hook is on: in this kernel the inlined points alone (never taken) cost
// measurable time, so production launches carry none of their code.
template <bool INCL, class C, bool PERTURB>
__global__ void __launch_bounds__(C::kThreads, 1)
    segscan_kernel(const uint32_t *in, const uint32_t *off, uint32_t nseg, uint32_t *out,
                   uint64_t n, uint32_t num_tiles, ScratchHeader *hdr, uint64_t *desc,
                   LaunchKnobs fault) {
    using Op = OpU32Add;
    constexpr int NW = C::kWarps, ITEMS = C::kItems, TILE = C::kTile;
    constexpr int SIN = C::kIn, SOUT = C::kOut, RING = C::kRing, LW = C::kLookers;
    constexpr int WE = C::kWarpElems;
    constexpr int AHEAD = C::kAhead;
    constexpr uint32_t NCONS = C::kConsumers;
    constexpr uint32_t kReducer0 = 1, kLooker0 = 1 + SIN, kReloader = 1 + SIN + LW,
                       kConsumer0 = 2 + SIN + LW;

    extern __shared__ __align__(128) unsigned char smem_raw[];
    const SegSmem<C> sm(smem_raw);
    const uint32_t warp = threadIdx.x >> 5, lane = threadIdx.x & 31u;
    // the kernel before may still be running: wait before reading anything
    // (no early trigger, as in the plain scan: the next kernel launches as
    // the blocks exit)
    pdl_wait();

    // offset sample: sample[i] = off[min(i * stride, N)]
    const uint64_t noff = uint64_t(nseg) + 1;
    const uint32_t stride = uint32_t((noff + kSample - 1) / kSample);
    const uint32_t nsample = uint32_t((noff + stride - 1) / stride);
    for (uint32_t i = threadIdx.x; i < nsample; i += blockDim.x)
        sm.sample()[i] = __ldg(off + min(uint64_t(i) * stride, uint64_t(nseg)));
    if (threadIdx.x == 0) {
        for (int s = 0; s < SIN; ++s) {
            mbar_init(sm.in_full(s), 1);
            mbar_init(sm.in_empty(s), 1);
            mbar_init(sm.id_ready(s), 1);
        }
        for (int o = 0; o < SOUT; ++o) {
            mbar_init(sm.out_full(o), 1);
            mbar_init(sm.out_empty(o), NW);
        }
        for (int i = 0; i < RING; ++i) {
            mbar_init(sm.info_ready(i), 1);
            mbar_init(sm.carry_ready(i), 1);
            mbar_init(sm.info_free(i), NW);
            mbar_init(sm.drawn(i), 1);
            *sm.heads_dirty(i) = 1u;  // bitmaps start uninitialised
        }
        *sm.abort_flag() = 0;
        *sm.end_iter() = kNoTile;
        const uint32_t lo = __ldg(off), last = __ldg(off + nseg);
        *sm.cover_lo() = lo;
        *sm.cover_hi() = uint32_t(min(uint64_t(last), n));
        fence_mbar_init();
    }
    __syncthreads();

    auto tile_extent = [&](uint32_t t, uint32_t &valid, uint32_t &bulk) {
        const uint64_t rem = n - uint64_t(t) * TILE;
        valid = rem < uint64_t(TILE) ? uint32_t(rem) : uint32_t(TILE);
        bulk = valid == uint32_t(TILE) ? valid : (valid & ~3u);
    };
    auto stop_at = [&](uint32_t k) { *reinterpret_cast<volatile uint32_t *>(sm.end_iter()) = k; };

    if (warp == 0) {
        // ------------------------------------------------------- producer
        // As in the plain scan: the tile of iteration k is drawn AHEAD
        // iterations early and prefetched into L2, so its bulk load is short.
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
                    else if (PERTURB) perturb(fault, t, kSiteDraw);
                }
                *reinterpret_cast<volatile uint32_t *>(sm.tile_id(gi)) = t;
                mbar_arrive(sm.drawn(gi));  // the look-back may start now
                ++taken;
                if (t == kNoTile) {
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
                stop_at(k - 1);
                return;
            }
            const uint32_t t = ld_volatile_smem(sm.tile_id(i));
            mbar_arrive(sm.id_ready(s));  // heads can be marked while the data is in flight
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
            const int w = warp_wait_or_end(sm.id_ready(s), use & 1u, k, sm.end_iter());
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
                // the load may still be writing the stage: wait for it first
                if (!warp_wait(sm.in_full(s), use & 1u) && lane == 0)
                    record_error(hdr, DWP_ERR_PIPELINE_TIMEOUT);
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
            const uint64_t tend = base + valid;
            uint32_t *heads = sm.heads(i);

            // -- S1: heads of this tile ------------------------------------
            // (the bitmap is cleared only if an earlier use of the slot set bits)
            if (*sm.heads_dirty(i)) {
                for (int q = int(lane); q < C::kHeadWords; q += 32) heads[q] = 0u;
            }
            __syncwarp();
            const uint32_t *smp = sm.sample();
            uint32_t a = 0, b = nsample;  // first sample >= base
            while (a < b) {
                const uint32_t m = (a + b) >> 1;
                if (uint64_t(smp[m]) < base) a = m + 1; else b = m;
            }
            uint32_t k0;
            if (a == 0) {
                k0 = 0;
            } else if (stride == 1u) {
                k0 = a;
            } else {
                const uint32_t lo = (a - 1) * stride + 1;
                const uint32_t hi = uint32_t(min(uint64_t(a) * stride, uint64_t(nseg) + 1));
                k0 = warp_lower_bound(off, lo, hi, uint32_t(base), lane);
            }
            uint32_t my_marks = 0;
            for (uint32_t kk = k0; kk <= nseg; kk += 32) {
                const uint64_t idx = uint64_t(kk) + lane;
                uint32_t p = 0xffffffffu;
                if (idx <= nseg && in_bounds(hdr, idx, 1, uint64_t(nseg) + 1))
                    p = stride == 1u ? smp[idx] : __ldg(off + idx);
                if (idx <= nseg && uint64_t(p) >= base && uint64_t(p) < tend) {
                    const uint32_t r = uint32_t(uint64_t(p) - base);
                    atomicOr(&heads[r >> 5], 1u << (r & 31u));
                    ++my_marks;
                }
                if (__any_sync(0xffffffffu, idx > nseg || uint64_t(p) >= tend)) break;
            }
            const bool tile_heads = __reduce_add_sync(0xffffffffu, my_marks) != 0u;
            __syncwarp();

            if (!warp_wait(sm.in_full(s), use & 1u)) {
                // the producer always completes the load it announced
                if (lane == 0) record_error(hdr, DWP_ERR_PIPELINE_TIMEOUT);
                return;
            }
            // -- per-thread (head, value) totals ---------------------------
            // Totals and head bits stay in registers until the stage is
            // freed: a shared-memory store between the loads would keep the
            // compiler from having the next rows' loads in flight.
            const uint32_t *buf = sm.in_data(s);
            uint32_t *pre = sm.prefix(i);
            unsigned char *ph = sm.phead(i);
            uint32_t tot[NW], thb[NW];
#pragma unroll
            for (int w2 = 0; w2 < NW; ++w2) {
                const uint32_t c = lane + 32u * w2;
                const uint32_t hb = tile_heads ? head_bits(heads, c * ITEMS, ITEMS) : 0u;
                uint32_t acc = 0;
                // vectors wherever the thread's items are all bulk-copied (a
                // ragged last tile too); element by element only for the
                // thread holding the 1-3 elements after the bulk part; heads
                // lie below the tile end, so threads past it hold nothing
                const bool vec = valid == uint32_t(TILE) || c * ITEMS + ITEMS <= bulk;
                if (vec && !hb) {
                    const uint4 *v4 = reinterpret_cast<const uint4 *>(buf);
#pragma unroll
                    for (int v = 0; v < ITEMS / 4; ++v) {
                        const uint4 q = v4[c * (ITEMS / 4) + v];
                        acc += (q.x + q.y) + (q.z + q.w);
                    }
                } else if (vec) {
                    const uint4 *v4 = reinterpret_cast<const uint4 *>(buf);
                    // only the items from the last head on count
                    const int from = hb ? 31 - __clz(hb) : 0;
#pragma unroll
                    for (int v = 0; v < ITEMS / 4; ++v) {
                        const uint4 q = v4[c * (ITEMS / 4) + v];
                        const uint32_t qq[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
                        for (int e = 0; e < 4; ++e)
                            if (4 * v + e >= from) acc += qq[e];
                    }
                } else if (c * ITEMS < valid) {
                    for (int j = 0; j < ITEMS; ++j) {
                        const uint32_t x = seg_elem(buf, in, base, c * ITEMS + j, bulk, valid, hdr, n);
                        acc = ((hb >> j) & 1u) ? x : acc + x;
                    }
                }
                tot[w2] = acc;
                thb[w2] = hb;
            }
            // the input stage is no longer needed
            __syncwarp();
            if (lane == 0) mbar_arrive(sm.in_empty(s));
#pragma unroll
            for (int w2 = 0; w2 < NW; ++w2) {
                const uint32_t c = lane + 32u * w2;
                pre[prefix_slot(c)] = tot[w2];
                if (tile_heads) ph[c] = thb[w2] ? 1 : 0;
            }
            __syncwarp();
            // lane l scans threads PER*l .. PER*l+PER-1 with the pair operator
            constexpr int PER = NCONS / 32;
            uint32_t mv[PER], mh = 0, rv = 0, rh = 0;
#pragma unroll
            for (int j = 0; j < PER; ++j) {
                const uint32_t c = lane * PER + j;
                mv[j] = rv;
                if (rh) mh |= 1u << j;
                const uint32_t hv = tile_heads ? ph[c] : 0u;
                const uint32_t v = pre[prefix_slot(c)];
                rv = hv ? v : rv + v;
                rh |= hv;
            }
            sm.lane_tot(i)[lane] = rv;
            if (tile_heads) sm.lane_head(i)[lane] = rh;
            __syncwarp();
            uint32_t ev = 0, eh = 0, av = 0, ah = 0;  // lane exclusive pair, tile aggregate
            if (tile_heads) {
#pragma unroll
                for (int l = 0; l < 32; ++l) {
                    const uint32_t v = sm.lane_tot(i)[l], h = sm.lane_head(i)[l];
                    if (uint32_t(l) < lane) {
                        ev = h ? v : ev + v;
                        eh |= h;
                    }
                    av = h ? v : av + v;
                    ah |= h;
                }
            } else {
#pragma unroll
                for (int l = 0; l < 32; ++l) {
                    const uint32_t v = sm.lane_tot(i)[l];
                    if (uint32_t(l) < lane) ev += v;
                    av += v;
                }
            }
            // each thread's exclusive pair: value in pre, head flag in ph
            // (lane l rewrites only its own PER slots)
#pragma unroll
            for (int j = 0; j < PER; ++j) {
                const uint32_t hj = (mh >> j) & 1u;
                pre[prefix_slot(lane * PER + j)] = hj ? mv[j] : ev + mv[j];
                if (tile_heads) ph[lane * PER + j] = (hj | eh) ? 1 : 0;
            }
            if (PERTURB) perturb(fault, t, kSiteAggregate);
            if (lane == 0) {
                if (t != fault.never_publish_tile && in_bounds(hdr, t, 1, num_tiles))
                    st_relaxed_gpu(desc + t, make_desc((t == 0 || ah) ? kPrefix : kAggregate, av));
                *sm.agg(i) = av;
                *sm.agg_head(i) = ah;
                *sm.first_head(i) = tile_heads ? (heads[0] & 1u) : 0u;
                *sm.has_heads(i) = tile_heads ? 1u : 0u;
                *sm.heads_dirty(i) = tile_heads ? 1u : 0u;
                *sm.lbres(i) = 0u;
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(sm.info_ready(i));
        }
    }

    if (warp >= kLooker0 && warp < kReloader) {
        // --------------------------------------------------- look-back warps
        const uint32_t j = warp - kLooker0;
        bool draining = false;
        for (uint32_t k = j;; k += LW) {
            const int i = int(k % RING);
            int w = warp_wait_or_end(sm.drawn(i), (k / RING) & 1u, k, sm.end_iter());
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
            // early: the look-back runs while the tile loads, before its heads
            // are known, and its carry is dropped if the tile's first row is a
            // head.  Only with the unbounded window: an intermediate carries
            // the tile's own aggregate, which needs the reduce first.
            const bool early = fault.lookback_window == 0u;
            uint32_t carry = 0;
            int rc = draining ? 1 : 0, early_rc = 0;
            if (early && rc == 0 && t != 0) {
                if (PERTURB) perturb(fault, t, kSiteLookback);
                early_rc = lookback<Op, C::kLookK>(desc, t, lane, fault.spin_limit, fault.fallback_polls,
                                                   SegRescue{in, off, nseg, n, uint32_t(TILE)}, hdr, 0u,
                                                   0u, false, &carry,
                                                   Backoff{DWP_SEG_LB_AFTER, DWP_SEG_LB_NS});
            }
            // the tile's heads and aggregate (or the reducer's verdict on it)
            w = warp_wait_or_end(sm.info_ready(i), (k / RING) & 1u, k, sm.end_iter());
            if (w != 2) {
                if (w == 0 && lane == 0) record_error(hdr, DWP_ERR_PIPELINE_TIMEOUT);
                return;
            }
            if (ld_volatile_smem(sm.lbres(i)) != 0u) rc = 1;  // the reducer gave the tile up
            const bool ah = ld_volatile_smem(sm.agg_head(i)) != 0u;
            const bool fh = ld_volatile_smem(sm.first_head(i)) != 0u;
            if (early) {
                if (fh) carry = 0;  // the tile restarts at its first row: no carry
                else if (rc == 0) rc = early_rc;
            }
            if (!early && rc == 0 && t != 0 && !fh) {
                if (PERTURB) perturb(fault, t, kSiteLookback);
                rc = lookback<Op, C::kLookK>(desc, t, lane, fault.spin_limit, fault.fallback_polls,
                                             SegRescue{in, off, nseg, n, uint32_t(TILE)},
                                             hdr, fault.lookback_window, *sm.agg(i),
                                             !ah && t != fault.never_publish_tile, &carry);
            }
            if (PERTURB && rc == 0) perturb(fault, t, kSitePrefix);
            if (lane == 0) {
                if (!in_bounds(hdr, t, 1, num_tiles)) {
                    // debug bounds build only: no descriptor to publish
                } else if (rc == 0) {
                    if (t != 0 && !ah && t != fault.never_publish_tile)
                        st_relaxed_gpu(desc + t, make_desc(kPrefix, carry + *sm.agg(i)));
                } else {
                    st_relaxed_gpu(desc + t, make_desc(kPoison, 0u));
                    if (rc == 2) record_error(hdr, DWP_ERR_LOOKBACK_TIMEOUT);
                    *reinterpret_cast<volatile uint32_t *>(sm.abort_flag()) = 1u;
                }
                *sm.carry(i) = carry;
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
    const uint32_t cw = warp - kConsumer0;
    const uint32_t c = cw * 32 + lane;
    const uint64_t cover_lo = *sm.cover_lo(), cover_hi = *sm.cover_hi();
    int pending = -1;
    for (uint32_t k = 0;; ++k) {
        const int i = int(k % RING), o = int(k % SOUT);
        const int w = warp_wait_or_end(sm.out_full(o), (k / SOUT) & 1u, k, sm.end_iter());
        if (w != 2) {
            if (w == 0 && lane == 0) record_error(hdr, DWP_ERR_PIPELINE_TIMEOUT);
            break;
        }
        const uint32_t t = ld_volatile_smem(sm.tile_id(i));
        if (t == kNoTile) break;
        uint32_t valid, bulk;
        tile_extent(t, valid, bulk);
        const uint64_t base = uint64_t(t) * TILE;
        // a tile wholly inside [cover_lo, cover_hi) is stored in bulk; any
        // other tile row by row, only the covered rows
        const bool covered = base >= cover_lo && base + valid <= cover_hi;
        const bool outside = base >= cover_hi || base + valid <= cover_lo;
        if (ld_volatile_smem(sm.lbres(i)) != 0u || outside) {
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
        uint32_t *buf = sm.out_data(o);
        const uint32_t p0 = c * ITEMS;
        const bool th = *sm.has_heads(i) != 0u;
        const uint32_t hb = th ? head_bits(sm.heads(i), p0, ITEMS) : 0u;
        const bool phd = th && sm.phead(i)[c] != 0;
        const uint32_t pv = sm.prefix(i)[prefix_slot(c)];
        uint32_t acc = phd ? pv : *sm.carry(i) + pv;
        __syncwarp();
        if (lane == 0) mbar_arrive(sm.info_free(i));  // the info slot has been read
        if (covered && (valid == uint32_t(TILE) || p0 + ITEMS <= bulk)) {
            uint4 *v4 = reinterpret_cast<uint4 *>(buf + p0);
#pragma unroll
            for (int v = 0; v < ITEMS / 4; ++v) {
                const uint4 q = v4[v];
                const uint32_t qq[4] = {q.x, q.y, q.z, q.w};
                uint32_t r[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    if ((hb >> (4 * v + e)) & 1u) acc = 0u;
                    if (INCL) {
                        acc += qq[e];
                        r[e] = acc;
                    } else {
                        r[e] = acc;
                        acc += qq[e];
                    }
                }
                v4[v] = make_uint4(r[0], r[1], r[2], r[3]);
            }
        } else if (p0 < valid) {
            for (int j = 0; j < ITEMS; ++j) {
                const uint32_t pos = p0 + j;
                const uint32_t x = seg_elem(buf, in, base, pos, bulk, valid, hdr, n);
                if ((hb >> j) & 1u) acc = 0u;
                uint32_t y;
                if (INCL) {
                    acc += x;
                    y = acc;
                } else {
                    y = acc;
                    acc += x;
                }
                const uint64_t g = base + pos;
                if (pos < valid && covered && pos < bulk)
                    buf[pos] = y;
                else if (pos < valid && g >= cover_lo && g < cover_hi && in_bounds(hdr, g, 1, n))
                    out[g] = y;
            }
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
            const uint32_t w0 = cw * WE;
            const uint32_t w1 = covered ? min(w0 + uint32_t(WE), bulk) : w0;
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

template <bool INCL>
cudaError_t launch_seg(const uint32_t *values, const uint32_t *offsets, uint32_t nseg,
                       uint32_t *out, uint64_t n, void *scratch, cudaStream_t stream,
                       const LaunchKnobs &fault) {
    using C = SegCfg;
    auto kern = fault.delay_threshold != 0u ? segscan_kernel<INCL, C, true> : segscan_kernel<INCL, C, false>;
    const int dev_blocks = device_blocks(reinterpret_cast<const void *>(kern), C::kThreads,
                                         C::kSmemBytes);
    if (dev_blocks <= 0) return cudaErrorInvalidConfiguration;
    const uint64_t tiles = (n + C::kTile - 1) / C::kTile;
    const uint32_t grid = uint32_t(tiles < uint64_t(dev_blocks) ? tiles : uint64_t(dev_blocks));
    auto *hdr = reinterpret_cast<ScratchHeader *>(scratch);
    auto *desc = reinterpret_cast<uint64_t *>(static_cast<unsigned char *>(scratch) + kHeaderBytes);
    return launch_pdl(kern, dim3(grid), dim3(C::kThreads), C::kSmemBytes, stream, values, offsets,
                      nseg, out, n, uint32_t(tiles), hdr, desc, fault);
}

}  // namespace

uint32_t segscan_tile_elems() { return SegCfg::kTile; }

cudaError_t launch_segscan(const uint32_t *values, const uint32_t *offsets, uint32_t nseg,
                           uint32_t *out, uint64_t n, bool inclusive, void *scratch,
                           cudaStream_t stream) {
    const LaunchKnobs fault = current_launch_knobs();
    return inclusive ? launch_seg<true>(values, offsets, nseg, out, n, scratch, stream, fault)
                     : launch_seg<false>(values, offsets, nseg, out, n, scratch, stream, fault);
}

}  // namespace dwp
