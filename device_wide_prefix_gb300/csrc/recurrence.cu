// First-order linear recurrence h[t] = a[t] h[t-1] + b[t], h[-1] = 0, as a
// single-pass chained scan with decoupled look-back, for sm_103a.
//
// "Parallel Prefix Sum (Scan), in depth", section "What scan builds": the
// recurrence looks sequential, but the pairs (a, b) compose associatively,
//     (a1, b1) then (a2, b2) = (a1 a2, a2 b1 + b2),
// so a scan of the pairs gives every h[t].  A pair is the affine map
// x -> a x + b, and "then" is map composition; it is not commutative, so
// every step here keeps operand order.  Arithmetic is f32, each
// a * x + b one fused multiply-add.
//
// The pipeline is the plain scan's (scan.cu), on two input streams:
//   producer warp    draws tile indices AHEAD iterations early, prefetches
//                    both tiles (a and b) into L2, and bulk loads them into
//                    the halves of one of SIN input stages;
//   reducer warps    one per input stage: each consumer thread's map over
//                    its ITEMS elements, and each thread's exclusive prefix
//                    map (lane-serial over consecutive threads, then a
//                    32-lane serial fold through shared memory), written to
//                    the tile's info slot; the tile map published at once;
//                    the input stage freed;
//   look-back warps  LW of them: an ordered look-back over the tile maps for
//                    the state h at the end of the previous tile (the carry),
//                    started when the tile is drawn and run while it loads,
//                    sleeping 128 ns before each poll; then the tile's end
//                    state published as its prefix.  Early start, the quieter
//                    polling and 16 warps instead of 4 measured 1-2% faster
//                    at 2^27 and 2^28 (with 8 warps the early start was 7%
//                    slower at 2^28);
//   reloader warp    brings both tiles back from L2 once the carry is known;
//   consumer warps   thread c starts from h = A_c carry + B_c (its exclusive
//                    map applied to the carry) and runs the recurrence over
//                    its ITEMS elements, writing h over the b half of the
//                    stage; one bulk store per warp.
//
// Descriptors: two 64-bit words per tile, each with the state in the high 32
// bits and f32 bits in the low 32.  Word 1 holds B (aggregate) or the end
// state h (prefix); word 0 holds A and is written once, before word 1's
// aggregate.  Every access is one single-copy-atomic 64-bit operation: a
// reader that finds word 1 in the aggregate state and word 0 not yet
// visible polls again.  A prefix needs only word 1: the map of everything
// before a tile is constant (its A is 0).
#include <cuda_runtime.h>

#include "device.cuh"
#include "launch.h"

namespace dwp {

namespace {

template <int NW_, int ITEMS_, int SIN_, int SOUT_, int RING_, int LW_, int AHEAD_>
struct RecConfig {
    static constexpr int kWarps = NW_;
    static constexpr int kItems = ITEMS_;
    static constexpr int kIn = SIN_;
    static constexpr int kOut = SOUT_;
    static constexpr int kRing = RING_;
    static constexpr int kLookers = LW_;
    static constexpr int kAhead = AHEAD_;
    static constexpr int kThreads = (2 + SIN_ + LW_ + NW_) * 32;
    static constexpr int kConsumers = NW_ * 32;
    static constexpr int kWarpElems = 32 * ITEMS_;
    static constexpr int kTile = NW_ * 32 * ITEMS_;
    static_assert(ITEMS_ % 4 == 0 && (ITEMS_ / 4) % 2 == 1, "ITEMS must be an odd multiple of 4");
    static_assert(NW_ >= 1 && NW_ <= 32, "");
    static_assert(kConsumers % 32 == 0, "");
    static_assert(RING_ % LW_ == 0, "a look-back warp must own every use of its info slots");
    static_assert(SOUT_ >= 2, "the reloader waits for the output stage of iteration k - SOUT");
    static_assert(RING_ >= SIN_ + SOUT_ + 2 + AHEAD_, "info ring shorter than the work in flight");
    // a stage: the a tile, then the b tile (h is written over b)
    static constexpr size_t kStageBytes = size_t(kTile) * 8;
    static constexpr int kPrefixWords = kConsumers + kConsumers / 8;
    // info slot: 4 mbarriers (32 B); tile id, carry, look-back result,
    // tile A, tile B, pad x3 (32 B); thread prefix maps, A then B
    static constexpr size_t kInfoBytes = 64 + 8 * size_t(kPrefixWords);
    static constexpr size_t kBarBytes = 16 * (SIN_ + SOUT_);
    // per-reducer scratch after the barriers: its 32 lane maps (32 A, 32 B)
    static constexpr size_t kWarpScratchBytes = 4 * 64 * size_t(SIN_);
    static constexpr size_t kSmemBytes =
        kStageBytes * (SIN_ + SOUT_) + kInfoBytes * RING_ + kBarBytes + 16 + kWarpScratchBytes;
    static_assert(kThreads <= 1024, "more than 1024 threads per block");
    static_assert(kSmemBytes <= 232448, "more than 227 KiB of shared memory per block");
};

#ifndef DWP_REC_WARPS
#define DWP_REC_WARPS 4
#endif
#ifndef DWP_REC_ITEMS
#define DWP_REC_ITEMS 36
#endif
#ifndef DWP_REC_IN
#define DWP_REC_IN 2
#endif
#ifndef DWP_REC_OUT
#define DWP_REC_OUT 3
#endif
#ifndef DWP_REC_RING
#define DWP_REC_RING 16
#endif
#ifndef DWP_REC_LOOKERS
#define DWP_REC_LOOKERS 16
#endif
#ifndef DWP_REC_AHEAD
#define DWP_REC_AHEAD 2
#endif
#ifndef DWP_REC_LB_AFTER
#define DWP_REC_LB_AFTER 0
#endif
#ifndef DWP_REC_LB_NS
#define DWP_REC_LB_NS 128
#endif
using RecCfg = RecConfig<DWP_REC_WARPS, DWP_REC_ITEMS, DWP_REC_IN, DWP_REC_OUT, DWP_REC_RING,
                         DWP_REC_LOOKERS, DWP_REC_AHEAD>;

template <class C>
struct RecSmem {
    unsigned char *base;
    __device__ explicit RecSmem(unsigned char *p) : base(p) {}
    __device__ float *in_a(int s) const {
        return reinterpret_cast<float *>(base + size_t(s) * C::kStageBytes);
    }
    __device__ float *in_b(int s) const { return in_a(s) + C::kTile; }
    __device__ float *out_a(int o) const {
        return reinterpret_cast<float *>(base + size_t(C::kIn + o) * C::kStageBytes);
    }
    __device__ float *out_b(int o) const { return out_a(o) + C::kTile; }
    __device__ unsigned char *info(int i) const {
        return base + C::kStageBytes * (C::kIn + C::kOut) + size_t(i) * C::kInfoBytes;
    }
    __device__ uint64_t *info_ready(int i) const { return reinterpret_cast<uint64_t *>(info(i)); }
    __device__ uint64_t *carry_ready(int i) const { return info_ready(i) + 1; }
    __device__ uint64_t *info_free(int i) const { return info_ready(i) + 2; }
    // the producer has written tile_id(i) (the tile is drawn)
    __device__ uint64_t *drawn(int i) const { return info_ready(i) + 3; }
    __device__ uint32_t *tile_id(int i) const { return reinterpret_cast<uint32_t *>(info(i) + 32); }
    __device__ float *carry(int i) const { return reinterpret_cast<float *>(tile_id(i) + 1); }
    __device__ uint32_t *lbres(int i) const { return tile_id(i) + 2; }
    __device__ float *agg_a(int i) const { return reinterpret_cast<float *>(tile_id(i) + 3); }
    __device__ float *agg_b(int i) const { return reinterpret_cast<float *>(tile_id(i) + 4); }
    __device__ float *pre_a(int i) const { return reinterpret_cast<float *>(info(i) + 64); }
    __device__ float *pre_b(int i) const { return pre_a(i) + C::kPrefixWords; }
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
    __device__ uint32_t *end_iter() const { return abort_flag() + 1; }
    // reducer r's 64-word scratch
    __device__ float *warp_scratch(int w) const {
        return reinterpret_cast<float *>(abort_flag() + 4) + 64 * w;
    }
};

// Element pos of a tile from the stage below `bulk`, from global memory
// below `valid` (the ragged tail the bulk copy cannot cover), else the
// identity map (a = 1, b = 0).
__device__ __forceinline__ void rec_elem(const float *sa, const float *sb, const float *ga,
                                         const float *gb, uint64_t base, uint32_t pos,
                                         uint32_t bulk, uint32_t valid, float &av, float &bv,
                                         ScratchHeader *hdr, uint64_t n) {
    if (pos < bulk) {
        av = sa[pos];
        bv = sb[pos];
    } else if (pos < valid && in_bounds(hdr, base + pos, 1, n)) {
        av = ga[base + pos];
        bv = gb[base + pos];
    } else {
        av = 1.0f;
        bv = 0.0f;
    }
}

// Fold 32 maps x -> a x + b, one per lane, into their composition by a
// shuffle tree; every lane gets the result.  LANE0_FIRST: lane 0's map is
// applied first and lane 31's last; otherwise the reverse.  After the step
// of width o, lane l holds the composite of lanes l .. l+o-1.  The map is
// not commutative, so each step composes the two halves in their order.
// (The look-back's fold lies on the path by which the prefix frontier
// advances; this tree replaced a serial fold by one lane through shared
// memory.)
template <bool LANE0_FIRST>
__device__ __forceinline__ void warp_compose(float a, float b, uint32_t lane, float &ra, float &rb) {
#pragma unroll
    for (uint32_t o = 1; o < 32u; o <<= 1) {
        const float a2 = __shfl_down_sync(0xffffffffu, a, o);
        const float b2 = __shfl_down_sync(0xffffffffu, b, o);
        if (lane + o < 32u) {
            if (LANE0_FIRST) {
                b = __fmaf_rn(a2, b, b2);  // (a, b) first, then (a2, b2)
            } else {
                b = __fmaf_rn(a, b2, b);   // (a2, b2) first, then (a, b)
            }
            a = __fmul_rn(a2, a);
        }
    }
    ra = __shfl_sync(0xffffffffu, a, 0);
    rb = __shfl_sync(0xffffffffu, b, 0);
}

// Decoupled Fallback for the recurrence: the two descriptor words tile p
// would publish, from a and b.  The map is not commutative, so lane l takes
// a contiguous run of the tile and the 32 runs are composed in order.
// Tile 0 publishes its end state (from h = 0) as a prefix.
struct RecRescue {
    const float *a;
    const float *b;
    uint64_t n;
    uint32_t tile;
    __device__ void operator()(uint32_t p, uint32_t lane, uint64_t &w0,
                               uint64_t &w1) const {
        const uint64_t t0 = uint64_t(p) * tile;
        const uint64_t e = min(n, t0 + uint64_t(tile));
        const uint64_t per = (e - t0 + 31u) / 32u;
        const uint64_t lo = t0 + uint64_t(lane) * per;
        const uint64_t hi = min(e, lo + per);
        float A = 1.0f, B = 0.0f;
        for (uint64_t q = lo; q < hi; ++q) {
            const float aq = a[q];
            B = __fmaf_rn(aq, B, b[q]);
            A = __fmul_rn(aq, A);
        }
        float TA, TB;
        warp_compose<true>(A, B, lane, TA, TB);
        if (p == 0) {
            w0 = 0ull;
            w1 = make_desc(kPrefix, __float_as_uint(TB));
        } else {
            w0 = make_desc(kAggregate, __float_as_uint(TA));
            w1 = make_desc(kAggregate, __float_as_uint(TB));
        }
    }
};

// Ordered decoupled look-back over two-word descriptors.  Lane l watches
// tile base - l of the current 32-tile window.  A lane is terminal when word
// 1 holds a prefix (or poison), ready when word 1 holds an aggregate and
// word 0 is visible, else it is polled again.  Once nothing nearer than the
// nearest terminal lane is unready, the maps from that lane to lane 0 are
// composed (farthest first); the terminal lane contributes the constant map
// to its end state.  Without a terminal lane the whole window's map is
// folded in and the window moves 32 tiles back.  Decoupled Fallback as in
// the commutative look-back (device.cuh), with two compare-and-swaps: word 0
// first, then word 1, whose swap decides who won.
// Returns 0 and the state at the end of tile t-1 in *carry_out; 1 poison;
// 2 poll limit.
__device__ __forceinline__ int lookback_affine(uint64_t *desc, uint32_t t, uint32_t lane,
                                               uint32_t spin_limit, uint32_t fallback_polls,
                                               const RecRescue &rescue, uint32_t *fallbacks,
                                               float *carry_out, const Backoff backoff) {
    float accA = 1.0f, accB = 0.0f;  // composition of the nearer windows, applied last
    int64_t base = static_cast<int64_t>(t) - 1;
    uint32_t polls = 0;
    while (true) {
        const int64_t idx = base - static_cast<int64_t>(lane);
        uint64_t w0 = 0ull, w1 = make_desc(kPrefix, __float_as_uint(0.0f));  // before tile 0: h = 0
        if (idx >= 0) {
            w1 = ld_relaxed_gpu(desc + 2 * idx + 1);
            w0 = ld_relaxed_gpu(desc + 2 * idx);
        }
        uint32_t tkey, stalled = 0;
        while (true) {
            const uint32_t s1 = desc_state(w1), s0 = desc_state(w0);
            const bool term = s1 == kPrefix || s1 == kPoison;
            const bool unready = !term && (s1 == kInvalid || s0 == kInvalid);
            tkey = __reduce_min_sync(0xffffffffu, term ? (lane << 1) | (s1 == kPoison ? 1u : 0u)
                                                       : 0xffffffffu);
            const uint32_t imin = __reduce_min_sync(0xffffffffu, unready ? lane : 0xffffffffu);
            if (tkey != 0xffffffffu ? imin > (tkey >> 1) : imin == 0xffffffffu) break;
            if (++polls >= spin_limit) return 2;
            const uint32_t lim = tkey != 0xffffffffu ? (tkey >> 1) : 32u;
            if (fallback_polls != 0u && ++stalled >= fallback_polls) {
                stalled = 0;
                uint32_t need = __ballot_sync(0xffffffffu, unready && lane < lim);
                while (need) {
                    const uint32_t j = uint32_t(__ffs(need)) - 1u;
                    need &= need - 1u;
                    const uint32_t p = static_cast<uint32_t>(base - static_cast<int64_t>(j));
                    uint64_t m0, m1;
                    rescue(p, lane, m0, m1);
                    unsigned long long g0 = 0ull, g1 = 0ull;
                    if (lane == 0) {
                        auto *d0 = reinterpret_cast<unsigned long long *>(desc + 2 * uint64_t(p));
                        if (m0 != 0ull) atomicCAS(d0, 0ull, static_cast<unsigned long long>(m0));
                        const unsigned long long old1 =
                            atomicCAS(d0 + 1, 0ull, static_cast<unsigned long long>(m1));
                        g1 = old1 == 0ull ? static_cast<unsigned long long>(m1) : old1;
                        if (old1 == 0ull) atomicAdd(fallbacks, 1u);
                        g0 = ld_relaxed_gpu(desc + 2 * uint64_t(p));
                    }
                    g0 = __shfl_sync(0xffffffffu, g0, 0);
                    g1 = __shfl_sync(0xffffffffu, g1, 0);
                    if (lane == j) {
                        w0 = g0;
                        w1 = g1;
                    }
                }
                continue;
            }
            if (polls > backoff.after) __nanosleep(polls > 256u ? 256u : backoff.ns);
            if (unready && lane < lim && idx >= 0) {
                w1 = ld_relaxed_gpu(desc + 2 * idx + 1);
                w0 = ld_relaxed_gpu(desc + 2 * idx);
            }
        }
        if (tkey != 0xffffffffu && (tkey & 1u)) return 1;
        const uint32_t last = tkey != 0xffffffffu ? (tkey >> 1) : 32u;
        // lane l's map; lanes past the terminal one are the identity
        float ma = 1.0f, mb = 0.0f;
        if (lane < last) {
            ma = __uint_as_float(desc_bits(w0));
            mb = __uint_as_float(desc_bits(w1));
        } else if (lane == last) {
            ma = 0.0f;
            mb = __uint_as_float(desc_bits(w1));
        }
        // lane 0 is the nearest tile and is applied last, the farthest
        // (lane 31) first
        float WA, WB;
        warp_compose<false>(ma, mb, lane, WA, WB);
        // total = (nearer windows) after (this window)
        accB = __fmaf_rn(accA, WB, accB);
        accA = __fmul_rn(accA, WA);
        if (tkey != 0xffffffffu) break;
        base -= 32;
    }
    *carry_out = accB;
    return 0;
}

// PERTURB compiles in the schedule-perturbation points of the test hook
// dwp_debug_set_delay.  Launches pick the variant without them unless the
// hook is on: in this kernel the inlined points alone (never taken) cost
// measurable time, so production launches carry none of their code.
template <bool INCL, class C, bool PERTURB>
__global__ void __launch_bounds__(C::kThreads, 1)
    recurrence_kernel(const float *ga, const float *gb, float *out, uint64_t n, uint32_t num_tiles,
                      ScratchHeader *hdr, uint64_t *desc, LaunchKnobs fault) {
    constexpr int NW = C::kWarps, ITEMS = C::kItems, TILE = C::kTile;
    constexpr int SIN = C::kIn, SOUT = C::kOut, RING = C::kRing, LW = C::kLookers;
    constexpr int WE = C::kWarpElems, AHEAD = C::kAhead;
    constexpr uint32_t NCONS = C::kConsumers;
    constexpr uint32_t kReducer0 = 1, kLooker0 = 1 + SIN, kReloader = 1 + SIN + LW,
                       kConsumer0 = 2 + SIN + LW;

    extern __shared__ __align__(128) unsigned char smem_raw[];
    const RecSmem<C> sm(smem_raw);
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
            mbar_init(sm.drawn(i), 1);
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
    auto stop_at = [&](uint32_t k) { *reinterpret_cast<volatile uint32_t *>(sm.end_iter()) = k; };

    if (warp == 0) {
        // ------------------------------------------------------- producer
        if (lane != 0) return;
        const uint64_t keep = l2_policy_evict_last();
        uint32_t taken = 0;
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
                    if (bulk && in_bounds(hdr, uint64_t(t) * TILE, bulk, n)) {
                        bulk_prefetch_l2(ga + uint64_t(t) * TILE, bulk * 4u, keep);
                        bulk_prefetch_l2(gb + uint64_t(t) * TILE, bulk * 4u, keep);
                    }
                }
            }
            if (ok && k >= uint32_t(SIN))
                ok = mbar_wait(sm.in_empty(s), ((k / SIN) - 1) & 1u, kPipeWaitLimit);
            if (!ok) {
                record_error(hdr, DWP_ERR_PIPELINE_TIMEOUT);
                for (uint32_t g = k; g < taken; ++g) {
                    const uint32_t t = ld_volatile_smem(sm.tile_id(int(g % RING)));
                    if (t != kNoTile && in_bounds(hdr, t, 1, num_tiles))
                        st_relaxed_gpu(desc + 2 * uint64_t(t) + 1, make_desc(kPoison, 0u));
                }
                stop_at(k - 1);
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
                mbar_arrive_expect_tx(sm.in_full(s), 2u * bulk * 4u);
                bulk_load_hint(sm.in_a(s), ga + uint64_t(t) * TILE, bulk * 4u, sm.in_full(s), keep);
                bulk_load_hint(sm.in_b(s), gb + uint64_t(t) * TILE, bulk * 4u, sm.in_full(s), keep);
            } else {
                mbar_arrive(sm.in_full(s));
            }
        }
    }

    if (warp >= kReducer0 && warp < kLooker0) {
        // -------------------------------------------------------- reducers
        const int s = int(warp - kReducer0);
        float *scr = sm.warp_scratch(s);
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
                if (lane == 0) {
                    if (in_bounds(hdr, t, 1, num_tiles))
                        st_relaxed_gpu(desc + 2 * uint64_t(t) + 1, make_desc(kPoison, 0u));
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
            const float *sa = sm.in_a(s), *sb = sm.in_b(s);
            float *pa = sm.pre_a(i), *pb = sm.pre_b(i);
            // map of consumer thread c = lane + 32*w2 over its ITEMS elements
            float tA[NW], tB[NW];
#pragma unroll
            for (int w2 = 0; w2 < NW; ++w2) {
                const uint32_t c = lane + 32u * w2;
                float A = 1.0f, B = 0.0f;
                // vectors wherever the thread's items are all bulk-copied (a
                // ragged last tile too; the test on `valid` first keeps the
                // usual full tile on one warp-uniform path), element by
                // element only for the thread holding the 1-3 elements after
                // the bulk part; a thread past the end keeps the identity map
                if (valid == uint32_t(TILE) || c * ITEMS + ITEMS <= bulk) {
                    const float4 *a4 = reinterpret_cast<const float4 *>(sa) + c * (ITEMS / 4);
                    const float4 *b4 = reinterpret_cast<const float4 *>(sb) + c * (ITEMS / 4);
#pragma unroll
                    for (int v = 0; v < ITEMS / 4; ++v) {
                        const float4 qa = a4[v], qb = b4[v];
                        B = __fmaf_rn(qa.x, B, qb.x);
                        B = __fmaf_rn(qa.y, B, qb.y);
                        B = __fmaf_rn(qa.z, B, qb.z);
                        B = __fmaf_rn(qa.w, B, qb.w);
                        A = __fmul_rn(__fmul_rn(__fmul_rn(qa.w, qa.z), __fmul_rn(qa.y, qa.x)), A);
                    }
                } else if (c * ITEMS < valid) {
                    for (int j = 0; j < ITEMS; ++j) {
                        float av, bv;
                        rec_elem(sa, sb, ga, gb, base, c * ITEMS + j, bulk, valid, av, bv, hdr, n);
                        B = __fmaf_rn(av, B, bv);
                        A = __fmul_rn(av, A);
                    }
                }
                tA[w2] = A;
                tB[w2] = B;
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(sm.in_empty(s));  // the input stage is no longer needed
#pragma unroll
            for (int w2 = 0; w2 < NW; ++w2) {
                pa[prefix_slot(lane + 32u * w2)] = tA[w2];
                pb[prefix_slot(lane + 32u * w2)] = tB[w2];
            }
            __syncwarp();
            // lane l composes the PER consecutive thread maps PER*l .. in order
            constexpr int PER = NCONS / 32;
            float mA[PER], mB[PER];
            float rA = 1.0f, rB = 0.0f;
#pragma unroll
            for (int j = 0; j < PER; ++j) {
                mA[j] = rA;
                mB[j] = rB;
                const float xa = pa[prefix_slot(lane * PER + j)], xb = pb[prefix_slot(lane * PER + j)];
                rB = __fmaf_rn(xa, rB, xb);
                rA = __fmul_rn(xa, rA);
            }
            scr[lane] = rA;
            scr[32 + lane] = rB;
            __syncwarp();
            // exclusive fold of the lane maps below this lane, and the tile map
            float eA = 1.0f, eB = 0.0f, gA = 1.0f, gB = 0.0f;
#pragma unroll
            for (int l = 0; l < 32; ++l) {
                const float xa = scr[l], xb = scr[32 + l];
                if (uint32_t(l) < lane) {
                    eB = __fmaf_rn(xa, eB, xb);
                    eA = __fmul_rn(xa, eA);
                }
                gB = __fmaf_rn(xa, gB, xb);
                gA = __fmul_rn(xa, gA);
            }
            // thread prefix = (lanes below) then (threads before it in this lane)
#pragma unroll
            for (int j = 0; j < PER; ++j) {
                pa[prefix_slot(lane * PER + j)] = __fmul_rn(mA[j], eA);
                pb[prefix_slot(lane * PER + j)] = __fmaf_rn(mA[j], eB, mB[j]);
            }
            if (PERTURB) perturb(fault, t, kSiteAggregate);
            if (lane == 0) {
                if (t != fault.never_publish_tile && in_bounds(hdr, t, 1, num_tiles)) {
                    if (t == 0) {
                        st_relaxed_gpu(desc + 1, make_desc(kPrefix, __float_as_uint(gB)));
                    } else {
                        st_relaxed_gpu(desc + 2 * uint64_t(t), make_desc(kAggregate, __float_as_uint(gA)));
                        if (PERTURB) perturb(fault, t, kSiteMidWord);
                        st_relaxed_gpu(desc + 2 * uint64_t(t) + 1,
                                       make_desc(kAggregate, __float_as_uint(gB)));
                    }
                }
                *sm.agg_a(i) = gA;
                *sm.agg_b(i) = gB;
                *sm.lbres(i) = 0u;
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(sm.info_ready(i));
        }
    }

    if (warp >= kLooker0 && warp < kReloader) {
        // --------------------------------------------------- look-back warps
        const uint32_t j = warp - kLooker0;
        const RecRescue rescue{ga, gb, n, uint32_t(TILE)};
        const Backoff backoff{DWP_REC_LB_AFTER, DWP_REC_LB_NS};
        bool draining = false;
        for (uint32_t k = j;; k += LW) {
            const int i = int(k % RING);
            // the look-back reads only predecessors' descriptors, so it
            // starts when the tile is drawn and runs while the tile loads
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
            float carry = 0.0f;
            int rc = draining ? 1 : 0;
            if (PERTURB && rc == 0) perturb(fault, t, kSiteLookback);
            if (rc == 0 && t != 0)
                rc = lookback_affine(desc, t, lane, fault.spin_limit, fault.fallback_polls, rescue,
                                     &hdr->fallbacks, &carry, backoff);
            // the tile's own map (or the reducer's verdict on it)
            w = warp_wait_or_end(sm.info_ready(i), (k / RING) & 1u, k, sm.end_iter());
            if (w != 2) {
                if (w == 0 && lane == 0) record_error(hdr, DWP_ERR_PIPELINE_TIMEOUT);
                return;
            }
            if (ld_volatile_smem(sm.lbres(i)) != 0u) rc = 1;
            if (PERTURB && rc == 0) perturb(fault, t, kSitePrefix);
            if (lane == 0) {
                if (!in_bounds(hdr, t, 1, num_tiles)) {
                    // debug bounds build only: no descriptor to publish
                } else if (rc == 0) {
                    if (t != 0 && t != fault.never_publish_tile)
                        st_relaxed_gpu(desc + 2 * uint64_t(t) + 1,
                                       make_desc(kPrefix, __float_as_uint(
                                                              __fmaf_rn(*sm.agg_a(i), carry, *sm.agg_b(i)))));
                } else {
                    st_relaxed_gpu(desc + 2 * uint64_t(t) + 1, make_desc(kPoison, 0u));
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
        const uint64_t drop = l2_policy_evict_first();
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
                mbar_arrive_expect_tx(sm.out_full(o), 2u * bulk * 4u);
                bulk_load_hint(sm.out_a(o), ga + uint64_t(t) * TILE, bulk * 4u, sm.out_full(o), drop);
                bulk_load_hint(sm.out_b(o), gb + uint64_t(t) * TILE, bulk * 4u, sm.out_full(o), drop);
            } else {
                mbar_arrive(sm.out_full(o));
            }
        }
    }

    if (warp < kConsumer0) return;
    // ---------------------------------------------------------- consumers
    const uint32_t cw = warp - kConsumer0;
    const uint32_t c = cw * 32 + lane;
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
        const float *sa = sm.out_a(o);
        float *sb = sm.out_b(o);
        const uint32_t p0 = c * ITEMS;
        // state entering this thread's elements: its exclusive map on the carry
        float h = __fmaf_rn(sm.pre_a(i)[prefix_slot(c)], *sm.carry(i), sm.pre_b(i)[prefix_slot(c)]);
        __syncwarp();
        if (lane == 0) mbar_arrive(sm.info_free(i));
        if (valid == uint32_t(TILE) || p0 + ITEMS <= bulk) {
            const float4 *a4 = reinterpret_cast<const float4 *>(sa + p0);
            float4 *b4 = reinterpret_cast<float4 *>(sb + p0);
#pragma unroll
            for (int v = 0; v < ITEMS / 4; ++v) {
                const float4 qa = a4[v], qb = b4[v];
                float4 r;
                if (INCL) {
                    h = __fmaf_rn(qa.x, h, qb.x); r.x = h;
                    h = __fmaf_rn(qa.y, h, qb.y); r.y = h;
                    h = __fmaf_rn(qa.z, h, qb.z); r.z = h;
                    h = __fmaf_rn(qa.w, h, qb.w); r.w = h;
                } else {
                    r.x = h; h = __fmaf_rn(qa.x, h, qb.x);
                    r.y = h; h = __fmaf_rn(qa.y, h, qb.y);
                    r.z = h; h = __fmaf_rn(qa.z, h, qb.z);
                    r.w = h; h = __fmaf_rn(qa.w, h, qb.w);
                }
                b4[v] = r;
            }
        } else if (p0 < valid) {
            for (int jj = 0; jj < ITEMS; ++jj) {
                const uint32_t pos = p0 + jj;
                float av, bv;
                rec_elem(sa, sb, ga, gb, base, pos, bulk, valid, av, bv, hdr, n);
                float y;
                if (INCL) {
                    h = __fmaf_rn(av, h, bv);
                    y = h;
                } else {
                    y = h;
                    h = __fmaf_rn(av, h, bv);
                }
                if (pos < bulk)
                    sb[pos] = y;
                else if (pos < valid && in_bounds(hdr, base + pos, 1, n))
                    out[base + pos] = y;
            }
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
            const uint32_t w0 = cw * WE;
            const uint32_t w1 = min(w0 + uint32_t(WE), bulk);
            if (w1 > w0 && in_bounds(hdr, base + w0, w1 - w0, n)) {
                bulk_store_hint(out + base + w0, sb + w0, (w1 - w0) * 4u, l2_policy_evict_first());
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
cudaError_t launch_rec(const float *a, const float *b, float *h, uint64_t n, void *scratch,
                       cudaStream_t stream, const LaunchKnobs &fault) {
    using C = RecCfg;
    auto kern = fault.delay_threshold != 0u ? recurrence_kernel<INCL, C, true> : recurrence_kernel<INCL, C, false>;
    const int dev_blocks = device_blocks(reinterpret_cast<const void *>(kern), C::kThreads,
                                         C::kSmemBytes);
    if (dev_blocks <= 0) return cudaErrorInvalidConfiguration;
    const uint64_t tiles = (n + C::kTile - 1) / C::kTile;
    const uint32_t grid = uint32_t(tiles < uint64_t(dev_blocks) ? tiles : uint64_t(dev_blocks));
    auto *hdr = reinterpret_cast<ScratchHeader *>(scratch);
    auto *desc = reinterpret_cast<uint64_t *>(static_cast<unsigned char *>(scratch) + kHeaderBytes);
    return launch_pdl(kern, dim3(grid), dim3(C::kThreads), C::kSmemBytes, stream, a, b, h, n,
                      uint32_t(tiles), hdr, desc, fault);
}

}  // namespace

uint32_t recurrence_tile_elems() { return RecCfg::kTile; }

cudaError_t launch_recurrence(const float *a, const float *b, float *h, uint64_t n, bool inclusive,
                              void *scratch, cudaStream_t stream) {
    LaunchKnobs fault = current_launch_knobs();
    // in place, the inputs of a stalled tile may already be output: no fallback
    if (h == a || h == b) fault.fallback_polls = 0u;
    return inclusive ? launch_rec<true>(a, b, h, n, scratch, stream, fault)
                     : launch_rec<false>(a, b, h, n, scratch, stream, fault);
}

}  // namespace dwp
