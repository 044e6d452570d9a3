// Stable stream compaction of 16-byte records by byte flags, single pass
// with decoupled look-back, for sm_103a.
//
// "Prefix scans and compaction", sections "Scan as an index generator" and
// "Worked example: Stable stream compaction"; "Parallel Prefix Sum (Scan),
// in depth", section "What scan builds": the exclusive scan of the keep
// flags is each kept record's output slot, so kept records keep their order
// and never share a slot; the output length is the flag total.
//
// The look-back needs only the flags (1 byte per 16-byte record), so the
// records stay out of shared memory until their output slots are known:
//   producer warp   takes a tile index from the atomic counter, loads the
//                   tile's flag bytes with one bulk copy into the tile's
//                   info slot, and asks L2 to prefetch the tile's records
//                   (bulk prefetch, evict-last);
//   tile warps      TW of them, iteration k taken by warp k % TW: each
//                   consumer thread's kept count and their exclusive prefix,
//                   the tile count published as the aggregate, a u32-add
//                   look-back for the number of records kept before the
//                   tile, the tile's inclusive count published; the last
//                   tile writes the total to *count;
//   loader warp     once a tile's output offset is known, loads its records
//                   (now in L2) with one bulk copy into a ring of SOUT
//                   output stages;
//   consumer warps  thread c owns IT contiguous records.  Each warp reads its
//                   records into registers, writes its kept ones to the front
//                   of its own chunk of the stage, in input order, and
//                   streams that block to its output slots with one bulk
//                   store.
// IT is odd, so 16-byte record reads at a thread stride of 16*IT bytes are
// free of bank conflicts.
#include <cuda_runtime.h>

#include "device.cuh"
#include "launch.h"

namespace dwp {

namespace {

template <int NW_, int IT_, int SOUT_, int RING_, int TW_, int LOOKK_>
struct CompactConfig {
    static constexpr int kWarps = NW_;
    static constexpr int kItems = IT_;  // records per consumer thread
    static constexpr int kOut = SOUT_;
    static constexpr int kRing = RING_;
    static constexpr int kTileWarps = TW_;
    static constexpr int kLookK = LOOKK_;
    static constexpr int kThreads = (2 + TW_ + NW_) * 32;
    static constexpr int kConsumers = NW_ * 32;
    static constexpr int kWarpRecs = 32 * IT_;
    static constexpr int kTile = NW_ * 32 * IT_;  // records per tile
    static_assert(IT_ % 2 == 1, "IT must be odd");
    static_assert(kTile % 16 == 0, "flag bytes of a tile must start 16-byte aligned");
    static_assert(NW_ >= 1 && NW_ <= 32, "");
    static_assert(RING_ % TW_ == 0, "a tile warp must own every use of its info slots");
    static_assert(SOUT_ >= 2, "the loader waits for the output stage of iteration k - SOUT");
    static constexpr size_t kRecBytes = size_t(kTile) * 16;
    static constexpr size_t kFlagBytes = (size_t(kTile) + 15) / 16 * 16;
    static constexpr int kPrefixWords = kConsumers + kConsumers / 8;
    // info slot: 3 mbarriers + pad (32 B); tile id, carry, look-back result,
    // tile count (16 B); flags; thread prefixes; lane totals 33 (+ pad to 16 B)
    static constexpr size_t kInfoBytes = (48 + kFlagBytes + 4 * (kPrefixWords + 33) + 15) / 16 * 16;
    static constexpr size_t kBarBytes = 16 * SOUT_;
    static constexpr size_t kSmemBytes = kRecBytes * SOUT_ + kInfoBytes * RING_ + kBarBytes + 16;
};

#ifndef DWP_CMP_WARPS
#define DWP_CMP_WARPS 16
#endif
#ifndef DWP_CMP_ITEMS
#define DWP_CMP_ITEMS 5
#endif
#ifndef DWP_CMP_OUT
#define DWP_CMP_OUT 4
#endif
#ifndef DWP_CMP_RING
#define DWP_CMP_RING 12
#endif
#ifndef DWP_CMP_TILEWARPS
#define DWP_CMP_TILEWARPS 12
#endif
#ifndef DWP_CMP_LOOKK
#define DWP_CMP_LOOKK 1
#endif
// Where the L2 prefetch of a tile's records is issued: 0 none, 1 by the
// producer when it draws the tile, 2 by the tile warp once the tile's count
// is published, 3 once its look-back is done (later points leave fewer
// prefetched lines waiting in L2 at once).
#ifndef DWP_CMP_PREFETCH
#define DWP_CMP_PREFETCH 2
#endif
using CmpCfg = CompactConfig<DWP_CMP_WARPS, DWP_CMP_ITEMS, DWP_CMP_OUT, DWP_CMP_RING,
                             DWP_CMP_TILEWARPS, DWP_CMP_LOOKK>;

template <class C>
struct CmpSmem {
    unsigned char *base;
    __device__ explicit CmpSmem(unsigned char *p) : base(p) {}
    __device__ uint4 *recs(int o) const {
        return reinterpret_cast<uint4 *>(base + size_t(o) * C::kRecBytes);
    }
    __device__ unsigned char *info(int i) const {
        return base + C::kRecBytes * C::kOut + size_t(i) * C::kInfoBytes;
    }
    __device__ uint64_t *flags_full(int i) const { return reinterpret_cast<uint64_t *>(info(i)); }
    __device__ uint64_t *carry_ready(int i) const { return flags_full(i) + 1; }
    __device__ uint64_t *info_free(int i) const { return flags_full(i) + 2; }
    __device__ uint32_t *tile_id(int i) const { return reinterpret_cast<uint32_t *>(info(i) + 32); }
    __device__ uint32_t *carry(int i) const { return tile_id(i) + 1; }
    __device__ uint32_t *lbres(int i) const { return tile_id(i) + 2; }
    __device__ uint32_t *tile_count(int i) const { return tile_id(i) + 3; }
    __device__ unsigned char *flags(int i) const { return info(i) + 48; }
    __device__ uint32_t *prefix(int i) const {
        return reinterpret_cast<uint32_t *>(flags(i) + C::kFlagBytes);
    }
    __device__ uint32_t *lane_tot(int i) const { return prefix(i) + C::kPrefixWords; }
    __device__ uint64_t *bars() const {
        return reinterpret_cast<uint64_t *>(base + C::kRecBytes * C::kOut + C::kInfoBytes * C::kRing);
    }
    __device__ uint64_t *out_full(int o) const { return bars() + o; }
    __device__ uint64_t *out_empty(int o) const { return bars() + C::kOut + o; }
    __device__ uint32_t *abort_flag() const {
        return reinterpret_cast<uint32_t *>(bars() + 2 * C::kOut);
    }
    __device__ uint32_t *end_iter() const { return abort_flag() + 1; }
};

// Bit j (j < 4) set when byte j of x is nonzero: the compare gives 0xff per
// nonzero byte; the multiply gathers the low bit of each byte into bits
// 24..27 (no partial product reaches them but these four).
__device__ __forceinline__ uint32_t nonzero_bytes4(uint32_t x) {
    return ((__vcmpne4(x, 0u) & 0x01010101u) * 0x01020408u) >> 24;
}

// Keep flag of record pos of a tile: from the slot below `fbulk`, from global
// memory below `valid`, else 0.
__device__ __forceinline__ bool keep_at(const unsigned char *sflags, const uint8_t *gflags,
                                        uint64_t base, uint32_t pos, uint32_t fbulk, uint32_t valid,
                                        ScratchHeader *hdr, uint64_t n) {
    if (pos < fbulk) return sflags[pos] != 0;
    if (pos < valid && in_bounds(hdr, base + pos, 1, n)) return gflags[base + pos] != 0;
    return false;
}

// Decoupled Fallback for compaction: the descriptor tile p would publish,
// the number of nonzero flags among its records, counted by one warp from
// the flag bytes (tile 0's count is its inclusive prefix).
template <int TILE>
struct CompactRescue {
    static_assert(TILE % 16 == 0, "full tiles are read as 16-byte vectors");
    const uint8_t *flags;
    uint64_t n;
    __device__ uint64_t operator()(uint32_t p, uint32_t lane) const {
        const uint64_t b = uint64_t(p) * TILE;
        const uint64_t e = min(n, b + uint64_t(TILE));
        uint32_t cnt = 0;
        if (e - b == uint64_t(TILE)) {
            const uint4 *v4 = reinterpret_cast<const uint4 *>(flags + b);
            for (uint32_t q = lane; q < uint32_t(TILE) / 16u; q += 32u) {
                const uint4 v = v4[q];
                // __vcmpne4: 0xff in every nonzero byte
                cnt += (__popc(__vcmpne4(v.x, 0u)) + __popc(__vcmpne4(v.y, 0u)) +
                        __popc(__vcmpne4(v.z, 0u)) + __popc(__vcmpne4(v.w, 0u))) >> 3;
            }
        } else {
            for (uint64_t q = b + lane; q < e; q += 32u) cnt += flags[q] != 0 ? 1u : 0u;
        }
        cnt = __reduce_add_sync(0xffffffffu, cnt);
        return make_desc(p == 0 ? kPrefix : kAggregate, cnt);
    }
};

template <class C>
__global__ void __launch_bounds__(C::kThreads, 1)
    compact_kernel(const uint4 *recs, const uint8_t *flags, uint64_t n, uint4 *out,
                   uint32_t *count, uint32_t num_tiles, ScratchHeader *hdr, uint64_t *desc,
                   LaunchKnobs fault) {
    using Op = OpU32Add;
    constexpr int NW = C::kWarps, IT = C::kItems, TILE = C::kTile;
    constexpr int SOUT = C::kOut, RING = C::kRing, TW = C::kTileWarps;
    constexpr int WR = C::kWarpRecs;
    constexpr uint32_t NCONS = C::kConsumers;
    constexpr uint32_t kTileWarp0 = 1, kLoader = 1 + TW, kConsumer0 = 2 + TW;

    extern __shared__ __align__(128) unsigned char smem_raw[];
    const CmpSmem<C> sm(smem_raw);
    const uint32_t warp = threadIdx.x >> 5, lane = threadIdx.x & 31u;
    if (threadIdx.x == 0) {
        for (int o = 0; o < SOUT; ++o) {
            mbar_init(sm.out_full(o), 1);
            mbar_init(sm.out_empty(o), NW);
        }
        for (int i = 0; i < RING; ++i) {
            mbar_init(sm.flags_full(i), 1);
            mbar_init(sm.carry_ready(i), 1);
            mbar_init(sm.info_free(i), NW);
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

    // valid records of tile t, and how many of its flag bytes the bulk copy
    // brings (a multiple of 16; the rest are read from global memory)
    auto tile_extent = [&](uint32_t t, uint32_t &valid, uint32_t &fbulk) {
        const uint64_t rem = n - uint64_t(t) * TILE;
        valid = rem < uint64_t(TILE) ? uint32_t(rem) : uint32_t(TILE);
        fbulk = valid & ~15u;
    };
    auto stop_at = [&](uint32_t k) { *reinterpret_cast<volatile uint32_t *>(sm.end_iter()) = k; };

    if (warp == 0) {
        // ------------------------------------------------------- producer
        if (lane != 0) return;
        const uint64_t keep = l2_policy_evict_last();
        for (uint32_t k = 0;; ++k) {
            const int i = int(k % RING);
            if (k >= uint32_t(RING) &&
                !mbar_wait(sm.info_free(i), ((k / RING) - 1) & 1u, kPipeWaitLimit)) {
                record_error(hdr, DWP_ERR_PIPELINE_TIMEOUT);
                stop_at(k - 1);
                return;
            }
            uint32_t t = kNoTile;
            if (ld_volatile_smem(sm.abort_flag()) == 0) {
                t = atomicAdd(&hdr->tile_counter, 1u);
                if (t >= num_tiles) t = kNoTile;
                else perturb(fault, t, kSiteDraw);
            }
            *reinterpret_cast<volatile uint32_t *>(sm.tile_id(i)) = t;
            if (t == kNoTile) {
                stop_at(k);
                mbar_arrive(sm.flags_full(i));
                return;
            }
            uint32_t valid, fbulk;
            tile_extent(t, valid, fbulk);
            const uint64_t base = uint64_t(t) * TILE;
            if (DWP_CMP_PREFETCH == 1 && in_bounds(hdr, base, valid, n))
                bulk_prefetch_l2(recs + base, valid * 16u, keep);
            if (fbulk && in_bounds(hdr, base, fbulk, n) && in_bounds(hdr, 0, fbulk, C::kFlagBytes)) {
                mbar_arrive_expect_tx(sm.flags_full(i), fbulk);
                bulk_load(sm.flags(i), flags + base, fbulk, sm.flags_full(i));
            } else {
                mbar_arrive(sm.flags_full(i));
            }
        }
    }

    if (warp >= kTileWarp0 && warp < kLoader) {
        // ----------------------------------------------------- tile warps
        const uint32_t j = warp - kTileWarp0;
        bool draining = false;
        for (uint32_t k = j;; k += TW) {
            const int i = int(k % RING);
            const int w = warp_wait_or_end(sm.flags_full(i), (k / RING) & 1u, k, sm.end_iter());
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
            if (draining) {
                if (lane == 0) {
                    if (in_bounds(hdr, t, 1, num_tiles)) st_relaxed_gpu(desc + t, make_desc(kPoison, 0u));
                    *sm.lbres(i) = 1u;
                    mbar_arrive(sm.carry_ready(i));
                }
                __syncwarp();
                continue;
            }
            uint32_t valid, fbulk;
            tile_extent(t, valid, fbulk);
            const uint64_t base = uint64_t(t) * TILE;
            const unsigned char *sf = sm.flags(i);
            uint32_t *pre = sm.prefix(i);
            uint32_t *lt = sm.lane_tot(i);
            // K1: lane l takes consumer threads PER*l .. PER*l + PER-1, whose
            // flags are the PER*IT contiguous bytes from PER*IT*l: read as
            // 16-byte vectors (a lane stride of 80 bytes, 5 times 16, so a
            // quarter warp hits 8 distinct bank groups), the keep mask and
            // count of each thread worked out in registers.  A ragged last
            // tile reads its flags one by one.
            constexpr int PER = NCONS / 32;
            static_assert(IT <= 5 && (PER * IT) % 16 == 0, "a thread's flags sit in one 8-byte window");
            static_assert(TILE < (1 << 24), "prefixes share a word with an 8-bit keep mask");
            uint32_t cntm[PER];  // kept count | keep mask << 24
            if (valid == uint32_t(TILE)) {
                const uint4 *fv = reinterpret_cast<const uint4 *>(sf) + lane * (PER * IT / 16);
                uint32_t wd[PER * IT / 4 + 1];
#pragma unroll
                for (int q = 0; q < PER * IT / 16; ++q) {
                    const uint4 x = fv[q];
                    wd[4 * q + 0] = x.x;
                    wd[4 * q + 1] = x.y;
                    wd[4 * q + 2] = x.z;
                    wd[4 * q + 3] = x.w;
                }
                wd[PER * IT / 4] = 0u;
#pragma unroll
                for (int j = 0; j < PER; ++j) {
                    const int lo = j * IT, w = lo >> 2, sh = (lo & 3) * 8;
                    const uint64_t v = ((uint64_t(wd[w + 1]) << 32) | wd[w]) >> sh;
                    const uint32_t m = (nonzero_bytes4(uint32_t(v)) | (nonzero_bytes4(uint32_t(v >> 32)) << 4)) &
                                       ((1u << IT) - 1u);
                    cntm[j] = uint32_t(__popc(m)) | (m << 24);
                }
            } else {
#pragma unroll
                for (int j = 0; j < PER; ++j) {
                    const uint32_t p0 = (lane * PER + j) * IT;
                    uint32_t m = 0;
                    for (int q = 0; q < IT; ++q)
                        if (keep_at(sf, flags, base, p0 + q, fbulk, valid, hdr, n)) m |= 1u << q;
                    cntm[j] = uint32_t(__popc(m)) | (m << 24);
                }
            }
            // K2: exclusive prefix of the counts, lane by lane
            uint32_t mine[PER], run = 0;
#pragma unroll
            for (int q = 0; q < PER; ++q) {
                mine[q] = run;
                run += cntm[q] & 0xffffffu;
            }
            lt[lane] = run;
            __syncwarp();
            uint32_t lane_excl = 0, total = 0;
#pragma unroll
            for (int l = 0; l < 32; ++l) {
                const uint32_t v = lt[l];
                if (uint32_t(l) < lane) lane_excl += v;
                total += v;
            }
            // each thread's exclusive prefix, its keep mask in the top byte
#pragma unroll
            for (int q = 0; q < PER; ++q)
                pre[prefix_slot(lane * PER + q)] = (lane_excl + mine[q]) | (cntm[q] & 0xff000000u);
            perturb(fault, t, kSiteAggregate);
            if (lane == 0 && t != fault.never_publish_tile && in_bounds(hdr, t, 1, num_tiles))
                st_relaxed_gpu(desc + t, make_desc(t == 0 ? kPrefix : kAggregate, total));
            if (DWP_CMP_PREFETCH == 2 && lane == 0 && total != 0u && in_bounds(hdr, base, valid, n))
                bulk_prefetch_l2(recs + base, valid * 16u, l2_policy_evict_last());
            uint32_t carry = 0;
            int rc = 0;
            perturb(fault, t, kSiteLookback);
            if (t != 0)
                rc = lookback<Op, C::kLookK>(desc, t, lane, fault.spin_limit, fault.fallback_polls,
                                             CompactRescue<TILE>{flags, n}, hdr,
                                             fault.lookback_window, total,
                                             t != fault.never_publish_tile, &carry);
            if (rc == 0) perturb(fault, t, kSitePrefix);
            if (DWP_CMP_PREFETCH == 3 && lane == 0 && rc == 0 && total != 0u && in_bounds(hdr, base, valid, n))
                bulk_prefetch_l2(recs + base, valid * 16u, l2_policy_evict_last());
            if (lane == 0) {
                if (!in_bounds(hdr, t, 1, num_tiles)) {
                    // debug bounds build only: no descriptor to publish
                } else if (rc == 0) {
                    if (t != 0 && t != fault.never_publish_tile)
                        st_relaxed_gpu(desc + t, make_desc(kPrefix, carry + total));
                    if (t == num_tiles - 1) *count = carry + total;  // K4: output length
                } else {
                    st_relaxed_gpu(desc + t, make_desc(kPoison, 0u));
                    if (rc == 2) record_error(hdr, DWP_ERR_LOOKBACK_TIMEOUT);
                    *reinterpret_cast<volatile uint32_t *>(sm.abort_flag()) = 1u;
                }
                *sm.carry(i) = carry;
                *sm.tile_count(i) = total;
                *sm.lbres(i) = uint32_t(rc);
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(sm.carry_ready(i));
            if (rc != 0) draining = true;
        }
    }

    if (warp == kLoader) {
        // ------------------------------------------------------------ loader
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
            if (t == kNoTile || ld_volatile_smem(sm.lbres(i)) != 0u ||
                ld_volatile_smem(sm.tile_count(i)) == 0u) {
                // nothing to load: sentinel, poisoned tile, or no record kept
                mbar_arrive(sm.out_full(o));
                if (t == kNoTile) return;
                continue;
            }
            uint32_t valid, fbulk;
            tile_extent(t, valid, fbulk);
            if (in_bounds(hdr, uint64_t(t) * TILE, valid, n) && in_bounds(hdr, 0, valid, TILE)) {
                mbar_arrive_expect_tx(sm.out_full(o), valid * 16u);
                bulk_load_hint(sm.recs(o), recs + uint64_t(t) * TILE, valid * 16u, sm.out_full(o), drop);
            } else {
                mbar_arrive(sm.out_full(o));
            }
        }
    }

    if (warp < kConsumer0) return;
    // ---------------------------------------------------------- consumers
    const uint32_t cw = warp - kConsumer0;
    const uint32_t c = cw * 32 + lane;
    const uint64_t drop = l2_policy_evict_first();
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
        uint32_t nkeep = 0, first = 0;  // this warp's kept records and its first output slot
        if (ld_volatile_smem(sm.lbres(i)) == 0u && *sm.tile_count(i) != 0u) {
            uint4 *region = sm.recs(o) + cw * WR;
            const uint32_t *pre = sm.prefix(i);
            const uint32_t wfirst = pre[prefix_slot(cw * 32)] & 0xffffffu;
            const uint32_t wend = cw + 1 < uint32_t(NW) ? pre[prefix_slot(cw * 32 + 32)] & 0xffffffu
                                                        : *sm.tile_count(i);
            nkeep = wend - wfirst;
            first = *sm.carry(i) + wfirst;
            // K3: read this thread's kept records (the keep mask rides in the
            // top byte of its prefix word), then (after the whole warp has
            // read) write them to their in-warp slots, in order
            const uint32_t pv = pre[prefix_slot(c)];
            const uint32_t keepm = pv >> 24;
            uint4 r[IT];
#pragma unroll
            for (int q = 0; q < IT; ++q)
                if ((keepm >> q) & 1u) r[q] = sm.recs(o)[c * IT + q];
            uint32_t slot = (pv & 0xffffffu) - wfirst;
            __syncwarp();
#pragma unroll
            for (int q = 0; q < IT; ++q)
                if ((keepm >> q) & 1u) region[slot++] = r[q];
            fence_proxy_async_smem();
        }
        __syncwarp();
        if (lane == 0) {
            mbar_arrive(sm.info_free(i));  // flags and prefixes have been read
            if (nkeep && in_bounds(hdr, first, nkeep, n) && in_bounds(hdr, 0, nkeep, WR)) {
                bulk_store_hint(out + first, sm.recs(o) + cw * WR, nkeep * 16u, drop);
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

}  // namespace

uint32_t compact_tile_records() { return CmpCfg::kTile; }

cudaError_t launch_compact(const void *records, const uint8_t *flags, uint64_t n, void *out,
                           uint32_t *count, void *scratch, cudaStream_t stream) {
    using C = CmpCfg;
    const LaunchKnobs fault = current_launch_knobs();
    auto kern = compact_kernel<C>;
    const int dev_blocks = device_blocks(reinterpret_cast<const void *>(kern), C::kThreads,
                                         C::kSmemBytes);
    if (dev_blocks <= 0) return cudaErrorInvalidConfiguration;
    const uint64_t tiles = (n + C::kTile - 1) / C::kTile;
    const uint32_t grid = uint32_t(tiles < uint64_t(dev_blocks) ? tiles : uint64_t(dev_blocks));
    auto *hdr = reinterpret_cast<ScratchHeader *>(scratch);
    auto *desc = reinterpret_cast<uint64_t *>(static_cast<unsigned char *>(scratch) + kHeaderBytes);
    return launch_pdl(kern, dim3(grid), dim3(C::kThreads), C::kSmemBytes, stream,
                      reinterpret_cast<const uint4 *>(records), flags, n,
                      reinterpret_cast<uint4 *>(out), count, uint32_t(tiles), hdr, desc, fault);
}

}  // namespace dwp
