// Stable stream compaction of 16-byte records by byte flags, single pass
// with decoupled look-back, for sm_103a.
//
// "Prefix scans and compaction", sections "Scan as an index generator" and
// "Worked example: Stable stream compaction"; "Parallel Prefix Sum (Scan),
// in depth", section "What scan builds": the exclusive scan of the keep
// flags is each kept record's output slot, so kept records keep their order
// and never share a slot; the output length is the flag total.
//
// The pipeline is the plain scan's (scan.cu), over counts:
//   producer warp   per tile, one bulk copy of the records and one of the
//                   flag bytes, completing on the same mbarrier;
//   tile warps      per tile: each consumer thread's kept count, their
//                   exclusive prefix, the tile count published as the
//                   aggregate, a u32-add look-back for the number of records
//                   kept before the tile, the tile's inclusive count
//                   published; the last tile writes the total to *count;
//   consumer warps  thread c owns IT contiguous records.  Each warp reads
//                   its records into registers, writes its kept ones to the
//                   front of its own chunk of the stage buffer, in input
//                   order, and streams that block to its output slots with
//                   one bulk store.
// IT is odd, so 16-byte record reads at a thread stride of 16*IT bytes are
// free of bank conflicts.
#include <cuda_runtime.h>

#include "device.cuh"
#include "launch.h"

namespace dwp {

namespace {

template <int NW_, int IT_, int STAGES_, int LOOKK_>
struct CompactConfig {
    static constexpr int kWarps = NW_;
    static constexpr int kItems = IT_;  // records per consumer thread
    static constexpr int kStages = STAGES_;
    static constexpr int kLookK = LOOKK_;
    static constexpr int kThreads = (1 + STAGES_ + NW_) * 32;
    static constexpr int kConsumers = NW_ * 32;
    static constexpr int kWarpRecs = 32 * IT_;
    static constexpr int kTile = NW_ * 32 * IT_;  // records per tile
    static_assert(IT_ % 2 == 1, "IT must be odd");
    static_assert(kTile % 16 == 0, "flag bytes of a tile must start 16-byte aligned");
    static_assert(NW_ >= 1 && NW_ <= 32, "");
    static constexpr size_t kRecBytes = size_t(kTile) * 16;
    static constexpr size_t kFlagBytes = (size_t(kTile) + 127) / 128 * 128;
    static constexpr size_t kStageBytes = kRecBytes + kFlagBytes;
    static constexpr int kPrefixWords = kConsumers + kConsumers / 8;
    // mbarriers 32 B; tile id, carry, look-back result, tile count 16 B;
    // prefixes; lane totals 33; look-back scratch 33
    static constexpr size_t kStageMeta = 48 + 4 * (kPrefixWords + 33 + 33);
    static constexpr size_t kSmemBytes = (kStageBytes + kStageMeta) * kStages + 16;
    static_assert(kStageBytes % 128 == 0, "stage buffers stay 128-byte aligned");
};

#ifndef DWP_CMP_WARPS
#define DWP_CMP_WARPS 16
#endif
#ifndef DWP_CMP_ITEMS
#define DWP_CMP_ITEMS 5
#endif
#ifndef DWP_CMP_STAGES
#define DWP_CMP_STAGES 4
#endif
using CmpCfg = CompactConfig<DWP_CMP_WARPS, DWP_CMP_ITEMS, DWP_CMP_STAGES, 4>;

template <class C>
struct CmpSmem {
    unsigned char *base;
    __device__ explicit CmpSmem(unsigned char *p) : base(p) {}
    __device__ uint4 *recs(int s) const {
        return reinterpret_cast<uint4 *>(base + size_t(s) * C::kStageBytes);
    }
    __device__ unsigned char *flags(int s) const {
        return base + size_t(s) * C::kStageBytes + C::kRecBytes;
    }
    __device__ unsigned char *meta(int s) const {
        return base + C::kStageBytes * C::kStages + size_t(s) * C::kStageMeta;
    }
    __device__ uint64_t *full(int s) const { return reinterpret_cast<uint64_t *>(meta(s)); }
    __device__ uint64_t *carry_ready(int s) const { return full(s) + 1; }
    __device__ uint64_t *empty(int s) const { return full(s) + 2; }
    __device__ uint32_t *tile_id(int s) const { return reinterpret_cast<uint32_t *>(meta(s) + 32); }
    __device__ uint32_t *carry(int s) const { return tile_id(s) + 1; }
    __device__ uint32_t *lbres(int s) const { return tile_id(s) + 2; }
    __device__ uint32_t *tile_count(int s) const { return tile_id(s) + 3; }
    __device__ uint32_t *prefix(int s) const { return tile_id(s) + 4; }
    __device__ uint32_t *lane_tot(int s) const { return prefix(s) + C::kPrefixWords; }
    __device__ uint32_t *lb_scratch(int s) const { return lane_tot(s) + 33; }
    __device__ uint32_t *abort_flag() const {
        return reinterpret_cast<uint32_t *>(base + (C::kStageBytes + C::kStageMeta) * C::kStages);
    }
    __device__ uint32_t *end_iter() const { return abort_flag() + 1; }
};

// Keep flag of record pos of a tile: from the stage below `fbulk`, from
// global memory below `valid`, else 0.
__device__ __forceinline__ bool keep_at(const unsigned char *sflags, const uint8_t *gflags,
                                        uint64_t base, uint32_t pos, uint32_t fbulk, uint32_t valid) {
    if (pos < fbulk) return sflags[pos] != 0;
    if (pos < valid) return gflags[base + pos] != 0;
    return false;
}

template <class C>
__global__ void __launch_bounds__(C::kThreads, 1)
    compact_kernel(const uint4 *recs, const uint8_t *flags, uint64_t n, uint4 *out,
                   uint32_t *count, uint32_t num_tiles, ScratchHeader *hdr, uint64_t *desc,
                   FaultConfig fault) {
    using Op = OpU32Add;
    constexpr int NW = C::kWarps, IT = C::kItems, STAGES = C::kStages, TILE = C::kTile;
    constexpr int WR = C::kWarpRecs;
    constexpr uint32_t NCONS = C::kConsumers;

    extern __shared__ __align__(128) unsigned char smem_raw[];
    const CmpSmem<C> sm(smem_raw);
    const uint32_t warp = threadIdx.x >> 5, lane = threadIdx.x & 31u;
    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(sm.full(s), 1);
            mbar_init(sm.carry_ready(s), 1);
            mbar_init(sm.empty(s), NW);
        }
        *sm.abort_flag() = 0;
        *sm.end_iter() = kNoTile;
        fence_mbar_init();
    }
    __syncthreads();

    // valid records of tile t, and how many of its flag bytes the bulk copy
    // brings (a multiple of 16; the rest are read from global memory)
    auto tile_extent = [&](uint32_t t, uint32_t &valid, uint32_t &fbulk) {
        const uint64_t rem = n - uint64_t(t) * TILE;
        valid = rem < uint64_t(TILE) ? uint32_t(rem) : uint32_t(TILE);
        fbulk = valid & ~15u;
    };

    if (warp == 0) {
        // ------------------------------------------------------- producer
        if (lane != 0) return;
        for (uint32_t k = 0;; ++k) {
            const int s = int(k % STAGES);
            if (k >= STAGES && !mbar_wait(sm.empty(s), ((k / STAGES) - 1) & 1u, kPipeWaitLimit)) {
                record_error(hdr, DWP_ERR_PIPELINE_TIMEOUT);
                *reinterpret_cast<volatile uint32_t *>(sm.end_iter()) = k - 1;
                return;
            }
            uint32_t t = kNoTile;
            if (ld_volatile_smem(sm.abort_flag()) == 0) {
                t = atomicAdd(&hdr->tile_counter, 1u);
                if (t >= num_tiles) t = kNoTile;
            }
            *reinterpret_cast<volatile uint32_t *>(sm.tile_id(s)) = t;
            if (t == kNoTile) {
                *reinterpret_cast<volatile uint32_t *>(sm.end_iter()) = k;
                mbar_arrive(sm.full(s));
                return;
            }
            uint32_t valid, fbulk;
            tile_extent(t, valid, fbulk);
            const uint64_t base = uint64_t(t) * TILE;
            mbar_arrive_expect_tx(sm.full(s), valid * 16u + fbulk);
            bulk_load(sm.recs(s), recs + base, valid * 16u, sm.full(s));
            if (fbulk) bulk_load(sm.flags(s), flags + base, fbulk, sm.full(s));
        }
    }

    if (warp <= uint32_t(STAGES)) {
        // ----------------------------------------------------- tile warps
        const int s = int(warp) - 1;
        bool draining = false;
        for (uint32_t use = 0;; ++use) {
            const int w = warp_wait_or_end(sm.full(s), use & 1u, use * STAGES + uint32_t(s),
                                           sm.end_iter());
            if (w != 2) {
                if (w == 0 && lane == 0) record_error(hdr, DWP_ERR_PIPELINE_TIMEOUT);
                return;
            }
            const uint32_t t = ld_volatile_smem(sm.tile_id(s));
            if (t == kNoTile) {
                if (lane == 0) mbar_arrive(sm.carry_ready(s));
                return;
            }
            if (!draining && ld_volatile_smem(sm.abort_flag()) != 0) draining = true;
            if (draining) {
                if (lane == 0) {
                    st_relaxed_gpu(desc + t, make_desc(kPoison, 0u));
                    *sm.lbres(s) = 1u;
                    mbar_arrive(sm.carry_ready(s));
                }
                __syncwarp();
                continue;
            }
            uint32_t valid, fbulk;
            tile_extent(t, valid, fbulk);
            const uint64_t base = uint64_t(t) * TILE;
            const unsigned char *sf = sm.flags(s);
            uint32_t *pre = sm.prefix(s);
            uint32_t *lt = sm.lane_tot(s);
            // K1: kept count of consumer thread c = lane + 32w (records c*IT ..)
#pragma unroll
            for (int w = 0; w < NW; ++w) {
                const uint32_t c = lane + 32u * w;
                uint32_t cnt = 0;
                if (valid == uint32_t(TILE)) {
#pragma unroll
                    for (int j = 0; j < IT; ++j) cnt += sf[c * IT + j] != 0;
                } else {
                    for (int j = 0; j < IT; ++j) cnt += keep_at(sf, flags, base, c * IT + j, fbulk, valid);
                }
                pre[prefix_slot(c)] = cnt;
            }
            __syncwarp();
            // K2: exclusive prefix of the counts (lane l: threads PER*l ..)
            constexpr int PER = NCONS / 32;
            uint32_t mine[PER], run = 0;
#pragma unroll
            for (int j = 0; j < PER; ++j) {
                mine[j] = run;
                run += pre[prefix_slot(lane * PER + j)];
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
#pragma unroll
            for (int j = 0; j < PER; ++j) pre[prefix_slot(lane * PER + j)] = lane_excl + mine[j];
            if (lane == 0 && t != fault.never_publish_tile)
                st_relaxed_gpu(desc + t, make_desc(t == 0 ? kPrefix : kAggregate, total));
            uint32_t carry = 0;
            int rc = 0;
            if (t != 0) rc = lookback<Op, C::kLookK>(desc, t, lane, fault.spin_limit, sm.lb_scratch(s), &carry);
            if (lane == 0) {
                if (rc == 0) {
                    if (t != 0 && t != fault.never_publish_tile)
                        st_relaxed_gpu(desc + t, make_desc(kPrefix, carry + total));
                    if (t == num_tiles - 1) *count = carry + total;  // K4: output length
                } else {
                    st_relaxed_gpu(desc + t, make_desc(kPoison, 0u));
                    if (rc == 2) record_error(hdr, DWP_ERR_LOOKBACK_TIMEOUT);
                    *reinterpret_cast<volatile uint32_t *>(sm.abort_flag()) = 1u;
                }
                *sm.carry(s) = carry;
                *sm.tile_count(s) = total;
                *sm.lbres(s) = uint32_t(rc);
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(sm.carry_ready(s));
            if (rc != 0) draining = true;
        }
    }

    // ---------------------------------------------------------- consumers
    const uint32_t cw = warp - 1 - STAGES;
    const uint32_t c = cw * 32 + lane;
    int pending = -1;
    for (uint32_t k = 0;; ++k) {
        const int s = int(k % STAGES);
        const uint32_t par = (k / STAGES) & 1u;
        const int w = warp_wait_or_end(sm.full(s), par, k, sm.end_iter());
        if (w != 2 || !warp_wait(sm.carry_ready(s), par)) {
            if (w != 1 && lane == 0) record_error(hdr, DWP_ERR_PIPELINE_TIMEOUT);
            break;
        }
        const uint32_t t = ld_volatile_smem(sm.tile_id(s));
        if (t == kNoTile) break;
        uint32_t nkeep = 0, first = 0;  // this warp's kept records and its first output slot
        if (ld_volatile_smem(sm.lbres(s)) == 0u) {
            uint32_t valid, fbulk;
            tile_extent(t, valid, fbulk);
            const uint64_t base = uint64_t(t) * TILE;
            uint4 *region = sm.recs(s) + cw * WR;
            const uint32_t *pre = sm.prefix(s);
            const uint32_t wfirst = pre[prefix_slot(cw * 32)];
            const uint32_t wend =
                cw + 1 < uint32_t(NW) ? pre[prefix_slot(cw * 32 + 32)] : *sm.tile_count(s);
            nkeep = wend - wfirst;
            first = *sm.carry(s) + wfirst;
            // K3: read this thread's records, then (after the whole warp has
            // read) write the kept ones to their in-warp slots, in order
            uint4 r[IT];
            uint32_t keepm = 0;
#pragma unroll
            for (int j = 0; j < IT; ++j) {
                const uint32_t pos = c * IT + j;
                if (pos < valid) r[j] = sm.recs(s)[pos];
                if (keep_at(sm.flags(s), flags, base, pos, fbulk, valid)) keepm |= 1u << j;
            }
            __syncwarp();
            uint32_t slot = pre[prefix_slot(c)] - wfirst;
#pragma unroll
            for (int j = 0; j < IT; ++j)
                if ((keepm >> j) & 1u) region[slot++] = r[j];
            fence_proxy_async_smem();
        }
        __syncwarp();
        if (lane == 0) {
            if (nkeep) {
                bulk_store(out + first, sm.recs(s) + cw * WR, nkeep * 16u);
                bulk_commit();
                bulk_wait_read<1>();
                if (pending >= 0) mbar_arrive(sm.empty(pending));
                pending = s;
            } else {
                bulk_wait_read<0>();
                if (pending >= 0) mbar_arrive(sm.empty(pending));
                mbar_arrive(sm.empty(s));
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
    const FaultConfig fault = current_fault_config();
    auto kern = compact_kernel<C>;
    const int dev_blocks = device_blocks(reinterpret_cast<const void *>(kern), C::kThreads,
                                         C::kSmemBytes);
    if (dev_blocks <= 0) return cudaErrorInvalidConfiguration;
    const uint64_t tiles = (n + C::kTile - 1) / C::kTile;
    const uint32_t grid = uint32_t(tiles < uint64_t(dev_blocks) ? tiles : uint64_t(dev_blocks));
    auto *hdr = reinterpret_cast<ScratchHeader *>(scratch);
    auto *desc = reinterpret_cast<uint64_t *>(static_cast<unsigned char *>(scratch) + kHeaderBytes);
    kern<<<grid, C::kThreads, C::kSmemBytes, stream>>>(
        reinterpret_cast<const uint4 *>(records), flags, n, reinterpret_cast<uint4 *>(out), count,
        uint32_t(tiles), hdr, desc, fault);
    return cudaGetLastError();
}

}  // namespace dwp
