// Single-pass chained scan with decoupled look-back for sm_103a.
//
// One persistent, warp-specialised launch ("Single-Pass Prefix Scan with
// Decoupled Look-Back"; "Parallel Prefix Sum (Scan), in depth", sections "A
// CUDA scan: warp, block, grid" and "Scanning a whole array: three grid
// strategies").  A block owns a ring of STAGES tile buffers in shared memory:
//
//   producer warp   takes tile indices from the atomic counter in the order
//                   tiles start and streams each tile global -> shared with
//                   one bulk (TMA) copy;
//   tile warps      one per stage.  For its tile: every consumer thread's
//                   total and their exclusive prefix (block layer), the
//                   aggregate published as soon as the data has landed, the
//                   look-back, the inclusive prefix published, the carry
//                   handed over.  With one warp per stage a block has up to
//                   STAGES look-backs in flight, so a slow predecessor
//                   delays only the tiles that need it;
//   consumer warps  warp w owns chunk w of every tile; each thread scans its
//                   ITEMS contiguous elements serially from carry + its
//                   in-tile prefix, writes them back in place, and the warp
//                   streams its chunk shared -> global with one bulk store.
//
// ITEMS is an odd multiple of 4, so the 16-byte shared-memory accesses of a
// quarter warp (thread stride 16*odd bytes) fall in 8 distinct bank groups.
// No block-wide barrier is used after set-up: warps meet only at mbarriers,
// and every wait is bounded.
#include <cuda_runtime.h>

#include "device.cuh"
#include "launch.h"

namespace dwp {

template <int NW_, int ITEMS_, int STAGES_, int LOOKK_, int MINB_>
struct ScanConfig {
    static constexpr int kWarps = NW_;        // consumer warps (one chunk of the tile each)
    static constexpr int kItems = ITEMS_;     // contiguous elements per consumer thread
    static constexpr int kStages = STAGES_;   // shared-memory ring depth = tile warps
    static constexpr int kLookK = LOOKK_;     // look-back sub-windows of 32 per round
    static constexpr int kMinBlocks = MINB_;  // resident blocks per SM the registers allow
    static constexpr int kThreads = (1 + STAGES_ + NW_) * 32;
    static constexpr int kConsumers = NW_ * 32;
    static constexpr int kWarpElems = 32 * ITEMS_;
    static constexpr int kTile = NW_ * 32 * ITEMS_;
    static_assert(ITEMS_ % 4 == 0 && (ITEMS_ / 4) % 2 == 1, "ITEMS must be an odd multiple of 4");
    static_assert(NW_ >= 1 && NW_ <= 32, "one 32-slot row of thread totals per consumer warp");
    static constexpr size_t kStageBytes = size_t(kTile) * 4;
    // Per stage after the data: 3 mbarriers (+pad, 32 B); tile id, aggregate,
    // carry, look-back result (16 B); thread prefixes, one word per consumer
    // thread plus one pad word per 8 (bank spread); 33 lane totals; 33 words
    // of look-back scratch.
    static constexpr int kPrefixWords = kConsumers + kConsumers / 8;
    static constexpr size_t kStageMeta = 48 + 4 * (kPrefixWords + 33 + 33);
    // + abort flag and end iteration
    static constexpr size_t kSmemBytes = (kStageBytes + kStageMeta) * kStages + 16;
};

#ifndef DWP_SCAN_WARPS
#define DWP_SCAN_WARPS 16
#endif
#ifndef DWP_SCAN_ITEMS
#define DWP_SCAN_ITEMS 20
#endif
#ifndef DWP_SCAN_STAGES
#define DWP_SCAN_STAGES 5
#endif
#ifndef DWP_SCAN_LOOKK
#define DWP_SCAN_LOOKK 4
#endif
#ifndef DWP_SCAN_MINB
#define DWP_SCAN_MINB 1
#endif
using ScanCfg = ScanConfig<DWP_SCAN_WARPS, DWP_SCAN_ITEMS, DWP_SCAN_STAGES, DWP_SCAN_LOOKK,
                           DWP_SCAN_MINB>;

// Shared-memory layout of one block.
template <class C>
struct ScanSmem {
    unsigned char *base;
    __device__ explicit ScanSmem(unsigned char *p) : base(p) {}
    __device__ uint32_t *data(int s) const {
        return reinterpret_cast<uint32_t *>(base + size_t(s) * C::kStageBytes);
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
    __device__ uint32_t *prefix(int s) const { return tile_id(s) + 4; }
    __device__ uint32_t *lane_tot(int s) const { return prefix(s) + C::kPrefixWords; }
    __device__ uint32_t *lb_scratch(int s) const { return lane_tot(s) + 33; }
    __device__ uint32_t *abort_flag() const {
        return reinterpret_cast<uint32_t *>(base + (C::kStageBytes + C::kStageMeta) * C::kStages);
    }
    // first ring iteration that holds no tile (set once by the producer)
    __device__ uint32_t *end_iter() const { return abort_flag() + 1; }
};

// Element pos of a tile: from the stage buffer below `bulk`, from global
// memory below `valid` (the ragged tail the bulk copy cannot cover), else the
// identity.
template <class Op>
__device__ __forceinline__ typename Op::T tile_elem(const uint32_t *buf, const typename Op::T *in,
                                                    uint64_t base, uint32_t pos, uint32_t bulk,
                                                    uint32_t valid) {
    if (pos < bulk) return Op::from_bits(buf[pos]);
    if (pos < valid) return in[base + pos];
    return Op::identity();
}

template <class Op, bool INCL, class C>
__global__ void __launch_bounds__(C::kThreads, C::kMinBlocks)
    scan_kernel(const typename Op::T *in, typename Op::T *out, uint64_t n, uint32_t num_tiles,
                ScratchHeader *hdr, uint64_t *desc, FaultConfig fault) {
    using T = typename Op::T;
    constexpr int NW = C::kWarps, ITEMS = C::kItems, STAGES = C::kStages, TILE = C::kTile;
    constexpr int WE = C::kWarpElems;
    constexpr uint32_t NCONS = C::kConsumers;

    extern __shared__ __align__(128) unsigned char smem_raw[];
    const ScanSmem<C> sm(smem_raw);
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

    auto tile_extent = [&](uint32_t t, uint32_t &valid, uint32_t &bulk) {
        const uint64_t rem = n - uint64_t(t) * TILE;
        valid = rem < uint64_t(TILE) ? uint32_t(rem) : uint32_t(TILE);
        bulk = valid == uint32_t(TILE) ? valid : (valid & ~3u);
    };

    if (warp == 0) {
        // ------------------------------------------------------- producer
        // Tile indices come from the atomic counter in the order tiles start
        // ("Scanning a whole array: three grid strategies"), so a tile only
        // ever waits for tiles that some running block already holds.
        if (lane != 0) return;
        for (uint32_t k = 0;; ++k) {
            const int s = int(k % STAGES);
            if (k >= STAGES && !mbar_wait(sm.empty(s), ((k / STAGES) - 1) & 1u, kPipeWaitLimit)) {
                record_error(hdr, DWP_ERR_PIPELINE_TIMEOUT);
                // the stage is still in use: leave it alone, and let every
                // warp waiting for iteration k or later stop
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
                // iteration k carries the sentinel to its tile warp and the
                // consumers; warps waiting for later iterations see end_iter
                *reinterpret_cast<volatile uint32_t *>(sm.end_iter()) = k;
                mbar_arrive(sm.full(s));
                return;
            }
            uint32_t valid, bulk;
            tile_extent(t, valid, bulk);
            const uint32_t bytes = bulk * 4u;
            if (bytes) {
                mbar_arrive_expect_tx(sm.full(s), bytes);
                bulk_load(sm.data(s), in + uint64_t(t) * TILE, bytes, sm.full(s));
            } else {
                mbar_arrive(sm.full(s));
            }
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
                // an earlier tile of this block gave up: poison this one so
                // no successor waits for it, and let the consumers skip it
                if (lane == 0) {
                    st_relaxed_gpu(desc + t, make_desc(kPoison, 0u));
                    *sm.lbres(s) = 1u;
                    mbar_arrive(sm.carry_ready(s));
                }
                __syncwarp();
                continue;
            }
            uint32_t valid, bulk;
            tile_extent(t, valid, bulk);
            const uint64_t base = uint64_t(t) * TILE;
            const uint32_t *buf = sm.data(s);
            uint32_t *pre = sm.prefix(s);
            uint32_t *lt = sm.lane_tot(s);
            // totals of consumer threads c = lane + 32*w, whose ITEMS
            // contiguous elements start at c*ITEMS
            T tot[NW];
            if (valid == uint32_t(TILE)) {
                const uint4 *v4 = reinterpret_cast<const uint4 *>(buf);
#pragma unroll
                for (int w = 0; w < NW; ++w) {
                    const uint32_t c = lane + 32u * w;
                    T acc = Op::identity();
#pragma unroll
                    for (int v = 0; v < ITEMS / 4; ++v) {
                        const uint4 q = v4[c * (ITEMS / 4) + v];
                        acc = Op::combine(acc, Op::combine(Op::combine(Op::from_bits(q.x), Op::from_bits(q.y)),
                                                           Op::combine(Op::from_bits(q.z), Op::from_bits(q.w))));
                    }
                    tot[w] = acc;
                }
            } else {
#pragma unroll
                for (int w = 0; w < NW; ++w) {
                    const uint32_t c = lane + 32u * w;
                    T acc = Op::identity();
                    for (int j = 0; j < ITEMS; ++j)
                        acc = Op::combine(acc, tile_elem<Op>(buf, in, base, c * ITEMS + j, bulk, valid));
                    tot[w] = acc;
                }
            }
#pragma unroll
            for (int w = 0; w < NW; ++w) pre[prefix_slot(lane + 32u * w)] = Op::to_bits(tot[w]);
            __syncwarp();
            // lane l scans the NW consecutive thread totals NW*l .. NW*l+NW-1
            // (padded slots; for NW = 8 word 9l+j, banks all distinct) ...
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
            if (lane == 0 && t != fault.never_publish_tile)
                st_relaxed_gpu(desc + t, make_desc(t == 0 ? kPrefix : kAggregate, Op::to_bits(agg)));
            // grid layer
            T carry = Op::identity();
            int rc = 0;
            if (t != 0)
                rc = lookback<Op, C::kLookK>(desc, t, lane, fault.spin_limit, sm.lb_scratch(s), &carry);
            if (lane == 0) {
                if (rc == 0) {
                    if (t != 0 && t != fault.never_publish_tile)
                        st_relaxed_gpu(desc + t, make_desc(kPrefix, Op::to_bits(Op::combine(carry, agg))));
                } else {
                    // give up on this tile: poison it so no successor waits
                    st_relaxed_gpu(desc + t, make_desc(kPoison, 0u));
                    if (rc == 2) record_error(hdr, DWP_ERR_LOOKBACK_TIMEOUT);
                    *reinterpret_cast<volatile uint32_t *>(sm.abort_flag()) = 1u;
                }
                *sm.carry(s) = Op::to_bits(carry);
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
    int pending = -1;  // lane 0: stage whose bulk store may still read smem
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
        if (ld_volatile_smem(sm.lbres(s)) != 0u) {
            if (lane == 0) {
                bulk_wait_read<0>();
                if (pending >= 0) mbar_arrive(sm.empty(pending));
                mbar_arrive(sm.empty(s));
                pending = -1;
            }
            __syncwarp();
            continue;
        }
        uint32_t valid, bulk;
        tile_extent(t, valid, bulk);
        const uint64_t base = uint64_t(t) * TILE;
        uint32_t *buf = sm.data(s);
        const uint32_t p0 = c * ITEMS;  // this thread's first element
        T acc = Op::combine(Op::from_bits(*sm.carry(s)), Op::from_bits(sm.prefix(s)[prefix_slot(c)]));
        if (valid == uint32_t(TILE)) {
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
        } else {
            for (int j = 0; j < ITEMS; ++j) {
                const uint32_t pos = p0 + j;
                const T xv = tile_elem<Op>(buf, in, base, pos, bulk, valid);
                T yv;
                if (INCL) {
                    acc = Op::combine(acc, xv);
                    yv = acc;
                } else {
                    yv = acc;
                    acc = Op::combine(acc, xv);
                }
                if (pos < bulk)
                    buf[pos] = Op::to_bits(yv);
                else if (pos < valid)
                    out[base + pos] = yv;
            }
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
            const uint32_t w0 = cw * WE;
            const uint32_t w1 = min(w0 + uint32_t(WE), bulk);
            if (w1 > w0) {
                bulk_store(out + base + w0, buf + w0, (w1 - w0) * 4u);
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

// ------------------------------------------------------------------ host

namespace {

template <class Op, bool INCL>
cudaError_t launch_one(const void *in, void *out, uint64_t n, void *scratch, cudaStream_t stream,
                       const FaultConfig &fault) {
    using C = ScanCfg;
    auto kern = scan_kernel<Op, INCL, C>;
    const int dev_blocks = device_blocks(reinterpret_cast<const void *>(kern), C::kThreads,
                                         C::kSmemBytes);
    if (dev_blocks <= 0) return cudaErrorInvalidConfiguration;
    const uint64_t tiles = (n + C::kTile - 1) / C::kTile;
    const uint32_t grid = uint32_t(tiles < uint64_t(dev_blocks) ? tiles : uint64_t(dev_blocks));
    auto *hdr = reinterpret_cast<ScratchHeader *>(scratch);
    auto *desc = reinterpret_cast<uint64_t *>(static_cast<unsigned char *>(scratch) + kHeaderBytes);
    kern<<<grid, C::kThreads, C::kSmemBytes, stream>>>(
        reinterpret_cast<const typename Op::T *>(in), reinterpret_cast<typename Op::T *>(out), n,
        uint32_t(tiles), hdr, desc, fault);
    return cudaGetLastError();
}

}  // namespace

uint32_t scan_tile_elems() { return ScanCfg::kTile; }

cudaError_t launch_scan(dwp_op op, bool inclusive, const void *in, void *out, uint64_t n,
                        void *scratch, cudaStream_t stream) {
    const FaultConfig fault = current_fault_config();
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
