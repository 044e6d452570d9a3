// Single-pass chained scan with decoupled look-back for sm_103a.
//
// One persistent, warp-specialised launch ("Single-Pass Prefix Scan with
// Decoupled Look-Back"; "Parallel Prefix Sum (Scan), in depth", sections "A
// CUDA scan: warp, block, grid" and "Scanning a whole array: three grid
// strategies"):
//
//   producer warp   takes tile indices from the atomic counter in the order
//                   tiles start, and streams each tile global -> shared with
//                   one bulk (TMA) copy into a ring of STAGES buffers;
//   consumer warps  per tile: thread-serial scan of ITEMS contiguous
//                   elements in registers, warp shuffle scan of the thread
//                   totals, block combine of the warp totals through shared
//                   memory; warp 0 publishes the tile aggregate, looks back
//                   32 predecessors per round and publishes the inclusive
//                   prefix; every thread folds the carry into its elements,
//                   writes them back in place and each warp streams its slice
//                   shared -> global with one bulk store.
//
// ITEMS is an odd multiple of 4 so the 16-byte shared-memory accesses of a
// quarter warp fall in 8 distinct bank groups (thread stride 16*odd bytes).
#include <cuda_runtime.h>

#include <mutex>

#include "device.cuh"
#include "launch.h"

namespace dwp {

constexpr uint32_t kNoTile = 0xffffffffu;

template <int NW_, int ITEMS_, int STAGES_>
struct ScanConfig {
    static constexpr int kWarps = NW_;
    static constexpr int kItems = ITEMS_;
    static constexpr int kStages = STAGES_;
    static constexpr int kThreads = (NW_ + 1) * 32;
    static constexpr int kConsumers = NW_ * 32;
    static constexpr int kWarpElems = 32 * ITEMS_;
    static constexpr int kTile = NW_ * 32 * ITEMS_;
    static_assert(ITEMS_ % 4 == 0 && (ITEMS_ / 4) % 2 == 1, "ITEMS must be an odd multiple of 4");
    // stage buffers, then full/empty barriers, tile ids, warp totals, carry,
    // look-back result, abort flag
    static constexpr size_t kStageBytes = size_t(kTile) * 4;
    static constexpr size_t kSmemBytes =
        kStageBytes * kStages + 16 * kStages + 4 * kStages + 4 * NW_ + 16;
};

#ifndef DWP_SCAN_WARPS
#define DWP_SCAN_WARPS 8
#endif
#ifndef DWP_SCAN_ITEMS
#define DWP_SCAN_ITEMS 20
#endif
#ifndef DWP_SCAN_STAGES
#define DWP_SCAN_STAGES 4
#endif
using ScanCfg = ScanConfig<DWP_SCAN_WARPS, DWP_SCAN_ITEMS, DWP_SCAN_STAGES>;

// barrier.red.and over the consumer threads: true iff every thread passed true.
__device__ __forceinline__ bool consumers_all(bool v, uint32_t nthreads) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 p, %1, 0;\n\t"
        "bar.red.and.pred q, 1, %2, p;\n\t"
        "selp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"(uint32_t(v)), "r"(nthreads)
        : "memory");
    return r != 0;
}

template <class Op, bool INCL, class C>
__global__ void __launch_bounds__(C::kThreads, 1)
    scan_kernel(const typename Op::T *in, typename Op::T *out, uint64_t n, uint32_t num_tiles,
                ScratchHeader *hdr, uint64_t *desc, FaultConfig fault) {
    using T = typename Op::T;
    constexpr int NW = C::kWarps, ITEMS = C::kItems, STAGES = C::kStages, TILE = C::kTile;
    constexpr uint32_t NCONS = C::kConsumers;

    extern __shared__ __align__(128) unsigned char smem[];
    T *stage_buf = reinterpret_cast<T *>(smem);
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + C::kStageBytes * STAGES);
    uint64_t *empty = full + STAGES;
    uint32_t *tile_id = reinterpret_cast<uint32_t *>(empty + STAGES);
    uint32_t *warp_tot = tile_id + STAGES;
    uint32_t *carry_sm = warp_tot + NW;
    uint32_t *lbres_sm = carry_sm + 1;
    uint32_t *abort_sm = carry_sm + 2;

    const uint32_t warp = threadIdx.x >> 5, lane = threadIdx.x & 31u;
    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], NW);
        }
        *abort_sm = 0;
        fence_mbar_init();
    }
    __syncthreads();

    // ------------------------------------------------------------- producer
    if (warp == NW) {
        if (lane != 0) return;
        for (uint32_t k = 0;; ++k) {
            const uint32_t s = k % STAGES;
            if (k >= STAGES && !mbar_wait(&empty[s], ((k / STAGES) - 1) & 1u, kPipeWaitLimit)) {
                // The consumers still hold stage s: leave it alone and stop.
                record_error(hdr, DWP_ERR_PIPELINE_TIMEOUT);
                return;
            }
            uint32_t t = kNoTile;
            if (ld_volatile_smem(abort_sm) == 0) {
                t = atomicAdd(&hdr->tile_counter, 1u);
                if (t >= num_tiles) t = kNoTile;
            }
            *reinterpret_cast<volatile uint32_t *>(&tile_id[s]) = t;
            if (t == kNoTile) {
                mbar_arrive(&full[s]);
                return;
            }
            const uint64_t base = uint64_t(t) * TILE;
            const uint64_t rem = n - base;
            const uint32_t valid = rem < uint64_t(TILE) ? uint32_t(rem) : uint32_t(TILE);
            const uint32_t bytes = (valid * uint32_t(sizeof(T))) & ~15u;
            if (bytes) {
                mbar_arrive_expect_tx(&full[s], bytes);
                bulk_load(stage_buf + size_t(s) * TILE, in + base, bytes, &full[s]);
            } else {
                mbar_arrive(&full[s]);
            }
        }
    }

    // ------------------------------------------------------------ consumers
    const uint32_t tid = threadIdx.x;  // 0 .. NCONS-1
    int pending = -1;                  // lane 0: stage whose bulk store may still read smem
    bool draining = false;
    for (uint32_t k = 0;; ++k) {
        const uint32_t s = k % STAGES;
        const bool ok = mbar_wait(&full[s], (k / STAGES) & 1u, kPipeWaitLimit);
        const uint32_t t = ld_volatile_smem(&tile_id[s]);
        const bool have = ok && t < num_tiles && !draining;
        T *buf = stage_buf + size_t(s) * TILE;
        const uint64_t base = uint64_t(t) * TILE;
        uint32_t valid = TILE, bulk_elems = TILE;

        T x[ITEMS];
        T thread_excl = Op::identity();
        if (have) {
            const uint64_t rem = n - base;
            if (rem < uint64_t(TILE)) {
                valid = uint32_t(rem);
                bulk_elems = valid & ~3u;
            }
            if (valid == uint32_t(TILE)) {
                const uint4 *src = reinterpret_cast<const uint4 *>(buf + tid * ITEMS);
#pragma unroll
                for (int v = 0; v < ITEMS / 4; ++v) {
                    const uint4 q = src[v];
                    x[4 * v + 0] = Op::from_bits(q.x);
                    x[4 * v + 1] = Op::from_bits(q.y);
                    x[4 * v + 2] = Op::from_bits(q.z);
                    x[4 * v + 3] = Op::from_bits(q.w);
                }
            } else {
#pragma unroll
                for (int j = 0; j < ITEMS; ++j) {
                    const uint32_t pos = tid * ITEMS + j;
                    x[j] = pos < bulk_elems ? buf[pos]
                                            : (pos < valid ? in[base + pos] : Op::identity());
                }
            }
            // thread-serial inclusive scan in registers
#pragma unroll
            for (int j = 1; j < ITEMS; ++j) x[j] = Op::combine(x[j - 1], x[j]);
            // warp layer over the thread totals
            const T winc = warp_inclusive_scan<Op>(x[ITEMS - 1], lane);
            const T up = __shfl_up_sync(0xffffffffu, winc, 1);
            thread_excl = lane ? up : Op::identity();
            if (lane == 31) warp_tot[warp] = Op::to_bits(winc);
        }
        // Barrier A: warp totals written; every thread's wait outcome combined
        // so the decision to stop is the same in every thread.
        if (!consumers_all(ok, NCONS)) {
            if (tid == 0) record_error(hdr, DWP_ERR_PIPELINE_TIMEOUT);
            break;
        }
        if (t >= num_tiles) break;

        if (draining) {
            // An earlier tile of this block gave up: mark this tile poisoned
            // so that no successor waits for it, and hand the stage back.
            if (tid == 0) st_release_gpu(desc + t, make_desc(kPoison, 0u));
            if (lane == 0) {
                bulk_wait_read<0>();
                if (pending >= 0) mbar_arrive(&empty[pending]);
                mbar_arrive(&empty[s]);
                pending = -1;
            }
            continue;
        }

        // block layer: this warp's exclusive prefix and the tile aggregate
        T warp_excl = Op::identity(), agg = Op::identity();
#pragma unroll
        for (int w = 0; w < NW; ++w) {
            const T wt = Op::from_bits(warp_tot[w]);
            if (w < int(warp)) warp_excl = Op::combine(warp_excl, wt);
            agg = Op::combine(agg, wt);
        }

        // grid layer: publish, look back, publish (warp 0)
        if (warp == 0) {
            const bool publish = (t != fault.never_publish_tile);
            T carry = Op::identity();
            int rc = 0;
            if (t == 0) {
                if (lane == 0 && publish) st_release_gpu(desc, make_desc(kPrefix, Op::to_bits(agg)));
            } else {
                if (lane == 0 && publish)
                    st_release_gpu(desc + t, make_desc(kAggregate, Op::to_bits(agg)));
                rc = lookback<Op>(desc, t, lane, fault.spin_limit, &carry);
                if (lane == 0) {
                    if (rc == 0) {
                        if (publish)
                            st_release_gpu(desc + t,
                                           make_desc(kPrefix, Op::to_bits(Op::combine(carry, agg))));
                    } else {
                        st_release_gpu(desc + t, make_desc(kPoison, 0u));
                        if (rc == 2) record_error(hdr, DWP_ERR_LOOKBACK_TIMEOUT);
                    }
                }
            }
            if (lane == 0) {
                *carry_sm = Op::to_bits(carry);
                *lbres_sm = uint32_t(rc);
            }
        }
        named_barrier(2, NCONS);  // Barrier B: carry and look-back result visible
        const T carry = Op::from_bits(*carry_sm);
        if (*lbres_sm != 0u) {
            draining = true;
            if (tid == 0) *reinterpret_cast<volatile uint32_t *>(abort_sm) = 1u;
            if (lane == 0) {
                bulk_wait_read<0>();
                if (pending >= 0) mbar_arrive(&empty[pending]);
                mbar_arrive(&empty[s]);
                pending = -1;
            }
            continue;
        }

        // fold the carry in and write back in place
        const T pre = Op::combine(Op::combine(carry, warp_excl), thread_excl);
        T y[ITEMS];
        if (INCL) {
#pragma unroll
            for (int j = 0; j < ITEMS; ++j) y[j] = Op::combine(pre, x[j]);
        } else {
            y[0] = pre;
#pragma unroll
            for (int j = 1; j < ITEMS; ++j) y[j] = Op::combine(pre, x[j - 1]);
        }
        if (valid == uint32_t(TILE)) {
            uint4 *dst = reinterpret_cast<uint4 *>(buf + tid * ITEMS);
#pragma unroll
            for (int v = 0; v < ITEMS / 4; ++v)
                dst[v] = make_uint4(Op::to_bits(y[4 * v + 0]), Op::to_bits(y[4 * v + 1]),
                                    Op::to_bits(y[4 * v + 2]), Op::to_bits(y[4 * v + 3]));
        } else {
#pragma unroll
            for (int j = 0; j < ITEMS; ++j) {
                const uint32_t pos = tid * ITEMS + j;
                if (pos < bulk_elems)
                    buf[pos] = y[j];
                else if (pos < valid)
                    out[base + pos] = y[j];
            }
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
            const uint32_t w0 = warp * C::kWarpElems;
            const uint32_t w1 = min(w0 + uint32_t(C::kWarpElems), bulk_elems);
            if (w1 > w0) {
                bulk_store(out + base + w0, buf + w0, (w1 - w0) * uint32_t(sizeof(T)));
                bulk_commit();
                bulk_wait_read<1>();
                if (pending >= 0) mbar_arrive(&empty[pending]);
                pending = int(s);
            } else {
                bulk_wait_read<0>();
                if (pending >= 0) mbar_arrive(&empty[pending]);
                mbar_arrive(&empty[s]);
                pending = -1;
            }
        }
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
