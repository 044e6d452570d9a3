// Device building blocks shared by the scan, segmented-scan and compaction
// kernels: sm_103a inline PTX for mbarriers, bulk (TMA) copies, proxy fences
// and acquire/release descriptor traffic; the associative operators; the
// warp and block scan layers; and the warp-parallel decoupled look-back.
#pragma once

#include <cstdint>

#include "common.h"

namespace dwp {

// ---------------------------------------------------------------------------
// Operators.  "Parallel Prefix Sum (Scan), in depth", "Inclusive, exclusive
// and associative": any associative operator; "Prefix scans and compaction",
// "Inclusive and exclusive scan": identities 0 for addition, lowest value for
// a maximum.  combine(a, b) keeps operand order: a covers earlier elements.

struct OpU32Add {
    using T = uint32_t;
    static __device__ __forceinline__ T identity() { return 0u; }
    static __device__ __forceinline__ T combine(T a, T b) { return a + b; }
    static __device__ __forceinline__ uint32_t to_bits(T v) { return v; }
    static __device__ __forceinline__ T from_bits(uint32_t b) { return b; }
};

struct OpU32Max {
    using T = uint32_t;
    static __device__ __forceinline__ T identity() { return 0u; }
    static __device__ __forceinline__ T combine(T a, T b) { return a > b ? a : b; }
    static __device__ __forceinline__ uint32_t to_bits(T v) { return v; }
    static __device__ __forceinline__ T from_bits(uint32_t b) { return b; }
};

struct OpF32Add {
    using T = float;
    static __device__ __forceinline__ T identity() { return 0.0f; }
    static __device__ __forceinline__ T combine(T a, T b) { return __fadd_rn(a, b); }
    static __device__ __forceinline__ uint32_t to_bits(T v) { return __float_as_uint(v); }
    static __device__ __forceinline__ T from_bits(uint32_t b) { return __uint_as_float(b); }
};

// ---------------------------------------------------------------------------
// Small PTX wrappers.

__device__ __forceinline__ uint32_t smem_addr(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count)
                 : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_addr(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Bounded wait for the phase with the given parity; false after `limit` polls.
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity, uint32_t limit) {
    for (uint32_t i = 0; i < limit; ++i) {
        if (mbar_try_wait(bar, parity)) return true;
        if (i >= 8) __nanosleep(64);
    }
    return false;
}

// Bulk global -> shared copy completing `bytes` on the mbarrier.  Addresses
// 16-byte aligned, bytes a nonzero multiple of 16.
__device__ __forceinline__ void bulk_load(void *smem_dst, const void *gmem_src, uint32_t bytes,
                                          uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
            "r"(smem_addr(smem_dst)),
        "l"(gmem_src), "r"(bytes), "r"(smem_addr(bar))
        : "memory");
}

// Bulk shared -> global copy in the current bulk async-group.
__device__ __forceinline__ void bulk_store(void *gmem_dst, const void *smem_src, uint32_t bytes) {
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(gmem_dst),
                 "r"(smem_addr(smem_src)), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void bulk_commit() {
    asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}

// Wait until at most N committed bulk groups are still reading shared memory.
template <int N>
__device__ __forceinline__ void bulk_wait_read() {
    asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}

// Wait until at most N committed bulk groups are incomplete (writes done).
template <int N>
__device__ __forceinline__ void bulk_wait_all() {
    asm volatile("cp.async.bulk.wait_group %0;" ::"n"(N) : "memory");
}

// Make this thread's generic-proxy shared-memory writes visible to the async
// proxy (bulk stores read shared memory through it).
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Barrier among the `nthreads` threads (a multiple of 32) that use `id`.
__device__ __forceinline__ void named_barrier(uint32_t id, uint32_t nthreads) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// Descriptor publication and reading: one 64-bit word, release store and
// acquire load at device (.gpu) scope ("Single-Pass Prefix Scan with
// Decoupled Look-Back", "The publication protocol in code": device scope
// suffices; the reader loads the whole word so flag and value never mix).
__device__ __forceinline__ void st_release_gpu(uint64_t *p, uint64_t v) {
    asm volatile("st.release.gpu.global.b64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}

__device__ __forceinline__ uint64_t ld_acquire_gpu(const uint64_t *p) {
    uint64_t v;
    asm volatile("ld.acquire.gpu.global.b64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}

// Plain (non-acquire) volatile read of a shared-memory word.
__device__ __forceinline__ uint32_t ld_volatile_smem(const uint32_t *p) {
    return *reinterpret_cast<const volatile uint32_t *>(p);
}

// Record a device-side error in the scratch status word (first error wins).
__device__ __forceinline__ void record_error(ScratchHeader *hdr, uint32_t code) {
    atomicCAS(&hdr->status, 0u, code);
}

// ---------------------------------------------------------------------------
// Tile descriptor ("Single-Pass Prefix Scan with Decoupled Look-Back",
// "Three states in a per-block descriptor"): state in the high 32 bits,
// 32-bit payload in the low 32 bits.  POISON marks a tile whose chain was
// abandoned after a timeout; readers treat it as terminal and propagate it.

enum : uint32_t { kInvalid = 0u, kAggregate = 1u, kPrefix = 2u, kPoison = 3u };

__device__ __forceinline__ uint64_t make_desc(uint32_t state, uint32_t bits) {
    return (static_cast<uint64_t>(state) << 32) | bits;
}
__device__ __forceinline__ uint32_t desc_state(uint64_t d) { return static_cast<uint32_t>(d >> 32); }
__device__ __forceinline__ uint32_t desc_bits(uint64_t d) { return static_cast<uint32_t>(d); }

// ---------------------------------------------------------------------------
// Warp layer: Hillis-Steele inclusive scan over the 32 lanes ("Parallel
// Prefix Sum (Scan), in depth", "Hillis-Steele: short span, too much work"
// and "A CUDA scan: warp, block, grid"): at distance d every lane >= d
// combines the value d lanes below it.

template <class Op>
__device__ __forceinline__ typename Op::T warp_inclusive_scan(typename Op::T v, uint32_t lane) {
#pragma unroll
    for (uint32_t d = 1; d < 32; d <<= 1) {
        typename Op::T other = __shfl_up_sync(0xffffffffu, v, d);
        if (lane >= d) v = Op::combine(other, v);
    }
    return v;
}

// ---------------------------------------------------------------------------
// Decoupled look-back, warp-parallel ("Single-Pass Prefix Scan with
// Decoupled Look-Back", "Three states in a per-block descriptor" and "Why
// the work stays linear"; "Parallel Prefix Sum (Scan), in depth", "Scanning
// a whole array: three grid strategies").
//
// Called by all 32 lanes of one warp for tile t > 0.  Lane l reads the
// descriptor of tile (base - l), so one round covers 32 predecessors.  The
// round is used once no lane nearer than the nearest terminal (prefix or
// poison) descriptor is still invalid; the values of the lanes up to and
// including that terminal lane are combined in tile order and folded in
// front of the running carry.  Without a terminal lane the window moves 32
// tiles back.  Returns the exclusive prefix of tile t in *carry_out.
// Result codes: 0 ok, 1 poison found, 2 spin limit reached.

template <class Op>
__device__ __forceinline__ int lookback(const uint64_t *desc, uint32_t t, uint32_t lane,
                                        uint32_t spin_limit, typename Op::T *carry_out) {
    using T = typename Op::T;
    T carry = Op::identity();
    int64_t base = static_cast<int64_t>(t) - 1;
    uint32_t polls = 0;
    while (true) {
        const int64_t idx = base - static_cast<int64_t>(lane);
        uint64_t d;
        uint32_t term_mask, first;
        while (true) {
            d = (idx >= 0) ? ld_acquire_gpu(desc + idx) : make_desc(kPrefix, Op::to_bits(Op::identity()));
            const uint32_t st = desc_state(d);
            term_mask = __ballot_sync(0xffffffffu, st == kPrefix || st == kPoison);
            const uint32_t inv_mask = __ballot_sync(0xffffffffu, st == kInvalid);
            first = term_mask ? (__ffs(term_mask) - 1) : 32u;
            const uint32_t needed = (first >= 31u) ? 0xffffffffu : ((2u << first) - 1u);
            if ((inv_mask & needed) == 0u) break;
            if (++polls >= spin_limit) return 2;
            if (polls > 4) __nanosleep(polls > 64 ? 256 : 32);
        }
        if (first < 32u) {
            const uint32_t fst = __shfl_sync(0xffffffffu, desc_state(d), first);
            if (fst == kPoison) return 1;
        }
        // Lanes 0..first hold, in reverse tile order, the aggregates and the
        // terminal prefix; combine them so that earlier tiles stay on the left.
        T v = (lane <= first) ? Op::from_bits(desc_bits(d)) : Op::identity();
#pragma unroll
        for (uint32_t o = 1; o < 32; o <<= 1) {
            const T earlier = __shfl_down_sync(0xffffffffu, v, o);
            if (lane + o < 32u) v = Op::combine(earlier, v);
        }
        const T window = __shfl_sync(0xffffffffu, v, 0);
        carry = Op::combine(window, carry);
        if (first < 32u) break;
        base -= 32;
    }
    *carry_out = carry;
    return 0;
}

}  // namespace dwp
