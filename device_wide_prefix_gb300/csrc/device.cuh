// Device building blocks shared by the kernels: sm_103a inline PTX for
// mbarriers, bulk (TMA) copies, proxy fences and descriptor traffic; the
// associative operators; the warp layer; and the warp-parallel decoupled
// look-back.
#pragma once

#include <cstdint>

#include "common.h"

namespace dwp {

constexpr uint32_t kNoTile = 0xffffffffu;

// ---------------------------------------------------------------------------
// Operators.  "Parallel Prefix Sum (Scan), in depth", "Inclusive, exclusive
// and associative": any associative operator; "Prefix scans and compaction",
// "Inclusive and exclusive scan": identities 0 for addition, lowest value for
// a maximum.  combine(a, b) keeps operand order: a covers earlier elements.
// warp_reduce combines one value per lane over the whole warp.

struct OpU32Add {
    static constexpr bool kCommutative = true;
    using T = uint32_t;
    static __device__ __forceinline__ T identity() { return 0u; }
    static __device__ __forceinline__ T combine(T a, T b) { return a + b; }
    static __device__ __forceinline__ uint32_t to_bits(T v) { return v; }
    static __device__ __forceinline__ T from_bits(uint32_t b) { return b; }
    // one redux instruction
    static __device__ __forceinline__ T warp_reduce(T v) { return __reduce_add_sync(0xffffffffu, v); }
};

struct OpU32Max {
    static constexpr bool kCommutative = true;
    using T = uint32_t;
    static __device__ __forceinline__ T identity() { return 0u; }
    static __device__ __forceinline__ T combine(T a, T b) { return a > b ? a : b; }
    static __device__ __forceinline__ uint32_t to_bits(T v) { return v; }
    static __device__ __forceinline__ T from_bits(uint32_t b) { return b; }
    static __device__ __forceinline__ T warp_reduce(T v) { return __reduce_max_sync(0xffffffffu, v); }
};

struct OpF32Add {
    static constexpr bool kCommutative = true;  // a + b == b + a exactly in IEEE
    using T = float;
    static __device__ __forceinline__ T identity() { return 0.0f; }
    static __device__ __forceinline__ T combine(T a, T b) { return __fadd_rn(a, b); }
    static __device__ __forceinline__ uint32_t to_bits(T v) { return __float_as_uint(v); }
    static __device__ __forceinline__ T from_bits(uint32_t b) { return __uint_as_float(b); }
    // No float redux instruction: a shuffle butterfly (xor 16, 8, 4, 2, 1),
    // then lane 0's sum goes to every lane, so all lanes return the same
    // bits.  The look-back's warp reduction lies on the path by which the
    // prefix frontier advances; the butterfly replaced a sum by one lane
    // through shared memory that cost 6% of a 2^28 scan.
    static __device__ __forceinline__ T warp_reduce(T v) {
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) v = __fadd_rn(v, __shfl_xor_sync(0xffffffffu, v, o));
        return __shfl_sync(0xffffffffu, v, 0);
    }
};

// ---------------------------------------------------------------------------
// Small PTX wrappers.

// Programmatic dependent launch.  Every kernel of the library is launched
// with programmatic stream serialisation, so it may start while the kernel
// before it on the stream is still running.  pdl_wait() blocks until that
// kernel (and, through its own wait, everything before it) has completed
// and its memory is visible; every kernel calls it before its first access
// to global memory.  pdl_trigger() lets the next kernel on the stream start
// its launch early; that kernel waits the same way before touching memory.
// The scratch-clear kernel and the short kernels trigger at once; the
// persistent look-back kernels do not (their blocks trigger as they exit),
// which measured faster on GB300 at every size.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

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

// L2 eviction-priority policies for bulk copies (createpolicy, sm_80+).
__device__ __forceinline__ uint64_t l2_policy_evict_last() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
    return p;
}
__device__ __forceinline__ uint64_t l2_policy_evict_first() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}

// bulk_load with an L2 eviction-priority policy for the lines it reads.
// Ask L2 to fetch [src, src + bytes) ahead of use, with an eviction priority.
__device__ __forceinline__ void bulk_prefetch_l2(const void *src, uint32_t bytes, uint64_t policy) {
    asm volatile("cp.async.bulk.prefetch.L2.global.L2::cache_hint [%0], %1, %2;" ::"l"(src),
                 "r"(bytes), "l"(policy)
                 : "memory");
}

__device__ __forceinline__ void bulk_load_hint(void *smem_dst, const void *gmem_src, uint32_t bytes,
                                               uint64_t *bar, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1], %2, [%3], %4;" ::"r"(smem_addr(smem_dst)),
        "l"(gmem_src), "r"(bytes), "r"(smem_addr(bar)), "l"(policy)
        : "memory");
}

// bulk_store with an L2 eviction-priority policy for the lines it writes.
__device__ __forceinline__ void bulk_store_hint(void *gmem_dst, const void *smem_src, uint32_t bytes,
                                                uint64_t policy) {
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group.L2::cache_hint [%0], [%1], %2, %3;" ::"l"(gmem_dst),
                 "r"(smem_addr(smem_src)), "r"(bytes), "l"(policy)
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

// Descriptor publication: one 64-bit device-scope atomic store of state and
// value together ("Single-Pass Prefix Scan with Decoupled Look-Back", "The
// publication protocol in code": device scope suffices, and because flag
// and payload travel in one word a reader can never see one without the
// other, so the word itself needs no fence).  The store is relaxed, not
// release: no reader consumes any other memory on the strength of the flag,
// and a release store (a full fence before it) was measured at about 0.8 us
// on GB300, on the serial path of every tile.
__device__ __forceinline__ void st_relaxed_gpu(uint64_t *p, uint64_t v) {
    asm volatile("st.relaxed.gpu.global.b64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}

// Device-scope atomic (relaxed) read of a descriptor word; never hoisted out
// of a polling loop ("Where the algorithm meets the hardware").
__device__ __forceinline__ uint64_t ld_relaxed_gpu(const uint64_t *p) {
    uint64_t v;
    asm volatile("ld.relaxed.gpu.global.b64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}

// Volatile read of a shared-memory word.
__device__ __forceinline__ uint32_t ld_volatile_smem(const uint32_t *p) {
    return *reinterpret_cast<const volatile uint32_t *>(p);
}

// Record a device-side error in the scratch status word (first error wins).
__device__ __forceinline__ void record_error(ScratchHeader *hdr, uint32_t code) {
    atomicCAS(&hdr->status, 0u, code);
}

// Debug bounds build (compile with -DDWP_DEBUG_BOUNDS=1).  Before each
// global access, the look-back kernels (plain and segmented scan,
// compaction, recurrence, segmented reduction) ask whether elements
// [first, first + count) lie inside a buffer of `extent` elements.  An access that would leave its buffer is skipped and
// DWP_ERR_BOUNDS is recorded in the status word: a checked run reports a bad
// index instead of faulting.  The default build compiles every check to
// `true`.
#ifndef DWP_DEBUG_BOUNDS
#define DWP_DEBUG_BOUNDS 0
#endif
__device__ __forceinline__ bool in_bounds(ScratchHeader *hdr, uint64_t first, uint64_t count,
                                          uint64_t extent) {
    if (!DWP_DEBUG_BOUNDS) return true;
    if (first <= extent && count <= extent - first) return true;
    record_error(hdr, DWP_ERR_BOUNDS);
    return false;
}

// ---------------------------------------------------------------------------
// Schedule perturbation, a test hook (dwp_debug_set_delay).  A missing
// ordering or synchronisation in a chained scan shows up only under rare
// interleavings ("Parallel Prefix Sum (Scan), in depth", section "Failure
// modes"), so a test can make a seeded subset of tiles sleep at their
// publication points to shuffle the order in which descriptors appear.
// Whether tile t sleeps at point `site` is decided by a hash of (seed, t,
// site) below `threshold`; the sleep is a second hash modulo max_ns + 1
// nanoseconds, timed on %globaltimer, and ends after a bounded number of
// polls whatever the timer says.  Warp-uniform when every lane passes the
// same arguments.  Off (threshold 0) it costs one compare.

// MurmurHash3's 32-bit finaliser (Appleby): a bijective avalanche mix.
__device__ __forceinline__ uint32_t fmix32(uint32_t h) {
    h ^= h >> 16;
    h *= 0x85ebca6bu;
    h ^= h >> 13;
    h *= 0xc2b2ae35u;
    h ^= h >> 16;
    return h;
}

__device__ __forceinline__ uint64_t global_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ void perturb(const LaunchKnobs &k, uint32_t t, uint32_t site) {
    if (k.delay_threshold == 0u) return;
    const uint32_t h = fmix32(k.delay_seed ^ fmix32(t * 8u + site + 1u));
    if (h >= k.delay_threshold) return;
    const uint32_t ns = fmix32(h ^ 0x9e3779b9u) % (k.delay_max_ns + 1u);
    const uint64_t t0 = global_ns();
    for (uint32_t i = 0; i < 4096u && global_ns() - t0 < ns; ++i) __nanosleep(32);
}

// Perturbation points.
enum : uint32_t {
    kSiteDraw = 0u,       // after a tile index is drawn, before its load
    kSiteAggregate = 1u,  // before the aggregate is published
    kSiteLookback = 2u,   // before the look-back starts
    kSitePrefix = 3u,     // before the inclusive prefix is published
    kSiteMidWord = 4u     // between the two words of a two-word descriptor
};

// ---------------------------------------------------------------------------
// Tile descriptor ("Single-Pass Prefix Scan with Decoupled Look-Back",
// "Three states in a per-block descriptor"): state in the high 32 bits,
// 32-bit payload in the low 32 bits.  POISON marks a tile whose chain was
// abandoned after a timeout; readers treat it as terminal and propagate it.

enum : uint32_t { kInvalid = 0u, kAggregate = 1u, kPrefix = 2u, kPoison = 3u };
// State kSpan0 + d (d >= 2): an intermediate published by a bounded-window
// look-back; its value combines the d tiles ending at this one.
constexpr uint32_t kSpan0 = 4u;

__device__ __forceinline__ uint64_t make_desc(uint32_t state, uint32_t bits) {
    return (static_cast<uint64_t>(state) << 32) | bits;
}
__device__ __forceinline__ uint32_t desc_state(uint64_t d) { return static_cast<uint32_t>(d >> 32); }
__device__ __forceinline__ uint32_t desc_bits(uint64_t d) { return static_cast<uint32_t>(d); }

// ---------------------------------------------------------------------------
// Ring-pipeline helpers shared by the kernels.

// Word index of consumer thread c's slot in a per-thread array: one pad word
// after every 8 spreads the banks when lane l reads slots 8l .. 8l+7.
__device__ __forceinline__ uint32_t prefix_slot(uint32_t c) { return c + (c >> 3); }

// Bounded mbarrier wait agreed by the whole warp (every lane polls).
__device__ __forceinline__ bool warp_wait(uint64_t *bar, uint32_t parity) {
    return __all_sync(0xffffffffu, mbar_wait(bar, parity, kPipeWaitLimit));
}

// Wait for ring iteration k's data, or learn that the producer stopped
// before iteration k (end_iter < k).  Warp-uniform result: 2 data ready,
// 1 ended, 0 poll limit reached.  Ready and ended cannot both hold for one k:
// the producer fills only iterations up to end_iter.
__device__ __forceinline__ int warp_wait_or_end(uint64_t *bar, uint32_t parity, uint32_t k,
                                                const uint32_t *end_iter) {
    uint32_t r = 0;
    for (uint32_t i = 0; i < kPipeWaitLimit; ++i) {
        if (mbar_try_wait(bar, parity)) {
            r = 2;
            break;
        }
        if (ld_volatile_smem(end_iter) < k) {
            r = 1;
            break;
        }
        if (i >= 8) __nanosleep(64);
    }
    return int(__reduce_max_sync(0xffffffffu, r));
}

// Warp-wide: the first index k in [lo, hi] with off[k] >= key, given that
// off[lo-1] < key (or lo == 0) and that hi is a valid answer (off[hi] >= key,
// or hi == N + 1).  Each round probes 32 evenly spaced indices below hi and
// keeps the sub-interval between the last probe below the key and the first
// one at or above it; probes stay inside [lo, hi), so inside offsets[0..N].
__device__ __forceinline__ uint32_t warp_lower_bound(const uint32_t *off, uint32_t lo, uint32_t hi,
                                                     uint32_t key, uint32_t lane) {
    while (lo < hi) {
        const uint32_t len = hi - lo;
        const uint32_t step = (len + 31u) / 32u;
        const uint64_t q = uint64_t(lo) + uint64_t(lane + 1u) * step - 1u;
        const bool probe = q < hi;
        const bool below = probe && __ldg(off + q) < key;
        const uint32_t c = __reduce_add_sync(0xffffffffu, below ? 1u : 0u);
        const uint32_t np = __reduce_add_sync(0xffffffffu, probe ? 1u : 0u);
        if (c < np) hi = lo + (c + 1u) * step - 1u;  // probe c is at or above the key
        lo = lo + c * step;                          // probes 0 .. c-1 are below it
    }
    return lo;
}

// ---------------------------------------------------------------------------
// Decoupled look-back, warp-parallel ("Single-Pass Prefix Scan with
// Decoupled Look-Back", "Three states in a per-block descriptor" and "Why
// the work stays linear"; "Parallel Prefix Sum (Scan), in depth", "Scanning
// a whole array: three grid strategies").
//
// Called by all 32 lanes of one warp for tile t > 0.  One round reads the
// K*32 nearest unread predecessors at once: position p = 32*i + lane is tile
// base - p, so a lane's K loads are independent and in flight together.  Two
// warp-wide min-reductions find the nearest terminal descriptor (prefix or
// poison) and the nearest invalid one; the round is used once nothing nearer
// than the terminal one is still invalid (invalid ones are re-polled).  The
// values up to and including the terminal descriptor are then combined and
// folded into the carry; without a terminal descriptor the window moves K*32
// tiles back.  Every plain-scan operator here is commutative (u32 add, u32
// max, and f32 add, whose a+b == b+a exactly), so values are combined per
// lane first and then across lanes; for f32 only the grouping changes, the
// run-to-run variation the method has anyway ("When not to use it").
// Warp collectives are kept to a few per poll: on a GB300 streaming at full
// bandwidth a dependent one was measured at several hundred cycles in the
// reducer.  The f32 sum of a window is still a shuffle butterfly: there a
// one-lane sum through shared memory measured slower (6% of a 2^28 scan).
//
// Decoupled Fallback ("GPU Prefix Sums", section "Decoupled Fallback"): with
// fallback_polls > 0, once a window has been polled fallback_polls times with
// a predecessor still unpublished, the warp stops waiting for it.  For each
// such predecessor p, `rescue(p, lane)` (called by all 32 lanes,
// same result on each) reduces tile p straight from the input and returns
// the descriptor p would publish; lane 0 installs it with a compare-and-swap
// against the invalid state.  So of several rescuers and the tile's own
// block, whichever writes first wins, and a lost swap hands back the winning
// descriptor (the same value for the integer operators; for f32 another
// grouping of the same sum).  Each swap won adds one to hdr->fallbacks.  The
// input must stay unmodified for the whole launch: callers disable the
// fallback (fallback_polls = 0) for an in-place scan.
//
// Bounded window ("Single-Pass Prefix Scan with Decoupled Look-Back",
// section "Why the work stays linear"): with window > 0 and `publish`, each
// time the look-back of tile t has folded `window` more tiles without
// reaching a prefix, lane 0 publishes an intermediate descriptor for t: the
// combination of everything folded so far with t's own aggregate `own`, and
// the number d of tiles it covers (t - d + 1 .. t), as state kSpan0 + d.  A
// look-back that meets an intermediate as the nearest stop of its window
// folds it and jumps d tiles back at once.  Publications and jumps are
// counted in hdr->intermediates and hdr->jumps.  Folds happen a window of K*32
// tiles at a time, so the effective window is a multiple of K*32.  A tile
// that has already published its prefix must pass publish = false.
//
// Returns 0 and the exclusive prefix of tile t in *carry_out; 1 if the
// nearest terminal descriptor is poison; 2 if the poll limit ran out.

// Back-off between a look-back's polls of a window: after the first
// `after` polls, sleep `ns` before each further one (256 ns from the 256th
// on).  Fewer polls leave L2 and the load/store path to the data streams;
// more polls notice a publication sooner.
struct Backoff {
    uint32_t after;
    uint32_t ns;
};
constexpr Backoff kBackoffDefault{8u, 64u};

template <class Op, int K, class Rescue>
__device__ __forceinline__ int lookback(uint64_t *desc, uint32_t t, uint32_t lane,
                                        uint32_t spin_limit, uint32_t fallback_polls,
                                        const Rescue &rescue, ScratchHeader *hdr,
                                        uint32_t window, uint32_t own, bool publish,
                                        typename Op::T *carry_out,
                                        const Backoff backoff = kBackoffDefault) {
    using T = typename Op::T;
    static_assert(Op::kCommutative, "the look-back combines per lane first");
    static_assert(K * 32 < (1 << 29), "window positions must fit the key");
    T carry = Op::identity();
    int64_t base = static_cast<int64_t>(t) - 1;
    uint32_t polls = 0;
    uint64_t next_pub = window;  // folded tiles at which the next intermediate goes out
    while (true) {
        uint64_t d[K];
#pragma unroll
        for (int i = 0; i < K; ++i) {
            const int64_t idx = base - 32 * i - static_cast<int64_t>(lane);
            d[i] = idx >= 0 ? ld_relaxed_gpu(desc + idx)
                            : make_desc(kPrefix, Op::to_bits(Op::identity()));
        }
        uint32_t tkey, imin, stalled = 0;
        while (true) {
            // key of the nearest stop = 4*position + kind (0 prefix, 1
            // poison, 2 intermediate)
            uint32_t my_t = 0xffffffffu, my_i = 0xffffffffu;
#pragma unroll
            for (int i = K - 1; i >= 0; --i) {
                const uint32_t st = desc_state(d[i]);
                const uint32_t p = 32u * i + lane;
                if (st == kPrefix) my_t = p << 2;
                else if (st == kPoison) my_t = (p << 2) | 1u;
                else if (st >= kSpan0) my_t = (p << 2) | 2u;
                if (st == kInvalid) my_i = p;
            }
            tkey = __reduce_min_sync(0xffffffffu, my_t);
            imin = __reduce_min_sync(0xffffffffu, my_i);
            if (tkey != 0xffffffffu ? imin > (tkey >> 2) : imin == 0xffffffffu) break;
            if (++polls >= spin_limit) return 2;
            const uint32_t lim = tkey != 0xffffffffu ? (tkey >> 2) : 32u * K;
            if (fallback_polls != 0u && ++stalled >= fallback_polls) {
                stalled = 0;
#pragma unroll
                for (int i = 0; i < K; ++i) {
                    const int64_t idx = base - 32 * i - static_cast<int64_t>(lane);
                    uint32_t need = __ballot_sync(
                        0xffffffffu, 32u * i + lane < lim && idx >= 0 && desc_state(d[i]) == kInvalid);
                    while (need) {
                        const uint32_t j = uint32_t(__ffs(need)) - 1u;
                        need &= need - 1u;
                        const uint32_t p = static_cast<uint32_t>(base - 32 * i - static_cast<int64_t>(j));
                        const uint64_t mine = rescue(p, lane);
                        unsigned long long got = 0ull;
                        if (lane == 0) {
                            const unsigned long long old = atomicCAS(
                                reinterpret_cast<unsigned long long *>(desc + p), 0ull,
                                static_cast<unsigned long long>(mine));
                            got = old == 0ull ? static_cast<unsigned long long>(mine) : old;
                            if (old == 0ull) atomicAdd(&hdr->fallbacks, 1u);
                        }
                        got = __shfl_sync(0xffffffffu, got, 0);
                        if (lane == j) d[i] = got;
                    }
                }
                continue;
            }
            if (polls > backoff.after) __nanosleep(polls > 256u ? 256u : backoff.ns);
#pragma unroll
            for (int i = 0; i < K; ++i) {
                const int64_t idx = base - 32 * i - static_cast<int64_t>(lane);
                if (32u * i <= lim && idx >= 0 && desc_state(d[i]) == kInvalid)
                    d[i] = ld_relaxed_gpu(desc + idx);
            }
        }
        const uint32_t kind = tkey != 0xffffffffu ? (tkey & 3u) : 3u;
        if (kind == 1u) return 1;
        const uint32_t last = tkey != 0xffffffffu ? (tkey >> 2) : 0xffffffffu;
        T acc = Op::identity();
        uint32_t span = 0;
#pragma unroll
        for (int i = 0; i < K; ++i) {
            if (32u * i + lane <= last) acc = Op::combine(acc, Op::from_bits(desc_bits(d[i])));
            if (32u * i + lane == last && kind == 2u) span = desc_state(d[i]) - kSpan0;
        }
        carry = Op::combine(Op::warp_reduce(acc), carry);
        if (kind == 0u) break;
        if (kind == 2u && lane == 0) atomicAdd(&hdr->jumps, 1u);
        // the intermediate at position `last` covers `span` tiles ending at it
        base -= kind == 2u ? int64_t(last) + int64_t(__reduce_max_sync(0xffffffffu, span)) : 32 * K;
        const uint64_t folded = uint64_t(int64_t(t) - 1 - base);
        if (window != 0u && publish && folded >= next_pub) {
            if (lane == 0) {
                st_relaxed_gpu(desc + t, make_desc(kSpan0 + uint32_t(folded) + 1u,
                                                   Op::to_bits(Op::combine(carry, Op::from_bits(own)))));
                atomicAdd(&hdr->intermediates, 1u);
            }
            next_pub = folded + window;
        }
    }
    *carry_out = carry;
    return 0;
}

// ---------------------------------------------------------------------------
// Decoupled Fallback for the plain scan: the descriptor tile p would
// publish, reduced by one warp straight from the input (tile 0's aggregate
// is its inclusive prefix).
template <class Op, int TILE>
struct ScanRescue {
    static_assert(TILE % 4 == 0, "full tiles are read as 16-byte vectors");
    const typename Op::T *in;
    uint64_t n;
    __device__ uint64_t operator()(uint32_t p, uint32_t lane) const {
        using T = typename Op::T;
        const uint64_t b = uint64_t(p) * TILE;
        const uint64_t e = min(n, b + uint64_t(TILE));
        T acc = Op::identity();
        if (e - b == uint64_t(TILE)) {
            const uint4 *v4 = reinterpret_cast<const uint4 *>(in + b);
            for (uint32_t q = lane; q < uint32_t(TILE) / 4u; q += 32u) {
                const uint4 v = v4[q];
                acc = Op::combine(acc, Op::combine(Op::combine(Op::from_bits(v.x), Op::from_bits(v.y)),
                                                   Op::combine(Op::from_bits(v.z), Op::from_bits(v.w))));
            }
        } else {
            for (uint64_t q = b + lane; q < e; q += 32u) acc = Op::combine(acc, in[q]);
        }
        const T tot = Op::warp_reduce(acc);
        return make_desc(p == 0 ? kPrefix : kAggregate, Op::to_bits(tot));
    }
};

}  // namespace dwp
