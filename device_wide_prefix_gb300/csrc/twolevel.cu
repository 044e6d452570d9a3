// Two-level (reduce, then scan) plain scan in three launches, for sm_103a.
//
// "Single-Pass Prefix Scan with Decoupled Look-Back", sections "The
// two-level decomposition" and "When not to use it": the older form that
// the single-pass scan improves on.  It needs neither descriptors nor any
// waiting on other blocks, and its two extra launches cost a few
// microseconds, so it stays useful for small inputs and as a comparison.
//   1. tl_reduce      block b reduces its chunk of CHUNK elements to one
//                     total, written to totals[b];
//   2. tl_scan_totals one block turns the totals into their exclusive scan,
//                     in place;
//   3. tl_scan        block b scans its chunk again from totals[b] and
//                     writes the outputs.
// Inside a block: ITEMS contiguous elements per thread scanned serially,
// the 32 thread totals of a warp by a shuffle scan, the warp totals through
// shared memory.  The input is read twice and the output written once;
// for the sizes this form is for, both fit in the 129 MB L2.
#include <cuda_runtime.h>

#include "device.cuh"
#include "launch.h"

namespace dwp {

namespace {

constexpr int kTlThreads = 256;
constexpr int kTlItems = 16;
constexpr int kTlChunk = kTlThreads * kTlItems;   // elements per block
constexpr int kTlTotThreads = 1024;               // the one block of step 2
constexpr int kTlTotItems = 16;                   // totals per thread in step 2
constexpr uint64_t kTlMaxBlocks = uint64_t(kTlTotThreads) * kTlTotItems;

// Inclusive Hillis-Steele scan of one value per lane ("Parallel Prefix Sum
// (Scan), in depth", section "Hillis-Steele: short span, too much work"):
// at step d = 1, 2, 4, 8, 16 every lane at or above d combines the value d
// lanes below it into its own.  With `steps` non-null, lane l also writes
// its value after step k (d = 2^k) to steps[32k + l], so a test can compare
// each step with the page's printed trace.
template <class Op>
__device__ __forceinline__ typename Op::T warp_incl_scan(typename Op::T v, uint32_t lane,
                                                        uint32_t *steps = nullptr) {
#pragma unroll
    for (int d = 1, k = 0; d < 32; d <<= 1, ++k) {
        const typename Op::T u = __shfl_up_sync(0xffffffffu, v, d);
        if (lane >= uint32_t(d)) v = Op::combine(u, v);
        if (steps) steps[32 * k + lane] = Op::to_bits(v);
    }
    return v;
}

// One warp runs warp_incl_scan over x[0 .. width) (the identity in the
// lanes past width) and writes the value of lanes 0 .. width-1 after each
// of the five steps to out[width * k + l].
__global__ void warp_scan_trace_kernel(const uint32_t *x, uint32_t width, uint32_t *out) {
    __shared__ uint32_t steps[5 * 32];
    pdl_wait();
    pdl_trigger();
    const uint32_t lane = threadIdx.x & 31u;
    const uint32_t v = lane < width ? x[lane] : OpU32Add::identity();
    warp_incl_scan<OpU32Add>(v, lane, steps);
    __syncwarp();
    for (uint32_t k = 0; k < 5; ++k)
        if (lane < width) out[width * k + lane] = steps[32 * k + lane];
}

// Exclusive scan of one value per thread over the block, in thread order;
// *total receives the block's combination.  `warp_tot` holds 32 words.
template <class Op>
__device__ __forceinline__ typename Op::T block_excl_scan(typename Op::T v, uint32_t *warp_tot,
                                                         typename Op::T *total) {
    using T = typename Op::T;
    const uint32_t lane = threadIdx.x & 31u, warp = threadIdx.x >> 5;
    const uint32_t nwarps = blockDim.x >> 5;
    const T incl = warp_incl_scan<Op>(v, lane);
    if (lane == 31) warp_tot[warp] = Op::to_bits(incl);
    __syncthreads();
    if (warp == 0) {
        T w = lane < nwarps ? Op::from_bits(warp_tot[lane]) : Op::identity();
        w = warp_incl_scan<Op>(w, lane);
        warp_tot[lane] = Op::to_bits(w);
    }
    __syncthreads();
    const T before = warp > 0 ? Op::from_bits(warp_tot[warp - 1]) : Op::identity();
    *total = Op::from_bits(warp_tot[nwarps - 1]);
    const T lane_excl = __shfl_up_sync(0xffffffffu, incl, 1);
    const T excl_in_warp = lane > 0 ? lane_excl : Op::identity();
    const T r = Op::combine(before, excl_in_warp);
    __syncthreads();  // warp_tot may be reused by the caller
    return r;
}

// This thread's ITEMS elements of block b's chunk (identity past n).
template <class Op>
__device__ __forceinline__ void load_items(const typename Op::T *in, uint64_t n, uint64_t first,
                                           typename Op::T (&v)[kTlItems]) {
    if (first + kTlItems <= n) {
        const uint4 *p = reinterpret_cast<const uint4 *>(in + first);
#pragma unroll
        for (int q = 0; q < kTlItems / 4; ++q) {
            const uint4 w = p[q];
            v[4 * q + 0] = Op::from_bits(w.x);
            v[4 * q + 1] = Op::from_bits(w.y);
            v[4 * q + 2] = Op::from_bits(w.z);
            v[4 * q + 3] = Op::from_bits(w.w);
        }
    } else {
#pragma unroll
        for (int j = 0; j < kTlItems; ++j) v[j] = first + j < n ? in[first + j] : Op::identity();
    }
}

template <class Op>
__global__ void __launch_bounds__(kTlThreads) tl_reduce(const typename Op::T *in, uint64_t n,
                                                        uint32_t *totals) {
    using T = typename Op::T;
    __shared__ uint32_t warp_tot[33];
    pdl_wait();
    pdl_trigger();
    const uint64_t first = uint64_t(blockIdx.x) * kTlChunk + uint64_t(threadIdx.x) * kTlItems;
    T v[kTlItems];
    load_items<Op>(in, n, first, v);
    T acc = Op::identity();
#pragma unroll
    for (int j = 0; j < kTlItems; ++j) acc = Op::combine(acc, v[j]);
    T total;
    block_excl_scan<Op>(acc, warp_tot, &total);
    if (threadIdx.x == 0) totals[blockIdx.x] = Op::to_bits(total);
}

template <class Op>
__global__ void __launch_bounds__(kTlTotThreads) tl_scan_totals(uint32_t *totals, uint32_t count) {
    using T = typename Op::T;
    __shared__ uint32_t warp_tot[33];
    pdl_wait();
    pdl_trigger();
    const uint32_t first = threadIdx.x * kTlTotItems;
    T v[kTlTotItems];
    T acc = Op::identity();
#pragma unroll
    for (int j = 0; j < kTlTotItems; ++j) {
        v[j] = first + j < count ? Op::from_bits(totals[first + j]) : Op::identity();
        acc = Op::combine(acc, v[j]);
    }
    T total;
    T run = block_excl_scan<Op>(acc, warp_tot, &total);
#pragma unroll
    for (int j = 0; j < kTlTotItems; ++j) {
        if (first + j < count) totals[first + j] = Op::to_bits(run);
        run = Op::combine(run, v[j]);
    }
}

template <class Op, bool INCL>
__global__ void __launch_bounds__(kTlThreads) tl_scan(const typename Op::T *in, typename Op::T *out,
                                                      uint64_t n, const uint32_t *totals) {
    using T = typename Op::T;
    __shared__ uint32_t warp_tot[33];
    pdl_wait();
    pdl_trigger();
    const uint64_t first = uint64_t(blockIdx.x) * kTlChunk + uint64_t(threadIdx.x) * kTlItems;
    T v[kTlItems];
    load_items<Op>(in, n, first, v);
    T acc = Op::identity();
#pragma unroll
    for (int j = 0; j < kTlItems; ++j) acc = Op::combine(acc, v[j]);
    T total;
    const T excl = block_excl_scan<Op>(acc, warp_tot, &total);
    T run = Op::combine(Op::from_bits(totals[blockIdx.x]), excl);
    T y[kTlItems];
#pragma unroll
    for (int j = 0; j < kTlItems; ++j) {
        if (INCL) {
            run = Op::combine(run, v[j]);
            y[j] = run;
        } else {
            y[j] = run;
            run = Op::combine(run, v[j]);
        }
    }
    if (first + kTlItems <= n) {
        uint4 *p = reinterpret_cast<uint4 *>(out + first);
#pragma unroll
        for (int q = 0; q < kTlItems / 4; ++q)
            p[q] = make_uint4(Op::to_bits(y[4 * q]), Op::to_bits(y[4 * q + 1]), Op::to_bits(y[4 * q + 2]),
                              Op::to_bits(y[4 * q + 3]));
    } else {
#pragma unroll
        for (int j = 0; j < kTlItems; ++j)
            if (first + j < n) out[first + j] = y[j];
    }
}

template <class Op, bool INCL>
cudaError_t launch_tl(const void *in, void *out, uint64_t n, void *scratch, cudaStream_t stream) {
    using T = typename Op::T;
    const uint64_t blocks = (n + kTlChunk - 1) / kTlChunk;
    auto *totals = reinterpret_cast<uint32_t *>(static_cast<unsigned char *>(scratch) + kHeaderBytes);
    const T *src = static_cast<const T *>(in);
    cudaError_t e = launch_pdl(tl_reduce<Op>, dim3(uint32_t(blocks)), dim3(kTlThreads), 0, stream,
                               src, n, totals);
    if (e == cudaSuccess)
        e = launch_pdl(tl_scan_totals<Op>, dim3(1), dim3(kTlTotThreads), 0, stream, totals,
                       uint32_t(blocks));
    if (e == cudaSuccess)
        e = launch_pdl(tl_scan<Op, INCL>, dim3(uint32_t(blocks)), dim3(kTlThreads), 0, stream, src,
                       static_cast<T *>(out), n, static_cast<const uint32_t *>(totals));
    return e;
}

}  // namespace

uint64_t two_level_max_n() { return kTlMaxBlocks * kTlChunk; }
uint32_t two_level_chunk() { return kTlChunk; }

cudaError_t launch_two_level(dwp_op op, bool inclusive, const void *in, void *out, uint64_t n,
                             void *scratch, cudaStream_t stream) {
    switch (op) {
        case DWP_U32_ADD:
            return inclusive ? launch_tl<OpU32Add, true>(in, out, n, scratch, stream)
                             : launch_tl<OpU32Add, false>(in, out, n, scratch, stream);
        case DWP_F32_ADD:
            return inclusive ? launch_tl<OpF32Add, true>(in, out, n, scratch, stream)
                             : launch_tl<OpF32Add, false>(in, out, n, scratch, stream);
        case DWP_U32_MAX:
            return inclusive ? launch_tl<OpU32Max, true>(in, out, n, scratch, stream)
                             : launch_tl<OpU32Max, false>(in, out, n, scratch, stream);
    }
    return cudaErrorInvalidValue;
}

}  // namespace dwp

extern "C" dwp_status dwp_debug_warp_scan_trace(const uint32_t *d_x, size_t width, uint32_t *d_steps,
                                                dwp_stream stream) {
    if (width == 0 || width > 32 || !d_x || !d_steps) return DWP_ERR_INVALID_VALUE;
    if (dwp::launch_pdl(dwp::warp_scan_trace_kernel, dim3(1), dim3(32), 0,
                        reinterpret_cast<cudaStream_t>(stream), d_x, uint32_t(width),
                        d_steps) != cudaSuccess) {
        cudaGetLastError();
        return DWP_ERR_CUDA;
    }
    return DWP_SUCCESS;
}
