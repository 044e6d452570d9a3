/*
 * dwp.h - device-wide single-pass prefix scan for NVIDIA GB300 (sm_103a).
 *
 * C ABI.  Every entry point takes plain device pointers and sizes, runs as
 * one stream-ordered launch sequence on the caller's stream and returns
 * without synchronising.  The library never allocates memory: the caller
 * owns inputs, outputs and scratch.
 *
 * Operation ("Parallel Prefix Sum (Scan), in depth", section "Inclusive,
 * exclusive and associative"): for an associative operator (+) with identity
 * e, the inclusive scan is y[i] = x[0] (+) ... (+) x[i]; the exclusive scan
 * is y[0] = e and y[i] = x[0] (+) ... (+) x[i-1].  Identities ("Prefix scans
 * and compaction", section "Inclusive and exclusive scan"): 0 for addition,
 * the lowest representable value (0 for u32) for a maximum.
 *
 * Method ("Single-Pass Prefix Scan with Decoupled Look-Back", sections
 * "Three states in a per-block descriptor" and "The publication protocol in
 * code"; "Parallel Prefix Sum (Scan), in depth", section "Scanning a whole
 * array: three grid strategies"): one pass over the data.  Tiles take their
 * index from an atomic counter, publish their aggregate in a 64-bit
 * descriptor (state and value in one word), look back over their
 * predecessors' descriptors until an inclusive prefix is found, publish
 * their own inclusive prefix and write their output.
 *
 * Scratch (two-call pattern, "Parallel Prefix Sum (Scan), in depth",
 * section "Use the library"): call once with d_scratch == NULL to receive
 * the required byte count in *scratch_bytes, then again with a device
 * buffer of at least that many bytes.  The scratch holds the tile counter,
 * a device-side status word and one 8-byte descriptor per tile; each call
 * clears the part it uses with a cudaMemsetAsync on `stream` before its
 * kernel.  Calls that share one scratch buffer must be ordered (same stream
 * or synchronised); overlapping calls on one scratch buffer race.
 *
 * Pointers: every data pointer and the scratch pointer must be 16-byte
 * aligned (DWP_ERR_MISALIGNED otherwise).  Sizes: n < 2^32.
 *
 * Errors: argument errors are reported before anything is enqueued.  A
 * launch error is DWP_ERR_CUDA.  Errors that arise on the device (a
 * look-back or pipeline wait that ran past its limit) are recorded in the
 * scratch status word and returned by dwp_read_status().  All device-side
 * waits are bounded: a kernel never hangs, it records an error and exits.
 */
#ifndef DWP_H
#define DWP_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* A CUDA stream handle; the same value as a cudaStream_t.  NULL means the
 * legacy default stream. */
typedef struct CUstream_st *dwp_stream;

typedef enum dwp_status {
    DWP_SUCCESS = 0,
    DWP_ERR_INVALID_VALUE = 1,     /* null pointer with n > 0, unknown op/mode, n >= 2^32 */
    DWP_ERR_MISALIGNED = 2,        /* a pointer is not 16-byte aligned */
    DWP_ERR_ALIASING = 3,          /* input, output or scratch ranges overlap (see each call) */
    DWP_ERR_SCRATCH_TOO_SMALL = 4, /* *scratch_bytes is below the size query's answer */
    DWP_ERR_CUDA = 5,              /* a CUDA runtime call or launch failed */
    DWP_ERR_LOOKBACK_TIMEOUT = 6,  /* device: a look-back spin ran past its limit */
    DWP_ERR_PIPELINE_TIMEOUT = 7,  /* device: a shared-memory pipeline wait ran past its limit */
    DWP_ERR_NO_DEVICE = 8,         /* no usable CUDA device */
    DWP_ERR_BOUNDS = 9             /* device, debug bounds build only: an access would have
                                      left its buffer and was skipped (never in the default build) */
} dwp_status;

/* Associative operators of the plain scans. */
typedef enum dwp_op {
    DWP_U32_ADD = 0, /* uint32 addition, wraps modulo 2^32; identity 0 */
    DWP_F32_ADD = 1, /* float32 addition in f32 arithmetic; identity +0.0f */
    DWP_U32_MAX = 2  /* uint32 maximum; identity 0 */
} dwp_op;

typedef enum dwp_mode {
    DWP_EXCLUSIVE = 0,
    DWP_INCLUSIVE = 1
} dwp_mode;

/*
 * Exclusive scan of n elements of d_in (uint32 or float32 per `op`) into
 * d_out.  Definition: "Parallel Prefix Sum (Scan), in depth", section
 * "Inclusive, exclusive and associative"; y[0] is the identity.
 *   op            DWP_U32_ADD, DWP_F32_ADD or DWP_U32_MAX
 *   d_in, d_out   device arrays of n 4-byte elements, contiguous.
 *                 d_out == d_in (exact in-place) is allowed; any other
 *                 overlap is DWP_ERR_ALIASING.
 *   n             element count, 0 <= n < 2^32; n == 0 enqueues only the
 *                 scratch clear.
 *   d_scratch     NULL for the size query, else a device buffer that does
 *                 not overlap d_in or d_out.
 *   scratch_bytes in: size of d_scratch; out (size query): size needed.
 *   stream        stream the work is enqueued on.
 * f32 results are not bit-reproducible from run to run: the grouping of the
 * partial sums depends on look-back timing ("Single-Pass Prefix Scan with
 * Decoupled Look-Back", section "When not to use it").
 */
dwp_status dwp_scan_exclusive(dwp_op op, const void *d_in, void *d_out, size_t n,
                              void *d_scratch, size_t *scratch_bytes, dwp_stream stream);

/* Inclusive scan; arguments as dwp_scan_exclusive.  y[i] includes x[i]. */
dwp_status dwp_scan_inclusive(dwp_op op, const void *d_in, void *d_out, size_t n,
                              void *d_scratch, size_t *scratch_bytes, dwp_stream stream);

/*
 * Segmented uint32 addition scan over CSR offsets ("GPUSegmentedScan",
 * sections "Prefix scans and segmented scans", "Contract" and
 * "Limitations"; "Parallel Prefix Sum (Scan), in depth", section "What scan
 * builds": the running total restarts at every segment boundary).
 *   d_values      device uint32[n], 16-byte aligned
 *   d_offsets     device uint32[num_segments + 1], 4-byte aligned; segment
 *                 s is rows [d_offsets[s], d_offsets[s+1]).  Offsets are
 *                 trusted: non-decreasing with d_offsets[num_segments] <= n
 *                 is a precondition the device does not check (no
 *                 readback); broken offsets give unspecified values but no
 *                 access out of range.  Repeated offsets are empty
 *                 segments and write no rows.
 *   num_segments  N, 0 <= N < 2^32 - 1 (N + 1 offsets are read).
 *   d_out         device uint32[n], 16-byte aligned.  Rows outside
 *                 [d_offsets[0], min(d_offsets[N], n)) are left unwritten.
 *                 Overlap with d_values, d_offsets or d_scratch is
 *                 DWP_ERR_ALIASING.
 *   n             row count, 0 <= n < 2^32.
 *   mode          DWP_EXCLUSIVE (a segment's first row is 0) or
 *                 DWP_INCLUSIVE.
 *   d_scratch, scratch_bytes, stream: as dwp_scan_exclusive (the size
 *                 query depends on n only).
 * u32 sums wrap modulo 2^32.  Results are bit-exact and deterministic.
 */
dwp_status dwp_segmented_scan_u32(const uint32_t *d_values, const uint32_t *d_offsets,
                                  size_t num_segments, uint32_t *d_out, size_t n,
                                  dwp_mode mode, void *d_scratch, size_t *scratch_bytes,
                                  dwp_stream stream);

/*
 * Stable stream compaction of 16-byte records by byte flags ("Prefix scans
 * and compaction", sections "Scan as an index generator" and "Worked
 * example: Stable stream compaction"; "Parallel Prefix Sum (Scan), in
 * depth", section "What scan builds").  Record i is kept when d_flags[i] is
 * nonzero and is written to slot (number of kept records before i) of
 * d_out, so kept records keep their input order; the number kept goes to
 * *d_count.
 *   d_records     device array of n records of 16 bytes each (opaque,
 *                 copied bit for bit), 16-byte aligned
 *   d_flags       device uint8[n], 16-byte aligned
 *   n             record count, 0 <= n < 2^32
 *   d_out         device array with room for n records, 16-byte aligned;
 *                 slots at and past the kept count are left unwritten.
 *   d_count       device uint32, 4-byte aligned: receives the kept count
 *                 (0 for n == 0).
 *   d_scratch, scratch_bytes, stream: as dwp_scan_exclusive.
 * Any overlap among d_out, d_count, d_scratch and the inputs is
 * DWP_ERR_ALIASING.  Results are bit-exact and deterministic.
 */
dwp_status dwp_compact_by_flags(const void *d_records, const uint8_t *d_flags, size_t n,
                                void *d_out, uint32_t *d_count, void *d_scratch,
                                size_t *scratch_bytes, dwp_stream stream);

/*
 * Scan for callers that cannot allocate device memory.  The source pages
 * have no counterpart to this entry point; it is a convenience of this
 * library.  Code that runs inside another framework's allocator hooks or
 * memory-pool callbacks (where cudaMalloc would re-enter that allocator),
 * or a plug-in whose host application owns all device memory, cannot hand
 * the other scan calls a scratch buffer.  This call uses instead a fixed
 * array of about 512 KiB that is part of the library's device image: every
 * GPU that loads libdwp.so holds it until the process exits.  The call
 * itself allocates and frees nothing.
 *   op, d_in, d_out, stream: as dwp_scan_exclusive.
 *   mode      DWP_EXCLUSIVE or DWP_INCLUSIVE.
 *   n         0 <= n <= DWP_SCAN_STATIC_MAX_N (2^28 elements); a larger n
 *             returns DWP_ERR_SCRATCH_TOO_SMALL before anything is enqueued.
 * Every call looks up the current device's address of the array
 * (cudaGetSymbolAddress), so the address stays right after a device or
 * context reset.  The first call on a device also loads the library's
 * device code there: make that first call before any stream capture.  Every
 * call on a device shares the one array, and each call clears the part it
 * uses on `stream` first, so calls must be ordered on the GPU: two calls
 * that overlap on the GPU (different streams, not synchronised) race and
 * give wrong results.  Device-side timeouts are recorded in the array's
 * status word: read it with dwp_read_static_status.  DWP_ERR_NO_DEVICE if
 * there is no current device; otherwise the errors of dwp_scan_exclusive.
 */
#define DWP_SCAN_STATIC_MAX_N 268435456u
dwp_status dwp_scan_static_scratch(dwp_op op, dwp_mode mode, const void *d_in, void *d_out,
                                   size_t n, dwp_stream stream);

/*
 * Device-side status of the most recent dwp_scan_static_scratch call on the
 * current device: what dwp_read_status returns for a caller-owned scratch
 * buffer, read from the built-in array.  Synchronises `stream` (order it
 * after the call).  Copies into host memory only; allocates nothing.
 */
dwp_status dwp_read_static_status(dwp_stream stream);

/*
 * The same scans as dwp_scan_exclusive / dwp_scan_inclusive (`mode` picks
 * one) by the two-level form in three launches: block totals, a one-block
 * scan of the totals, then each block scans its chunk again from its total
 * ("Single-Pass Prefix Scan with Decoupled Look-Back", sections "The
 * two-level decomposition" and "When not to use it").  No descriptors and
 * no spinning; the input is read twice.  For small inputs and for
 * comparison with the single-pass scan.
 *   n            at most 2^26 (DWP_ERR_INVALID_VALUE above).
 *   d_scratch    NULL: *scratch_bytes receives the size needed (128 bytes
 *                plus 4 bytes per 4096-element block).
 * Pointers, alignment, in-place use and errors as for dwp_scan_exclusive.
 */
dwp_status dwp_scan_two_level(dwp_op op, dwp_mode mode, const void *d_in, void *d_out, size_t n,
                              void *d_scratch, size_t *scratch_bytes, dwp_stream stream);

/*
 * Stable compaction in three stages, for comparison with the fused
 * dwp_compact_by_flags ("Prefix scans and compaction", section "Worked
 * example: Stable stream compaction": compare an implementation that
 * materialises the flags and their prefixes with a fused one; section
 * "Common errors": the cost of materialising predicates and prefixes).
 * Same arguments, output and count as dwp_compact_by_flags; the output is
 * bit for bit the same.  The stages, in three launches plus the scan's
 * scratch clear: u32 flags f[i] = (d_flags[i] != 0) written to scratch;
 * dwp_scan_exclusive of f into offsets in scratch; a scatter that reads f,
 * the offsets and each kept record and writes it to its slot.  Memory
 * traffic is about 21 bytes per record plus the kept records' sectors and
 * output, against 17 plus the output for the fused kernel.
 *   d_scratch  NULL: *scratch_bytes receives the size needed (the scan's
 *              scratch plus 8 bytes per record).  Otherwise at least that
 *              many bytes, 16-byte aligned, overlapping no other argument;
 *              dwp_read_status on it reports the scan's device status.
 * Errors as for dwp_compact_by_flags.
 */
dwp_status dwp_compact_by_flags_staged(const void *d_records, const uint8_t *d_flags, size_t n,
                                       void *d_out, uint32_t *d_count, void *d_scratch,
                                       size_t *scratch_bytes, dwp_stream stream);

/*
 * Segmented u32 addition reduction over CSR offsets ("GPUSegmentedScan"
 * (luma.gl), section "Composition", which names the segmented reduction
 * beside the segmented scan; the segments are those of "Contract"):
 * d_out[s] = d_values[offsets[s]] + ... + d_values[offsets[s+1] - 1],
 * wrapping modulo 2^32, and 0 for an empty segment.
 *   d_values     n u32 (device, 16-byte aligned).
 *   d_offsets    num_segments + 1 u32 (device, 4-byte aligned),
 *                non-decreasing, d_offsets[num_segments] <= n.  Trusted, as
 *                for dwp_segmented_scan_u32: other offsets give unspecified
 *                sums, but every access stays inside the arrays.
 *   d_out        num_segments u32 (device, 4-byte aligned), overlapping no
 *                other argument.
 *   d_scratch    NULL: *scratch_bytes receives the size needed (128 bytes:
 *                a tile counter and the status word; this operation keeps
 *                no per-tile state).  Otherwise at least that many bytes,
 *                16-byte aligned, overlapping no other argument.
 * The call clears d_out and the scratch on `stream` and launches one kernel;
 * n == 0 or num_segments == 0 launches nothing.  Segment pieces that cross a
 * tile edge are added with atomics: the result is exact (u32 addition wraps
 * and commutes) and does not depend on the order.  Errors as for
 * dwp_segmented_scan_u32.
 */
dwp_status dwp_segmented_reduce_u32(const uint32_t *d_values, const uint32_t *d_offsets,
                                    size_t num_segments, uint32_t *d_out, size_t n,
                                    void *d_scratch, size_t *scratch_bytes, dwp_stream stream);

/*
 * First-order linear recurrence ("Parallel Prefix Sum (Scan), in depth",
 * section "What scan builds"): h[t] = a[t] * h[t-1] + b[t] with h[-1] = 0,
 * computed as a single-pass scan of the pairs (a[t], b[t]) under
 * (a1, b1) then (a2, b2) = (a1 a2, a2 b1 + b2).
 *   d_a, d_b  n f32 coefficients and inputs (device, 16-byte aligned).
 *   d_h       n f32 outputs (device, 16-byte aligned).  DWP_INCLUSIVE
 *             writes h[t]; DWP_EXCLUSIVE writes the state before step t,
 *             h[t-1] (0 at t = 0).  d_h may equal d_a or d_b exactly (in
 *             place); any other overlap with them is DWP_ERR_ALIASING.
 *   d_scratch NULL: *scratch_bytes receives the size needed (a 128-byte
 *             header plus 16 bytes per tile) and nothing else happens.
 *             Otherwise at least that many bytes, 16-byte aligned, owned by
 *             the caller, overlapping no other argument.
 * Arithmetic is f32 with one fused multiply-add per step; the grouping
 * differs from the sequential loop, so results agree with it to f32
 * rounding, not bit for bit.  Errors as for dwp_scan_exclusive; the
 * Decoupled Fallback applies except in place.
 */
dwp_status dwp_linear_recurrence_f32(const float *d_a, const float *d_b, float *d_h, size_t n,
                                     dwp_mode mode, void *d_scratch, size_t *scratch_bytes,
                                     dwp_stream stream);

/*
 * Device-side status of the most recent call that used d_scratch.
 * Synchronises `stream`, then reads the status word.  Returns DWP_SUCCESS,
 * DWP_ERR_LOOKBACK_TIMEOUT or DWP_ERR_PIPELINE_TIMEOUT (and, in a library
 * built with -DDWP_DEBUG_BOUNDS=1, DWP_ERR_BOUNDS); DWP_ERR_CUDA if the
 * synchronisation or the read fails; DWP_ERR_INVALID_VALUE for NULL.
 */
dwp_status dwp_read_status(const void *d_scratch, dwp_stream stream);

/*
 * Decoupled Fallback count of the most recent call that used d_scratch
 * ("GPU Prefix Sums", section "Decoupled Fallback").  A tile whose
 * look-back waits too long on a predecessor that has not published reduces
 * that predecessor's input itself and publishes the result with a
 * compare-and-swap; *count receives the number of such swaps that won.  It
 * is 0 in a healthy run: the fallback starts only after thousands of polls
 * (milliseconds).  Synchronises `stream`.  DWP_ERR_INVALID_VALUE for a NULL
 * argument; DWP_ERR_CUDA if the synchronisation or the read fails.
 */
dwp_status dwp_read_fallbacks(const void *d_scratch, dwp_stream stream, uint32_t *count);

/*
 * Look-back counters of the most recent call that used d_scratch (plain
 * scan, segmented scan or compaction): Decoupled Fallbacks won (as
 * dwp_read_fallbacks), intermediate descriptors published by a bounded
 * look-back window ("Single-Pass Prefix Scan with Decoupled Look-Back",
 * section "Why the work stays linear"; see dwp_set_lookback_window), and
 * look-back steps that jumped over such an intermediate.  Any output pointer
 * may be NULL.  Synchronises `stream`.  DWP_ERR_INVALID_VALUE for a NULL
 * d_scratch; DWP_ERR_CUDA if the synchronisation or the read fails.
 */
dwp_status dwp_read_lookback_stats(const void *d_scratch, dwp_stream stream, uint32_t *fallbacks,
                                   uint32_t *intermediates, uint32_t *jumps);

/* Static, NUL-terminated name of a status code. */
const char *dwp_status_string(dwp_status status);

/* Library version: major * 10000 + minor * 100 + patch. */
int dwp_version(void);

/*
 * Look-back window, a tuning setting for every later call in this process
 * ("Single-Pass Prefix Scan with Decoupled Look-Back", section "Why the work
 * stays linear"): 0 (the default) lets a look-back follow the chain of
 * predecessors as far as it goes.  tiles > 0 bounds it: each time a tile's
 * look-back has folded `tiles` more predecessors without reaching a prefix,
 * it publishes an intermediate descriptor (the sum so far with its own
 * aggregate, and how many tiles that covers), and a later look-back that
 * meets it jumps over that many tiles at once.  Folds go 32 tiles at a
 * time, so the window is effectively rounded up to a multiple of 32.
 * Applies to the plain and segmented scans and to compaction; results do not
 * depend on it (bit for bit for the integer operations).  Not thread-safe;
 * affects every device.  Always DWP_SUCCESS.
 */
dwp_status dwp_set_lookback_window(uint32_t tiles);

/*
 * Test hook, not for production use.  For every later call in this process
 * until reset:
 *   - the tile with index `never_publish_tile` does its work but never
 *     publishes its descriptor (UINT32_MAX disables this);
 *   - look-back spins give up after `spin_limit` polls (0 restores the
 *     default, about a second of polling);
 *   - a look-back takes the Decoupled Fallback after `fallback_polls` polls
 *     on an unpublished predecessor (0 restores the default, 4096 polls;
 *     UINT32_MAX disables the fallback).
 * With the fallback on, the successors of the silent tile reduce its input
 * themselves and the call succeeds with correct output (see
 * dwp_read_fallbacks).  With it off, or for an in-place scan (where the
 * fallback is always off: the silent tile's input may already have been
 * overwritten), they record DWP_ERR_LOOKBACK_TIMEOUT in the scratch status
 * and exit instead of waiting forever.  Not thread-safe; affects every
 * device.
 */
dwp_status dwp_debug_set_fault(uint32_t never_publish_tile, uint32_t spin_limit,
                               uint32_t fallback_polls);

/*
 * Test hook, not for production use: the step-by-step trace of the warp
 * layer's Hillis-Steele scan ("Parallel Prefix Sum (Scan), in depth",
 * section "Hillis-Steele: short span, too much work"), the shuffle scan that
 * dwp_scan_two_level runs on every warp.  One warp loads d_x[0 .. width)
 * (u32 addition; lanes past width hold 0) and runs the scan; after step k
 * (k = 0..4, offset d = 2^k) lane l writes its running value to
 * d_steps[width * k + l] for l < width.  So the page's 8-element trace can
 * be checked step by step on the device.
 *   d_x      device uint32[width];   d_steps  device uint32[5 * width]
 *   width    1 .. 32 (DWP_ERR_INVALID_VALUE otherwise, or for NULL pointers)
 * Asynchronous on `stream`; DWP_ERR_CUDA if the launch fails.
 */
dwp_status dwp_debug_warp_scan_trace(const uint32_t *d_x, size_t width, uint32_t *d_steps,
                                     dwp_stream stream);

/*
 * Test hook, not for production use: schedule perturbation for every later
 * call of the look-back kernels (plain and segmented scan, compaction,
 * linear recurrence) in this process until reset.  A missing ordering step
 * in a chained scan shows only under rare interleavings ("Parallel Prefix
 * Sum (Scan), in depth", section "Failure modes"); this makes a seeded
 * subset of tiles sleep at their publication points (after drawing the
 * tile index, before publishing the aggregate, before the look-back, before
 * publishing the prefix, and between the two words of a two-word
 * descriptor), so that descriptors appear in other orders than the
 * hardware's usual one.  Results must not change.
 *   seed          selects the subset and the sleep lengths
 *   fraction_ppm  share of (tile, point) pairs that sleep, in parts per
 *                 million (0 switches the hook off; at most 1000000)
 *   max_ns        longest sleep, at most 100000 ns
 * Every sleep is bounded.  DWP_ERR_INVALID_VALUE for arguments out of
 * range.  Not thread-safe; affects every device.
 */
dwp_status dwp_debug_set_delay(uint32_t seed, uint32_t fraction_ppm, uint32_t max_ns);

#ifdef __cplusplus
}
#endif

#endif /* DWP_H */
