/*
 * Sequential CPU oracle for the device-wide prefix scan library.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may call, link or
 * load this file: only the tests, the package's smoke check and the CPU
 * baseline leg of the benchmark use it.  It shares no code, header, table or
 * helper with the CUDA path.
 *
 * Every function is the plain definition of what it computes, one element
 * after another, in the order the definition states.  There is no blocking,
 * no tiling and no reordering.
 *
 * Definitions followed:
 *   - "Parallel Prefix Sum (Scan), in depth", section "Inclusive, exclusive
 *     and associative": inclusive y[i] = x[0] (+) ... (+) x[i]; exclusive
 *     y[0] = identity, y[i] = x[0] (+) ... (+) x[i-1].
 *   - "Prefix scans and compaction", section "Inclusive and exclusive scan":
 *     the additive identity is 0; for an integer maximum, the lowest
 *     representable value (0 for unsigned 32-bit).
 *   - "Prefix scans and compaction", sections "Scan as an index generator"
 *     and "Worked example: Stable stream compaction": kept record i goes to
 *     output[exclusive prefix of the flags at i]; the output length is the
 *     flag total.
 *   - "GPUSegmentedScan" (luma.gl), sections "Prefix scans and segmented
 *     scans" and "Contract": segment s is rows [offsets[s], offsets[s+1]),
 *     the running total restarts at every segment, empty segments write
 *     nothing.
 *   - "Parallel Prefix Sum (Scan), in depth", section "What scan builds": the
 *     first-order linear recurrence h[t] = a[t] h[t-1] + b[t].
 *   - "GPUSegmentedScan" (luma.gl), section "Composition": the segmented
 *     reduction it names beside the segmented scan, read as one u32 sum per
 *     segment of the same CSR offsets.
 *
 * Readings where the pages leave a step open (each also listed in the
 * design notes):
 *   - u32 addition wraps modulo 2^32 (unsigned arithmetic).
 *   - f32 addition: inputs are f32, the reference accumulates in double and
 *     returns double values; alongside it returns the running sum of |x|
 *     (double), which the tests turn into the tolerance
 *     1e-4 * sum|x| + 1e-6.
 *   - segmented rows outside [offsets[0], offsets[N]) are left untouched.
 *   - compaction flags are bytes, nonzero means keep.
 *   - segmented reduction: out[s] is the wrapping u32 sum of rows
 *     [offsets[s], offsets[s+1]); an empty segment gives 0, the identity.
 *   - linear recurrence: the state before the first step is 0 (the page's
 *     worked example starts from it); inputs are f32, the reference runs
 *     the loop in double; exclusive output is the state before each step;
 *     alongside it the same recurrence on |a| and |b|, which the tests turn
 *     into the tolerance 1e-4 * g + 1e-6.
 */
#include <stddef.h>
#include <stdint.h>
#include <string.h>

/* Plain scan with u32 addition (wraps modulo 2^32). */
void oracle_scan_u32_add(const uint32_t *x, uint64_t n, int inclusive, uint32_t *y)
{
    uint32_t acc = 0u; /* additive identity */
    for (uint64_t i = 0; i < n; ++i) {
        uint32_t xi = x[i];
        if (!inclusive)
            y[i] = acc;
        acc = acc + xi;
        if (inclusive)
            y[i] = acc;
    }
}

/* Plain scan with u32 maximum; identity 0, the lowest u32 value. */
void oracle_scan_u32_max(const uint32_t *x, uint64_t n, int inclusive, uint32_t *y)
{
    uint32_t acc = 0u;
    for (uint64_t i = 0; i < n; ++i) {
        uint32_t xi = x[i];
        if (!inclusive)
            y[i] = acc;
        acc = (xi > acc) ? xi : acc;
        if (inclusive)
            y[i] = acc;
    }
}

/*
 * Plain scan with addition of f32 inputs, accumulated in double.
 * y[i]    : the exact-order double prefix (exclusive or inclusive).
 * absy[i] : the double prefix of |x| over the same index range, for the
 *           tolerance.  Either output pointer may be NULL.
 */
void oracle_scan_f32_add(const float *x, uint64_t n, int inclusive, double *y, double *absy)
{
    double acc = 0.0, aacc = 0.0;
    for (uint64_t i = 0; i < n; ++i) {
        double xi = (double)x[i];
        if (!inclusive) {
            if (y) y[i] = acc;
            if (absy) absy[i] = aacc;
        }
        acc = acc + xi;
        aacc = aacc + (xi < 0.0 ? -xi : xi);
        if (inclusive) {
            if (y) y[i] = acc;
            if (absy) absy[i] = aacc;
        }
    }
}

/*
 * Segmented u32 addition scan over CSR offsets (num_segments + 1 entries).
 * For every segment s the running total starts again from 0 over rows
 * offsets[s] .. offsets[s+1]-1.  Rows no segment covers are not written.
 * Offsets are assumed non-decreasing with offsets[num_segments] <= n; the
 * loop clamps to n so that a broken precondition cannot write out of range.
 */
void oracle_segmented_scan_u32(const uint32_t *values, const uint32_t *offsets,
                               uint64_t num_segments, uint64_t n, int inclusive,
                               uint32_t *out)
{
    for (uint64_t s = 0; s < num_segments; ++s) {
        uint64_t lo = offsets[s], hi = offsets[s + 1];
        if (hi > n) hi = n;
        uint32_t acc = 0u;
        for (uint64_t i = lo; i < hi; ++i) {
            if (!inclusive)
                out[i] = acc;
            acc = acc + values[i];
            if (inclusive)
                out[i] = acc;
        }
    }
}

/*
 * Stable stream compaction of fixed-size records by byte flags.
 * Record i (record_bytes bytes) is copied to slot k of out, where k is the
 * number of kept records before i.  Returns the number kept.
 */
uint64_t oracle_compact(const void *records, const uint8_t *flags, uint64_t n,
                        uint64_t record_bytes, void *out)
{
    const unsigned char *src = (const unsigned char *)records;
    unsigned char *dst = (unsigned char *)out;
    uint64_t k = 0;
    for (uint64_t i = 0; i < n; ++i) {
        if (flags[i] != 0) {
            memcpy(dst + k * record_bytes, src + i * record_bytes, (size_t)record_bytes);
            ++k;
        }
    }
    return k;
}

/*
 * First-order linear recurrence h[t] = a[t] * h[t-1] + b[t], h[-1] = 0, as
 * the sequential loop the definition states, in double from f32 inputs.
 * Inclusive: y[t] = h[t].  Exclusive: y[t] = h[t-1], so y[0] = 0.
 * mag[t] (if not NULL) runs the same loop on magnitudes over the same range:
 * g[t] = |a[t]| * g[t-1] + |b[t]|, g[-1] = 0.
 */
void oracle_linear_recurrence_f32(const float *a, const float *b, uint64_t n, int inclusive,
                                  double *y, double *mag)
{
    double h = 0.0, g = 0.0;
    for (uint64_t t = 0; t < n; ++t) {
        double at = (double)a[t], bt = (double)b[t];
        if (!inclusive) {
            if (y) y[t] = h;
            if (mag) mag[t] = g;
        }
        h = at * h + bt;
        g = (at < 0.0 ? -at : at) * g + (bt < 0.0 ? -bt : bt);
        if (inclusive) {
            if (y) y[t] = h;
            if (mag) mag[t] = g;
        }
    }
}

/*
 * Segmented u32 addition reduction over CSR offsets (num_segments + 1
 * entries): out[s] = values[offsets[s]] + ... + values[offsets[s+1] - 1],
 * wrapping modulo 2^32, and 0 for an empty segment.  Offsets are assumed
 * non-decreasing with offsets[num_segments] <= n; the loop clamps to n so
 * that a broken precondition cannot read out of range.
 */
void oracle_segmented_reduce_u32(const uint32_t *values, const uint32_t *offsets,
                                 uint64_t num_segments, uint64_t n, uint32_t *out)
{
    for (uint64_t s = 0; s < num_segments; ++s) {
        uint64_t first = offsets[s], end = offsets[s + 1];
        if (end > n)
            end = n;
        uint32_t acc = 0u;
        for (uint64_t i = first; i < end; ++i)
            acc = acc + values[i];
        out[s] = acc;
    }
}
