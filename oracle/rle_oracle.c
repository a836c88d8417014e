/*
 * rle_oracle.c -- sequential CPU oracle for the producers of offsets.
 *
 * TEST INFRASTRUCTURE ONLY: used by tests/ and nothing in the product path.
 * It shares no code with the CUDA library.
 *
 * oracle_rle follows GPURunLengthEncode and GPUUnique (luma.gl API reference),
 * "What is run-length encoding?" and "Contract".  Each maximal run of
 * adjacent equal uint32 values in the ordered input becomes one run.  The
 * outputs are the run's value, its length and the index where it starts.
 * Runs keep first-occurrence order.  Equal values that are not adjacent start
 * new runs.  Empty input gives zero runs.  The offsets take one more entry,
 * n, so that they delimit the runs as "Why RLE matters for GPU grouping"
 * describes (lengths [3,2,4] correspond to offsets [0,3,5,9]).
 *
 * oracle_flags_to_offsets follows GPUSegmentedReduction, "What is an
 * offset-delimited segment?" (GPUSegmentedLayout materialises offsets from
 * segment-start flags).  Every index whose flag is non-zero starts a
 * segment.  The offsets list those indices in order, then n.  Rows before
 * the first flag belong to no segment, as a first offset above 0 allows.
 */
#include <stdint.h>

/* Returns the number of runs (>= 0), or -1 on a bad argument.  Any output
 * pointer may be NULL.  values / lengths hold at least n entries, offsets
 * at least n + 1. */
int64_t oracle_rle(const uint32_t *keys, int64_t n, uint32_t *values, uint32_t *lengths,
                   int64_t *offsets)
{
    if (n < 0 || (n > 0 && keys == 0))
        return -1;
    int64_t runs = 0;
    int64_t start = 0;
    for (int64_t i = 0; i <= n; ++i) {
        /* a run ends before i when i == n or keys[i] differs from keys[i-1] */
        int ends_here = i > 0 && (i == n || keys[i] != keys[i - 1]);
        if (ends_here) {
            if (values)
                values[runs] = keys[start];
            if (lengths)
                lengths[runs] = (uint32_t)(i - start);
            if (offsets)
                offsets[runs] = start;
            runs += 1;
            start = i;
        }
    }
    if (offsets)
        offsets[runs] = n;
    return runs;
}

/* Returns the number of segments (>= 0), or -1 on a bad argument.  offsets
 * holds at least n + 1 entries. */
int64_t oracle_flags_to_offsets(const uint8_t *flags, int64_t n, int64_t *offsets)
{
    if (n < 0 || (n > 0 && flags == 0) || offsets == 0)
        return -1;
    int64_t count = 0;
    for (int64_t i = 0; i < n; ++i) {
        if (flags[i] != 0) {
            offsets[count] = i;
            count += 1;
        }
    }
    offsets[count] = n;
    return count;
}
