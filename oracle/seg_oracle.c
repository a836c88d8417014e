/*
 * seg_oracle.c -- CPU oracle for segmented reduction over offset-delimited
 * (CSR indptr) segments.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the slow, obviously correct
 * definition that the CUDA library is checked against.  It shares no code,
 * header, constant or helper with the CUDA library, and only the test suite,
 * the smoke check and the benchmark's CPU-baseline leg may load it.
 *
 * What it computes (the plain definition, one segment at a time):
 *
 *   GPUSegmentedReduction (luma.gl docs), "What is an offset-delimited
 *   segment?": segment s owns the half-open row range [offsets[s],
 *   offsets[s+1]); S segments need S+1 offsets; repeated offsets are empty
 *   segments.  "Contract": output row s reduces input[o_s .. o_{s+1}), the
 *   first offset may be non-zero, values are uint32 / sint32 / float32, the
 *   operations are sum / min / max, and an empty segment produces zero.
 *
 *   graph-reduce README (HF kernels hub), "API" and "Method": src is [N, ...]
 *   reduced over dimension 0 (so an [N, F] tensor is reduced per column),
 *   min / max also return the source row that produced the value, ties go to
 *   the lower row, mean is the segment sum divided by its length and an empty
 *   mean is 0.  Its "Correctness" section gives -1 as the arg of an empty
 *   segment.
 *
 * Readings taken where the pages are silent or disagree:
 *   - empty min / max give 0 (the luma contract) with arg -1 (graph-reduce);
 *   - the arg is the absolute row index into values, as int64;
 *   - integer sums wrap modulo 2^32 for both uint32 and sint32;
 *   - uint32 compares unsigned, sint32 signed, float32 by IEEE '<' / '>'
 *     (so -0.0 and +0.0 tie and the lower row wins);
 *   - float32 sums accumulate in double in row order and are rounded to
 *     float once; mean = (float)sum / (float)length, both in float;
 *   - mean is defined for float32 only.
 *
 * No blocking, no reordering, no parallelism: one sequential loop.
 *
 * The CPU baseline of the benchmark also times this same loop on all host
 * cores: compiled a second time with ORC_PARALLEL_SEGMENTS and -fopenmp, the
 * (segment, column) iterations, which write disjoint outputs and each run
 * the same sequential inner loop, are shared among threads.  Each output is
 * then computed exactly as in the sequential build.  The parity checks use
 * the sequential build only.
 */
#include <stdint.h>
#include <string.h>
#ifdef ORC_PARALLEL_SEGMENTS
#include <omp.h>
#endif

/* Codes private to this file (the Python wrapper passes them). */
#define ORC_DT_U32 0
#define ORC_DT_S32 1
#define ORC_DT_F32 2

#define ORC_OFF_U32 0
#define ORC_OFF_I64 1

#define ORC_SUM 0
#define ORC_MIN 1
#define ORC_MAX 2
#define ORC_MEAN 3

#define ORC_OK 0
#define ORC_BAD_ARGUMENT (-1)
#define ORC_BAD_OFFSETS (-2)
#define ORC_MEAN_ON_INTEGER (-3)

static int64_t offset_at(const void *offsets, int off_dtype, int64_t s)
{
    if (off_dtype == ORC_OFF_U32)
        return (int64_t)((const uint32_t *)offsets)[s];
    return ((const int64_t *)offsets)[s];
}

/* Checks the producer's invariants: nondecreasing and inside [0, N]. */
static int check_offsets(const void *offsets, int off_dtype, int64_t S,
                         int64_t N)
{
    for (int64_t s = 0; s <= S; ++s) {
        int64_t o = offset_at(offsets, off_dtype, s);
        if (o < 0 || o > N)
            return ORC_BAD_OFFSETS;
        if (s > 0 && o < offset_at(offsets, off_dtype, s - 1))
            return ORC_BAD_OFFSETS;
    }
    return ORC_OK;
}

static void reduce_u32(const uint32_t *v, int64_t F, int64_t b, int64_t e,
                       int64_t f, int op, uint32_t *out, int64_t *arg)
{
    if (op == ORC_SUM) {
        uint32_t acc = 0u;                 /* unsigned: wraps mod 2^32 */
        for (int64_t r = b; r < e; ++r)
            acc += v[r * F + f];
        *out = acc;
        return;
    }
    uint32_t best = v[b * F + f];
    int64_t best_row = b;
    for (int64_t r = b + 1; r < e; ++r) {
        uint32_t x = v[r * F + f];
        if ((op == ORC_MIN && x < best) || (op == ORC_MAX && x > best)) {
            best = x;
            best_row = r;
        }
    }
    *out = best;
    *arg = best_row;
}

static void reduce_s32(const int32_t *v, int64_t F, int64_t b, int64_t e,
                       int64_t f, int op, int32_t *out, int64_t *arg)
{
    if (op == ORC_SUM) {
        uint32_t acc = 0u;                 /* two's complement wrap */
        for (int64_t r = b; r < e; ++r)
            acc += (uint32_t)v[r * F + f];
        memcpy(out, &acc, sizeof acc);
        return;
    }
    int32_t best = v[b * F + f];
    int64_t best_row = b;
    for (int64_t r = b + 1; r < e; ++r) {
        int32_t x = v[r * F + f];
        if ((op == ORC_MIN && x < best) || (op == ORC_MAX && x > best)) {
            best = x;
            best_row = r;
        }
    }
    *out = best;
    *arg = best_row;
}

static void reduce_f32(const float *v, int64_t F, int64_t b, int64_t e,
                       int64_t f, int op, float *out, int64_t *arg)
{
    if (op == ORC_SUM || op == ORC_MEAN) {
        double acc = 0.0;
        for (int64_t r = b; r < e; ++r)
            acc += (double)v[r * F + f];
        float sum = (float)acc;
        if (op == ORC_SUM) {
            *out = sum;
        } else {
            float len = (float)(e - b);
            *out = sum / len;
        }
        return;
    }
    float best = v[b * F + f];
    int64_t best_row = b;
    for (int64_t r = b + 1; r < e; ++r) {
        float x = v[r * F + f];
        if ((op == ORC_MIN && x < best) || (op == ORC_MAX && x > best)) {
            best = x;
            best_row = r;
        }
    }
    *out = best;
    *arg = best_row;
}

/*
 * values   : [num_values, F] row-major, element type `dtype`
 * offsets  : [S + 1], element type `off_dtype`
 * out      : [S, F], element type `dtype`
 * out_arg  : [S, F] int64, or NULL; written only for min / max
 * Returns ORC_OK, or a negative code (nothing is written then).
 */
int oracle_seg_reduce(const void *values, int dtype, int64_t F,
                      int64_t num_values, const void *offsets, int off_dtype,
                      int64_t S, int op, void *out, int64_t *out_arg)
{
    if (F < 1 || S < 0 || num_values < 0)
        return ORC_BAD_ARGUMENT;
    if (dtype < ORC_DT_U32 || dtype > ORC_DT_F32)
        return ORC_BAD_ARGUMENT;
    if (off_dtype != ORC_OFF_U32 && off_dtype != ORC_OFF_I64)
        return ORC_BAD_ARGUMENT;
    if (op < ORC_SUM || op > ORC_MEAN)
        return ORC_BAD_ARGUMENT;
    if (op == ORC_MEAN && dtype != ORC_DT_F32)
        return ORC_MEAN_ON_INTEGER;
    if (S > 0 && (offsets == 0 || out == 0))
        return ORC_BAD_ARGUMENT;
    if (S > 0) {
        int rc = check_offsets(offsets, off_dtype, S, num_values);
        if (rc != ORC_OK)
            return rc;
    }

    int with_arg = (op == ORC_MIN || op == ORC_MAX) && out_arg != 0;
#ifdef ORC_PARALLEL_SEGMENTS
#pragma omp parallel for collapse(2) schedule(dynamic, 64)
#endif
    for (int64_t s = 0; s < S; ++s) {
        for (int64_t f = 0; f < F; ++f) {
            int64_t b = offset_at(offsets, off_dtype, s);
            int64_t e = offset_at(offsets, off_dtype, s + 1);
            int64_t o = s * F + f;
            int64_t arg = -1;
            if (e == b) {
                /* empty segment: value 0, arg -1 */
                if (dtype == ORC_DT_F32)
                    ((float *)out)[o] = 0.0f;
                else
                    ((uint32_t *)out)[o] = 0u;
            } else if (dtype == ORC_DT_U32) {
                reduce_u32((const uint32_t *)values, F, b, e, f, op,
                           (uint32_t *)out + o, &arg);
            } else if (dtype == ORC_DT_S32) {
                reduce_s32((const int32_t *)values, F, b, e, f, op,
                           (int32_t *)out + o, &arg);
            } else {
                reduce_f32((const float *)values, F, b, e, f, op,
                           (float *)out + o, &arg);
            }
            if (with_arg)
                out_arg[o] = arg;
        }
    }
    return ORC_OK;
}

/* Threads the loop above runs on: 1 in the sequential build. */
int oracle_threads(void)
{
#ifdef ORC_PARALLEL_SEGMENTS
    return omp_get_max_threads();
#else
    return 1;
#endif
}
