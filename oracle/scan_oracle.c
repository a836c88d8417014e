/*
 * scan_oracle.c -- CPU oracle for the segmented scan over CSR offsets.
 *
 * TEST INFRASTRUCTURE ONLY: used by tests/ and the benchmark's CPU-baseline
 * leg, nothing in the product path.  It shares no code with the CUDA library.
 *
 * The pages name a segmented scan (GPUSegmentedScan, next to GPUScan in the
 * luma.gl GPURunLengthEncode page) without defining it.  The plain reading,
 * built on the segments of GPUSegmentedReduction ("What is an
 * offset-delimited segment?", "Contract"): for every row r of segment s,
 * i.e. offsets[s] <= r < offsets[s+1],
 *   inclusive: out[r] = op(values[offsets[s]], ..., values[r]);
 *   exclusive (sum only): out[r] = sum(values[offsets[s]], ..., values[r-1]),
 *     0 for the segment's first row;
 * and out[r] = 0 for a row in no segment (before offsets[0] or from
 * offsets[S] on).  op is sum (uint32 / sint32 wrap modulo 2^32; float32
 * accumulates in double in row order, each output rounded to float once),
 * min or max (uint32 unsigned, sint32 signed, float32 by IEEE '<' / '>').
 *
 * One pass over each segment in row order.
 */
#include <stdint.h>

#define SN_U32 0
#define SN_S32 1
#define SN_F32 2
#define SN_SUM 0
#define SN_MIN 1
#define SN_MAX 2

/* Returns 0, -1 on a bad argument, -2 when the offsets are not nondecreasing
 * within [0, N].  offsets: int64 [S + 1]; out: [N] of the dtype. */
int oracle_seg_scan(const void *values, int dtype, int64_t N, const int64_t *offsets, int64_t S,
                    int op, int exclusive, void *out)
{
    if (N < 0 || S < 0 || offsets == 0 || (N > 0 && (values == 0 || out == 0)))
        return -1;
    if (dtype < SN_U32 || dtype > SN_F32 || op < SN_SUM || op > SN_MAX || (exclusive && op != SN_SUM))
        return -1;
    for (int64_t s = 0; s <= S; ++s) {
        if (offsets[s] < 0 || offsets[s] > N || (s > 0 && offsets[s] < offsets[s - 1]))
            return -2;
    }
    for (int64_t r = 0; r < N; ++r) {
        if (dtype == SN_F32)
            ((float *)out)[r] = 0.0f;
        else
            ((uint32_t *)out)[r] = 0u;
    }
    for (int64_t s = 0; s < S; ++s) {
        const int64_t b = offsets[s], e = offsets[s + 1];
        double dacc = 0.0;
        uint32_t uacc = 0u;
        for (int64_t r = b; r < e; ++r) {
            if (op == SN_SUM) {
                if (dtype == SN_F32) {
                    const double before = dacc;
                    dacc += (double)((const float *)values)[r];
                    ((float *)out)[r] = (float)(exclusive ? before : dacc);
                } else {
                    const uint32_t before = uacc;
                    uacc += ((const uint32_t *)values)[r];
                    ((uint32_t *)out)[r] = exclusive ? before : uacc;
                }
                continue;
            }
            /* running min / max: the previous output unless this row is better */
            if (r == b) {
                if (dtype == SN_F32)
                    ((float *)out)[r] = ((const float *)values)[r];
                else
                    ((uint32_t *)out)[r] = ((const uint32_t *)values)[r];
                continue;
            }
            if (dtype == SN_F32) {
                const float x = ((const float *)values)[r], y = ((float *)out)[r - 1];
                ((float *)out)[r] = (op == SN_MIN ? x < y : x > y) ? x : y;
            } else if (dtype == SN_S32) {
                const int32_t x = ((const int32_t *)values)[r], y = ((int32_t *)out)[r - 1];
                ((int32_t *)out)[r] = (op == SN_MIN ? x < y : x > y) ? x : y;
            } else {
                const uint32_t x = ((const uint32_t *)values)[r], y = ((uint32_t *)out)[r - 1];
                ((uint32_t *)out)[r] = (op == SN_MIN ? x < y : x > y) ? x : y;
            }
        }
    }
    return 0;
}
