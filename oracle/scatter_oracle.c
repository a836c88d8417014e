/*
 * scatter_oracle.c -- CPU oracle for the unsorted scatter path.
 *
 * TEST INFRASTRUCTURE ONLY: used by tests/ and the benchmark's CPU-baseline
 * leg, nothing in the product path.  It shares no code with the CUDA library.
 *
 * graph-reduce README (HF kernels hub), "API": scatter_sum / scatter_add sum
 * the rows of src [N, F] into the output row named by index[r] (int64, [N]);
 * scatter_mean divides by the number of rows sent there, and an output that
 * received none is 0; scatter_max / scatter_min return (values, arg), the arg
 * being the source row.  "Method": ties go to the lower row.
 *
 * Readings where the pages are silent (the same as the segmented path's):
 *   - an output that receives no row gives 0, and arg -1 for max / min;
 *   - an index outside [0, dim_size) sends its row nowhere;
 *   - float32 sums accumulate in double and are rounded to float once;
 *     mean = (float)sum / (float)count;
 *   - integer sums wrap modulo 2^32; uint32 compares unsigned, sint32
 *     signed, float32 by IEEE '<' / '>' (NaN inputs are not defined);
 *   - mean is defined for float32 only.
 *
 * One pass over the rows in order, no reordering.
 */
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define SC_U32 0
#define SC_S32 1
#define SC_F32 2
#define SC_SUM 0
#define SC_MIN 1
#define SC_MAX 2
#define SC_MEAN 3

/* Returns 0, -1 on a bad argument, -3 for mean on integers, -4 when out of
 * memory.  out: [D, F] of the dtype; arg: [D, F] int64 or NULL (min / max). */
int oracle_scatter(const void *src, int dtype, int64_t F, int64_t N, const int64_t *index,
                   int64_t D, int op, void *out, int64_t *arg)
{
    if (F < 1 || N < 0 || D < 0 || (N > 0 && (src == 0 || index == 0)) || (D > 0 && out == 0))
        return -1;
    if (dtype < SC_U32 || dtype > SC_F32 || op < SC_SUM || op > SC_MEAN)
        return -1;
    if (op == SC_MEAN && dtype != SC_F32)
        return -3;
    const int64_t cells = D * F;
    int64_t *count = (int64_t *)calloc((size_t)(D > 0 ? D : 1), sizeof(int64_t));
    double *acc = (double *)calloc((size_t)(cells > 0 ? cells : 1), sizeof(double));
    uint32_t *iacc = (uint32_t *)calloc((size_t)(cells > 0 ? cells : 1), sizeof(uint32_t));
    int64_t *best = (int64_t *)malloc((size_t)(cells > 0 ? cells : 1) * sizeof(int64_t));
    if (!count || !acc || !iacc || !best) {
        free(count); free(acc); free(iacc); free(best);
        return -4;
    }
    for (int64_t c = 0; c < cells; ++c)
        best[c] = -1;
    for (int64_t r = 0; r < N; ++r) {
        const int64_t d = index[r];
        if (d < 0 || d >= D)
            continue;
        count[d] += 1;
        for (int64_t f = 0; f < F; ++f) {
            const int64_t c = d * F + f;
            const int64_t i = r * F + f;
            if (op == SC_SUM || op == SC_MEAN) {
                if (dtype == SC_F32)
                    acc[c] += (double)((const float *)src)[i];
                else
                    iacc[c] += ((const uint32_t *)src)[i];
                continue;
            }
            /* min / max: replace only when strictly better, so the first
             * (lowest) row holding the extreme stays */
            if (best[c] < 0) {
                best[c] = r;
                continue;
            }
            const int64_t j = best[c] * F + f;
            int better;
            if (dtype == SC_F32) {
                const float x = ((const float *)src)[i], y = ((const float *)src)[j];
                better = op == SC_MIN ? x < y : x > y;
            } else if (dtype == SC_S32) {
                const int32_t x = ((const int32_t *)src)[i], y = ((const int32_t *)src)[j];
                better = op == SC_MIN ? x < y : x > y;
            } else {
                const uint32_t x = ((const uint32_t *)src)[i], y = ((const uint32_t *)src)[j];
                better = op == SC_MIN ? x < y : x > y;
            }
            if (better)
                best[c] = r;
        }
    }
    for (int64_t d = 0; d < D; ++d) {
        for (int64_t f = 0; f < F; ++f) {
            const int64_t c = d * F + f;
            if (op == SC_SUM || op == SC_MEAN) {
                if (dtype == SC_F32) {
                    float s = (float)acc[c];
                    if (op == SC_MEAN)
                        s = count[d] > 0 ? s / (float)count[d] : 0.0f;
                    ((float *)out)[c] = s;
                } else {
                    ((uint32_t *)out)[c] = iacc[c];
                }
            } else {
                const int64_t b = best[c];
                if (dtype == SC_F32)
                    ((float *)out)[c] = b < 0 ? 0.0f : ((const float *)src)[b * F + f];
                else
                    ((uint32_t *)out)[c] = b < 0 ? 0u : ((const uint32_t *)src)[b * F + f];
                if (arg)
                    arg[c] = b;
            }
        }
    }
    free(count); free(acc); free(iacc); free(best);
    return 0;
}
