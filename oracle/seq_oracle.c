/*
 * seq_oracle.c -- sequential CPU oracle for the input-order float32 mode.
 *
 * TEST INFRASTRUCTURE ONLY: used by tests/ and nothing in the product path.
 * It shares no code with the CUDA library.
 *
 * graph-reduce README (HF kernels hub), "Correctness": the CSR path is
 * bitwise equal to torch.segment_reduce because its summation order is
 * fixed; empty outputs are 0 for sum and mean.  The plain reading of a fixed
 * order that a user can reproduce is the input order: the sum of segment s
 * in column f starts from 0.0f and adds values[r, f] for r = offsets[s],
 * offsets[s] + 1, ..., offsets[s+1] - 1, each addition rounded to float32
 * (round to nearest even).  The mean is that float32 sum divided by the
 * segment length as a float32, one more rounding; an empty segment gives 0.
 *
 * Built with -ffp-contract=off and without fast-math, so every '+' below is
 * one IEEE float32 addition in the order written.
 */
#include <stdint.h>

/* Returns 0, -1 on a bad argument, -2 when the offsets are not
 * nondecreasing within [0, N].  values: [N, F] row-major float32; offsets:
 * [S + 1] int64; out: [S, F] float32. */
int oracle_seg_sequential_f32(const float *values, int64_t N, int64_t F, const int64_t *offsets,
                              int64_t S, int mean, float *out)
{
    if (N < 0 || F < 1 || S < 0 || (S > 0 && (offsets == 0 || out == 0)) || (N > 0 && values == 0))
        return -1;
    for (int64_t s = 0; s <= S; ++s) {
        if (offsets[s] < 0 || offsets[s] > N || (s > 0 && offsets[s] < offsets[s - 1]))
            return -2;
    }
    for (int64_t s = 0; s < S; ++s) {
        const int64_t b = offsets[s], e = offsets[s + 1];
        for (int64_t f = 0; f < F; ++f) {
            float acc = 0.0f;
            for (int64_t r = b; r < e; ++r)
                acc = acc + values[r * F + f];
            if (mean)
                acc = e > b ? acc / (float)(e - b) : 0.0f;
            out[s * F + f] = acc;
        }
    }
    return 0;
}
