// seg_seq.cuh -- the input-order float32 mode: per segment and column, a sum
// that starts at 0.0f and adds the rows in order, each addition rounded to
// float32 (graph-reduce README, "Correctness": a fixed summation order, the
// one that makes its CSR path bitwise equal to torch.segment_reduce); mean is
// that sum divided by the length as a float32; an empty segment gives 0.
//
// The order is a single chain of dependent additions per (segment, column),
// so each thread owns one chain: thread i takes segment i / F, column i % F.
// A warp then reads 32 adjacent columns of one row (coalesced) when F >= 32,
// and 32 adjacent segments' rows when F == 1.  Loads are issued eight rows
// ahead of the additions.  The time of a call is bounded below by its
// longest segment: about one float32 addition latency per row.
#pragma once
#include <cstdint>
#include <cuda_runtime.h>

namespace segred {

constexpr int SEQ_NT = 256;    // threads per CTA
constexpr int SEQ_AHEAD = 8;   // rows loaded before they are added

struct SeqParams {
    const float* values;   // [N, F]
    const void* offsets;   // [S + 1], uint32 or int64
    int32_t off64;         // 1: int64 offsets
    int32_t mean;          // 1: divide by the length
    int64_t N, F, S;
    float* out;            // [S, F]
};

// Enqueue the launch on `stream` (S * F > 0).
cudaError_t launch_sequential(const SeqParams& p, cudaStream_t stream);

}  // namespace segred
