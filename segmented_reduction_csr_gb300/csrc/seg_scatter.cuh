// seg_scatter.cuh -- the unsorted scatter path (graph-reduce README, "API" and
// "Method"): row r of src [N, F] goes to output row index[r]; sum / mean add
// it there, max / min keep the extreme and the lowest row that holds it.
//
// One atomic per element (per four elements for float32 sums with 128-bit
// vector reductions), as the page's method, except that max and min skip
// the atomic of an element that the output's current word already beats
// (read from L2 just before; about ln n of n random candidates win).  For
// max and min the value and its row settle inside one 64-bit atomic: the value's bits made monotone
// (float32: negative values complemented, others with the sign bit set;
// int32: the sign bit flipped; uint32: as is) in the high half, and the row
// in the low half -- complemented for max, so that the largest word holds
// the maximum and, among equal values, the lowest row; as is for min.
// -0.0 is taken as +0.0 there (IEEE compares them equal, so the lower row
// must win); the finishing pass turns the word's high half back into the
// value, and reads a float32 zero back from the winning row of src, so the
// output keeps its sign bit.
//
// Float32 sums and means are not deterministic: the order in which the
// atomics land varies from run to run.  Integer sums (modulo 2^32) and max /
// min are.
#pragma once
#include <cstdint>
#include <cuda_runtime.h>

namespace segred {

constexpr int SC_NT = 256;        // threads per CTA
constexpr int SC_ITEMS = 4;       // (row, column chunk) items per thread

struct ScatterParams {
    const void* src;           // [N, F]
    const int64_t* index;      // [N]
    int64_t N, F, D;           // rows, columns, output rows
    int32_t dtype;             // 0 uint32, 1 int32, 2 float32
    int32_t op;                // 0 sum, 1 min, 2 max, 3 mean
    int32_t vec;               // columns per item: 4 (16-byte aligned src, out, F % 4 == 0) or 1
    void* out;                 // [D, F]
    int64_t* arg;              // [D, F] or nullptr
    unsigned long long* word;  // scratch [D, F]: packed (value, row) for max / min
    uint32_t* count;           // scratch [D]: rows received, for mean
};

// Enqueue the launches on `stream`; D * F > 0.
cudaError_t launch_scatter(const ScatterParams& p, cudaStream_t stream);

}  // namespace segred
