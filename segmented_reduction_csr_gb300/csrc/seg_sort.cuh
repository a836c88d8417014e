// seg_sort.cuh -- a stable sort of the scatter path's rows by destination, the
// first half of the deterministic scatter (graph-reduce README,
// "Correctness": the atomic path's order is not fixed; sorting the rows by
// destination and reducing the contiguous groups is).
//
// Keys are the destinations, with every index outside [0, D) mapped to D so
// that those rows sort last; values are the row numbers.  A least
// significant digit radix sort, 8 bits a pass, as many passes as D needs.
// Each pass:
//  1. histogram: CTA t counts the digits of tile t (RS_SORT_TILE keys) in
//     shared memory and writes them digit-major: hist[digit * T + t];
//  2. scan: CTA d scans digit d's row of the histogram (the tiles' exclusive
//     prefix within the digit) and its total;
//  3. scatter: CTA t ranks its keys stably -- in row order, 256 at a time,
//     peers of a digit found with a warp match, warps in order -- and writes
//     key and value to digit base + tile prefix + rank.
// Then offsets[d] = lower bound of d in the sorted keys (d = 0 .. D), the
// rows are gathered in sorted order, and the segmented reduction runs over
// them with those offsets.
#pragma once
#include <cstdint>
#include <cuda_runtime.h>

namespace segred {

constexpr int SORT_NT = 256;                       // threads per CTA
constexpr int SORT_ITEMS = 8;                      // keys per thread per tile
constexpr int SORT_TILE = SORT_NT * SORT_ITEMS;    // 2,048 keys
constexpr int SORT_RADIX = 256;                    // 8-bit digits

struct SortParams {
    const int64_t* index;    // [N] destinations (the first pass reads them)
    int64_t N, D;
    int64_t tiles;           // ceil(N / SORT_TILE)
    uint32_t* keys[2];       // scratch [N] each: ping-pong
    uint32_t* vals[2];       // scratch [N] each: row numbers
    uint32_t* hist;          // scratch [SORT_RADIX * tiles]: counts, then exclusive prefixes
    uint32_t* total;         // scratch [SORT_RADIX]
    int passes;              // ceil(bits of D / 8)
};

// Scratch bytes of the sort for N rows.
inline int64_t sort_scratch_bytes(int64_t N) {
    const int64_t tiles = (N + SORT_TILE - 1) / SORT_TILE;
    return 16 * N + 4 * SORT_RADIX * tiles + 4 * SORT_RADIX + 1024;
}

// Enqueue the passes; keys[(passes - 1) % 2] / vals[(passes - 1) % 2] then
// hold the sorted keys and row numbers.
cudaError_t launch_sort(const SortParams& p, cudaStream_t stream);

// offsets[d] = #{sorted keys < d} for d = 0 .. D (int64, D + 1 entries).
cudaError_t launch_bucket_offsets(const uint32_t* sorted, int64_t N, int64_t D, int64_t* offsets,
                                  cudaStream_t stream);

// dst[i, :] = src[perm[i], :] for i < N (F 32-bit columns per row).
cudaError_t launch_gather_rows(const void* src, const uint32_t* perm, int64_t N, int64_t F, void* dst,
                               cudaStream_t stream);

// arg[i] = arg[i] < 0 ? -1 : perm[arg[i]] for i < n.
cudaError_t launch_map_args(int64_t* arg, const uint32_t* perm, int64_t n, cudaStream_t stream);

}  // namespace segred
