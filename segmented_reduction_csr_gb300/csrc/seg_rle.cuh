// seg_rle.cuh -- producers of offsets: run-length encoding of an ordered
// uint32 vector (GPURunLengthEncode / GPUUnique, luma.gl API reference:
// "What is run-length encoding?", "Contract") and offsets from segment-start
// flags (GPUSegmentedLayout, named on GPUSegmentedReduction's page).
//
// A run starts at index i when i == 0 or keys[i] != keys[i-1]; a flagged
// segment starts at i when flags[i] != 0.  Three launches follow the page's
// outline (detect boundaries, scan them to dense indices, materialise):
//
//  1. count: CTA b owns a contiguous range of tiles of RLE_TILE elements; it
//     counts the starts in its range and notes its first start;
//  2. scan: one CTA turns the per-CTA counts into each CTA's first run index
//     and finds, for each CTA, the first start after its range (n if none);
//     it writes the run count and offsets[count] = n;
//  3. write: CTA b walks its tiles in order.  Per tile, a block scan of the
//     threads' start counts places each start in shared memory; the block
//     then writes offsets, values and lengths coalesced.  A run's length is
//     the next start minus its own; the last run of a tile gets its length
//     when the next start turns up (a later tile, or the first start after
//     the range found by the scan).
//
// The launches take no lock and read no answer on the host.
#pragma once
#include <cstdint>
#include <cuda_runtime.h>

namespace segred {

constexpr int RLE_NT = 256;                   // threads per CTA (count and write)
constexpr int RLE_PER = 16;                   // elements per thread per tile
constexpr int RLE_TILE = RLE_NT * RLE_PER;    // elements per tile
constexpr int RLE_MAX_CTAS = 1024;            // the scan pass is one CTA of this many threads
constexpr int RLE_CTAS_PER_SM = 4;

struct RleParams {
    const uint32_t* keys;    // run-length input, or nullptr
    const uint8_t* flags;    // flags input, or nullptr
    int64_t n;
    int64_t tiles;           // ceil(n / RLE_TILE)
    int32_t ctas;            // CTAs of the count and write launches (<= RLE_MAX_CTAS)
    int32_t vec;             // 1: the input is 16-byte aligned (128-bit loads)
    uint32_t* values;        // [>= n] or nullptr
    uint32_t* lengths;       // [>= n] or nullptr
    int64_t* offsets;        // [>= n + 1] or nullptr
    int64_t* count;          // [1]
    int64_t* cta_count;      // scratch [ctas]
    int64_t* cta_first;      // scratch [ctas]
    int64_t* cta_base;       // scratch [ctas]
    int64_t* cta_next;       // scratch [ctas]
};

// Scratch bytes the three launches need for `ctas` CTAs.
inline int64_t rle_scratch_bytes(int32_t ctas) { return int64_t(4) * 8 * ctas; }

// Enqueue the three launches on `stream`.  The caller has checked the
// arguments; returns the first launch error.
cudaError_t launch_rle(const RleParams& p, cudaStream_t stream);

}  // namespace segred
