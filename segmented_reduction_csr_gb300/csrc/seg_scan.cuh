// seg_scan.cuh -- segmented scan over CSR offsets: for every row r of
// segment s (offsets[s] <= r < offsets[s+1]) the inclusive sum / min / max
// of values[offsets[s] .. r], or the exclusive sum of values[offsets[s] ..
// r - 1]; rows in no segment give 0.  (The pages name a segmented scan,
// GPUSegmentedScan, beside GPUScan; the segments are GPUSegmentedReduction's.)
//
// Launches, each reading what the previous one wrote:
//  1. zero a start bitmap (bit r: a segment starts at row r);
//  2. set the bit of every offset (one atomic OR per offset);
//  3. scan: CTA b owns a contiguous range of tiles (RS_TILE rows: 16 per
//     thread) and scans them in order, carrying the open segment from tile
//     to tile in registers: a per-thread scan with resets at the start
//     bits, then a segmented scan over the lanes and the warps.  Rows are
//     written without the part of their segment that lies in earlier CTAs.
//     The CTA records its aggregate -- whether its range holds a start, and
//     the reduction of its rows after the last start -- and the row of its
//     first start.  The CTA that arrives last on a generation-tagged ticket
//     scans the aggregates into each CTA's carry-in (float32 sums as
//     compensated float pairs);
//  4. fix-up: the rows of each range before its first start belong to a
//     segment that began in an earlier range; they get the carry-in added
//     (float32 sums as a two-float carry, so the rounding stays that of one
//     addition).  Segments shorter than a range touch a few rows here; a
//     segment that spans whole ranges is read and written once more.
#pragma once
#include <cstdint>
#include <cuda_runtime.h>

#include "seg_common.cuh"   // PartPair

namespace segred {

constexpr int RS_NT = 128;
constexpr int RS_PER = 16;
constexpr int RS_TILE = RS_NT * RS_PER;    // 2,048 rows
constexpr int RS_MAX_CTAS = 1024;

struct ScanParams {
    const void* values;        // [N] of the dtype
    const void* offsets;       // [S + 1], uint32 or int64
    int32_t off64;
    int32_t dtype;             // 0 uint32, 1 int32, 2 float32
    int32_t op;                // 0 sum, 1 min, 2 max
    int32_t exclusive;         // sum only
    int32_t vec;               // 1: values and out 16-byte aligned (128-bit loads and stores)
    int64_t N, S;
    void* out;                 // [N]
    int64_t tiles;             // ceil(N / RS_TILE)
    int32_t sm_count;
    int32_t ctas;              // set by launch_scan: one wave of scan CTAs, at most RS_MAX_CTAS
    uint32_t gen;
    unsigned long long* ticket;
    unsigned long long* bitmap;   // scratch [N / 64 + 1]
    PartPair* cta_aggf;           // scratch [ctas]: float32 sums (hi, lo)
    uint32_t* cta_aggi;           // scratch [ctas]: other ops (value bits)
    int32_t* cta_flag;            // scratch [ctas]: the range holds a start
    int64_t* cta_first;           // scratch [ctas]: first start row of the range (or its end)
    PartPair* carryf;             // scratch [ctas]
    uint32_t* carryi;             // scratch [ctas]
};

inline int64_t rs_bitmap_words(int64_t N) { return N / 64 + 1; }

// Enqueue the launches on `stream`; N > 0.
cudaError_t launch_scan(const ScanParams& p, cudaStream_t stream);

}  // namespace segred
