// seg_rle.cuh -- producers of offsets: run-length encoding of an ordered
// uint32 vector (GPURunLengthEncode / GPUUnique, luma.gl API reference:
// "What is run-length encoding?", "Contract") and offsets from segment-start
// flags (GPUSegmentedLayout, named on GPUSegmentedReduction's page).
//
// A run starts at index i when i == 0 or keys[i] != keys[i-1]; a flagged
// segment starts at i when flags[i] != 0.  Two launches follow the page's
// outline (detect boundaries, scan them to dense indices, materialise):
//
//  1. count: CTA b owns a contiguous range of tiles (RLE_TILE elements
//     each); it marks the starts, writes them as a bitmap (bit i: element i
//     starts a run; n/8 bytes, small enough to stay in L2), and records per
//     tile the number of starts, and per CTA their total and the first one;
//  2. write: one CTA per tile (the hardware balances tiles dense in starts
//     against empty ones).  Its first run index and the first start after it
//     come from one round of loads over the per-CTA words and its count
//     CTA's per-tile words, with a block-wide sum and minimum; a block scan
//     ranks the tile's starts into shared memory, then offsets, values (a
//     gather of keys[start]) and lengths (the next start minus this one) go
//     out coalesced.  The last tile's CTA writes the run count and
//     offsets[count] = n.
//
// The count CTAs used to scan the per-CTA counts in the last of them to
// finish, while the other SMs idled (on 64M flags, SMs active 31 K of 45 K
// elapsed cycles under ncu); each write CTA now sums what it needs itself.
// A persistent write pass (one CTA per count range, tiles in order) was
// slower on the skewed keys, whose starts crowd into few ranges.
//
// The input is read once in full (count pass); the write pass reads the
// bitmap and, for run-length encoding, the keys at run starts only.  A
// single pass that scans with a decoupled look-back over per-tile states was
// slower on GB300: under full streaming load every look-back poll of L2
// waits about as long as a DRAM load, and the look-back sits on each tile's
// critical path.
//
// The launches take no lock and read no answer on the host.
#pragma once
#include <cstdint>
#include <cuda_runtime.h>

namespace segred {

constexpr int RLE_NT = 256;                    // threads per CTA (count and write)
constexpr int RLE_TILE = RLE_NT * 64;          // elements per tile: one 64-bit bitmap word per thread
constexpr int RLE_KEYS_PER = 16;               // count pass: uint32 keys per thread per step (4 steps a tile)
constexpr int RLE_FLAGS_PER = 64;              // count pass: flag bytes per thread per step (1 step a tile)
constexpr int RLE_MAX_CTAS = 1024;             // CTAs of each launch, at most
constexpr int RLE_CTAS_PER_SM = 4;

struct RleParams {
    const uint32_t* keys;    // run-length input, or nullptr
    const uint8_t* flags;    // flags input, or nullptr
    int64_t n;
    int64_t tiles;           // ceil(n / RLE_TILE)
    int32_t ctas;            // CTAs of the count and write launches (<= RLE_MAX_CTAS)
    int32_t vec;             // 1: the input is 16-byte aligned (128-bit loads)
    int32_t flags_mode;      // 1: flags to offsets, 0: run-length encoding
    uint32_t* values;        // [>= n] or nullptr
    uint32_t* lengths;       // [>= n] or nullptr
    int64_t* offsets;        // [>= n + 1] or nullptr
    int64_t* count;          // [1]
    int64_t* cta_count;      // scratch [ctas]
    int64_t* cta_first;      // scratch [ctas]
    int32_t* tile_count;     // scratch [tiles]
    int64_t* tile_first;     // scratch [tiles]
    unsigned long long* bitmap;  // scratch [tiles * RLE_NT]: bit i set when element i starts
};

// Once per device: the kernels' shared-memory carveout.
cudaError_t configure_rle();

// Scratch bytes of the per-CTA arrays (for RLE_MAX_CTAS CTAs) and of the
// per-tile arrays and bitmap for `tiles` tiles.
constexpr int64_t RLE_CTA_SCRATCH = int64_t(2) * 8 * RLE_MAX_CTAS;
inline int64_t rle_tile_bytes(int64_t tiles) {
    return ((tiles * 12 + 255) / 256) * 256 + tiles * RLE_NT * 8;
}

// Enqueue the launches on `stream` (count and write; one small kernel when n == 0).  The caller has checked the
// arguments; returns the first launch error.
cudaError_t launch_rle(const RleParams& p, cudaStream_t stream);

}  // namespace segred
