// seg_rle.cuh -- producers of offsets: run-length encoding of an ordered
// uint32 vector (GPURunLengthEncode / GPUUnique, luma.gl API reference:
// "What is run-length encoding?", "Contract") and offsets from segment-start
// flags (GPUSegmentedLayout, named on GPUSegmentedReduction's page).
//
// A run starts at index i when i == 0 or keys[i] != keys[i-1]; a flagged
// segment starts at i when flags[i] != 0.  Three launches follow the page's
// outline (detect boundaries, scan them to dense indices, materialise):
//
//  1. count: CTA b owns a contiguous range of tiles (RLE_TILE elements
//     each); it marks the starts, writes them as a bitmap (bit i: element i
//     starts a run; n/8 bytes, small enough to stay in L2), and records per
//     tile the number of starts and the first one, and per CTA their total
//     and the first;
//  2. scan: the last count CTA to finish (a generation-tagged ticket tells
//     it) turns the per-CTA counts into each CTA's first run index and
//     finds, for each CTA, the first start after its range (n if none); it
//     writes the run count and offsets[count] = n;
//  3. write: one CTA per tile.  It finds its first run index (its count CTA's
//     base plus the counts of the tiles before it in that range) and the
//     first start after it, ranks its starts with a block scan into shared
//     memory, then writes offsets, values (a gather of keys[start]) and
//     lengths (the next start minus this one) coalesced.  One CTA per tile
//     lets the hardware balance tiles dense in starts against empty ones.
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
constexpr int RLE_MAX_CTAS = 1024;             // the scan pass is one CTA of this many threads
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
    int64_t* cta_base;       // scratch [ctas]
    int64_t* cta_next;       // scratch [ctas]
    int32_t* tile_count;     // scratch [tiles]
    int64_t* tile_first;     // scratch [tiles]
    unsigned long long* bitmap;  // scratch [tiles * RLE_NT]: bit i set when element i starts
    unsigned long long* ticket;  // scratch: arrivals of the count CTAs, (generation << 32) | count
    uint32_t gen;                // call generation (> 0)
};

// Once per device: the kernels' shared-memory carveout.
cudaError_t configure_rle();

// Scratch bytes of the per-CTA arrays (for RLE_MAX_CTAS CTAs) and of the
// per-tile arrays and bitmap for `tiles` tiles.
constexpr int64_t RLE_CTA_SCRATCH = int64_t(4) * 8 * RLE_MAX_CTAS;
inline int64_t rle_tile_bytes(int64_t tiles) {
    return ((tiles * 12 + 255) / 256) * 256 + tiles * RLE_NT * 8;
}

// Enqueue the launches on `stream` (count and write; one small kernel when n == 0).  The caller has checked the
// arguments; returns the first launch error.
cudaError_t launch_rle(const RleParams& p, cudaStream_t stream);

}  // namespace segred
