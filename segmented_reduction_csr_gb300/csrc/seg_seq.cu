// seg_seq.cu -- the input-order float32 mode (see seg_seq.cuh).
#include "ptx.cuh"
#include "seg_seq.cuh"

namespace segred {
namespace {

constexpr int64_t SEQ_LONG = 512;      // longer segments take the long-segment paths
constexpr int SEQ_RING = 8;            // F == 1 warp path: blocks of 32 rows in flight per lane
constexpr int64_t SEQ_PF_BYTES = 16 << 10;   // L2 prefetch: span of one request
constexpr int64_t SEQ_PF_AHEAD = 64 << 10;   // L2 prefetch: distance ahead of the additions

template <class OffT>
__device__ __forceinline__ int64_t clamped(const OffT* off, int64_t s, int64_t N) {
    int64_t o = static_cast<int64_t>(__ldg(off + s));
    o = o < 0 ? 0 : o;
    return o > N ? N : o;
}

// Ask L2 for the bytes [a, a + SEQ_PF_BYTES) of the values, clipped to the
// array and rounded inward to 16-byte boundaries.
__device__ __forceinline__ void prefetch_bytes(const SeqParams& p, int64_t a) {
    const uint64_t base = reinterpret_cast<uint64_t>(p.values);
    const uint64_t end = (base + static_cast<uint64_t>(p.N * p.F) * 4) & ~uint64_t(15);
    const uint64_t lo = (base + static_cast<uint64_t>(a) + 15) & ~uint64_t(15);
    uint64_t hi = (base + static_cast<uint64_t>(a + SEQ_PF_BYTES)) & ~uint64_t(15);
    hi = hi < end ? hi : end;
    if (hi > lo) bulk_prefetch_l2(reinterpret_cast<const void*>(lo), static_cast<uint32_t>(hi - lo));
}

// One thread's chain: rows [b, e) of one column, loads SEQ_AHEAD rows ahead.
template <int AHEAD>
__device__ __forceinline__ float thread_chain(const SeqParams& p, const float* __restrict__ col,
                                              int64_t b, int64_t e, bool prefetch) {
    float acc = 0.0f;
    int64_t r = b;
    int64_t next_pf = b * p.F * 4;
    for (; r + AHEAD <= e; r += AHEAD) {
        if (prefetch && r * p.F * 4 >= next_pf) {
            prefetch_bytes(p, next_pf + SEQ_PF_AHEAD);
            next_pf += SEQ_PF_BYTES;
        }
        float x[AHEAD];
#pragma unroll
        for (int k = 0; k < AHEAD; ++k) x[k] = __ldg(col + (r + k) * p.F);
#pragma unroll
        for (int k = 0; k < AHEAD; ++k) acc = __fadd_rn(acc, x[k]);
    }
    for (; r < e; ++r) acc = __fadd_rn(acc, __ldg(col + r * p.F));
    return acc;
}

// F == 1, one long segment [b, e) run by the whole warp: each lane loads one
// row of a block of 32, SEQ_RING blocks ahead, and the chain takes the 32
// values in order by shuffles (every lane keeps the same sum).
__device__ __forceinline__ float warp_chain(const SeqParams& p, int64_t b, int64_t e, int lane) {
    const float* __restrict__ v = p.values;
    float ring[SEQ_RING];
#pragma unroll
    for (int k = 0; k < SEQ_RING; ++k) {
        const int64_t r = b + 32 * k + lane;
        ring[k] = r < e ? __ldg(v + r) : 0.0f;
    }
    if (lane == 0) prefetch_bytes(p, b * 4 + SEQ_PF_BYTES);
    int64_t next_pf = b * 4 + 2 * SEQ_PF_BYTES;
    float acc = 0.0f;
    for (int64_t blk = b; blk < e; blk += 32 * SEQ_RING) {
        if (lane == 0 && (blk + 32 * SEQ_RING) * 4 >= next_pf - SEQ_PF_AHEAD) {
            prefetch_bytes(p, next_pf);
            next_pf += SEQ_PF_BYTES;
        }
#pragma unroll
        for (int k = 0; k < SEQ_RING; ++k) {
            const int64_t cur = blk + 32 * k;
            if (cur >= e) break;
            const int64_t left = e - cur;
            if (left >= 32) {
#pragma unroll
                for (int j = 0; j < 32; ++j) acc = __fadd_rn(acc, __shfl_sync(0xffffffffu, ring[k], j));
            } else {
#pragma unroll
                for (int j = 0; j < 32; ++j) {
                    const float x = __shfl_sync(0xffffffffu, ring[k], j);
                    if (j < left) acc = __fadd_rn(acc, x);
                }
            }
            const int64_t r = cur + 32 * SEQ_RING + lane;
            ring[k] = r < e ? __ldg(v + r) : 0.0f;
        }
    }
    return acc;
}

__device__ __forceinline__ float finish(const SeqParams& p, float acc, int64_t len) {
    if (p.mean) return len > 0 ? __fdiv_rn(acc, __ll2float_rn(len)) : 0.0f;
    return acc;
}

template <class OffT>
__global__ void __launch_bounds__(SEQ_NT) seg_seq_kernel(const SeqParams p) {
    const int64_t i = static_cast<int64_t>(blockIdx.x) * SEQ_NT + threadIdx.x;
    const bool valid = i < p.S * p.F;
    const int lane = threadIdx.x & 31;
    const OffT* off = static_cast<const OffT*>(p.offsets);
    const int64_t s = valid ? i / p.F : 0, f = valid ? i - s * p.F : 0;
    const int64_t b = valid ? clamped(off, s, p.N) : 0;
    const int64_t e0 = valid ? clamped(off, s + 1, p.N) : 0;
    const int64_t e = e0 > b ? e0 : b;
    if (p.F == 1) {
        const bool is_long = e - b > SEQ_LONG;
        if (valid && !is_long) p.out[i] = finish(p, thread_chain<SEQ_AHEAD>(p, p.values, b, e, false), e - b);
        // the warp's long segments, one after another, each by all 32 lanes
        unsigned m = __ballot_sync(0xffffffffu, valid && is_long);
        while (m) {
            const int owner = __ffs(m) - 1;
            m &= m - 1;
            const int64_t bo = __shfl_sync(0xffffffffu, b, owner);
            const int64_t eo = __shfl_sync(0xffffffffu, e, owner);
            const float acc = warp_chain(p, bo, eo, lane);
            if (lane == owner) p.out[i] = finish(p, acc, eo - bo);
        }
        return;
    }
    if (!valid) return;
    // rows: one column's chain per thread; the segment's first column asks L2
    // for the rows ahead when the segment is long
    const bool prefetch = f == 0 && e - b > SEQ_LONG;
    p.out[i] = finish(p, thread_chain<2 * SEQ_AHEAD>(p, p.values + f, b, e, prefetch), e - b);
}

}  // namespace

cudaError_t launch_sequential(const SeqParams& p, cudaStream_t stream) {
    const int64_t items = p.S * p.F;
    const unsigned grid = static_cast<unsigned>((items + SEQ_NT - 1) / SEQ_NT);
    if (p.off64) seg_seq_kernel<int64_t><<<grid, SEQ_NT, 0, stream>>>(p);
    else seg_seq_kernel<uint32_t><<<grid, SEQ_NT, 0, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace segred
