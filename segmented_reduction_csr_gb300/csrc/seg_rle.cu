// seg_rle.cu -- the kernels of the offsets producers (run-length encoding,
// unique, flags to offsets) and their launcher; the passes are described in
// seg_rle.cuh.
#include "seg_rle.cuh"

namespace segred {
namespace {

constexpr int64_t kNone = INT64_MAX;   // "no start seen"
constexpr int kWarps = RLE_NT / 32;

// Shared-memory slot of the k-th start of a tile: one pad word per 32
// entries, so that the all-starts case (thread t writing slots 16t + j)
// spreads a warp's stores over all 32 banks.
__device__ __forceinline__ int pad_slot(int k) { return k + (k >> 5); }
constexpr int kSlots = RLE_TILE + RLE_TILE / 32 + 1;

// My RLE_PER elements starting at `base`: their keys (0 past n) and a bit
// mask of the ones that start a run (bit j: element base + j).
__device__ __forceinline__ uint32_t load_starts(const RleParams& p, int64_t base,
                                                uint32_t (&k)[RLE_PER]) {
    const int lane = threadIdx.x & 31;
    uint32_t bits = 0;
    if (p.keys != nullptr) {
        if (p.vec && base + RLE_PER <= p.n) {
            const uint4* q = reinterpret_cast<const uint4*>(p.keys + base);
#pragma unroll
            for (int v = 0; v < RLE_PER / 4; ++v) {
                const uint4 w = __ldg(q + v);
                k[4 * v] = w.x;
                k[4 * v + 1] = w.y;
                k[4 * v + 2] = w.z;
                k[4 * v + 3] = w.w;
            }
        } else {
#pragma unroll
            for (int j = 0; j < RLE_PER; ++j) k[j] = base + j < p.n ? __ldg(p.keys + base + j) : 0u;
        }
        // the key before my first element: the previous lane's last one, or a load
        uint32_t before = __shfl_up_sync(0xffffffffu, k[RLE_PER - 1], 1);
        if (lane == 0) before = base > 0 && base - 1 < p.n ? __ldg(p.keys + base - 1) : 0u;
#pragma unroll
        for (int j = 0; j < RLE_PER; ++j) {
            const uint32_t prev = j == 0 ? before : k[j - 1];
            const bool start = base + j < p.n && (base + j == 0 || k[j] != prev);
            bits |= static_cast<uint32_t>(start) << j;
        }
    } else {
        uint32_t w[RLE_PER / 4];
        if (p.vec && base + RLE_PER <= p.n) {
            const uint4 v = __ldg(reinterpret_cast<const uint4*>(p.flags + base));
            w[0] = v.x, w[1] = v.y, w[2] = v.z, w[3] = v.w;
        } else {
#pragma unroll
            for (int q = 0; q < RLE_PER / 4; ++q) {
                uint32_t x = 0;
#pragma unroll
                for (int b = 0; b < 4; ++b) {
                    const int64_t i = base + 4 * q + b;
                    if (i < p.n) x |= static_cast<uint32_t>(__ldg(p.flags + i)) << (8 * b);
                }
                w[q] = x;
            }
        }
#pragma unroll
        for (int j = 0; j < RLE_PER; ++j) {
            k[j] = 0;
            bits |= static_cast<uint32_t>(((w[j / 4] >> (8 * (j % 4))) & 0xffu) != 0) << j;
        }
    }
    return bits;
}

// Tiles [t0, t1) of CTA b: contiguous, every CTA at least one tile.
__device__ __forceinline__ void cta_tiles(const RleParams& p, int64_t& t0, int64_t& t1) {
    t0 = p.tiles * blockIdx.x / p.ctas;
    t1 = p.tiles * (blockIdx.x + 1) / p.ctas;
}

__global__ void __launch_bounds__(RLE_NT) rle_count_kernel(const RleParams p) {
    __shared__ int64_t s_cnt[kWarps];
    __shared__ int64_t s_first[kWarps];
    int64_t t0, t1;
    cta_tiles(p, t0, t1);
    int64_t cnt = 0, first = kNone;
#pragma unroll 2
    for (int64_t t = t0; t < t1; ++t) {
        const int64_t base = t * RLE_TILE + static_cast<int64_t>(threadIdx.x) * RLE_PER;
        uint32_t k[RLE_PER];
        const uint32_t bits = load_starts(p, base, k);
        cnt += __popc(bits);
        if (bits != 0 && first == kNone) first = base + (__ffs(bits) - 1);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        cnt += __shfl_xor_sync(0xffffffffu, cnt, o);
        const int64_t f = __shfl_xor_sync(0xffffffffu, first, o);
        first = f < first ? f : first;
    }
    if ((threadIdx.x & 31) == 0) {
        s_cnt[threadIdx.x >> 5] = cnt;
        s_first[threadIdx.x >> 5] = first;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        int64_t c = 0, f = kNone;
        for (int w = 0; w < kWarps; ++w) {
            c += s_cnt[w];
            f = s_first[w] < f ? s_first[w] : f;
        }
        p.cta_count[blockIdx.x] = c;
        p.cta_first[blockIdx.x] = f;
    }
}

// One CTA of RLE_MAX_CTAS threads; thread b handles CTA b's entries.
__global__ void __launch_bounds__(RLE_MAX_CTAS) rle_scan_kernel(const RleParams p) {
    constexpr int W = RLE_MAX_CTAS / 32;
    __shared__ int64_t s_sum[W];
    __shared__ int64_t s_min[RLE_MAX_CTAS + 1];
    const int b = threadIdx.x, lane = b & 31, warp = b >> 5;
    const int64_t c = b < p.ctas ? p.cta_count[b] : 0;
    const int64_t f = b < p.ctas ? p.cta_first[b] : kNone;
    // exclusive sum of the counts
    int64_t inc = c;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int64_t y = __shfl_up_sync(0xffffffffu, inc, o);
        if (lane >= o) inc += y;
    }
    if (lane == 31) s_sum[warp] = inc;
    s_min[b] = f;
    if (b == 0) s_min[RLE_MAX_CTAS] = kNone;
    __syncthreads();
    int64_t before = 0, total = 0;
    for (int w = 0; w < W; ++w) {
        const int64_t x = s_sum[w];
        before += w < warp ? x : 0;
        total += x;
    }
    // suffix minimum of the first starts, by doubling
    for (int o = 1; o < RLE_MAX_CTAS; o <<= 1) {
        const int64_t y = b + o < RLE_MAX_CTAS ? s_min[b + o] : kNone;
        __syncthreads();
        if (y < s_min[b]) s_min[b] = y;
        __syncthreads();
    }
    if (b < p.ctas) {
        const int64_t nx = s_min[b + 1];
        p.cta_base[b] = before + inc - c;
        p.cta_next[b] = nx < p.n ? nx : p.n;
    }
    if (b == 0) {
        *p.count = total;
        if (p.offsets != nullptr) p.offsets[total] = p.n;
    }
}

__global__ void __launch_bounds__(RLE_NT) rle_write_kernel(const RleParams p) {
    __shared__ uint32_t s_rel[kSlots];
    __shared__ uint32_t s_val[kSlots];
    __shared__ int s_warp[kWarps];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int64_t t0, t1;
    cta_tiles(p, t0, t1);
    int64_t run = p.cta_base[blockIdx.x];   // index of the next run to write
    int64_t pend_r = -1, pend_i = 0;       // thread 0: the run still without a length
    for (int64_t t = t0; t < t1; ++t) {
        const int64_t tile0 = t * RLE_TILE;
        const int64_t base = tile0 + static_cast<int64_t>(threadIdx.x) * RLE_PER;
        uint32_t k[RLE_PER];
        const uint32_t bits = load_starts(p, base, k);
        // block exclusive sum of the start counts
        const int c = __popc(bits);
        int inc = c;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, inc, o);
            if (lane >= o) inc += y;
        }
        if (lane == 31) s_warp[warp] = inc;
        __syncthreads();
        int before = inc - c, total = 0;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) {
            const int x = s_warp[w];
            before += w < warp ? x : 0;
            total += x;
        }
        // my starts, in order, into their slots
        int slot = before;
#pragma unroll
        for (int j = 0; j < RLE_PER; ++j) {
            if ((bits >> j) & 1u) {
                s_rel[pad_slot(slot)] = threadIdx.x * RLE_PER + j;
                s_val[pad_slot(slot)] = k[j];
                ++slot;
            }
        }
        __syncthreads();
        for (int q = threadIdx.x; q < total; q += RLE_NT) {
            const int64_t r = run + q;
            const uint32_t rel = s_rel[pad_slot(q)];
            if (p.offsets != nullptr) p.offsets[r] = tile0 + rel;
            if (p.values != nullptr) p.values[r] = s_val[pad_slot(q)];
            if (p.lengths != nullptr && q + 1 < total) p.lengths[r] = s_rel[pad_slot(q + 1)] - rel;
        }
        if (threadIdx.x == 0 && total > 0) {
            const int64_t first = tile0 + s_rel[pad_slot(0)];
            if (p.lengths != nullptr && pend_r >= 0)
                p.lengths[pend_r] = static_cast<uint32_t>(first - pend_i);
            pend_r = run + total - 1;
            pend_i = tile0 + s_rel[pad_slot(total - 1)];
        }
        run += total;
        __syncthreads();
    }
    if (threadIdx.x == 0 && p.lengths != nullptr && pend_r >= 0)
        p.lengths[pend_r] = static_cast<uint32_t>(p.cta_next[blockIdx.x] - pend_i);
}

}  // namespace

cudaError_t launch_rle(const RleParams& p, cudaStream_t stream) {
    if (p.ctas > 0) {
        rle_count_kernel<<<p.ctas, RLE_NT, 0, stream>>>(p);
        const cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    rle_scan_kernel<<<1, RLE_MAX_CTAS, 0, stream>>>(p);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    if (p.ctas > 0 && (p.values != nullptr || p.lengths != nullptr || p.offsets != nullptr)) {
        rle_write_kernel<<<p.ctas, RLE_NT, 0, stream>>>(p);
        e = cudaGetLastError();
    }
    return e;
}

}  // namespace segred
