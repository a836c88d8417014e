// seg_rle.cu -- the kernels of the offsets producers (run-length encoding,
// unique, flags to offsets) and their launcher; the passes are described in
// seg_rle.cuh.
#include "seg_common.cuh"
#include "seg_rle.cuh"

namespace segred {
namespace {

constexpr int64_t kNone = INT64_MAX;   // "no start seen"
constexpr int kWarps = RLE_NT / 32;

// One thread's share of a tile as loaded: RLE_KEYS_PER keys (plus, for lane
// 0, the key just before them), or RLE_FLAGS_PER flag bytes as 32-bit words.
template <bool FLAGS>
struct Raw {
    static constexpr int PER = FLAGS ? RLE_FLAGS_PER : RLE_KEYS_PER;
    static constexpr int WORDS = FLAGS ? RLE_FLAGS_PER / 4 : RLE_KEYS_PER;
    uint32_t w[WORDS];
    uint32_t before;   // keys: the key before w[0] (lane 0 only; other lanes take it by shuffle)
};

template <bool FLAGS>
__device__ __forceinline__ void load_raw(const RleParams& p, int64_t base, Raw<FLAGS>& r) {
    constexpr int PER = Raw<FLAGS>::PER;
    if constexpr (FLAGS) {
        if (p.vec && base + PER <= p.n) {
            const uint4* q = reinterpret_cast<const uint4*>(p.flags + base);
#pragma unroll
            for (int v = 0; v < PER / 16; ++v) {
                const uint4 x = __ldcs(q + v);
                r.w[4 * v] = x.x, r.w[4 * v + 1] = x.y, r.w[4 * v + 2] = x.z, r.w[4 * v + 3] = x.w;
            }
        } else {
#pragma unroll
            for (int q = 0; q < PER / 4; ++q) {
                uint32_t x = 0;
#pragma unroll
                for (int b = 0; b < 4; ++b) {
                    const int64_t i = base + 4 * q + b;
                    if (i < p.n) x |= static_cast<uint32_t>(__ldg(p.flags + i)) << (8 * b);
                }
                r.w[q] = x;
            }
        }
        r.before = 0;
    } else {
        if (p.vec && base + PER <= p.n) {
            const uint4* q = reinterpret_cast<const uint4*>(p.keys + base);
#pragma unroll
            for (int v = 0; v < PER / 4; ++v) {
                const uint4 x = __ldcs(q + v);
                r.w[4 * v] = x.x, r.w[4 * v + 1] = x.y, r.w[4 * v + 2] = x.z, r.w[4 * v + 3] = x.w;
            }
        } else {
#pragma unroll
            for (int j = 0; j < PER; ++j) r.w[j] = base + j < p.n ? __ldg(p.keys + base + j) : 0u;
        }
        r.before = (threadIdx.x & 31) == 0 && base > 0 && base - 1 < p.n ? __ldg(p.keys + base - 1) : 0u;
    }
}

// The mask of my elements that start a run / segment (bit j: element base + j).
template <bool FLAGS>
__device__ __forceinline__ unsigned long long start_bits(const RleParams& p, int64_t base,
                                                         const Raw<FLAGS>& r) {
    unsigned long long bits = 0;
    if constexpr (FLAGS) {
        // four flag bytes at a time: the high bit of each non-zero byte
        // ((b & 0x7f) + 0x7f carries into bit 7 for b in 1..0x7f; b >= 0x80
        // has it already), then one multiply gathers bits 7, 15, 23 and 31
        // into bits 21..24 (the partial products never overlap)
#pragma unroll
        for (int q = 0; q < RLE_FLAGS_PER / 4; ++q) {
            const uint32_t w = r.w[q];
            const uint32_t hi = (((w & 0x7f7f7f7fu) + 0x7f7f7f7fu) | w) & 0x80808080u;
            const uint32_t nib = ((hi >> 7) * 0x204081u) >> 21 & 0xfu;
            bits |= static_cast<unsigned long long>(nib) << (4 * q);
        }
    } else {
        // the key before my first one: the previous lane's last key, or lane 0's load
        uint32_t before = __shfl_up_sync(0xffffffffu, r.w[RLE_KEYS_PER - 1], 1);
        if ((threadIdx.x & 31) == 0) before = r.before;
#pragma unroll
        for (int j = 0; j < RLE_KEYS_PER; ++j) {
            const uint32_t prev = j == 0 ? before : r.w[j - 1];
            const bool start = base + j < p.n && (base + j == 0 || r.w[j] != prev);
            bits |= static_cast<unsigned long long>(start) << j;
        }
    }
    return bits;
}

// Tiles [t0, t1) of CTA b: contiguous, every CTA at least one tile.
__device__ __forceinline__ void cta_tiles(const RleParams& p, int64_t& t0, int64_t& t1) {
    t0 = p.tiles * blockIdx.x / p.ctas;
    t1 = p.tiles * (blockIdx.x + 1) / p.ctas;
}

template <bool FLAGS>
__global__ void __launch_bounds__(RLE_NT) rle_count_kernel(const RleParams p) {
    constexpr int PER = Raw<FLAGS>::PER;
    constexpr int STEP = RLE_NT * PER;        // elements per step
    constexpr int SPT = RLE_TILE / STEP;      // steps per tile
    __shared__ int s_cnt[2][kWarps];          // by tile parity: thread 0 reads one while
    __shared__ int64_t s_first[2][kWarps];    // the warps fill the other
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int64_t t0, t1;
    cta_tiles(p, t0, t1);
    const int64_t s0 = t0 * SPT, s1 = t1 * SPT;
    int64_t cta_cnt = 0, cta_first = kNone;   // thread 0: the CTA's totals
    int tc = 0;                               // my starts in the current tile
    int64_t tf = kNone;                       // my first start in it
    const int64_t mine = static_cast<int64_t>(threadIdx.x) * PER;
    Raw<FLAGS> cur;
    load_raw<FLAGS>(p, s0 * STEP + mine, cur);
    for (int64_t st = s0; st < s1; ++st) {
        Raw<FLAGS> nxt;
        if (st + 1 < s1) load_raw<FLAGS>(p, (st + 1) * STEP + mine, nxt);
        const int64_t base = st * STEP + mine;
        const unsigned long long bits = start_bits<FLAGS>(p, base, cur);
        // my PER bits of the bitmap (bit i: element i), little-endian within its words
        if constexpr (FLAGS) p.bitmap[st * RLE_NT + threadIdx.x] = bits;
        else reinterpret_cast<uint16_t*>(p.bitmap)[st * RLE_NT + threadIdx.x] = static_cast<uint16_t>(bits);
        tc += __popcll(bits);
        if (bits != 0 && tf == kNone) tf = base + (__ffsll(static_cast<long long>(bits)) - 1);
        cur = nxt;
        if ((st + 1) % SPT == 0) {
            // the tile is done: its count and first start
            const int64_t t = st / SPT;
            const int par = static_cast<int>(t & 1);
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
                tc += __shfl_xor_sync(0xffffffffu, tc, o);
                const int64_t f = __shfl_xor_sync(0xffffffffu, tf, o);
                tf = f < tf ? f : tf;
            }
            if (lane == 0) {
                s_cnt[par][warp] = tc;
                s_first[par][warp] = tf;
            }
            __syncthreads();
            if (threadIdx.x == 0) {
                int c = 0;
                int64_t f = kNone;
#pragma unroll
                for (int w = 0; w < kWarps; ++w) {
                    c += s_cnt[par][w];
                    f = s_first[par][w] < f ? s_first[par][w] : f;
                }
                p.tile_count[t] = c;
                p.tile_first[t] = f;
                cta_cnt += c;
                cta_first = f < cta_first ? f : cta_first;
            }
            tc = 0;
            tf = kNone;
        }
    }
    if (threadIdx.x == 0) {
        p.cta_count[blockIdx.x] = cta_cnt;
        p.cta_first[blockIdx.x] = cta_first;
    }
}

// Shared-memory slot of the k-th start of a tile.  Start positions are
// 16-bit: one pad word per 32 words keeps the all-starts case (thread t
// writing slots 64 t + j) free of bank conflicts.
__device__ __forceinline__ int rel_slot(int k) { return k + 2 * (k >> 6); }

// The count CTA b whose range [t0, t1) holds tile t (the inverse of
// cta_tiles).  Below 2^21 tiles every product fits 32 bits and the divisions
// are 32-bit ones.
__device__ __forceinline__ void owner_of(const RleParams& p, int64_t t, int64_t& b, int64_t& t0, int64_t& t1) {
    if (p.tiles < (int64_t(1) << 21)) {
        const uint32_t T = static_cast<uint32_t>(p.tiles), C = static_cast<uint32_t>(p.ctas);
        const uint32_t bb = ((static_cast<uint32_t>(t) + 1) * C + T - 1) / T - 1;
        b = bb;
        t0 = T * bb / C;
        t1 = T * (bb + 1) / C;
    } else {
        b = ((t + 1) * p.ctas + p.tiles - 1) / p.tiles - 1;
        t0 = p.tiles * b / p.ctas;
        t1 = p.tiles * (b + 1) / p.ctas;
    }
}

// CTA t writes the runs that start in tile t (one CTA per tile lets the
// hardware balance tiles dense in starts against empty ones).  Its first run
// index is the counts of the count CTAs before its owner b plus those of b's
// tiles before t; the first start after it is the earliest first start of
// b's later tiles and of the later count CTAs.  Both come from one round of
// loads, spread over the block, and a block-wide sum and minimum.  Thread i
// owns bitmap word i (elements tile0 + 64 i + [0, 64)); a block scan ranks
// the starts into shared memory, then offsets, values (a gather of
// keys[start]) and lengths (the next start minus this one) go out
// coalesced.  A tile without starts returns at once, except the last tile,
// whose CTA writes the run count and offsets[count] = n.
__global__ void __launch_bounds__(RLE_NT) rle_write_kernel(const RleParams p) {
    __shared__ uint16_t s_rel[RLE_TILE + 2 * (RLE_TILE / 64) + 2];
    __shared__ int s_warp[kWarps];
    __shared__ int64_t s_sum[kWarps], s_min[kWarps];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int64_t t = blockIdx.x;
    const bool last_tile = t == p.tiles - 1;
    const bool outputs = p.values != nullptr || p.lengths != nullptr || p.offsets != nullptr;
    const int cnt = (outputs || last_tile) ? __ldcg(p.tile_count + t) : 0;
    if (!last_tile && (!outputs || cnt == 0)) return;
    const int64_t tile0 = t * RLE_TILE;
    const unsigned long long word = outputs ? __ldcg(p.bitmap + t * RLE_NT + threadIdx.x) : 0ull;
    int64_t b, t0, t1;
    owner_of(p, t, b, t0, t1);
    int64_t before = 0, after = kNone;
    for (int64_t i = threadIdx.x; i < p.ctas; i += RLE_NT) {
        if (i < b) {
            before += __ldcg(p.cta_count + i);
        } else if (i > b) {
            const int64_t f = __ldcg(p.cta_first + i);
            after = f < after ? f : after;
        }
    }
    for (int64_t i = t0 + threadIdx.x; i < t1; i += RLE_NT) {
        if (i < t) {
            before += __ldcg(p.tile_count + i);
        } else if (i > t) {
            const int64_t f = __ldcg(p.tile_first + i);
            after = f < after ? f : after;
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        before += __shfl_xor_sync(0xffffffffu, before, o);
        const int64_t f = __shfl_xor_sync(0xffffffffu, after, o);
        after = f < after ? f : after;
    }
    if (lane == 0) {
        s_sum[warp] = before;
        s_min[warp] = after;
    }
    // block exclusive sum of the start counts
    const int c = __popcll(word);
    int inc = c;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, inc, o);
        if (lane >= o) inc += y;
    }
    if (lane == 31) s_warp[warp] = inc;
    __syncthreads();
    int64_t run = 0, next = kNone;
    int slot = inc - c, total = 0;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) {
        run += s_sum[w];
        next = s_min[w] < next ? s_min[w] : next;
        const int x = s_warp[w];
        slot += w < warp ? x : 0;
        total += x;
    }
    next = next < p.n ? next : p.n;
    if (last_tile && threadIdx.x == 0) {
        *p.count = run + cnt;
        if (p.offsets != nullptr) p.offsets[run + cnt] = p.n;
    }
    if (total == 0) return;
    // my starts, in order, into their slots
    unsigned long long bits = word;
    while (bits) {
        const int j = __ffsll(static_cast<long long>(bits)) - 1;
        bits &= bits - 1;
        s_rel[rel_slot(slot++)] = static_cast<uint16_t>(threadIdx.x * 64 + j);
    }
    __syncthreads();
    const uint32_t* __restrict__ keys = p.keys;
    uint32_t* __restrict__ values = p.values;
    uint32_t* __restrict__ lengths = p.lengths;
    int64_t* __restrict__ offsets = p.offsets;
#pragma unroll 4
    for (int q = threadIdx.x; q < total; q += RLE_NT) {
        const int64_t r = run + q;
        const int64_t pos = tile0 + s_rel[rel_slot(q)];
        if (offsets != nullptr) offsets[r] = pos;
        if (values != nullptr) values[r] = __ldg(keys + pos);
        if (lengths != nullptr) {
            const int64_t end = q + 1 < total ? tile0 + s_rel[rel_slot(q + 1)] : next;
            lengths[r] = static_cast<uint32_t>(end - pos);
        }
    }
}

__global__ void rle_empty_kernel(const RleParams p) {
    *p.count = 0;
    if (p.offsets != nullptr) p.offsets[0] = 0;
}

template <bool FLAGS>
cudaError_t launch_mode(const RleParams& p, cudaStream_t stream) {
    if (p.ctas == 0) {
        rle_empty_kernel<<<1, 1, 0, stream>>>(p);
        return cudaGetLastError();
    }
    rle_count_kernel<FLAGS><<<p.ctas, RLE_NT, 0, stream>>>(p);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    // the write pass also writes the count, so it runs even with no outputs
    rle_write_kernel<<<static_cast<unsigned>(p.tiles), RLE_NT, 0, stream>>>(p);
    return cudaGetLastError();
}

template <class K>
cudaError_t max_carveout(K kernel) {
    return cudaFuncSetAttribute(kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                                cudaSharedmemCarveoutMaxShared);
}

}  // namespace

cudaError_t configure_rle() {
    // all shared memory for the carveout, so that more write CTAs fit per SM
    return max_carveout(rle_write_kernel);
}

cudaError_t launch_rle(const RleParams& p, cudaStream_t stream) {
    return p.flags_mode ? launch_mode<true>(p, stream) : launch_mode<false>(p, stream);
}

}  // namespace segred
