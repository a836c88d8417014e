// seg_sort.cu -- the stable radix sort of the deterministic scatter and its
// helpers (see seg_sort.cuh).
#include "seg_sort.cuh"

namespace segred {
namespace {

constexpr int kWarps = SORT_NT / 32;
constexpr unsigned FULL = 0xffffffffu;

// The key of row r: its destination, or D for one outside [0, D).
__device__ __forceinline__ uint32_t key_of(const SortParams& p, int64_t r) {
    const int64_t d = __ldg(p.index + r);
    return static_cast<uint32_t>(d >= 0 && d < p.D ? d : p.D);
}

// Pass `pass` reads the index (pass 0) or buffer (pass - 1) & 1, and writes
// buffer pass & 1.
__device__ __forceinline__ void load_kv(const SortParams& p, int pass, int64_t r, uint32_t& k, uint32_t& v) {
    if (pass == 0) {
        k = key_of(p, r);
        v = static_cast<uint32_t>(r);
    } else {
        k = p.keys[(pass - 1) & 1][r];
        v = p.vals[(pass - 1) & 1][r];
    }
}

// Exclusive sum of x over the SORT_NT threads; `total` gets the sum.
__device__ __forceinline__ uint32_t block_exclusive(uint32_t x, uint32_t& total, uint32_t* sw) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    uint32_t inc = x;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t y = __shfl_up_sync(FULL, inc, o);
        if (lane >= o) inc += y;
    }
    if (lane == 31) sw[warp] = inc;
    __syncthreads();
    uint32_t before = 0;
    total = 0;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) {
        before += w < warp ? sw[w] : 0u;
        total += sw[w];
    }
    __syncthreads();
    return before + inc - x;
}

__global__ void __launch_bounds__(SORT_NT) sort_hist_kernel(const SortParams p, int pass) {
    __shared__ uint32_t h[SORT_RADIX];
    const int shift = 8 * pass;
    h[threadIdx.x] = 0;
    __syncthreads();
    const int64_t tile0 = static_cast<int64_t>(blockIdx.x) * SORT_TILE;
#pragma unroll
    for (int k = 0; k < SORT_ITEMS; ++k) {
        const int64_t r = tile0 + static_cast<int64_t>(k) * SORT_NT + threadIdx.x;
        if (r < p.N) {
            uint32_t key, val;
            load_kv(p, pass, r, key, val);
            atomicAdd(&h[(key >> shift) & (SORT_RADIX - 1)], 1u);
        }
    }
    __syncthreads();
    p.hist[static_cast<int64_t>(threadIdx.x) * p.tiles + blockIdx.x] = h[threadIdx.x];
}

// CTA d: the tiles' exclusive prefix within digit d, and the digit's total.
__global__ void __launch_bounds__(SORT_NT) sort_scan_kernel(const SortParams p) {
    __shared__ uint32_t sw[kWarps];
    uint32_t* row = p.hist + static_cast<int64_t>(blockIdx.x) * p.tiles;
    uint32_t carry = 0;
    for (int64_t c0 = 0; c0 < p.tiles; c0 += SORT_NT) {
        const int64_t i = c0 + threadIdx.x;
        const uint32_t x = i < p.tiles ? row[i] : 0u;
        uint32_t chunk;
        const uint32_t ex = block_exclusive(x, chunk, sw);
        if (i < p.tiles) row[i] = carry + ex;
        carry += chunk;
    }
    if (threadIdx.x == 0) p.total[blockIdx.x] = carry;
}

// CTA t: each key of tile t to digit base + tile prefix + its stable rank.
__global__ void __launch_bounds__(SORT_NT) sort_scatter_kernel(const SortParams p, int pass) {
    __shared__ uint32_t s_base[SORT_RADIX];
    __shared__ uint32_t s_run[SORT_RADIX];
    __shared__ uint32_t s_w[kWarps][SORT_RADIX];
    __shared__ uint32_t sw[kWarps];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int shift = 8 * pass;
    const int dig = threadIdx.x;   // the digit this thread keeps the books of
    uint32_t all;
    const uint32_t dbase = block_exclusive(p.total[dig], all, sw);
    s_base[dig] = dbase + p.hist[static_cast<int64_t>(dig) * p.tiles + blockIdx.x];
    s_run[dig] = 0;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) s_w[w][dig] = 0;
    __syncthreads();
    uint32_t* kout = p.keys[pass & 1];
    uint32_t* vout = p.vals[pass & 1];
    const int64_t tile0 = static_cast<int64_t>(blockIdx.x) * SORT_TILE;
    const uint32_t lt = (1u << lane) - 1u;
    for (int k = 0; k < SORT_ITEMS; ++k) {
        // rows in order: round k holds rows tile0 + 256 k .. + 255, in thread order
        const int64_t r = tile0 + static_cast<int64_t>(k) * SORT_NT + threadIdx.x;
        const bool valid = r < p.N;
        uint32_t key = 0, val = 0;
        if (valid) load_kv(p, pass, r, key, val);
        // a value no real digit has, different in every lane, for the rows past N
        const uint32_t d = valid ? (key >> shift) & (SORT_RADIX - 1) : SORT_RADIX + lane;
        const uint32_t peers = __match_any_sync(FULL, d);
        const uint32_t rank = __popc(peers & lt);
        if (valid && lane == __ffs(peers) - 1) s_w[warp][d] = __popc(peers);
        __syncthreads();
        if (valid) {
            uint32_t before = s_run[d];
            for (int w = 0; w < warp; ++w) before += s_w[w][d];
            const uint32_t pos = s_base[d] + before + rank;
            kout[pos] = key;
            vout[pos] = val;
        }
        __syncthreads();
        uint32_t add = 0;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) {
            add += s_w[w][dig];
            s_w[w][dig] = 0;
        }
        s_run[dig] += add;
        __syncthreads();
    }
}

__global__ void __launch_bounds__(SORT_NT) bucket_offsets_kernel(const uint32_t* sorted, int64_t N, int64_t D,
                                                                 int64_t* offsets) {
    const int64_t stride = static_cast<int64_t>(gridDim.x) * SORT_NT;
    for (int64_t d = static_cast<int64_t>(blockIdx.x) * SORT_NT + threadIdx.x; d <= D; d += stride) {
        int64_t lo = 0, hi = N;   // first i with sorted[i] >= d
        while (lo < hi) {
            const int64_t mid = (lo + hi) >> 1;
            if (static_cast<int64_t>(__ldg(sorted + mid)) < d) lo = mid + 1;
            else hi = mid;
        }
        offsets[d] = lo;
    }
}

template <int VEC>
__global__ void __launch_bounds__(SORT_NT) gather_rows_kernel(const uint32_t* src, const uint32_t* perm,
                                                              int64_t N, int64_t F, uint32_t* dst) {
    const int64_t chunks = F / VEC;
    const int64_t items = N * chunks;
    const int64_t stride = static_cast<int64_t>(gridDim.x) * SORT_NT;
    for (int64_t it = static_cast<int64_t>(blockIdx.x) * SORT_NT + threadIdx.x; it < items; it += stride) {
        const int64_t i = it / chunks, c = it - i * chunks;
        const int64_t r = __ldg(perm + i);
        if constexpr (VEC == 4) {
            reinterpret_cast<uint4*>(dst + i * F)[c] = __ldg(reinterpret_cast<const uint4*>(src + r * F) + c);
        } else {
            dst[i * F + c] = __ldg(src + r * F + c);
        }
    }
}

__global__ void __launch_bounds__(SORT_NT) map_args_kernel(int64_t* arg, const uint32_t* perm, int64_t n) {
    const int64_t stride = static_cast<int64_t>(gridDim.x) * SORT_NT;
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * SORT_NT + threadIdx.x; i < n; i += stride) {
        const int64_t a = arg[i];
        arg[i] = a < 0 ? -1 : static_cast<int64_t>(__ldg(perm + a));
    }
}

unsigned grid_for(int64_t work, int64_t per_cta) {
    const int64_t g = (work + per_cta - 1) / per_cta;
    return static_cast<unsigned>(g < 1 ? 1 : (g > (int64_t(1) << 20) ? (int64_t(1) << 20) : g));
}

}  // namespace

cudaError_t launch_sort(const SortParams& p, cudaStream_t stream) {
    if (p.tiles == 0) return cudaSuccess;
    for (int pass = 0; pass < p.passes; ++pass) {
        sort_hist_kernel<<<static_cast<unsigned>(p.tiles), SORT_NT, 0, stream>>>(p, pass);
        sort_scan_kernel<<<SORT_RADIX, SORT_NT, 0, stream>>>(p);
        sort_scatter_kernel<<<static_cast<unsigned>(p.tiles), SORT_NT, 0, stream>>>(p, pass);
    }
    return cudaGetLastError();
}

cudaError_t launch_bucket_offsets(const uint32_t* sorted, int64_t N, int64_t D, int64_t* offsets,
                                  cudaStream_t stream) {
    bucket_offsets_kernel<<<grid_for(D + 1, SORT_NT), SORT_NT, 0, stream>>>(sorted, N, D, offsets);
    return cudaGetLastError();
}

cudaError_t launch_gather_rows(const void* src, const uint32_t* perm, int64_t N, int64_t F, void* dst,
                               cudaStream_t stream) {
    if (N == 0) return cudaSuccess;
    const bool vec = F % 4 == 0 && reinterpret_cast<uintptr_t>(src) % 16 == 0 &&
                     reinterpret_cast<uintptr_t>(dst) % 16 == 0;
    const int64_t items = N * (vec ? F / 4 : F);
    if (vec)
        gather_rows_kernel<4><<<grid_for(items, SORT_NT * 4), SORT_NT, 0, stream>>>(
            static_cast<const uint32_t*>(src), perm, N, F, static_cast<uint32_t*>(dst));
    else
        gather_rows_kernel<1><<<grid_for(items, SORT_NT * 4), SORT_NT, 0, stream>>>(
            static_cast<const uint32_t*>(src), perm, N, F, static_cast<uint32_t*>(dst));
    return cudaGetLastError();
}

cudaError_t launch_map_args(int64_t* arg, const uint32_t* perm, int64_t n, cudaStream_t stream) {
    if (n == 0) return cudaSuccess;
    map_args_kernel<<<grid_for(n, SORT_NT * 4), SORT_NT, 0, stream>>>(arg, perm, n);
    return cudaGetLastError();
}

}  // namespace segred
