// seg_scatter.cu -- the kernels of the unsorted scatter path (see seg_scatter.cuh).
#include "seg_scatter.cuh"

namespace segred {
namespace {

__global__ void __launch_bounds__(SC_NT) sc_fill_kernel(uint32_t* a, int64_t na, uint32_t va,
                                                        unsigned long long* b, int64_t nb,
                                                        unsigned long long vb) {
    const int64_t stride = static_cast<int64_t>(gridDim.x) * SC_NT;
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * SC_NT + threadIdx.x; i < na; i += stride) a[i] = va;
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * SC_NT + threadIdx.x; i < nb; i += stride) b[i] = vb;
}

__device__ __forceinline__ void red_add_v4(float* a, float4 v) {
    asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(a), "f"(v.x), "f"(v.y), "f"(v.z),
                 "f"(v.w)
                 : "memory");
}

// Item `it` of a thread's SC_ITEMS (it = first + k * SC_NT) as (row, chunk):
// one 64-bit division per thread, then steps of SC_NT items.
struct ItemWalk {
    int64_t r, c;
    int64_t dr, dc, chunks;
    __device__ __forceinline__ ItemWalk(int64_t first, int64_t chunks_) : chunks(chunks_) {
        r = first / chunks;
        c = first - r * chunks;
        dr = SC_NT / chunks;
        dc = SC_NT - dr * chunks;
    }
    __device__ __forceinline__ void next() {
        r += dr;
        c += dc;
        if (c >= chunks) {
            c -= chunks;
            r += 1;
        }
    }
};

// sum / mean: item = (row, chunk of VEC columns); SC_ITEMS items per thread,
// all loads issued before the atomics.
template <int DT, int VEC>
__global__ void __launch_bounds__(SC_NT) sc_add_kernel(const ScatterParams p) {
    const int64_t chunks = p.F / VEC;
    const int64_t items = p.N * chunks;
    const int64_t first = (static_cast<int64_t>(blockIdx.x) * SC_NT * SC_ITEMS) + threadIdx.x;
    int64_t dst[SC_ITEMS], col[SC_ITEMS];
    float4 fv[SC_ITEMS];
    uint32_t iv[SC_ITEMS];
    ItemWalk iw(first, chunks);
#pragma unroll
    for (int k = 0; k < SC_ITEMS; ++k, iw.next()) {
        const int64_t it = first + static_cast<int64_t>(k) * SC_NT;
        dst[k] = -1;
        if (it < items) {
            // the row's values load whatever its index says (the row is in
            // bounds), so the two loads overlap instead of one waiting on the other
            const int64_t r = iw.r, c = iw.c;
            dst[k] = __ldg(p.index + r);
            col[k] = c * VEC;
            if constexpr (DT == 2 && VEC == 4)
                fv[k] = __ldg(reinterpret_cast<const float4*>(static_cast<const float*>(p.src) + r * p.F) + c);
            else if constexpr (DT == 2)
                fv[k].x = __ldg(static_cast<const float*>(p.src) + r * p.F + c);
            else
                iv[k] = __ldg(static_cast<const uint32_t*>(p.src) + r * p.F + c);
        }
    }
#pragma unroll
    for (int k = 0; k < SC_ITEMS; ++k) {
        if (dst[k] >= p.D) dst[k] = -1;   // outside [0, D): the row goes nowhere
        if (p.count != nullptr && dst[k] >= 0 && col[k] == 0) atomicAdd(p.count + dst[k], 1u);
    }
#pragma unroll
    for (int k = 0; k < SC_ITEMS; ++k) {
        if (dst[k] < 0) continue;
        if constexpr (DT == 2 && VEC == 4)
            red_add_v4(static_cast<float*>(p.out) + dst[k] * p.F + col[k], fv[k]);
        else if constexpr (DT == 2)
            atomicAdd(static_cast<float*>(p.out) + dst[k] * p.F + col[k], fv[k].x);
        else
            atomicAdd(static_cast<uint32_t*>(p.out) + dst[k] * p.F + col[k], iv[k]);
    }
}

// The value's bits in an order-preserving unsigned form (-0.0 as +0.0).
template <int DT>
__device__ __forceinline__ uint32_t monotone(uint32_t bits) {
    if constexpr (DT == 2) {
        if (bits == 0x80000000u) bits = 0u;
        return (bits & 0x80000000u) ? ~bits : (bits | 0x80000000u);
    } else if constexpr (DT == 1) {
        return bits ^ 0x80000000u;
    } else {
        return bits;
    }
}

// The value bits back from their monotone form (+0.0 for a -0.0 that went in).
template <int DT>
__device__ __forceinline__ uint32_t unmonotone(uint32_t m) {
    if constexpr (DT == 2) {
        return (m & 0x80000000u) ? (m & 0x7fffffffu) : ~m;
    } else if constexpr (DT == 1) {
        return m ^ 0x80000000u;
    } else {
        return m;
    }
}

// max / min: item = (row, chunk of VEC columns); the packed word settles
// value and row.  An output cell receives many candidates but its word
// changes rarely (about ln n times for n candidates in random order), so
// each candidate first reads the value half of the cell's word from L2 and
// issues its atomic only if that value does not already beat it.  The read
// may be stale, never ahead: words only grow (max) or shrink (min), so a
// candidate it rules out cannot win.
template <int DT, bool MAX, int VEC>
__global__ void __launch_bounds__(SC_NT) sc_ext_kernel(const ScatterParams p) {
    const int64_t chunks = p.F / VEC;
    const int64_t items = p.N * chunks;
    const int64_t first = (static_cast<int64_t>(blockIdx.x) * SC_NT * SC_ITEMS) + threadIdx.x;
    int64_t cell[SC_ITEMS];
    uint32_t m[SC_ITEMS][VEC];   // monotone value bits
    uint32_t lo[SC_ITEMS];       // the row as packed (complemented for max)
    ItemWalk iw(first, chunks);
#pragma unroll
    for (int k = 0; k < SC_ITEMS; ++k, iw.next()) {
        const int64_t it = first + static_cast<int64_t>(k) * SC_NT;
        cell[k] = -1;
        if (it < items) {
            // value and index load together (the row is in bounds either way)
            const int64_t r = iw.r, c = iw.c;
            const int64_t d = __ldg(p.index + r);
            const uint32_t* src = static_cast<const uint32_t*>(p.src) + r * p.F + c * VEC;
            if constexpr (VEC == 4) {
                const uint4 b4 = __ldg(reinterpret_cast<const uint4*>(src));
                m[k][0] = b4.x, m[k][1] = b4.y, m[k][2] = b4.z, m[k][3] = b4.w;
            } else {
                m[k][0] = __ldg(src);
            }
            lo[k] = MAX ? ~static_cast<uint32_t>(r) : static_cast<uint32_t>(r);
            cell[k] = d >= 0 && d < p.D ? d * p.F + c * VEC : -1;
        }
    }
    // the cells' current words, high halves only (the value): a candidate
    // whose value is strictly beaten cannot win; a tie on the value goes to
    // the atomic, which settles the row
    uint32_t hi[SC_ITEMS][VEC];
#pragma unroll
    for (int k = 0; k < SC_ITEMS; ++k) {
        if (cell[k] < 0) continue;
        const uint32_t* wp = reinterpret_cast<const uint32_t*>(p.word + cell[k]) + 1;
        if constexpr (VEC == 4) {
            const uint4 a = __ldcg(reinterpret_cast<const uint4*>(wp - 1));
            const uint4 b = __ldcg(reinterpret_cast<const uint4*>(wp - 1) + 1);
            hi[k][0] = a.y, hi[k][1] = a.w, hi[k][2] = b.y, hi[k][3] = b.w;
        } else {
            hi[k][0] = __ldcg(wp);
        }
    }
#pragma unroll
    for (int k = 0; k < SC_ITEMS; ++k) {
        if (cell[k] < 0) continue;
#pragma unroll
        for (int v = 0; v < VEC; ++v) {
            const uint32_t mv = monotone<DT>(m[k][v]);
            if (MAX ? mv < hi[k][v] : mv > hi[k][v]) continue;
            const unsigned long long w = (static_cast<unsigned long long>(mv) << 32) | lo[k];
            // no return value wanted: a reduction, not an atomic that waits
            if (MAX)
                asm volatile("red.relaxed.gpu.global.max.u64 [%0], %1;" ::"l"(p.word + cell[k] + v), "l"(w) : "memory");
            else
                asm volatile("red.relaxed.gpu.global.min.u64 [%0], %1;" ::"l"(p.word + cell[k] + v), "l"(w) : "memory");
        }
    }
}

// max / min: the winning row's value and the row (0 and -1 when none).  The
// value comes back from the word's high half; only a float32 zero is read
// again from src, so that a -0.0 keeps its sign bit.
template <int DT, bool MAX>
__global__ void __launch_bounds__(SC_NT) sc_ext_finish_kernel(const ScatterParams p) {
    const int64_t cells = p.D * p.F;
    const int64_t stride = static_cast<int64_t>(gridDim.x) * SC_NT;
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * SC_NT + threadIdx.x; i < cells; i += stride) {
        const unsigned long long w = p.word[i];
        const bool none = MAX ? w == 0ull : w == ~0ull;
        const uint32_t lo = static_cast<uint32_t>(w);
        const uint32_t m = static_cast<uint32_t>(w >> 32);
        const int64_t row = none ? -1 : static_cast<int64_t>(MAX ? ~lo : lo);
        uint32_t v = none ? 0u : unmonotone<DT>(m);
        if (DT == 2 && !none && m == 0x80000000u)
            v = __ldg(static_cast<const uint32_t*>(p.src) + row * p.F + i % p.F);
        static_cast<uint32_t*>(p.out)[i] = v;
        if (p.arg != nullptr) p.arg[i] = row;
    }
}

__global__ void __launch_bounds__(SC_NT) sc_mean_finish_kernel(const ScatterParams p) {
    const int64_t cells = p.D * p.F;
    const int64_t stride = static_cast<int64_t>(gridDim.x) * SC_NT;
    float* out = static_cast<float*>(p.out);
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * SC_NT + threadIdx.x; i < cells; i += stride) {
        // (32-bit division where the cells allow: the 64-bit one is a long subroutine)
        const int64_t row = cells <= int64_t(UINT32_MAX) ? static_cast<int64_t>(static_cast<uint32_t>(i) /
                                                                                static_cast<uint32_t>(p.F))
                                                         : i / p.F;
        const uint32_t n = p.count[row];
        out[i] = n > 0 ? __fdiv_rn(out[i], __uint2float_rn(n)) : 0.0f;
    }
}

unsigned grid_for(int64_t work, int64_t per_cta) {
    const int64_t g = (work + per_cta - 1) / per_cta;
    return static_cast<unsigned>(g < 1 ? 1 : (g > (int64_t(1) << 30) ? (int64_t(1) << 30) : g));
}

template <int DT>
cudaError_t launch_dt(const ScatterParams& p, cudaStream_t stream) {
    const int64_t cells = p.D * p.F;
    const unsigned gcells = grid_for(cells, SC_NT * 8);
    const int64_t per = int64_t(SC_NT) * SC_ITEMS;
    if (p.op == 0 || p.op == 3) {
        sc_fill_kernel<<<gcells, SC_NT, 0, stream>>>(static_cast<uint32_t*>(p.out), cells, 0u, nullptr, 0, 0ull);
        if (p.op == 3) sc_fill_kernel<<<grid_for(p.D, SC_NT * 8), SC_NT, 0, stream>>>(p.count, p.D, 0u, nullptr, 0, 0ull);
        if (p.N > 0) {
            if (DT == 2 && p.vec == 4)
                sc_add_kernel<DT, 4><<<grid_for(p.N * (p.F / 4), per), SC_NT, 0, stream>>>(p);
            else
                sc_add_kernel<DT, 1><<<grid_for(p.N * p.F, per), SC_NT, 0, stream>>>(p);
        }
        if (p.op == 3) sc_mean_finish_kernel<<<gcells, SC_NT, 0, stream>>>(p);
        return cudaGetLastError();
    }
    const bool mx = p.op == 2;
    sc_fill_kernel<<<gcells, SC_NT, 0, stream>>>(nullptr, 0, 0u, p.word, cells, mx ? 0ull : ~0ull);
    if (p.N > 0) {
        // four columns an item when rows allow 16-byte loads (the word array
        // is the library's own, 256-byte aligned)
        const bool v4 = p.F % 4 == 0 && reinterpret_cast<uintptr_t>(p.src) % 16 == 0;
        const unsigned g = grid_for(p.N * (v4 ? p.F / 4 : p.F), per);
        if (mx && v4) sc_ext_kernel<DT, true, 4><<<g, SC_NT, 0, stream>>>(p);
        else if (mx) sc_ext_kernel<DT, true, 1><<<g, SC_NT, 0, stream>>>(p);
        else if (v4) sc_ext_kernel<DT, false, 4><<<g, SC_NT, 0, stream>>>(p);
        else sc_ext_kernel<DT, false, 1><<<g, SC_NT, 0, stream>>>(p);
    }
    if (mx) sc_ext_finish_kernel<DT, true><<<gcells, SC_NT, 0, stream>>>(p);
    else sc_ext_finish_kernel<DT, false><<<gcells, SC_NT, 0, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_scatter(const ScatterParams& p, cudaStream_t stream) {
    if (p.dtype == 2) return launch_dt<2>(p, stream);
    if (p.dtype == 1) return launch_dt<1>(p, stream);
    return launch_dt<0>(p, stream);
}

}  // namespace segred
