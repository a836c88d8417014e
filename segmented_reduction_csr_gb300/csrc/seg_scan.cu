// seg_scan.cu -- the segmented scan (see seg_scan.cuh).
#include <climits>

#include "seg_common.cuh"
#include "seg_scan.cuh"

namespace segred {
namespace {

constexpr int kWarps = RS_NT / 32;

template <int DT> struct ScanType;
template <> struct ScanType<0> { using T = uint32_t; };
template <> struct ScanType<1> { using T = int32_t; };
template <> struct ScanType<2> { using T = float; };

template <class T>
__device__ __forceinline__ T from_word(uint32_t w) {
    if constexpr (std::is_floating_point<T>::value) return __uint_as_float(w);
    else return static_cast<T>(w);
}
template <class T>
__device__ __forceinline__ uint32_t to_word(T v) {
    if constexpr (std::is_floating_point<T>::value) return __float_as_uint(v);
    else return static_cast<uint32_t>(v);
}

// The identity of the op: 0 for sum, the largest value for min, the
// smallest for max.
template <int DT, int OP>
__device__ __forceinline__ typename ScanType<DT>::T identity() {
    using T = typename ScanType<DT>::T;
    if constexpr (OP == 0) return T(0);
    else if constexpr (DT == 2) return __int_as_float(OP == 1 ? 0x7f800000 : static_cast<int>(0xff800000u));
    else if constexpr (DT == 1) return OP == 1 ? INT_MAX : INT_MIN;
    else return OP == 1 ? UINT_MAX : 0u;
}

// op(a, b) with a the earlier rows: sum (integers wrap modulo 2^32), min, max.
template <int DT, int OP, class T>
__device__ __forceinline__ T apply(T a, T b) {
    if constexpr (OP == 0) {
        if constexpr (DT == 2) return __fadd_rn(a, b);
        else return static_cast<T>(static_cast<uint32_t>(a) + static_cast<uint32_t>(b));
    } else if constexpr (OP == 1) {
        return b < a ? b : a;
    } else {
        return b > a ? b : a;
    }
}

// Segmented pair (f: a segment starts inside, v: the reduction after the last
// start, or of everything when none): (f1, v1) then (f2, v2).
template <int DT, int OP, class T>
__device__ __forceinline__ void combine(bool f1, T v1, bool& f2, T& v2) {
    v2 = f2 ? v2 : apply<DT, OP>(v1, v2);
    f2 = f1 || f2;
}

template <class OffT>
__device__ __forceinline__ int64_t offset_at(const ScanParams& p, int64_t s) {
    int64_t o = static_cast<int64_t>(__ldg(static_cast<const OffT*>(p.offsets) + s));
    o = o < 0 ? 0 : o;
    return o > p.N ? p.N : o;
}

__device__ __forceinline__ int64_t bound_at(const ScanParams& p, int64_t s) {
    return p.off64 ? offset_at<int64_t>(p, s) : offset_at<uint32_t>(p, s);
}

__global__ void __launch_bounds__(RS_NT) rs_zero_kernel(unsigned long long* a, int64_t n) {
    const int64_t stride = static_cast<int64_t>(gridDim.x) * RS_NT;
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * RS_NT + threadIdx.x; i < n; i += stride) a[i] = 0ull;
}

// One bit per offset inside [0, N): the row where a segment starts (the end
// offset marks where the rows in no segment begin).  A thread takes
// RS_FLAG_RUN consecutive offsets (sorted, so mostly in few words) and
// issues one atomic OR per word it touches.
constexpr int RS_FLAG_RUN = 8;

__global__ void __launch_bounds__(RS_NT) rs_flag_kernel(const ScanParams p) {
    const int64_t stride = static_cast<int64_t>(gridDim.x) * RS_NT * RS_FLAG_RUN;
    for (int64_t s0 = (static_cast<int64_t>(blockIdx.x) * RS_NT + threadIdx.x) * RS_FLAG_RUN; s0 <= p.S;
         s0 += stride) {
        int64_t word = -1;
        unsigned long long bits = 0;
#pragma unroll
        for (int k = 0; k < RS_FLAG_RUN; ++k) {
            const int64_t s = s0 + k;
            if (s > p.S) break;
            const int64_t o = bound_at(p, s);
            if (o >= p.N) break;   // nondecreasing: the rest are at N too
            if ((o >> 6) != word) {
                if (word >= 0) atomicOr(p.bitmap + word, bits);
                word = o >> 6;
                bits = 0;
            }
            bits |= 1ull << (o & 63);
        }
        if (word >= 0) atomicOr(p.bitmap + word, bits);
    }
}

__device__ __forceinline__ void cta_tiles(const ScanParams& p, int64_t& t0, int64_t& t1) {
    t0 = p.tiles * blockIdx.x / p.ctas;
    t1 = p.tiles * (blockIdx.x + 1) / p.ctas;
}

template <int DT>
__device__ __forceinline__ void load_tile(const ScanParams& p, int64_t base, typename ScanType<DT>::T (&v)[RS_PER],
                                          uint32_t& flags) {
    using T = typename ScanType<DT>::T;
    if (p.vec && base + RS_PER <= p.N) {
        const uint4* q = reinterpret_cast<const uint4*>(static_cast<const T*>(p.values) + base);
#pragma unroll
        for (int k = 0; k < RS_PER / 4; ++k) {
            const uint4 w = __ldcs(q + k);
            v[4 * k] = from_word<T>(w.x);
            v[4 * k + 1] = from_word<T>(w.y);
            v[4 * k + 2] = from_word<T>(w.z);
            v[4 * k + 3] = from_word<T>(w.w);
        }
    } else {
#pragma unroll
        for (int j = 0; j < RS_PER; ++j)
            v[j] = base + j < p.N ? __ldg(static_cast<const T*>(p.values) + base + j) : T(0);
    }
    static_assert(RS_PER == 8 || RS_PER == 16 || RS_PER == 32, "a thread's start bits lie in one bitmap word");
    constexpr unsigned long long kMask = (1ull << RS_PER) - 1;
    flags = base < p.N ? static_cast<uint32_t>((__ldcg(p.bitmap + (base >> 6)) >> (base & 63)) & kMask) : 0u;
}

// Scan pass: CTA b scans its tiles in order, carrying the open segment.
template <int DT, int OP, bool EXCL>
__global__ void __launch_bounds__(RS_NT, 8) rs_scan_kernel(const ScanParams p) {
    using T = typename ScanType<DT>::T;
    __shared__ T s_wv[kWarps];
    __shared__ int s_wf[kWarps];
    __shared__ long long s_wfirst[kWarps];
    __shared__ int s_last;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int64_t t0, t1;
    cta_tiles(p, t0, t1);
    const int64_t lo = bound_at(p, 0), hi = bound_at(p, p.S);
    const T id = identity<DT, OP>();
    bool cf = false;          // the carry across this CTA's tiles (block-uniform)
    T cv = id;
    int64_t first = LLONG_MAX;   // the range's first start row
    const int64_t mine = static_cast<int64_t>(threadIdx.x) * RS_PER;
    T cur[RS_PER];
    uint32_t cflags;
    load_tile<DT>(p, t0 * RS_TILE + mine, cur, cflags);
    for (int64_t t = t0; t < t1; ++t) {
        T nxt[RS_PER];
        uint32_t nflags = 0;
        if (t + 1 < t1) load_tile<DT>(p, (t + 1) * RS_TILE + mine, nxt, nflags);
        const int64_t base = t * RS_TILE + mine;
        // my rows: an inclusive scan that restarts at each start bit
        T incl[RS_PER];
        T acc = id;
#pragma unroll
        for (int j = 0; j < RS_PER; ++j) {
            acc = ((cflags >> j) & 1u) ? cur[j] : apply<DT, OP>(acc, cur[j]);
            incl[j] = acc;
        }
        bool f = cflags != 0;
        T v = acc;
        // segmented inclusive scan over the lanes
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const bool f2 = __shfl_up_sync(0xffffffffu, f, o);
            const T v2 = __shfl_up_sync(0xffffffffu, v, o);
            if (lane >= o) combine<DT, OP>(f2, v2, f, v);
        }
        bool ef = __shfl_up_sync(0xffffffffu, f, 1);
        T ev = __shfl_up_sync(0xffffffffu, v, 1);
        if (lane == 0) {
            ef = false;
            ev = id;
        }
        // first start row of the tile, per warp (until the range's first is known)
        const bool want_first = first == LLONG_MAX;
        if (want_first) {
            long long myfirst = cflags ? base + (__ffs(cflags) - 1) : LLONG_MAX;
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
                const long long y = __shfl_xor_sync(0xffffffffu, myfirst, o);
                myfirst = y < myfirst ? y : myfirst;
            }
            if (lane == 0) s_wfirst[warp] = myfirst;
        }
        if (lane == 31) {
            s_wf[warp] = f;
            s_wv[warp] = v;
        }
        __syncthreads();
        // the warps before mine, then the carry from the CTA's earlier tiles
        bool pf = false;
        T pv = id;
        bool tf = false;
        T tv = id;
        long long tfirst = LLONG_MAX;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) {
            const bool wf = s_wf[w] != 0;
            const T wv = s_wv[w];
            if (w < warp) {
                bool f2 = wf;
                T v2 = wv;
                combine<DT, OP>(pf, pv, f2, v2);
                pf = f2;
                pv = v2;
            }
            bool f2 = wf;
            T v2 = wv;
            combine<DT, OP>(tf, tv, f2, v2);
            tf = f2;
            tv = v2;
            if (want_first) tfirst = s_wfirst[w] < tfirst ? s_wfirst[w] : tfirst;
        }
        combine<DT, OP>(pf, pv, ef, ev);        // the warps before mine, then the lanes before me
        bool xf = ef;
        T xv = ev;
        combine<DT, OP>(cf, cv, xf, xv);        // the CTA's earlier tiles come first
        // outputs: my rows before my first start get the prefix
        T outv[RS_PER];
        bool seen = false;
#pragma unroll
        for (int j = 0; j < RS_PER; ++j) {
            seen = seen || ((cflags >> j) & 1u);
            outv[j] = seen ? incl[j] : apply<DT, OP>(xv, incl[j]);
        }
        if constexpr (EXCL) {
            // the sum of the segment's rows before each row (0 at a start)
            T prev = xv;
#pragma unroll
            for (int j = 0; j < RS_PER; ++j) {
                const T inc = outv[j];
                outv[j] = ((cflags >> j) & 1u) ? T(0) : prev;
                prev = inc;
            }
        }
        const int64_t tile0 = t * RS_TILE;
        if (tile0 < lo || tile0 + RS_TILE > hi) {   // the tile reaches rows in no segment
#pragma unroll
            for (int j = 0; j < RS_PER; ++j)
                if (base + j < lo || base + j >= hi) outv[j] = T(0);
        }
        T* out = static_cast<T*>(p.out) + base;
        if (p.vec && base + RS_PER <= p.N) {
#pragma unroll
            for (int k = 0; k < RS_PER / 4; ++k) {
                uint4 w;
                w.x = to_word(outv[4 * k]);
                w.y = to_word(outv[4 * k + 1]);
                w.z = to_word(outv[4 * k + 2]);
                w.w = to_word(outv[4 * k + 3]);
                __stcs(reinterpret_cast<uint4*>(out) + k, w);
            }
        } else {
#pragma unroll
            for (int j = 0; j < RS_PER; ++j)
                if (base + j < p.N) out[j] = outv[j];
        }
        // the carry into the next tile: (cf, cv) then the whole tile
        combine<DT, OP>(cf, cv, tf, tv);
        cf = tf;
        cv = tv;
        if (want_first) first = tfirst;
        for (int j = 0; j < RS_PER; ++j) cur[j] = nxt[j];
        cflags = nflags;
        __syncthreads();
    }
    if (threadIdx.x == 0) {
        const int64_t rend = t1 * RS_TILE < p.N ? t1 * RS_TILE : p.N;
        p.cta_flag[blockIdx.x] = cf ? 1 : 0;
        if constexpr (DT == 2 && OP == 0) p.cta_aggf[blockIdx.x] = PartPair{cv, 0.0f};
        else p.cta_aggi[blockIdx.x] = to_word(cv);
        p.cta_first[blockIdx.x] = first < rend ? first : rend;
        // the arrival releases the words above
        s_last = ticket_last(ticket_take(p.ticket, 0, p.gen), p.gen, p.ctas) ? 1 : 0;
    }
    __syncthreads();
    if (!s_last) return;
    fence_acq_rel_gpu();
    // the last CTA: each CTA's carry-in, a segmented exclusive scan of the
    // aggregates (float32 sums as compensated pairs: no FP64, which issues
    // far slower than FP32 on this part); thread i takes CTAs PER i .. PER i + PER - 1
    constexpr int PER = RS_MAX_CTAS / RS_NT;
    constexpr bool kPair = DT == 2 && OP == 0;
    using A = typename std::conditional<kPair, PartPair, T>::type;
    __shared__ A s_av[kWarps];
    __shared__ int s_af[kWarps];
    A aid;
    if constexpr (kPair) aid = PartPair{0.0f, 0.0f};
    else aid = id;
    auto shfl_up_a = [&](A v, int o) -> A {
        if constexpr (kPair)
            return PartPair{__shfl_up_sync(0xffffffffu, v.hi, o), __shfl_up_sync(0xffffffffu, v.lo, o)};
        else
            return __shfl_up_sync(0xffffffffu, v, o);
    };
    bool af[PER];
    A av[PER];
    bool mf = false;
    A mv = aid;
#pragma unroll
    for (int k = 0; k < PER; ++k) {
        const int i = threadIdx.x * PER + k;
        af[k] = i < p.ctas && __ldcg(p.cta_flag + i) != 0;
        if (i < p.ctas) {
            if constexpr (kPair) {
                const float2 a = __ldcg(reinterpret_cast<const float2*>(p.cta_aggf + i));
                av[k] = PartPair{a.x, a.y};
            }
            else av[k] = from_word<T>(__ldcg(p.cta_aggi + i));
        } else {
            av[k] = aid;
        }
        bool f2 = af[k];
        A v2 = av[k];
        if constexpr (kPair) { v2 = f2 ? v2 : pair_add(mv, v2); f2 = mf || f2; }
        else combine<DT, OP>(mf, mv, f2, v2);
        mf = f2;
        mv = v2;
    }
    bool f = mf;
    A v = mv;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const bool f2 = __shfl_up_sync(0xffffffffu, f, o);
        const A v2 = shfl_up_a(v, o);
        if (lane >= o) {
            if constexpr (kPair) { v = f ? v : pair_add(v2, v); f = f2 || f; }
            else combine<DT, OP>(f2, v2, f, v);
        }
    }
    bool ef = __shfl_up_sync(0xffffffffu, f, 1);
    A ev = shfl_up_a(v, 1);
    if (lane == 0) {
        ef = false;
        ev = aid;
    }
    if (lane == 31) {
        s_af[warp] = f;
        s_av[warp] = v;
    }
    __syncthreads();
    bool pf = false;
    A pv = aid;
    for (int w = 0; w < warp; ++w) {
        bool f2 = s_af[w];
        A v2 = s_av[w];
        if constexpr (kPair) { v2 = f2 ? v2 : pair_add(pv, v2); f2 = pf || f2; }
        else combine<DT, OP>(pf, pv, f2, v2);
        pf = f2;
        pv = v2;
    }
    if constexpr (kPair) { ev = ef ? ev : pair_add(pv, ev); ef = pf || ef; }
    else combine<DT, OP>(pf, pv, ef, ev);
#pragma unroll
    for (int k = 0; k < PER; ++k) {
        const int i = threadIdx.x * PER + k;
        if (i < p.ctas) {
            if constexpr (kPair) p.carryf[i] = ev;
            else p.carryi[i] = to_word(ev);
        }
        bool f2 = af[k];
        A v2 = av[k];
        if constexpr (kPair) { v2 = f2 ? v2 : pair_add(ev, v2); f2 = ef || f2; }
        else combine<DT, OP>(ef, ev, f2, v2);
        ef = f2;
        ev = v2;
    }
}

// Fix-up: CTA t adds the carry-in of its scan range to the rows of tile t
// that lie before the range's first start (and inside [offsets[0], offsets[S])).
template <int DT, int OP>
__global__ void __launch_bounds__(RS_NT) rs_fix_kernel(const ScanParams p) {
    using T = typename ScanType<DT>::T;
    const int64_t t = blockIdx.x;
    const int64_t b = ((t + 1) * p.ctas + p.tiles - 1) / p.tiles - 1;
    const int64_t r0 = (p.tiles * b / p.ctas) * RS_TILE;
    const int64_t lo = bound_at(p, 0), hi = bound_at(p, p.S);
    int64_t a = t * RS_TILE, e = (t + 1) * RS_TILE;
    e = e < p.N ? e : p.N;
    const int64_t first = __ldcg(p.cta_first + b);
    a = a > r0 ? a : r0;
    a = a > lo ? a : lo;
    e = e < first ? e : first;
    e = e < hi ? e : hi;
    if (a >= e) return;
    T* out = static_cast<T*>(p.out);
    if constexpr (DT == 2 && OP == 0) {
        // the carry as a normalised pair: ch = hi + lo rounded, cl what that
        // rounding dropped, so that ch + (cl + x) rounds like one addition
        const float2 c2 = __ldcg(reinterpret_cast<const float2*>(p.carryf + b));
        const PartPair c{c2.x, c2.y};
        const float ch = c.hi + c.lo;
        const float cl = c.lo - (ch - c.hi);
        for (int64_t r = a + threadIdx.x; r < e; r += RS_NT) out[r] = __fadd_rn(ch, __fadd_rn(cl, out[r]));
    } else {
        const T c = from_word<T>(__ldcg(p.carryi + b));
        for (int64_t r = a + threadIdx.x; r < e; r += RS_NT) out[r] = apply<DT, OP>(c, out[r]);
    }
}

unsigned grid_for(int64_t work, int64_t per_cta) {
    const int64_t g = (work + per_cta - 1) / per_cta;
    return static_cast<unsigned>(g < 1 ? 1 : (g > 65535 * 16 ? 65535 * 16 : g));
}

template <int DT, int OP, bool EXCL>
cudaError_t launch_op(ScanParams p, cudaStream_t stream) {
    // one wave of scan CTAs: as many as fit on the GPU at once
    static const int per_sm = [] {
        int n = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, rs_scan_kernel<DT, OP, EXCL>, RS_NT, 0) != cudaSuccess)
            n = 1;
        return n < 1 ? 1 : n;
    }();
    int64_t ctas = int64_t(p.sm_count) * per_sm;
    ctas = ctas < RS_MAX_CTAS ? ctas : RS_MAX_CTAS;
    p.ctas = static_cast<int32_t>(ctas < p.tiles ? ctas : p.tiles);
    const int64_t words = rs_bitmap_words(p.N);
    rs_zero_kernel<<<grid_for(words, RS_NT * 8), RS_NT, 0, stream>>>(p.bitmap, words);
    rs_flag_kernel<<<grid_for(p.S + 1, RS_NT * RS_FLAG_RUN), RS_NT, 0, stream>>>(p);
    rs_scan_kernel<DT, OP, EXCL><<<p.ctas, RS_NT, 0, stream>>>(p);
    rs_fix_kernel<DT, OP><<<static_cast<unsigned>(p.tiles), RS_NT, 0, stream>>>(p);
    return cudaGetLastError();
}

template <int DT>
cudaError_t launch_dt(const ScanParams& p, cudaStream_t stream) {
    if (p.op == 0) return p.exclusive ? launch_op<DT, 0, true>(p, stream) : launch_op<DT, 0, false>(p, stream);
    if (p.op == 1) return launch_op<DT, 1, false>(p, stream);
    return launch_op<DT, 2, false>(p, stream);
}

}  // namespace

cudaError_t launch_scan(const ScanParams& p, cudaStream_t stream) {
    if (p.dtype == 2) return launch_dt<2>(p, stream);
    if (p.dtype == 1) return launch_dt<1>(p, stream);
    return launch_dt<0>(p, stream);
}

}  // namespace segred
