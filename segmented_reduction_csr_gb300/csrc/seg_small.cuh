// seg_small.cuh -- the small-input kernel: F == 1 reductions of at most
// SM_MAXR rows over at most SM_MAXS segments (GPUSegmentedReduction's
// "Contract", as the other kernels), in one CTA and one launch.
//
// At this size a call is bound by its latency, not by bandwidth: the whole
// input is a few tens of kilobytes.  The CTA copies every row and the
// offsets into shared memory (per-thread asynchronous copies, all in flight
// at once: one memory round trip), then:
//  * every segment of at most 32 rows is reduced by one thread, reading its
//    rows from shared memory in order;
//  * every longer segment is reduced by one warp: lane l folds rows l,
//    l + 32, ... in order (float sums in blocks of 32 rows, each folded into
//    a compensated pair), then a fixed butterfly combines the lanes (min /
//    max keep the lower row on ties).
// The short pass puts the longer segments on a shared-memory list, so the
// warps visit only those.  No scratch, no global atomics, no cross-CTA
// combine; every order is fixed by the offsets, so float results are
// reproducible run to run.
#pragma once
#include "seg_common.cuh"

namespace segred {

constexpr int SM_NT = 1024;                 // threads of the one CTA
constexpr int SM_MAXR = 16384;              // rows, at most
constexpr int SM_MAXS = 4096;               // segments, at most
constexpr uint32_t SM_SMEM = SM_MAXR * 4 + (SM_MAXS + 1) * 8 + 16;

template <class T, int OP, class OffT>
__global__ void __launch_bounds__(SM_NT, 1) seg_small_kernel(const Params p) {
    using RD = Red<T, OP>;
    constexpr unsigned FULL = 0xffffffffu;
    constexpr bool kFloatSum = OP == OP_SUM && kIsFloat<T>;
    constexpr int KO = (SM_MAXS + 1 + SM_NT - 1) / SM_NT;
    extern __shared__ __align__(1024) unsigned char smem[];   // aligned as the other kernels declare it
    OffT* sraw = reinterpret_cast<OffT*>(smem);                            // [S + 1] offsets as given
    int32_t* so = reinterpret_cast<int32_t*>(smem);                         // ... then clamped to [0, N]
    uint32_t* sv = reinterpret_cast<uint32_t*>(smem + (SM_MAXS + 1) * 8);  // rows [0, N)
    __shared__ int32_t slong[SM_MAXR / 33 + 1];                             // the segments of > 32 rows
    __shared__ int32_t snlong;
    const int tid = threadIdx.x;
    const int lane = tid & 31;
    const int warp = tid >> 5;
    const int64_t N = p.N;
    const int S = static_cast<int>(p.S);
    const int nr = static_cast<int>(N);   // N <= SM_MAXR: the planner checked
    const OffT* offs = static_cast<const OffT*>(p.offsets);
    const uint32_t* vals = static_cast<const uint32_t*>(p.values);

    // the offsets and every row, by per-thread asynchronous copies, all in
    // flight at once
    for (int i = tid; i <= S; i += SM_NT) cp_async_small<sizeof(OffT)>(sraw + i, offs + i);
    for (int i = tid; i < nr; i += SM_NT) cp_async_small<4>(sv + i, vals + i);
    cp_async_commit();
    if (tid == 0) snlong = 0;
    cp_async_wait_all();
    __syncthreads();
    {
        // offsets clamped to [0, N] as 32-bit rows, in place: all read, then written
        int32_t w[KO];
#pragma unroll
        for (int k = 0; k < KO; ++k) {
            const int i = tid + k * SM_NT;
            w[k] = i <= S ? static_cast<int32_t>(clamp_off(sraw[i], N)) : 0;
        }
        __syncthreads();
#pragma unroll
        for (int k = 0; k < KO; ++k) {
            const int i = tid + k * SM_NT;
            if (i <= S) so[i] = w[k];
        }
    }
    __syncthreads();

    T* out = static_cast<T*>(p.out);
    const bool want_arg = (OP != OP_SUM) && p.out_arg != nullptr;

    // ---- short segments: a thread each; the longer ones go on a list ---------------
    for (int s = tid; s < S; s += SM_NT) {
        const int b = so[s];
        const int e = so[s + 1] > b ? so[s + 1] : b;   // (a decreasing pair: empty)
        if (e - b > 32) {
            slong[atomicAdd(&snlong, 1)] = s;
            continue;
        }
        Acc<T> a = RD::ident();
        for (int r = b; r < e; ++r) RD::add(a, from_bits<T>(sv[r]), r);
        T v;
        int64_t arg;
        finish_acc<T, OP>(a, e - b, p.mean, 0, v, arg);
        out[s] = v;
        if (want_arg) p.out_arg[s] = arg;
    }
    __syncthreads();

    // ---- long segments: a warp each ------------------------------------------------
    const int nlong = snlong;
    for (int k = warp; k < nlong; k += SM_NT / 32) {
        const int s = slong[k];
        const int b = so[s], e = so[s + 1];
        Acc<T> a = RD::ident();
        CarryF2 c{0.0f, 0.0f};
        for (int r0 = b; r0 < e; r0 += 32 * 32) {
            // a block of up to 32 rows per lane, folded into the pair afterwards
            Acc<T> blk = RD::ident();
            const int r1 = r0 + 32 * 32 < e ? r0 + 32 * 32 : e;
            for (int r = r0 + lane; r < r1; r += 32) RD::add(blk, from_bits<T>(sv[r]), r);
            if constexpr (kFloatSum)
                c = two_sum_add(c, blk.v);
            else
                a = RD::comb(a, blk);
        }
        if constexpr (kFloatSum) a.v = c.hi + c.lo;
        // lanes hold interleaved rows: combine with the lower row on ties
#pragma unroll
        for (int o = 16; o >= 1; o >>= 1) {
            Acc<T> other;
            other.v = from_bits<T>(__shfl_xor_sync(FULL, bits_of(a.v), o));
            other.row = OP == OP_SUM ? -1 : __shfl_xor_sync(FULL, a.row, o);
            if constexpr (OP == OP_SUM) {
                a = (lane & o) ? RD::comb(other, a) : RD::comb(a, other);
            } else {
                const bool ob = (OP == OP_MIN) ? (other.v < a.v) : (other.v > a.v);
                const bool ab = (OP == OP_MIN) ? (a.v < other.v) : (a.v > other.v);
                if (a.row < 0 || (other.row >= 0 && (ob || (!ab && other.row < a.row)))) a = other;
            }
        }
        if (lane == 0) {
            T v;
            int64_t arg;
            finish_acc<T, OP>(a, e - b, p.mean, 0, v, arg);
            out[s] = v;
            if (want_arg) p.out_arg[s] = arg;
        }
    }
}

}  // namespace segred
