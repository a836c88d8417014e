// seg_common.cuh -- pieces shared by the segmented-reduction kernels (sm_103a):
// launch parameters, element arithmetic, the merge-path CTA partition, the
// bulk-copy producer, bounded waits and the cross-CTA ticket combine.
//
// What it computes: GPUSegmentedReduction (luma.gl), "Contract" -- segment s
// reduces rows [offsets[s], offsets[s+1]) to a sum, min or max, an empty
// segment gives 0; graph-reduce README, "API" / "Method" / "Correctness" --
// [N, F] rows reduce per column, min / max also return the source row (ties to
// the lower row, -1 when empty), mean = sum / length.
//
// The kernels (seg_scalar.cuh, seg_rows2.cuh) cut the merged sequence of
// rows and segment ends into equal-weight units, one per warp, and combine
// the segments that cross units through per-unit partials and an atomic
// ticket (never a wait).  This file holds what they share: the launch
// parameters, element arithmetic, the partial format, the bulk-copy stream
// geometry, bounded waits and the ticket.
#pragma once
#include <climits>
#include <cstdint>
#include <type_traits>

#include "ptx.cuh"

namespace segred {

enum : int { OP_SUM = 0, OP_MIN = 1, OP_MAX = 2 };

constexpr uint64_t WAIT_LIMIT_NS = 2000000000ull;

constexpr unsigned STATUS_CONSUMER_TIMEOUT = 1u;
constexpr unsigned STATUS_DRAIN_TIMEOUT = 4u;

struct Params {
    const void* values;
    const void* offsets;
    void* out;
    int64_t* out_arg;
    int64_t N;        // rows in values
    int64_t S;        // segments
    int32_t F;        // columns
    int32_t G;        // row kernel: column slices
    int32_t K;        // rows per lane per tile / rows in flight (informational)
    int32_t max_ends; // segment ends per tile (informational)
    int32_t P;        // CTAs in the grid
    int32_t mean;     // finalise sums as means
    void* ws_parts;   // unit tail partials, then unit head partials
    unsigned long long* ws_tickets;  // one per unit: (generation << 32) | arrivals
    unsigned int* status;            // device status word
    uint32_t gen;                    // call generation, > 0, increasing per scratch buffer
};

// One cross-CTA partial: a float sum as a compensated pair (hi, lo), an
// integer sum, or a (value, absolute row) pair.  No double arithmetic: FP64
// issues far slower than FP32 on this part, and a combine over hundreds of
// partials sat on the critical path.
struct PartPair {
    float hi, lo;
};
struct PartElem {
    union {
        unsigned long long w;   // the raw 8 bytes (copies and shuffles)
        PartPair c;
        uint32_t u;
        int32_t i;
        float f;
    } v;
    int64_t row;
};
static_assert(sizeof(PartElem) == 16, "scratch element layout");


// ---------------------------------------------------------------------------
// Element arithmetic.

template <class T>
constexpr bool kIsFloat = std::is_floating_point<T>::value;

template <class T>
struct Acc {
    T v;
    int32_t row;  // CTA-relative source row for min / max, -1 = no row yet
};

__device__ __forceinline__ float add_wrap(float a, float b) { return a + b; }
__device__ __forceinline__ uint32_t add_wrap(uint32_t a, uint32_t b) { return a + b; }
__device__ __forceinline__ int32_t add_wrap(int32_t a, int32_t b) {
    return static_cast<int32_t>(static_cast<uint32_t>(a) + static_cast<uint32_t>(b));
}

template <class T, int OP>
struct Red {
    __device__ __forceinline__ static Acc<T> ident() {
        Acc<T> a;
        a.v = T(0);
        a.row = -1;
        return a;
    }
    // Rows arrive in increasing order, so a strict compare keeps the lower row on ties.
    __device__ __forceinline__ static void add(Acc<T>& a, T x, int32_t row) {
        if constexpr (OP == OP_SUM) {
            a.v = add_wrap(a.v, x);
        } else {
            const bool better = (OP == OP_MIN) ? (x < a.v) : (x > a.v);
            if (a.row < 0 || better) {
                a.v = x;
                a.row = row;
            }
        }
    }
    // `e` covers lower rows than `l`.
    __device__ __forceinline__ static Acc<T> comb(const Acc<T>& e, const Acc<T>& l) {
        if constexpr (OP == OP_SUM) {
            Acc<T> r;
            r.v = add_wrap(e.v, l.v);
            r.row = -1;
            return r;
        } else {
            const bool better = (OP == OP_MIN) ? (l.v < e.v) : (l.v > e.v);
            return (l.row >= 0 && (e.row < 0 || better)) ? l : e;
        }
    }
};

// Running value of the segment that is still open at a tile boundary.
template <class T, int OP>
struct Carry {
    using C = Acc<T>;
    __device__ __forceinline__ static C ident() { return Red<T, OP>::ident(); }
    __device__ __forceinline__ static C from(const Acc<T>& a) { return a; }
    __device__ __forceinline__ static C then(const C& c, const Acc<T>& a) {
        return Red<T, OP>::comb(c, a);
    }
};
// The scalar kernel's float-sum carry: a compensated pair (hi + lo) kept
// with TwoSum (Knuth), so a long chain of tile partials stays within a few
// units of 2^-48 of the exact sum while using only float32 arithmetic.
struct CarryF2 {
    float hi, lo;
};
__device__ __forceinline__ CarryF2 two_sum_add(const CarryF2& c, float a) {
    const float s = c.hi + a;
    const float bb = s - c.hi;
    const float err = (c.hi - (s - bb)) + (a - bb);
    return CarryF2{s, c.lo + err};
}
template <class T, int OP>
struct ScalarCarry : Carry<T, OP> {};
template <>
struct ScalarCarry<float, OP_SUM> {
    using C = CarryF2;
    __device__ __forceinline__ static C ident() { return C{0.0f, 0.0f}; }
    __device__ __forceinline__ static C from(const Acc<float>& a) { return C{a.v, 0.0f}; }
    __device__ __forceinline__ static C then(const C& c, const Acc<float>& a) {
        return two_sum_add(c, a.v);
    }
};

template <class T>
__device__ __forceinline__ uint32_t bits_of(T x) {
    return *reinterpret_cast<uint32_t*>(&x);
}
template <class T>
__device__ __forceinline__ T from_bits(uint32_t b) {
    return *reinterpret_cast<T*>(&b);
}

// Final value / arg of a segment from a float32 (or integer) accumulator.
template <class T, int OP>
__device__ __forceinline__ void finish_acc(const Acc<T>& a, int64_t len, int mean, int64_t row_base,
                                           T& v, int64_t& arg) {
    if constexpr (OP == OP_SUM) {
        v = a.v;
        if constexpr (kIsFloat<T>) {
            if (mean) v = len > 0 ? a.v / static_cast<float>(len) : 0.0f;
        }
        arg = -1;
    } else {
        v = a.row >= 0 ? a.v : T(0);
        arg = a.row >= 0 ? row_base + a.row : -1;
    }
}
template <class T, int OP>
__device__ __forceinline__ PartElem to_part(const Acc<T>& a, int64_t row_base) {
    PartElem p;
    p.v.u = bits_of(a.v);
    p.row = (OP != OP_SUM && a.row >= 0) ? row_base + a.row : -1;
    return p;
}
__device__ __forceinline__ void finish_carry(const CarryF2& c, int64_t len, int mean, float& v) {
    const float s = c.hi + c.lo;
    v = mean ? (len > 0 ? s / static_cast<float>(len) : 0.0f) : s;
}
__device__ __forceinline__ PartElem to_part(const CarryF2& c) {
    PartElem p;
    p.v.c = PartPair{c.hi, c.lo};
    p.row = -1;
    return p;
}
// (a.hi + a.lo) + (b.hi + b.lo) as a pair: TwoSum of the high parts, the
// rounding error and both low parts carried in lo.
__device__ __forceinline__ PartPair pair_add(const PartPair& a, const PartPair& b) {
    const float s = a.hi + b.hi;
    const float bb = s - a.hi;
    const float err = (a.hi - (s - bb)) + (b.hi - bb);
    return PartPair{s, (a.lo + b.lo) + err};
}
template <class T, int OP>
__device__ __forceinline__ PartElem part_comb(const PartElem& e, const PartElem& l) {
    PartElem r;
    if constexpr (OP == OP_SUM) {
        if constexpr (kIsFloat<T>) {
            r.v.c = pair_add(e.v.c, l.v.c);
        } else {
            r.v.u = e.v.u + l.v.u;
        }
        r.row = -1;
        return r;
    } else {
        const T ev = from_bits<T>(e.v.u), lv = from_bits<T>(l.v.u);
        const bool better = (OP == OP_MIN) ? (lv < ev) : (lv > ev);
        return (l.row >= 0 && (e.row < 0 || better)) ? l : e;
    }
}
template <class T, int OP>
__device__ __forceinline__ void finish_part(const PartElem& p, int64_t len, int mean, T& v,
                                            int64_t& arg) {
    if constexpr (OP == OP_SUM) {
        if constexpr (kIsFloat<T>) {
            const float f = p.v.c.hi + p.v.c.lo;
            v = mean ? (len > 0 ? f / static_cast<float>(len) : 0.0f) : f;
        } else {
            v = from_bits<T>(p.v.u);
        }
        arg = -1;
    } else {
        v = p.row >= 0 ? from_bits<T>(p.v.u) : T(0);
        arg = p.row;
    }
}

// ---------------------------------------------------------------------------
// Geometry of one streamed byte range [BA, BE) of a device buffer.

struct Stream {
    uint64_t A0;   // BA rounded down to 16: byte A0 + k lands at ring offset k mod ring size
    uint64_t AE;   // BE rounded up to 16
    uint64_t BA, BE;
    uint64_t TA, TE;  // 16-byte-aligned interior of the whole buffer (bulk-copy region)
    int64_t nch;      // chunks
};

__device__ __forceinline__ Stream make_stream(uint64_t buf, uint64_t buf_bytes, uint64_t ba,
                                              uint64_t be, uint32_t chunk) {
    Stream s;
    s.BA = ba;
    s.BE = be;
    s.A0 = ba & ~uint64_t(15);
    s.AE = (be + 15) & ~uint64_t(15);
    s.TA = (buf + 15) & ~uint64_t(15);
    s.TE = (buf + buf_bytes) & ~uint64_t(15);
    s.nch = be > ba ? static_cast<int64_t>((s.AE - s.A0 + chunk - 1) / chunk) : 0;
    return s;
}

// Producer side: copy chunk m of stream `s` (chunk bytes from A0) to `dst`.
__device__ __forceinline__ void issue_chunk_to(const Stream& s, int64_t m, uint32_t chunk,
                                               unsigned char* dst, uint64_t* full, uint64_t policy) {
    const uint64_t cs = s.A0 + static_cast<uint64_t>(m) * chunk;
    const uint64_t ce = cs + chunk < s.AE ? cs + chunk : s.AE;
    const uint64_t ts = cs > s.TA ? cs : s.TA;
    const uint64_t te = ce < s.TE ? ce : s.TE;
    const uint32_t tx = te > ts ? static_cast<uint32_t>(te - ts) : 0u;
    // Needed bytes outside the bulk-copy region: at most 12 at either end of the buffer.
    const uint64_t f0 = cs > s.BA ? cs : s.BA;
    const uint64_t f1 = ce < s.BE ? ce : s.BE;
    if (tx == 0) {
        for (uint64_t b = f0; b < f1; b += 4)
            *reinterpret_cast<uint32_t*>(dst + (b - cs)) = ld_global_u32(b);
    } else {
        for (uint64_t b = f0; b < (f1 < ts ? f1 : ts); b += 4)
            *reinterpret_cast<uint32_t*>(dst + (b - cs)) = ld_global_u32(b);
        for (uint64_t b = (f0 > te ? f0 : te); b < f1; b += 4)
            *reinterpret_cast<uint32_t*>(dst + (b - cs)) = ld_global_u32(b);
    }
    mbar_arrive_expect_tx(full, tx);
    if (tx) bulk_load(dst + (ts - cs), reinterpret_cast<const void*>(ts), tx, full, policy);
}

// Same, into a power-of-two ring: byte A0 + k lands at ring offset k mod ring_bytes.
__device__ __forceinline__ void issue_chunk(const Stream& s, int64_t m, unsigned char* ring,
                                            uint32_t ring_bytes, uint32_t chunk, uint64_t* full,
                                            uint64_t policy) {
    const uint64_t cs = s.A0 + static_cast<uint64_t>(m) * chunk;
    issue_chunk_to(s, m, chunk, ring + ((cs - s.A0) & (ring_bytes - 1)), full, policy);
}

// Wait for a phase with a time limit; records `code` in the status word on expiry.
__device__ __forceinline__ bool wait_bounded_for(uint64_t* bar, uint32_t parity, unsigned int* status,
                                                 unsigned code, uint64_t limit_ns) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    for (;;) {
        for (int k = 0; k < 8; ++k)
            if (mbar_try_wait(bar, parity)) return true;
        if (globaltimer_ns() - t0 > limit_ns) {
            atomicOr(status, code);
            return false;
        }
    }
}

__device__ __forceinline__ bool wait_bounded(uint64_t* bar, uint32_t parity, unsigned int* status,
                                             unsigned code) {
    return wait_bounded_for(bar, parity, status, code, WAIT_LIMIT_NS);
}

template <class OffT>
__device__ __forceinline__ int64_t clamp_off(OffT raw, int64_t N) {
    int64_t o = static_cast<int64_t>(raw);
    o = o < 0 ? 0 : o;
    return o > N ? N : o;
}

// At kernel start each CTA asks L2 for its 1/P slice of the offsets array
// (when the array is small enough to stay there): the boundary search and the
// units' own offsets loads then find it in L2 instead of each paying a DRAM
// round trip.  The bytes are read once either way.
constexpr uint64_t OFFSETS_PREFETCH_MAX = 32ull << 20;

__device__ __forceinline__ void prefetch_offsets_slice(const void* offsets, uint64_t bytes, int cta, int P,
                                                       int tid, int nth) {
    if (bytes > OFFSETS_PREFETCH_MAX) return;
    const uint64_t base = reinterpret_cast<uint64_t>(offsets);
    const uint64_t ta = (base + 15) & ~uint64_t(15);
    const uint64_t te = (base + bytes) & ~uint64_t(15);
    if (te <= ta) return;
    const uint64_t per = ((te - ta) / P + 4095) & ~uint64_t(4095);
    const uint64_t a = ta + per * static_cast<uint64_t>(cta);
    const uint64_t b = a + per < te ? a + per : te;
    for (uint64_t c = a + static_cast<uint64_t>(tid) * 4096; c < b; c += static_cast<uint64_t>(nth) * 4096) {
        const uint64_t e = c + 4096 < b ? c + 4096 : b;
        bulk_prefetch_l2(reinterpret_cast<const void*>(c), static_cast<uint32_t>(e - c));
    }
}

// Cross-unit arrival for the segment whose end lies in unit q, in two halves
// so that the caller can go on working while the atomic is in flight.
// Tickets carry the call generation in the high half: a stale count left by
// an earlier call is reset by the max, never used.  ticket_take returns the
// old ticket value (the caller's own earlier writes are released with it);
// ticket_last tells whether that arrival was the last of `expected`.  The
// last arriver runs fence_acq_rel_gpu() before it reads the others' partials.
__device__ __forceinline__ unsigned long long ticket_take(unsigned long long* tickets, int q, uint32_t gen) {
    const unsigned long long base = static_cast<unsigned long long>(gen) << 32;
    red_max_relaxed_gpu(&tickets[q], base);
    return atom_add_release_gpu(&tickets[q], 1ull);
}
__device__ __forceinline__ bool ticket_last(unsigned long long old, uint32_t gen, int expected) {
    return old == (static_cast<unsigned long long>(gen) << 32) + static_cast<unsigned long long>(expected - 1);
}

__device__ __forceinline__ PartElem load_part(const PartElem* src) {
    const longlong2 raw = __ldcg(reinterpret_cast<const longlong2*>(src));
    PartElem pe;
    pe.v.w = static_cast<unsigned long long>(raw.x);
    pe.row = raw.y;
    return pe;
}

}  // namespace segred
