// seg_rows2.cuh -- the row kernel: [N, F] row tensors (F > 1) of uint32,
// int32 or float32, reduced per column (graph-reduce README, "API": the
// per-edge to per-node message-passing shape).
//
// Work split.  The columns are cut into slices of 32 * VEC (one VEC-wide
// vector per lane), and for every slice the merged sequence of rows and
// segment ends (a row weighs 1, an end RW_CW_SUM, or RW_CW_ARG when it also
// stores int64 rows) is cut into ranges of equal weight.  A warp owns one (slice, range) unit; one CTA of RW_NW warps per
// SM.  A CTA finds the range boundaries its warps need with one cooperative
// search (the same weighted merge-path search as the scalar kernel).
//
// Per warp.  Every lane reads its columns of each row of the range with a
// VEC-wide read-only global load, 16 (VEC = 4) or 32 rows ahead of use (a
// register ring: 8 KiB per warp in flight for VEC >= 2), and folds them into its
// accumulators.  Segment boundaries are the same for all lanes, so the warp
// takes them together: when row r reaches the end of the current segment,
// each lane finishes its columns and stores them (consecutive lanes store
// consecutive columns).  Segment ends come from a window of 32 offsets held
// one per lane, with the next 32 already loading.  Float sums add a block of
// rows in float32 and fold each block into a compensated pair (TwoSum), so
// long segments stay far inside the error bound.
//
// A segment that crosses ranges leaves per-unit partials in scratch; the
// last unit to arrive (atomic ticket, no waiting) combines them in range
// order, so float results are reproducible.
#pragma once
#include "seg_common.cuh"

namespace segred {

constexpr int RW_NW = 8;                      // warps (units) per CTA
constexpr int RW_NTHREADS = RW_NW * 32;
// Merge-path weight of a segment end, in rows.  Measured on 10M x 128 f32
// with evenly spaced ends: an end costs about 1.9 rows of time for a sum and
// about 5 for a max that also stores its int64 rows (three times the bytes).
constexpr int RW_CW_SUM = 2;
constexpr int RW_CW_ARG = 5;
constexpr int RW_NDIAG = RW_NW + 1;           // range boundaries per CTA (at most)
constexpr int RW_GRID = 1024;                 // first-round probes, shared by all CTAs
constexpr int RW_PROBES = 56;                 // later-round probes per boundary
constexpr int RW_MIN_ITEMS = 128;             // weighted items per range, at least
constexpr int64_t RW_ADOPT = 512;             // rows of a cut-crossing segment a range adopts
constexpr int RW_NSR = 3;                     // staged rows: shared-memory stages per warp
constexpr uint32_t RW_CB = 8192;              // staged rows: bytes per stage
static_assert(RW_NDIAG * RW_PROBES <= 2 * RW_NTHREADS, "two probes per thread per round");

struct RowsSearchSmem {
    int64_t graw[RW_GRID];
    int64_t D[RW_NDIAG], lo[RW_NDIAG], hi[RW_NDIAG], R[RW_NDIAG];
    int cnt[RW_NDIAG];
    int64_t o0, oS;
};
constexpr uint32_t RW_SMEM = ((sizeof(RowsSearchSmem) + 127) / 128) * 128;
constexpr uint32_t RW_SMEM_STAGED = RW_NW * RW_NSR * RW_CB + RW_NW * RW_NSR * 8;
static_assert(RW_SMEM <= RW_SMEM_STAGED && RW_SMEM_STAGED <= 227 * 1024, "staged rows fit one CTA per SM");
// Offsets arrays up to this size are copied whole into a staged CTA's shared
// memory (behind the search scratch) and searched there.
constexpr uint32_t RW_SMALL_OFFS = 96 * 1024;
static_assert(RW_SMEM + RW_SMALL_OFFS <= RW_SMEM_STAGED, "the offsets fit beside the search scratch");

// VEC consecutive 32-bit elements, read once: no L1 allocation, L2 evict-first.
template <int VEC>
__device__ __forceinline__ void ld_stream(uint32_t (&x)[VEC], const uint32_t* p, uint64_t pol) {
    if constexpr (VEC == 4) {
        asm volatile("ld.global.nc.L1::no_allocate.L2::cache_hint.v4.b32 {%0, %1, %2, %3}, [%4], %5;"
                     : "=r"(x[0]), "=r"(x[1]), "=r"(x[2]), "=r"(x[3])
                     : "l"(p), "l"(pol));
    } else if constexpr (VEC == 2) {
        asm volatile("ld.global.nc.L1::no_allocate.L2::cache_hint.v2.b32 {%0, %1}, [%2], %3;"
                     : "=r"(x[0]), "=r"(x[1])
                     : "l"(p), "l"(pol));
    } else {
        asm volatile("ld.global.nc.L1::no_allocate.L2::cache_hint.b32 %0, [%1], %2;"
                     : "=r"(x[0])
                     : "l"(p), "l"(pol));
    }
}

// A lane's VEC output columns: one vector store when `vec` (the caller
// checked alignment), else one store per column.
template <int VEC>
__device__ __forceinline__ void store_cols(uint32_t* dst, const uint32_t (&r)[VEC], bool vec) {
    if constexpr (VEC == 4) {
        if (vec) {
            *reinterpret_cast<uint4*>(dst) = make_uint4(r[0], r[1], r[2], r[3]);
            return;
        }
    } else if constexpr (VEC == 2) {
        if (vec) {
            *reinterpret_cast<uint2*>(dst) = make_uint2(r[0], r[1]);
            return;
        }
    }
#pragma unroll
    for (int v = 0; v < VEC; ++v) dst[v] = r[v];
}
template <int VEC>
__device__ __forceinline__ void store_args(int64_t* dst, const int64_t (&a)[VEC], bool vec) {
    if constexpr (VEC >= 2) {
        if (vec) {
#pragma unroll
            for (int v = 0; v < VEC; v += 2)
                *reinterpret_cast<longlong2*>(dst + v) = make_longlong2(a[v], a[v + 1]);
            return;
        }
    }
#pragma unroll
    for (int v = 0; v < VEC; ++v) dst[v] = a[v];
}

// Last arriver of a segment that crosses ranges pc .. qc of slice `slice`:
// tails of ranges pc .. qc-1, then the head of range qc, in range order.
template <class T, int OP, int VEC>
__device__ __forceinline__ void rows_combine_store(const Params& p, const uint32_t* pv, const int64_t* pr,
                                                   int64_t U, int NSL, int slice, int64_t pc, int64_t qc,
                                                   int64_t s, int64_t len, int lane) {
    constexpr int SLW = 32 * VEC;
    const int F = p.F;
    const int c0 = slice * SLW + lane * VEC;
    if (c0 >= F) return;
    CarryF2 ds[VEC];   // float sums: a compensated pair (no FP64, which issues far slower)
    T tv[VEC];
    int64_t trow[VEC];
#pragma unroll
    for (int v = 0; v < VEC; ++v) {
        ds[v] = CarryF2{0.0f, 0.0f};
        tv[v] = T(0);
        trow[v] = -1;
    }
    // Partials are read KB units at a time (all loads of a batch in flight
    // together: a long segment has hundreds of them) and folded in order.
    constexpr int KB = OP == OP_SUM ? 16 : 8;
    for (int64_t k0 = pc; k0 <= qc; k0 += KB) {
        uint32_t b[KB][VEC];
        int64_t rr[OP == OP_SUM ? 1 : KB][VEC];
#pragma unroll
        for (int j = 0; j < KB; ++j) {
            const int64_t k = k0 + j;
            if (k <= qc) {
                const int64_t at = ((k < qc ? 0 : U) + k * NSL + slice) * SLW + lane * VEC;
#pragma unroll
                for (int v = 0; v < VEC; ++v) {
                    b[j][v] = __ldcg(&pv[at + v]);
                    if constexpr (OP != OP_SUM) rr[j][v] = __ldcg(&pr[at + v]);
                }
            }
        }
#pragma unroll
        for (int j = 0; j < KB; ++j) {
            if (k0 + j <= qc) {
#pragma unroll
                for (int v = 0; v < VEC; ++v) {
                    if constexpr (OP == OP_SUM) {
                        if constexpr (kIsFloat<T>) ds[v] = two_sum_add(ds[v], __uint_as_float(b[j][v]));
                        else tv[v] = add_wrap(tv[v], from_bits<T>(b[j][v]));
                    } else {
                        const T x = from_bits<T>(b[j][v]);
                        const bool better = (OP == OP_MIN) ? (x < tv[v]) : (x > tv[v]);
                        if (rr[j][v] >= 0 && (trow[v] < 0 || better)) {
                            tv[v] = x;
                            trow[v] = rr[j][v];
                        }
                    }
                }
            }
        }
    }
    T* out = static_cast<T*>(p.out);
#pragma unroll
    for (int v = 0; v < VEC; ++v) {
        T r;
        if constexpr (OP == OP_SUM && kIsFloat<T>) {
            const float f = ds[v].hi + ds[v].lo;
            r = p.mean ? (len > 0 ? f / static_cast<float>(len) : 0.0f) : f;
        } else {
            r = (OP != OP_SUM && trow[v] < 0) ? T(0) : tv[v];
        }
        out[s * F + c0 + v] = r;
        if (OP != OP_SUM && p.out_arg != nullptr) p.out_arg[s * F + c0 + v] = trow[v];
    }
}

template <class T, int OP, class OffT, int VEC, bool STAGED>
__global__ void __launch_bounds__(RW_NTHREADS, 1) seg_rows2_kernel(const Params p) {
    constexpr int PD = STAGED ? 1 : (VEC == 4 ? 16 : 32);   // rows in flight per lane (register ring)
    constexpr int SLW = 32 * VEC;    // columns per slice
    constexpr unsigned FULL = 0xffffffffu;
    constexpr bool kFloatSum = OP == OP_SUM && kIsFloat<T>;
    using RD = Red<T, OP>;

    extern __shared__ __align__(1024) unsigned char smem[];
    const int tid = threadIdx.x;
    const int lane = tid & 31;
    const int warp = tid >> 5;
    const int cta = blockIdx.x;
    const int64_t N = p.N;
    const int64_t S = p.S;
    const int F = p.F;
    const int NSL = p.G;                               // column slices
    const int64_t U = static_cast<int64_t>(p.P) * RW_NW;
    const int64_t CW = (OP != OP_SUM && p.out_arg != nullptr) ? RW_CW_ARG : RW_CW_SUM;
    const int64_t NR = U / NSL;                        // ranges per slice
    const OffT* offs = static_cast<const OffT*>(p.offsets);

    // ranges this CTA's warps own: rg_lo .. rg_hi
    const int64_t u_first = static_cast<int64_t>(cta) * RW_NW;
    const int64_t rg_lo = u_first / NSL;
    if (rg_lo >= NR) return;   // the whole CTA is idle
    int64_t rg_hi = (u_first + RW_NW - 1) / NSL;
    rg_hi = rg_hi < NR - 1 ? rg_hi : NR - 1;
    const int nb = static_cast<int>(rg_hi - rg_lo) + 2;   // boundaries rg_lo .. rg_hi + 1

    // ---- range boundaries: weighted merge path ---------------------------------
    // End s sits at key(s) = (offsets[s+1] - o0) + CW s; a cut at D takes
    // the I(D) = #{s : key(s) < D} ends before it and the rows before both
    // D - CW I and the start of segment I.
    // A small offsets array (staged shapes) is copied whole into shared
    // memory and each boundary is a binary search there: no probe rounds.
    RowsSearchSmem* ss = reinterpret_cast<RowsSearchSmem*>(smem);
    OffT* soffs = reinterpret_cast<OffT*>(smem + RW_SMEM);
    const bool small = STAGED && static_cast<uint64_t>(S + 1) * sizeof(OffT) <= RW_SMALL_OFFS;
    if (small) {
        for (int64_t i = tid; i <= S; i += RW_NTHREADS) cp_async_small<sizeof(OffT)>(soffs + i, offs + i);
        cp_async_commit();
        cp_async_wait_all();
    } else {
        prefetch_offsets_slice(p.offsets, static_cast<uint64_t>(S + 1) * sizeof(OffT), cta, p.P, tid, RW_NTHREADS);
        if (tid == 0) ss->o0 = clamp_off(__ldg(&offs[0]), N);
        if (tid == 1) ss->oS = clamp_off(__ldg(&offs[S]), N);
        for (int m = tid; m < RW_GRID; m += RW_NTHREADS) {
            const int64_t sm = static_cast<int64_t>(m) * S / RW_GRID;
            ss->graw[m] = clamp_off(__ldg(&offs[sm + 1]), N);
        }
    }
    __syncthreads();
    const int64_t o0 = small ? clamp_off(soffs[0], N) : ss->o0;
    const int64_t oS_raw = small ? clamp_off(soffs[S], N) : ss->oS;
    const int64_t oS = oS_raw < o0 ? o0 : oS_raw;
    const int64_t nrows = oS - o0;
    const int64_t total = nrows + CW * S;
    const int64_t Wr = (total + NR - 1) / NR;
    if (tid < nb) {
        const int64_t rg = rg_lo + tid;
        const int64_t D = rg * Wr < total ? rg * Wr : total;
        int64_t lo = D > nrows ? (D - nrows + CW - 1) / CW : 0;
        int64_t hi = (D + CW - 1) / CW;
        hi = hi < S ? hi : S;
        if (small) {
            // I = #{s : key(s) < D}: the first s in [lo, hi) with key(s) >= D
            while (lo < hi) {
                const int64_t mid = (lo + hi) >> 1;
                if (clamp_off(soffs[mid + 1], N) - o0 + CW * mid < D)
                    lo = mid + 1;
                else
                    hi = mid;
            }
            hi = lo;
        } else {
            int a = 0, b = RW_GRID;
            while (a < b) {
                const int mid = (a + b) >> 1;
                const int64_t sm = static_cast<int64_t>(mid) * S / RW_GRID;
                if (ss->graw[mid] - o0 + CW * sm < D)
                    a = mid + 1;
                else
                    b = mid;
            }
            const int64_t lower = a > 0 ? static_cast<int64_t>(a - 1) * S / RW_GRID + 1 : 0;
            const int64_t upper = a < RW_GRID ? static_cast<int64_t>(a) * S / RW_GRID : S;
            lo = lo > lower ? lo : lower;
            hi = hi < upper ? hi : upper;
            if (hi < lo) hi = lo;
        }
        ss->D[tid] = D;
        ss->lo[tid] = lo;
        ss->hi[tid] = hi;
        ss->cnt[tid] = 0;
    }
    __syncthreads();
    for (int round = 0; round < (small ? 0 : 64); ++round) {
#pragma unroll
        for (int u = 0; u < 2; ++u) {
            const int pidx = tid + u * RW_NTHREADS;
            const int k = pidx / RW_PROBES;
            const int mm = pidx - k * RW_PROBES;
            if (k < nb) {
                const int64_t lo = ss->lo[k], hi = ss->hi[k];
                const int64_t len = hi - lo;
                if (len > 0) {
                    const int64_t step = (len + RW_PROBES - 1) / RW_PROBES;
                    const int64_t s = lo + mm * step;
                    if (s < hi && clamp_off(__ldg(&offs[s + 1]), N) - o0 + CW * s < ss->D[k])
                        atomicAdd(&ss->cnt[k], 1);
                }
            }
        }
        __syncthreads();
        bool open = false;
        if (tid < nb) {
            int64_t lo = ss->lo[tid], hi = ss->hi[tid];
            const int64_t len = hi - lo;
            if (len > 0) {
                const int64_t step = (len + RW_PROBES - 1) / RW_PROBES;
                const int64_t c = ss->cnt[tid];
                if (c == 0) {
                    hi = lo;
                } else {
                    const int64_t last = lo + (c - 1) * step;
                    hi = last + step < hi ? last + step : hi;
                    lo = last + 1 < hi ? last + 1 : hi;
                }
                ss->lo[tid] = lo;
                ss->hi[tid] = hi;
                ss->cnt[tid] = 0;
                open = lo < hi;
            }
        }
        if (!__syncthreads_or(open)) break;
    }
    if (tid < nb) {
        const int64_t I = ss->lo[tid];
        const int64_t oI = I > 0 ? clamp_off(small ? soffs[I] : __ldg(&offs[I]), N) - o0 : 0;
        int64_t R = ss->D[tid] - CW * I;
        R = R < oI ? oI : R;
        R = R < 0 ? 0 : (R > nrows ? nrows : R);
        ss->R[tid] = o0 + R;
    }
    __syncthreads();
    const int64_t u_me = u_first + warp;
    const int slice = static_cast<int>(u_me % NSL);
    const int64_t rg = u_me / NSL;
    const int bi = static_cast<int>(rg < NR ? rg - rg_lo : 0);
    const int64_t Dlo = ss->D[bi], Dhi = ss->D[bi + 1];
    const int64_t Iu = ss->lo[bi];
    const int64_t Iu2 = ss->lo[bi + 1] > Iu ? ss->lo[bi + 1] : Iu;
    const int64_t Rc = ss->R[bi];                           // the cuts' rows
    const int64_t Rc2 = ss->R[bi + 1] > Rc ? ss->R[bi + 1] : Rc;
    // the offsets of the segments that cross the cuts, while a shared copy lives
    int64_t off_Iu = 0, off_Iu1 = 0, off_Iu2 = 0, off_Iu21 = 0;
    if (small) {
        off_Iu = clamp_off(soffs[Iu], N);
        off_Iu1 = Iu < S ? clamp_off(soffs[Iu + 1], N) : 0;
        off_Iu2 = Iu2 < S ? clamp_off(soffs[Iu2], N) : 0;
        off_Iu21 = Iu2 < S ? clamp_off(soffs[Iu2 + 1], N) : 0;
    }
    __syncthreads();   // the search scratch is dead from here on (staged rows reuse it)
    if (rg >= NR || Dlo >= Dhi) return;
    // Offsets of the segment that crosses each cut, and adoption: a segment
    // that crosses just one cut with at most RW_ADOPT rows before it is taken
    // whole by the range that holds its end (which starts at the segment's
    // first row; the range before it stops there), so it needs no partial
    // and no ticket.  Both sides decide it from the same cut and offsets.
    if (!small) {
        off_Iu = clamp_off(__ldg(&offs[Iu]), N);
        off_Iu1 = Iu < S ? clamp_off(__ldg(&offs[Iu + 1]), N) : 0;
        off_Iu2 = Iu2 < S ? clamp_off(__ldg(&offs[Iu2]), N) : 0;
        off_Iu21 = Iu2 < S ? clamp_off(__ldg(&offs[Iu2 + 1]), N) : 0;
    }
    bool adopt_head = false, give_tail = false;
    if (Iu < Iu2 && off_Iu < Rc && Rc - off_Iu <= RW_ADOPT && rg > 0)
        adopt_head = (off_Iu - o0 + CW * Iu) / Wr == rg - 1;
    if (Iu2 < S && off_Iu2 < Rc2 && Rc2 - off_Iu2 <= RW_ADOPT) {
        const int64_t f = off_Iu2 - o0 + CW * Iu2;
        const int64_t e = (off_Iu21 > off_Iu2 ? off_Iu21 : off_Iu2) - o0 + CW * Iu2;
        give_tail = f / Wr == rg && e / Wr == rg + 1;
    }
    const int64_t Ru = adopt_head ? off_Iu : Rc;
    const int64_t Ru2 = give_tail ? (off_Iu2 > Ru ? off_Iu2 : Ru) : Rc2;

    // ---- per-warp state ----------------------------------------------------------
    const int c0 = slice * SLW + lane * VEC;   // my first column
    const bool active = c0 < F;
    const int32_t nR = static_cast<int32_t>(Ru2 - Ru);
    const uint64_t pol = policy_evict_first();
    const uint32_t* vp = static_cast<const uint32_t*>(p.values) + Ru * F + (active ? c0 : 0);
    T* out = static_cast<T*>(p.out);
    uint32_t* pv = static_cast<uint32_t*>(p.ws_parts);             // [2U][SLW] partial values
    int64_t* pr = reinterpret_cast<int64_t*>(pv + 2 * U * SLW);     // [2U][SLW] partial rows
    const int mean = p.mean;
    const bool want_arg = (OP != OP_SUM) && p.out_arg != nullptr;
    // one VEC-wide store per lane where the output rows allow it (every
    // lane's first column is then a multiple of VEC)
    const bool vec_out = VEC > 1 && F % VEC == 0 && reinterpret_cast<uintptr_t>(p.out) % (4 * VEC) == 0;
    const bool vec_arg = VEC > 1 && F % 2 == 0 && reinterpret_cast<uintptr_t>(p.out_arg) % 16 == 0;

    // register ring: xb[d] holds row r0 + d
    uint32_t xb[PD][VEC];
#pragma unroll
    for (int d = 0; d < PD; ++d) {
#pragma unroll
        for (int v = 0; v < VEC; ++v) xb[d][v] = 0u;
        if (!STAGED && active && d < nR) ld_stream<VEC>(xb[d], vp + static_cast<int64_t>(d) * F, pol);
    }

    // an absolute offset as a row relative to Ru, clamped to [-1, nR + 1]
    auto rel = [&](int64_t x) -> int32_t {
        x -= Ru;
        return static_cast<int32_t>(x < -1 ? -1 : (x > nR + 1 ? nR + 1 : x));
    };
    // segment ends: lane l holds E of segment eb + l (current window) and
    // of eb + 32 + l (next window, loading)
    int64_t eb = Iu;
    int32_t EB = eb + lane < Iu2 ? rel(__ldg(&offs[eb + lane + 1])) : INT32_MAX;
    int32_t EN = eb + 32 + lane < Iu2 ? rel(__ldg(&offs[eb + 32 + lane + 1])) : INT32_MAX;
    int k = 0;
    int32_t ecur = __shfl_sync(FULL, EB, 0);
    int64_t s = Iu;
    bool head_pending = Iu < S && off_Iu < Ru;
    int32_t bst = rel(off_Iu);   // start of segment s

    // accumulators for my VEC columns
    T acc[VEC];
    int32_t arow[VEC];     // min / max: row relative to Ru, -1 = none yet
    float blk[VEC];        // float sums: the current block of rows
    CarryF2 car[VEC];      // float sums: everything before the block
#pragma unroll
    for (int v = 0; v < VEC; ++v) {
        acc[v] = T(0);
        arow[v] = -1;
        blk[v] = 0.0f;
        car[v] = CarryF2{0.0f, 0.0f};
    }
    auto reset = [&]() {
#pragma unroll
        for (int v = 0; v < VEC; ++v) {
            acc[v] = T(0);
            arow[v] = -1;
            blk[v] = 0.0f;
            car[v] = CarryF2{0.0f, 0.0f};
        }
    };
    // my partial of the current segment, as stored in scratch
    auto part_bits = [&](int v) -> uint32_t {
        if constexpr (kFloatSum) {
            const CarryF2 c = two_sum_add(car[v], blk[v]);
            return __float_as_uint(c.hi + c.lo);
        } else {
            return bits_of(acc[v]);
        }
    };
    auto write_part = [&](int64_t slot) {   // slot: unit index in [0, 2U)
        if (!active) return;
        const int64_t at = slot * SLW + lane * VEC;
#pragma unroll
        for (int v = 0; v < VEC; ++v) {
            pv[at + v] = part_bits(v);
            if constexpr (OP != OP_SUM) pr[at + v] = arow[v] >= 0 ? Ru + arow[v] : -1;
        }
    };
    // The head segment (begun in an earlier range) goes to scratch as soon as
    // it ends; its ticket is taken outside the row loop.
    bool head_saved = false;
    // finish segment s, which ends at row e (relative), and move to s + 1
    auto emit = [&](int32_t e) {
        if (head_pending && s == Iu) {
            write_part(U + u_me);
            head_saved = true;
            head_pending = false;
        } else if (active) {
            const int32_t len = e > bst ? e - bst : 0;
            uint32_t r[VEC];
            int64_t a[VEC];
#pragma unroll
            for (int v = 0; v < VEC; ++v) {
                a[v] = -1;
                if constexpr (kFloatSum) {
                    const CarryF2 c = two_sum_add(car[v], blk[v]);
                    const float f = c.hi + c.lo;
                    r[v] = __float_as_uint(mean ? (len > 0 ? f / static_cast<float>(len) : 0.0f) : f);
                } else if constexpr (OP == OP_SUM) {
                    r[v] = bits_of(acc[v]);
                } else {
                    r[v] = bits_of(arow[v] >= 0 ? acc[v] : T(0));
                    a[v] = arow[v] >= 0 ? Ru + arow[v] : -1;
                }
            }
            store_cols<VEC>(reinterpret_cast<uint32_t*>(out) + s * F + c0, r, vec_out);
            if (want_arg) store_args<VEC>(p.out_arg + s * F + c0, a, vec_arg);
        }
        reset();
        bst = e;
        ++s;
        if (++k == 32) {
            EB = EN;
            eb += 32;
            EN = eb + 32 + lane < Iu2 ? rel(__ldg(&offs[eb + 32 + lane + 1])) : INT32_MAX;
            k = 0;
        }
        ecur = __shfl_sync(FULL, EB, k);
    };
    // the head's ticket (its partial is out); the answer is read when the
    // range is done, so the atomic's latency hides behind the rows
    bool head_taken = false;
    unsigned long long head_ticket = 0;   // lane 0
    auto head_flush = [&]() {
        __threadfence();
        __syncwarp();   // every lane's partial is out before the ticket
        if (lane == 0) head_ticket = ticket_take(p.ws_tickets, static_cast<int>(u_me), p.gen);
        head_taken = true;
        head_saved = false;
    };
    // fold row r (relative), whose VEC elements are x
    auto add_row = [&](const uint32_t (&x)[VEC], int32_t r) {
#pragma unroll
        for (int v = 0; v < VEC; ++v) {
            const T xv = from_bits<T>(x[v]);
            if constexpr (kFloatSum) {
                blk[v] += xv;
            } else if constexpr (OP == OP_SUM) {
                acc[v] = add_wrap(acc[v], xv);
            } else {
                const bool better = (OP == OP_MIN) ? (xv < acc[v]) : (xv > acc[v]);
                if (arow[v] < 0 || better) {
                    acc[v] = xv;
                    arow[v] = r;
                }
            }
        }
    };
    // the same once the segment has a row (min / max: no "first row" test,
    // one compare and two selects per element)
    auto add_row_seen = [&](const uint32_t (&x)[VEC], int32_t r) {
        if constexpr (OP == OP_SUM) {
            add_row(x, r);
        } else {
#pragma unroll
            for (int v = 0; v < VEC; ++v) {
                const T xv = from_bits<T>(x[v]);
                const bool better = (OP == OP_MIN) ? (xv < acc[v]) : (xv > acc[v]);
                acc[v] = better ? xv : acc[v];
                arow[v] = better ? r : arow[v];
            }
        }
    };
    // register ring: row r is the value loaded PD rows ago; then load row r + PD
    auto take_row = [&](int d, int32_t r) {
        uint32_t x[VEC];
#pragma unroll
        for (int v = 0; v < VEC; ++v) x[v] = xb[d][v];
        if (active && r + PD < nR) ld_stream<VEC>(xb[d], vp + static_cast<int64_t>(r + PD) * F, pol);
        add_row(x, r);
    };
    auto fold_block = [&]() {
        if constexpr (kFloatSum) {
#pragma unroll
            for (int v = 0; v < VEC; ++v) {
                car[v] = two_sum_add(car[v], blk[v]);
                blk[v] = 0.0f;
            }
        }
    };

    if constexpr (STAGED) {
        // Rows of 16-byte multiples, one column slice: the range is one
        // contiguous byte run, streamed in chunks of RPC whole rows through
        // RW_NSR stages of this warp's shared memory by 1-D bulk copies (lane
        // 0 issues).  An L2 prefetch further ahead measured slower here: the
        // copies already keep enough bytes in flight.
        const uint32_t rowb = static_cast<uint32_t>(F) * 4;
        const int32_t RPC = static_cast<int32_t>(RW_CB / rowb);
        unsigned char* ring = smem + warp * (RW_NSR * RW_CB);
        uint64_t* bars = reinterpret_cast<uint64_t*>(smem + RW_NW * RW_NSR * RW_CB) + warp * RW_NSR;
        const int64_t nch = (nR + RPC - 1) / RPC;
        const uint64_t src0 = reinterpret_cast<uint64_t>(p.values) + static_cast<uint64_t>(Ru) * rowb;
        auto chunk_bytes = [&](int64_t k) -> uint32_t {
            const int64_t rb = k * RPC;
            const int64_t re = rb + RPC < nR ? rb + RPC : nR;
            return static_cast<uint32_t>((re - rb) * rowb);
        };
        auto issue = [&](int64_t k) {   // lane 0
            uint64_t* bar = &bars[k % RW_NSR];
            const uint32_t nb = chunk_bytes(k);
            mbar_arrive_expect_tx(bar, nb);
            bulk_load(ring + (k % RW_NSR) * RW_CB, reinterpret_cast<const void*>(src0 + k * RPC * rowb), nb, bar,
                      pol);
        };
        if (lane == 0) {
            for (int k = 0; k < RW_NSR; ++k) mbar_init(&bars[k], 1);
            fence_mbarrier_init();
            for (int64_t k = 0; k < RW_NSR && k < nch; ++k) issue(k);
        }
        __syncwarp();
        int64_t k = 0;
        bool ok = true;
        for (; k < nch; ++k) {
            ok = __all_sync(FULL, wait_bounded(&bars[k % RW_NSR], static_cast<uint32_t>((k / RW_NSR) & 1),
                                               p.status, STATUS_CONSUMER_TIMEOUT));
            if (!ok) break;
            const int32_t rb = static_cast<int32_t>(k * RPC);
            const int32_t re = rb + RPC < nR ? rb + RPC : nR;
            const unsigned char* st = ring + (k % RW_NSR) * RW_CB + lane * VEC * 4;   // row rb, my columns
            auto lrow = [&](int32_t r, uint32_t (&x)[VEC]) {
                const unsigned char* q = st + static_cast<uint32_t>(r - rb) * rowb;
                if constexpr (VEC == 4) {
                    const uint4 w = *reinterpret_cast<const uint4*>(q);
                    x[0] = w.x, x[1] = w.y, x[2] = w.z, x[3] = w.w;
                } else if constexpr (VEC == 2) {
                    const uint2 w = *reinterpret_cast<const uint2*>(q);
                    x[0] = w.x, x[1] = w.y;
                } else {
                    x[0] = *reinterpret_cast<const uint32_t*>(q);
                }
            };
            auto srow = [&](int32_t r) {
                uint32_t x[VEC];
                lrow(r, x);
                add_row(x, r);
            };
            for (int32_t r1 = rb; r1 < re; r1 += 32) {
                const int32_t r2 = r1 + 32 < re ? r1 + 32 : re;
                if (ecur >= r2 || s >= Iu2) {
                    if (active) {
                        // no segment ends in these rows: after the segment's
                        // first row (all lanes alike) the plain compare suffices
                        int32_t r = r1;
                        if (OP != OP_SUM && arow[0] < 0) srow(r++);
#pragma unroll 8
                        for (; r < r2; ++r) {
                            uint32_t x[VEC];
                            lrow(r, x);
                            add_row_seen(x, r);
                        }
                    }
                } else {
#pragma unroll 2
                    for (int32_t r = r1; r < r2; ++r) {
                        while (ecur <= r && s < Iu2) emit(ecur);
                        if (active) srow(r);
                    }
                    if (head_saved) head_flush();
                }
                fold_block();
            }
            __syncwarp();   // every lane is done with the stage before it is refilled
            if (lane == 0 && k + RW_NSR < nch) issue(k + RW_NSR);
        }
        if (!ok) {
            // a wait ran out (recorded in the status word): let every copy land, then stop
            if (lane == 0)
                for (int64_t j = k; j < nch && j < k + RW_NSR; ++j)
                    wait_bounded(&bars[j % RW_NSR], static_cast<uint32_t>((j / RW_NSR) & 1), p.status,
                                 STATUS_DRAIN_TIMEOUT);
            return;
        }
    } else {
    // L2 prefetch: lane d asks for row r + d of the block RW_PFB blocks ahead,
    // the bytes of my slice rounded out to 16 bytes inside the buffer
    const uint64_t vbase = reinterpret_cast<uint64_t>(p.values);
    const uint64_t vTA = (vbase + 15) & ~uint64_t(15);
    const uint64_t vTE = (vbase + static_cast<uint64_t>(N) * F * 4) & ~uint64_t(15);
    const int ncol = F - slice * SLW < SLW ? F - slice * SLW : SLW;
    auto prefetch_row = [&](int32_t r) {
        if (r >= nR) return;
        const uint64_t a = vbase + (static_cast<uint64_t>(Ru + r) * F + slice * SLW) * 4;
        uint64_t lo = a & ~uint64_t(15);
        uint64_t hi = (a + static_cast<uint64_t>(ncol) * 4 + 15) & ~uint64_t(15);
        lo = lo < vTA ? vTA : lo;
        hi = hi > vTE ? vTE : hi;
        if (hi > lo) bulk_prefetch_l2(reinterpret_cast<const void*>(lo), static_cast<uint32_t>(hi - lo));
    };
    constexpr int RW_PFB = 4;   // blocks of PD rows prefetched ahead
#pragma unroll 1
    for (int b = 1; b <= RW_PFB; ++b)
        if (lane < PD) prefetch_row(b * PD + lane);

    for (int32_t r0 = 0; r0 < nR; r0 += PD) {
        if (lane < PD) prefetch_row(r0 + (RW_PFB + 1) * PD + lane);
        if (ecur >= r0 + PD || s >= Iu2) {
            // no segment ends inside this block of rows
            if (r0 + PD <= nR) {
#pragma unroll
                for (int d = 0; d < PD; ++d) take_row(d, r0 + d);
            } else {
#pragma unroll
                for (int d = 0; d < PD; ++d)
                    if (r0 + d < nR) take_row(d, r0 + d);
            }
        } else {
#pragma unroll
            for (int d = 0; d < PD; ++d) {
                const int32_t r = r0 + d;
                if (r < nR) {
                    while (ecur <= r && s < Iu2) emit(ecur);
                    take_row(d, r);
                }
            }
            if (head_saved) head_flush();
        }
        fold_block();   // the block of PD rows into the compensated pair
    }
    }
    // segments that end at the range's last row (and, for malformed offsets, any left)
    while (s < Iu2) emit(ecur < nR ? ecur : nR);
    if (head_saved) head_flush();

    // ---- the segment still open at the end of the range ---------------------------
    // Its partial and ticket go out first; while that atomic is in flight the
    // head ticket is read, and its segment combined if this range came last.
    bool tail_taken = false;
    unsigned long long tail_ticket = 0;
    int64_t tpc = 0, tqc = 0, tob = 0;
    if (Iu2 < S) {
        tob = off_Iu2;
        if (tob < Ru2) {
            write_part(u_me);
            __threadfence();
            __syncwarp();   // every lane's partial is out before the ticket
            if (lane == 0) {
                const int64_t oe = off_Iu21;
                const int64_t f = tob - o0 + CW * Iu2;
                const int64_t e = (oe > tob ? oe : tob) - o0 + CW * Iu2;
                tpc = f / Wr;
                tqc = e / Wr;
                tpc = tpc < 0 ? 0 : (tpc > rg ? rg : tpc);
                tqc = tqc <= rg ? rg + 1 : tqc;
                if (tqc < NR) tail_ticket = ticket_take(p.ws_tickets, static_cast<int>(tqc * NSL + slice), p.gen);
            }
            tpc = __shfl_sync(FULL, tpc, 0);
            tqc = __shfl_sync(FULL, tqc, 0);
            tail_taken = tqc < NR;
        }
    }
    if (head_taken) {
        int64_t pc = (off_Iu - o0 + CW * Iu) / Wr;
        pc = pc < 0 ? 0 : (pc > rg ? rg : pc);
        const bool last =
            __shfl_sync(FULL, lane == 0 && ticket_last(head_ticket, p.gen, static_cast<int>(rg - pc + 1)), 0);
        if (last) {
            fence_acq_rel_gpu();
            rows_combine_store<T, OP, VEC>(p, pv, pr, U, NSL, slice, pc, rg, Iu,
                                           off_Iu1 > off_Iu ? off_Iu1 - off_Iu : 0, lane);
        }
    }
    if (tail_taken) {
        const bool last =
            __shfl_sync(FULL, lane == 0 && ticket_last(tail_ticket, p.gen, static_cast<int>(tqc - tpc + 1)), 0);
        if (last) {
            fence_acq_rel_gpu();
            rows_combine_store<T, OP, VEC>(p, pv, pr, U, NSL, slice, tpc, tqc, Iu2,
                                           off_Iu21 > tob ? off_Iu21 - tob : 0, lane);
        }
    }
}

}  // namespace segred
