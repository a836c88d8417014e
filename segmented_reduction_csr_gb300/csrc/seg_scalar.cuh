// seg_scalar.cuh -- the scalar kernel: F == 1 vectors of uint32, int32 or
// float32 (GPUSegmentedReduction's "packed scalar values").
//
// Work split.  The merge path of rows and segment ends is cut into units of
// equal length, one unit per warp (SW_NW warps per CTA, one CTA per SM).  A
// CTA finds the SW_NW + 1 unit boundaries it needs with one cooperative
// search; after that every warp runs on its own: no CTA barrier in the main
// loop, so the latency of one warp's steps hides behind the others.
//
// Per warp.  Lane 0 streams the unit's rows (SW_VCHUNK-byte chunks, SW_NSV
// stages) and offsets (a SW_NSO-stage ring) into the warp's shared memory
// with 1-D bulk copies, refilling a stage as soon as the warp is done with it.
// A tile is the rows of one chunk plus the segment ends that fall in them (at
// most SW_EMAX ends; a chunk with more is split into several tiles):
//
//  1. marks: every lane takes segment ends and sets the bit of the row where
//     the next segment starts (a 20-bit word per lane), plus the tile's first row;
//  2. rows: lane l owns rows [20 l, 20 l + 20) of the chunk, loads them with
//     128-bit shared loads (the 80-byte lane stride makes them conflict free),
//     runs an inclusive segmented scan in registers (sum: restart at a mark;
//     min / max: strict compare, restart at a mark; rows arrive in order so
//     ties keep the lower row) and writes the running values back;  a
//     segmented shuffle scan over the lanes gives each lane the running value
//     of the rows before it;
//  3. ends: every lane takes a segment end; its result is the running value at
//     the segment's last row, joined with the owning lane's prefix (a shuffle)
//     when the segment started in an earlier lane, and with the warp's carry
//     when it started in an earlier tile.  Consecutive lanes store consecutive
//     segments.  The carry of the segment left open is taken the same way.
//
// A segment that crosses units leaves per-unit partials in scratch; the last
// unit to arrive (atomic ticket, no waiting) combines them in unit order with
// a lane-parallel tree, so float results are reproducible.
#pragma once
#include "seg_common.cuh"

namespace segred {

constexpr int SW_NW = 16;                      // warps (units) per CTA
constexpr int SW_NTHREADS = SW_NW * 32;
constexpr int SW_KR = 20;                      // rows per lane per tile (SW_KR / 4 odd)
constexpr int SW_TROWS = 32 * SW_KR;           // rows per value chunk
constexpr uint32_t SW_VCHUNK = SW_TROWS * 4;   // bytes per value chunk
constexpr int SW_NSV = 3;                      // value stages per warp
constexpr uint32_t SW_OCHUNK = 512;            // bytes per offsets chunk
constexpr int SW_NSO = 4;                      // offsets stages per warp
constexpr uint32_t SW_ORING = SW_OCHUNK * SW_NSO;
constexpr int SW_EMAX = 64;                    // segment ends per tile (two per lane)
constexpr int SW_NDIAG = SW_NW + 1;            // unit boundaries per CTA
constexpr int SW_GRID = 1024;                  // first-round probes, shared by all CTAs
constexpr int SW_PROBES = 60;                  // later-round probes per boundary
static_assert((SW_KR / 4) % 2 == 1, "conflict-free 128-bit row loads need SW_KR / 4 odd");
static_assert(SW_NDIAG * SW_PROBES <= 2 * SW_NTHREADS, "two probes per thread per round");
static_assert((SW_EMAX + 1) * 8 + SW_OCHUNK <= SW_ORING, "offsets ring holds a tile's window");
static_assert(SW_EMAX == 64, "each lane holds two of a tile's segment ends");

// Per-warp shared memory.
struct WarpSmem {
    static constexpr uint32_t vstage = 0;
    static constexpr uint32_t oring = SW_NSV * SW_VCHUNK;
    static constexpr uint32_t marks = oring + SW_ORING;
    static constexpr uint32_t argr = marks + 32 * 4;
    static constexpr uint32_t bars = argr + SW_TROWS * 2;
    static constexpr uint32_t bytes = ((bars + (SW_NSV + SW_NSO) * 8 + 1023) / 1024) * 1024;
};
constexpr uint32_t SW_SMEM = SW_NW * WarpSmem::bytes;

// Search scratch (aliases the warps' memory before they start).
struct SearchSmem {
    int64_t graw[SW_GRID];
    int64_t D[SW_NDIAG], lo[SW_NDIAG], hi[SW_NDIAG];
    int cnt[SW_NDIAG];
    int64_t o0, oS;
};
static_assert(sizeof(SearchSmem) <= SW_SMEM, "search scratch fits");

// Last arriver of a multi-unit segment: partials tails[pc .. qc-1] then
// heads[qc], combined by the whole warp: lane l folds a contiguous block in
// order, then lanes fold pairwise in order (a fixed tree), lane 0 stores.
template <class T, int OP>
__device__ __forceinline__ void warp_combine_store(const Params& p, const PartElem* tails,
                                                   const PartElem* heads, int pc, int qc, int64_t s,
                                                   int64_t len, int lane) {
    const int n = qc - pc + 1;
    const int per = (n + 31) / 32;
    PartElem a;
    a.v.d = 0.0;
    a.row = -1;
    bool have = false;
    for (int t = 0; t < per; ++t) {
        const int k = pc + lane * per + t;
        if (k <= qc) {
            const PartElem pe = load_part(k < qc ? &tails[k] : &heads[qc]);
            a = have ? part_comb<T, OP>(a, pe) : pe;
            have = true;
        }
    }
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        PartElem b;
        b.v.d = __longlong_as_double(__shfl_down_sync(0xffffffffu, __double_as_longlong(a.v.d), o));
        b.row = __shfl_down_sync(0xffffffffu, a.row, o);
        const bool bh = __shfl_down_sync(0xffffffffu, have, o);
        if ((lane & (2 * o - 1)) == 0 && bh) {
            a = have ? part_comb<T, OP>(a, b) : b;
            have = true;
        }
    }
    if (lane == 0) {
        T v;
        int64_t ar;
        finish_part<T, OP>(a, len, p.mean, v, ar);
        static_cast<T*>(p.out)[s] = v;
        if (OP != OP_SUM && p.out_arg != nullptr) p.out_arg[s] = ar;
    }
}

template <class T, int OP, class OffT>
__global__ void __launch_bounds__(SW_NTHREADS, 1) seg_scalar_kernel(const Params p) {
    using RD = Red<T, OP>;
    using CO = Carry<T, OP>;
    using C = typename CO::C;
    constexpr uint32_t OSZ = sizeof(OffT);

    extern __shared__ __align__(1024) unsigned char smem[];
    const int tid = threadIdx.x;
    const int lane = tid & 31;
    const int warp = tid >> 5;
    const int cta = blockIdx.x;
    const int64_t N = p.N;
    const int64_t S = p.S;
    const OffT* offs = static_cast<const OffT*>(p.offsets);
    const int64_t U = static_cast<int64_t>(p.P) * SW_NW;   // units in the grid

    // ---- a2: unit boundaries ---------------------------------------------------
    // I(D) = #{s : key(s) < D}, key(s) = (offsets[s+1] - o0) + s.  Round 1
    // reads a fixed grid of SW_GRID keys that every CTA shares (so it hits L2);
    // then each boundary narrows its bracket with SW_PROBES probes per round.
    SearchSmem* ss = reinterpret_cast<SearchSmem*>(smem);
    if (tid == 0) ss->o0 = clamp_off(__ldg(&offs[0]), N);
    if (tid == 1) ss->oS = clamp_off(__ldg(&offs[S]), N);
    for (int m = tid; m < SW_GRID; m += SW_NTHREADS) {
        const int64_t sm = static_cast<int64_t>(m) * S / SW_GRID;
        ss->graw[m] = clamp_off(__ldg(&offs[sm + 1]), N);
    }
    __syncthreads();
    const int64_t o0 = ss->o0;
    const int64_t oS = ss->oS < o0 ? o0 : ss->oS;
    const int64_t nrows = oS - o0;
    const int64_t total = nrows + S;
    const int64_t Wu = (total + U - 1) / U;
    if (tid < SW_NDIAG) {
        const int64_t u = static_cast<int64_t>(cta) * SW_NW + tid;
        const int64_t D = u * Wu < total ? u * Wu : total;
        int64_t lo = D - nrows > 0 ? D - nrows : 0;
        int64_t hi = D < S ? D : S;
        int a = 0, b = SW_GRID;   // c = #{m : key(s_m) < D}
        while (a < b) {
            const int mid = (a + b) >> 1;
            const int64_t sm = static_cast<int64_t>(mid) * S / SW_GRID;
            if (ss->graw[mid] - o0 + sm < D)
                a = mid + 1;
            else
                b = mid;
        }
        const int64_t lower = a > 0 ? static_cast<int64_t>(a - 1) * S / SW_GRID + 1 : 0;
        const int64_t upper = a < SW_GRID ? static_cast<int64_t>(a) * S / SW_GRID : S;
        lo = lo > lower ? lo : lower;
        hi = hi < upper ? hi : upper;
        if (hi < lo) hi = lo;
        ss->D[tid] = D;
        ss->lo[tid] = lo;
        ss->hi[tid] = hi;
        ss->cnt[tid] = 0;
    }
    __syncthreads();
    for (int round = 0; round < 64; ++round) {
#pragma unroll
        for (int u = 0; u < 2; ++u) {
            const int pidx = tid + u * SW_NTHREADS;
            const int k = pidx / SW_PROBES;
            const int mm = pidx - k * SW_PROBES;
            if (k < SW_NDIAG) {
                const int64_t lo = ss->lo[k], hi = ss->hi[k];
                const int64_t len = hi - lo;
                if (len > 0) {
                    const int64_t step = (len + SW_PROBES - 1) / SW_PROBES;
                    const int64_t s = lo + mm * step;
                    if (s < hi && clamp_off(__ldg(&offs[s + 1]), N) - o0 + s < ss->D[k])
                        atomicAdd(&ss->cnt[k], 1);
                }
            }
        }
        __syncthreads();
        bool open = false;
        if (tid < SW_NDIAG) {
            int64_t lo = ss->lo[tid], hi = ss->hi[tid];
            const int64_t len = hi - lo;
            if (len > 0) {
                const int64_t step = (len + SW_PROBES - 1) / SW_PROBES;
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
    // my unit: merge positions [D_w, D_w+1), ends [Iu, Iu2), rows [Ru, Ru2)
    const int64_t u_me = static_cast<int64_t>(cta) * SW_NW + warp;
    const int64_t Dlo = ss->D[warp], Dhi = ss->D[warp + 1];
    const int64_t Iu = ss->lo[warp];
    const int64_t Iu2 = ss->lo[warp + 1] > Iu ? ss->lo[warp + 1] : Iu;
    int64_t Ru = Dlo - Iu + o0;
    Ru = Ru < o0 ? o0 : (Ru > oS ? oS : Ru);
    int64_t Ru2 = Dhi - Iu2 + o0;
    Ru2 = Ru2 < Ru ? Ru : (Ru2 > oS ? oS : Ru2);
    __syncthreads();   // the search scratch is dead from here on
    if (Dlo >= Dhi) return;

    // ---- per-warp state ----------------------------------------------------------
    unsigned char* wbase = smem + warp * WarpSmem::bytes;
    unsigned char* vst = wbase + WarpSmem::vstage;
    unsigned char* oring = wbase + WarpSmem::oring;
    uint32_t* marks = reinterpret_cast<uint32_t*>(wbase + WarpSmem::marks);
    int16_t* argr = reinterpret_cast<int16_t*>(wbase + WarpSmem::argr);
    uint64_t* fv = reinterpret_cast<uint64_t*>(wbase + WarpSmem::bars);
    uint64_t* fo = fv + SW_NSV;
    T* out = static_cast<T*>(p.out);
    PartElem* tails = static_cast<PartElem*>(p.ws_parts);
    PartElem* heads = tails + U;
    const int mean = p.mean;
    const bool want_arg = (OP != OP_SUM) && p.out_arg != nullptr;

    const uint64_t vbase = reinterpret_cast<uint64_t>(p.values);
    const uint64_t obase = reinterpret_cast<uint64_t>(p.offsets);
    const Stream vs = make_stream(vbase, static_cast<uint64_t>(N) * 4, vbase + Ru * 4, vbase + Ru2 * 4,
                                  SW_VCHUNK);
    const Stream os = make_stream(obase, static_cast<uint64_t>(S + 1) * OSZ, obase + Iu * OSZ,
                                  obase + (Iu2 + 1) * OSZ, SW_OCHUNK);
    const int64_t vrow0 = static_cast<int64_t>(vs.A0 - vbase) / 4;   // row of chunk 0's first byte
    const uint64_t policy = policy_evict_first();

    marks[lane] = 0u;
    if (lane == 0) {
        for (int k = 0; k < SW_NSV + SW_NSO; ++k) mbar_init(&fv[k], 1);
        fence_mbarrier_init();
    }
    __syncwarp();
    int64_t v_issued = 0, o_issued = 0;       // lane 0's counters (kept uniform by shuffles)
    if (lane == 0) {
        for (; v_issued < SW_NSV && v_issued < vs.nch; ++v_issued)
            issue_chunk_to(vs, v_issued, SW_VCHUNK, vst + (v_issued % SW_NSV) * SW_VCHUNK,
                           &fv[v_issued % SW_NSV], policy);
        for (; o_issued < SW_NSO && o_issued < os.nch; ++o_issued)
            issue_chunk(os, o_issued, oring, SW_ORING, SW_OCHUNK, &fo[o_issued % SW_NSO], policy);
    }

    auto off_w = [&](int64_t s) -> int64_t {
        const uint32_t at = static_cast<uint32_t>((obase + static_cast<uint64_t>(s) * OSZ) - os.A0) &
                            (SW_ORING - 1);
        return clamp_off(*reinterpret_cast<const OffT*>(oring + at), N);
    };
    int64_t ow = 0, odone = 0;   // offsets chunks waited for / handed back
    bool ok = true;
    // wait until offsets entry x is in the ring (uniform across the warp)
    auto wait_offsets = [&](int64_t x) {
        const int64_t need =
            static_cast<int64_t>((obase + static_cast<uint64_t>(x + 1) * OSZ - 1 - os.A0) / SW_OCHUNK);
        if (ow <= need && ow < os.nch) {
            if (lane == 0)
                for (; ok && ow <= need && ow < os.nch; ++ow)
                    ok = wait_bounded(&fo[ow % SW_NSO], static_cast<uint32_t>((ow / SW_NSO) & 1), p.status,
                                      STATUS_CONSUMER_TIMEOUT);
            ok = __shfl_sync(0xffffffffu, ok, 0);
            ow = __shfl_sync(0xffffffffu, ow, 0);
            __syncwarp();
        }
    };

    C carry = CO::ident();
    const int64_t off_Iu = clamp_off(__ldg(&offs[Iu]), N);
    bool head_pending = (Iu < S) && off_Iu < Ru;
    int64_t m = 0;            // current value chunk
    bool m_ready = false;
    int64_t es = Iu;          // next segment end
    int64_t b_es = off_Iu;    // offsets[es]
    int64_t j = Ru;           // next row

    while (ok) {
        const bool lastc = m + 1 >= vs.nch;
        const int64_t crow0 = vrow0 + m * SW_TROWS;
        const int64_t rl = lastc ? Ru2 : (crow0 + SW_TROWS < Ru2 ? crow0 + SW_TROWS : Ru2);
        if (m < vs.nch && !m_ready) {
            if (lane == 0)
                ok = wait_bounded(&fv[m % SW_NSV], static_cast<uint32_t>((m / SW_NSV) & 1), p.status,
                                  STATUS_CONSUMER_TIMEOUT);
            ok = __shfl_sync(0xffffffffu, ok, 0);
            __syncwarp();
            m_ready = true;
            if (!ok) break;
        }
        const int64_t rem = Iu2 - es;
        const int ncand = static_cast<int>(rem < SW_EMAX ? rem : SW_EMAX);
        wait_offsets(es + ncand);
        if (!ok) break;
        // Lane l holds ends es + l and es + 32 + l: E = offsets[s + 1] (the
        // segment's end, which is the next segment's start), B = offsets[s].
        int64_t E[2], B[2];
        bool have[2];
#pragma unroll
        for (int k = 0; k < 2; ++k) {
            const int idx = 32 * k + lane;
            have[k] = idx < ncand;
            E[k] = have[k] ? off_w(es + idx + 1) : INT64_MAX;
        }
        {
            const int64_t up0 = __shfl_up_sync(0xffffffffu, E[0], 1);
            const int64_t up1 = __shfl_up_sync(0xffffffffu, E[1], 1);
            const int64_t last0 = __shfl_sync(0xffffffffu, E[0], 31);
            B[0] = lane == 0 ? b_es : up0;
            B[1] = lane == 0 ? last0 : up1;
        }
        // ends of this tile: a prefix of those whose segment ends by row rl
        // (all of them on the unit's last chunk)
        int n_e = ncand;
        if (!lastc) {
            const unsigned b0 = __ballot_sync(0xffffffffu, have[0] && E[0] <= rl);
            int run = b0 == 0xffffffffu ? 32 : __ffs(~b0) - 1;
            if (run == 32) {
                const unsigned b1 = __ballot_sync(0xffffffffu, have[1] && E[1] <= rl);
                run += b1 == 0xffffffffu ? 32 : __ffs(~b1) - 1;
            }
            n_e = run < ncand ? run : ncand;
        }
        int64_t tr1 = rl;
        if (n_e == SW_EMAX && es + n_e < Iu2) {
            const int64_t x = __shfl_sync(0xffffffffu, E[1], 31);   // rows up to the last included end
            tr1 = x < j ? j : (x > rl ? rl : x);
        }
        if (n_e == 0 && j >= tr1) {
            // nothing left in this chunk
            if (lastc) break;
            __syncwarp();
            if (lane == 0 && v_issued < vs.nch) {
                issue_chunk_to(vs, v_issued, SW_VCHUNK, vst + (v_issued % SW_NSV) * SW_VCHUNK,
                               &fv[v_issued % SW_NSV], policy);
                ++v_issued;
            }
            ++m;
            m_ready = false;
            continue;
        }

        // ---- one tile: rows [j, tr1) of chunk m, ends [es, es + n_e) ----------------
        unsigned char* stage = vst + (m % SW_NSV) * SW_VCHUNK;
        const int32_t jr = static_cast<int32_t>(j - crow0);       // rows relative to the chunk
        const int32_t tr = static_cast<int32_t>(tr1 - crow0);
        const bool has_rows = tr1 > j && m < vs.nch;
        const int32_t crow_u = static_cast<int32_t>(crow0 - Ru);  // chunk row 0, relative to the unit
        Acc<T> X = RD::ident();   // running value of the rows before my lane's rows
        if (has_rows) {
            // 1. marks: the segment after each of this tile's ends starts at its E
#pragma unroll
            for (int k = 0; k < 2; ++k) {
                if (32 * k + lane < n_e && E[k] >= j && E[k] < tr1) {
                    const int32_t rr = static_cast<int32_t>(E[k] - crow0);
                    atomicOr(&marks[rr / SW_KR], 1u << (rr % SW_KR));
                }
            }
            if (lane == 0) atomicOr(&marks[jr / SW_KR], 1u << (jr % SW_KR));
            __syncwarp();
            // 2. rows
            const uint32_t w = marks[lane];
            marks[lane] = 0u;
            uint32_t xb[SW_KR];
#pragma unroll
            for (int q = 0; q < SW_KR / 4; ++q) {
                const uint4 u4 = *reinterpret_cast<const uint4*>(stage + lane * (SW_KR * 4) + 16 * q);
                xb[4 * q + 0] = u4.x;
                xb[4 * q + 1] = u4.y;
                xb[4 * q + 2] = u4.z;
                xb[4 * q + 3] = u4.w;
            }
            const int32_t lrow0 = lane * SW_KR;              // my first row, relative to the chunk
            Acc<T> acc = RD::ident();
            int16_t rr[OP == OP_SUM ? 1 : SW_KR];
#pragma unroll
            for (int k = 0; k < SW_KR; ++k) {
                const T x = from_bits<T>(xb[k]);
                const bool reset = (w >> k) & 1u;
                if constexpr (OP == OP_SUM) {
                    acc.v = reset ? x : add_wrap(acc.v, x);
                } else {
                    const bool better = (OP == OP_MIN) ? (x < acc.v) : (x > acc.v);
                    if (reset || acc.row < 0 || better) {
                        acc.v = x;
                        acc.row = crow_u + lrow0 + k;
                    }
                    rr[k] = static_cast<int16_t>(acc.row - crow_u);
                }
                xb[k] = bits_of(acc.v);
            }
            // write the running values back over rows < tr1 (later rows are the
            // next tile's input; earlier rows are finished)
            const int32_t hi = tr - lrow0;
            if (hi >= SW_KR) {
#pragma unroll
                for (int q = 0; q < SW_KR / 4; ++q)
                    *reinterpret_cast<uint4*>(stage + lane * (SW_KR * 4) + 16 * q) =
                        make_uint4(xb[4 * q], xb[4 * q + 1], xb[4 * q + 2], xb[4 * q + 3]);
                if constexpr (OP != OP_SUM) {
#pragma unroll
                    for (int q = 0; q < SW_KR / 2; ++q)
                        *reinterpret_cast<uint32_t*>(&argr[lrow0 + 2 * q]) =
                            (static_cast<uint32_t>(static_cast<uint16_t>(rr[2 * q + 1])) << 16) |
                            static_cast<uint16_t>(rr[2 * q]);
                }
            } else if (hi > 0) {
#pragma unroll
                for (int k = 0; k < SW_KR; ++k) {
                    if (k < hi) {
                        *reinterpret_cast<uint32_t*>(stage + (lrow0 + k) * 4) = xb[k];
                        if constexpr (OP != OP_SUM) argr[lrow0 + k] = rr[k];
                    }
                }
            }
            // segmented scan of the lane totals; X = exclusive prefix
            Acc<T> inc = acc;
            bool fi = w != 0u;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                Acc<T> pv;
                pv.v = from_bits<T>(__shfl_up_sync(0xffffffffu, bits_of(inc.v), o));
                if constexpr (OP != OP_SUM) pv.row = __shfl_up_sync(0xffffffffu, inc.row, o);
                else pv.row = -1;
                const bool pf = __shfl_up_sync(0xffffffffu, fi, o);
                if (lane >= o) {
                    if (!fi) inc = RD::comb(pv, inc);
                    fi = fi || pf;
                }
            }
            X.v = from_bits<T>(__shfl_up_sync(0xffffffffu, bits_of(inc.v), 1));
            if constexpr (OP != OP_SUM) X.row = __shfl_up_sync(0xffffffffu, inc.row, 1);
            if (lane == 0) X = RD::ident();
            __syncwarp();
        }
        // running value at chunk row `k` (jr <= k < tr) of the run starting at
        // chunk row `st`: the lane's running value there, joined with the owning
        // lane's prefix when the run began in an earlier lane (every lane calls
        // this together: it shuffles)
        auto running_at = [&](int32_t k, int32_t st) -> Acc<T> {
            if (!has_rows) return RD::ident();   // uniform across the warp
            k = k < jr ? jr : (k >= tr ? tr - 1 : k);
            const int o = k / SW_KR;
            Acc<T> Xo;
            Xo.v = from_bits<T>(__shfl_sync(0xffffffffu, bits_of(X.v), o));
            if constexpr (OP != OP_SUM) Xo.row = __shfl_sync(0xffffffffu, X.row, o);
            else Xo.row = -1;
            Acc<T> P;
            P.v = *reinterpret_cast<const T*>(stage + k * 4);
            if constexpr (OP == OP_SUM) {
                P.row = -1;
            } else {
                P.row = static_cast<int32_t>(argr[k]) + crow_u;
            }
            return st < o * SW_KR ? RD::comb(Xo, P) : P;
        };
        // 3. ends
#pragma unroll
        for (int k = 0; k < 2; ++k) {
            if (k == 1 && n_e <= 32) break;
            const int idx = 32 * k + lane;
            const bool valid = idx < n_e;
            const int64_t s = es + idx;
            const int64_t ob = valid ? B[k] : j;
            const int64_t oe = valid ? E[k] : j;
            const bool rows_here = valid && has_rows && oe > ob && oe - 1 >= j;
            const int32_t kl = rows_here ? static_cast<int32_t>(oe - 1 - crow0) : jr;
            const int32_t st = static_cast<int32_t>((ob > j ? ob : j) - crow0);
            const Acc<T> P = running_at(kl, st);
            const int64_t len = oe > ob ? oe - ob : 0;
            bool last = false;
            int pc = 0;
            if (valid) {
                if (head_pending && s == Iu) {
                    // began in an earlier unit: leave the head partial, join the ticket
                    const C R = rows_here ? CO::then(carry, P) : carry;
                    if constexpr (OP == OP_SUM && kIsFloat<T>) heads[u_me] = to_part(R);
                    else heads[u_me] = to_part<T, OP>(R, Ru);
                    __threadfence();
                    const int64_t f = ob - o0 + Iu;
                    pc = static_cast<int>(f / Wu);
                    pc = pc < 0 ? 0 : (pc > u_me ? static_cast<int>(u_me) : pc);
                    last = ticket_arrive(p.ws_tickets, static_cast<int>(u_me),
                                         static_cast<int>(u_me) - pc + 1, p.gen);
                    if (last) __threadfence();
                } else {
                    T v;
                    int64_t a;
                    if (len == 0) {
                        v = T(0);
                        a = -1;
                    } else if (ob >= j) {
                        finish_acc<T, OP>(P, len, mean, Ru, v, a);   // began in this tile
                    } else {
                        const C R = rows_here ? CO::then(carry, P) : carry;
                        if constexpr (OP == OP_SUM && kIsFloat<T>) {
                            finish_carry(R, len, mean, v);
                            a = -1;
                        } else {
                            finish_acc<T, OP>(R, len, mean, Ru, v, a);
                        }
                    }
                    out[s] = v;
                    if (want_arg) p.out_arg[s] = a;
                }
            }
            if (head_pending && k == 0) {
                // the unit's first end sat on lane 0
                last = __shfl_sync(0xffffffffu, last, 0);
                pc = __shfl_sync(0xffffffffu, pc, 0);
                const int64_t hl = __shfl_sync(0xffffffffu, len, 0);
                if (last)
                    warp_combine_store<T, OP>(p, tails, heads, pc, static_cast<int>(u_me), Iu, hl, lane);
            }
        }
        if (n_e > 0) head_pending = false;
        // the segment left open, es + n_e, starts at offsets[es + n_e]
        {
            const int l = (n_e - 1) & 31;
            const int64_t e0 = __shfl_sync(0xffffffffu, E[0], l);
            const int64_t e1 = __shfl_sync(0xffffffffu, E[1], l);
            const int64_t bo = n_e == 0 ? b_es : (n_e <= 32 ? e0 : e1);
            const int64_t sto = bo > j ? bo : j;
            const bool rows_open = has_rows && sto < tr1;
            const Acc<T> P = running_at(tr - 1, static_cast<int32_t>(sto - crow0));
            if (rows_open)
                carry = bo < j ? CO::then(carry, P) : CO::from(P);
            else if (!(bo < j))
                carry = CO::ident();
            b_es = bo;
        }
        j = tr1;
        es += n_e;
        __syncwarp();
        // hand back offsets chunks that hold only entries before es
        if (lane == 0) {
            while (odone < ow && os.A0 + static_cast<uint64_t>(odone + 1) * SW_OCHUNK <=
                                     obase + static_cast<uint64_t>(es) * OSZ) {
                if (o_issued < os.nch) {
                    issue_chunk(os, o_issued, oring, SW_ORING, SW_OCHUNK, &fo[o_issued % SW_NSO], policy);
                    ++o_issued;
                }
                ++odone;
            }
        }
        odone = __shfl_sync(0xffffffffu, odone, 0);
        o_issued = __shfl_sync(0xffffffffu, o_issued, 0);
    }
    v_issued = __shfl_sync(0xffffffffu, v_issued, 0);

    // ---- a6: the segment still open at the end of the unit -------------------------
    if (ok && Iu2 < S) {
        const int64_t ob = clamp_off(__ldg(&offs[Iu2]), N);
        if (ob < Ru2) {
            bool last = false;
            int pc = 0, qc = 0;
            if (lane == 0) {
                if constexpr (OP == OP_SUM && kIsFloat<T>) tails[u_me] = to_part(carry);
                else tails[u_me] = to_part<T, OP>(carry, Ru);
                __threadfence();
                const int64_t oe = clamp_off(__ldg(&offs[Iu2 + 1]), N);
                const int64_t f = ob - o0 + Iu2;
                const int64_t e = (oe > ob ? oe : ob) - o0 + Iu2;
                pc = static_cast<int>(f / Wu);
                qc = static_cast<int>(e / Wu);
                pc = pc < 0 ? 0 : (pc > u_me ? static_cast<int>(u_me) : pc);
                qc = qc <= u_me ? static_cast<int>(u_me) + 1 : qc;
                last = qc < U && ticket_arrive(p.ws_tickets, qc, qc - pc + 1, p.gen);
                if (last) __threadfence();
            }
            last = __shfl_sync(0xffffffffu, last, 0);
            pc = __shfl_sync(0xffffffffu, pc, 0);
            qc = __shfl_sync(0xffffffffu, qc, 0);
            if (last) {
                const int64_t oe = clamp_off(__ldg(&offs[Iu2 + 1]), N);
                warp_combine_store<T, OP>(p, tails, heads, pc, qc, Iu2, oe > ob ? oe - ob : 0, lane);
            }
        }
    }
    // every copy this warp started must land before it exits
    if (lane == 0) {
        for (int64_t k = m + (m_ready ? 1 : 0); k < v_issued; ++k)
            wait_bounded(&fv[k % SW_NSV], static_cast<uint32_t>((k / SW_NSV) & 1), p.status,
                         STATUS_DRAIN_TIMEOUT);
        for (int64_t k = ow; k < o_issued; ++k)
            wait_bounded(&fo[k % SW_NSO], static_cast<uint32_t>((k / SW_NSO) & 1), p.status,
                         STATUS_DRAIN_TIMEOUT);
    }
}

}  // namespace segred
