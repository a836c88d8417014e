// seg_scalar.cuh -- the scalar kernel: F == 1 vectors of uint32, int32 or
// float32 (GPUSegmentedReduction's "packed scalar values").
//
// Work split.  Rows and segment ends form one merged sequence in which a row
// weighs 1 and a segment end weighs SW_CW (an end costs about that many rows
// of work: its offsets load, its lookup and its store).  The sequence is cut
// into units of equal weight, one unit per warp (SW_NW warps per CTA, one CTA
// per SM), so skewed length distributions balance.  A CTA finds the SW_NW + 1
// unit boundaries it needs with one cooperative search; after that every warp
// runs on its own: no CTA barrier in the main loop.
//
// Per warp.  Lane 0 streams the unit's rows (SW_VCHUNK-byte chunks, SW_NSV
// stages) into the warp's shared memory with 1-D bulk copies, refilling a
// stage as soon as the warp is done with it.  The segment ends of the next
// tile are copied by every lane (per-thread async copies, one entry each)
// into the other half of a double buffer while the current tile runs.
// A tile is the rows of one chunk plus the segment ends that fall in them (up
// to SW_EMAXT ends; a chunk with more, which takes many empty segments, is
// split into several tiles):
//
//  * a chunk that no segment end touches is summed as a whole: every lane
//    folds its rows, then a fixed butterfly over the lanes;
//  * otherwise: start flags (a byte per row: the tile's first row and, for
//    each segment end, the row where the next segment starts); an inclusive
//    segmented scan of each lane's SW_KR rows, a quad at a time (128-bit
//    shared loads; the 144-byte lane stride keeps them conflict free), with
//    the running values written back over the rows; a segmented shuffle scan
//    of the lane totals, whose exclusive prefixes go to shared memory.  Then
//    lanes take 32 segment ends at a time: the running value at the segment's last row,
//    joined with the owning lane's prefix when the segment started in an
//    earlier lane, and with the warp's carry when it started in an earlier
//    tile.  Consecutive lanes store consecutive segments.
//
// The carry of the segment left open at a tile's end is kept by every lane;
// float sums carry a compensated pair (TwoSum), so long chains of tiles add
// no float32 error.  Rows are int32 offsets from the unit's first row (the
// planner keeps a unit below 2^31 rows).
//
// A segment that crosses units leaves per-unit partials in scratch; the last
// unit to arrive (atomic ticket, no waiting) combines them in unit order with
// a lane-parallel tree, so float results are reproducible.
#pragma once
#include "seg_common.cuh"

namespace segred {

constexpr int SW_NW = 16;                      // warps (units) per CTA
constexpr int SW_NTHREADS = SW_NW * 32;
constexpr int SW_CW = 24;                      // merge-path weight of a segment end, in rows
constexpr int SW_KR = 36;                      // rows per lane per tile
constexpr int SW_Q = SW_KR / 4;                // quads per lane
constexpr int SW_TROWS = 32 * SW_KR;           // rows per value chunk
constexpr uint32_t SW_VCHUNK = SW_TROWS * 4;   // bytes per value chunk
constexpr int SW_NSV = 2;                      // value stages per warp
constexpr int SW_EMAXT = 160;                  // segment ends per tile
constexpr int64_t SW_ADOPT = 1152;             // rows of a cut-crossing segment a unit adopts
constexpr int SW_NDIAG = SW_NW + 1;            // unit boundaries per CTA
constexpr int SW_GRID = 512;                   // first-round probes, shared by all CTAs
constexpr int SW_PROBES = 60;                  // later-round probes per boundary
static_assert(SW_Q % 2 == 1, "conflict-free 128-bit row loads need SW_KR / 4 odd");
constexpr int SW_PROBE_PASSES = (SW_NDIAG * SW_PROBES + SW_NTHREADS - 1) / SW_NTHREADS;   // per thread per round
static_assert(SW_EMAXT % 32 == 0, "ends are taken 32 at a time");

// Per-warp shared memory.
struct WarpSmem {
    static constexpr uint32_t vstage = 0;
    static constexpr uint32_t obuf = SW_NSV * SW_VCHUNK;    // [2][SW_EMAXT] offsets (8 bytes each)
    static constexpr uint32_t xs = obuf + 2 * SW_EMAXT * 8; // [32] lane prefix values
    static constexpr uint32_t xr = xs + 32 * 4;             // [32] lane prefix rows
    static constexpr uint32_t argr = xr + 32 * 4;           // [SW_TROWS] int16; start flags
    static constexpr uint32_t bars = argr + SW_TROWS * 2;
    static constexpr uint32_t bytes = ((bars + SW_NSV * 8 + 127) / 128) * 128;
};
constexpr uint32_t SW_SMEM = SW_NW * WarpSmem::bytes;
static_assert(SW_SMEM <= 227 * 1024, "one CTA per SM");

// Search scratch (aliases the warps' memory before they start).
struct SearchSmem {
    int64_t graw[SW_GRID];
    int64_t D[SW_NDIAG], lo[SW_NDIAG], hi[SW_NDIAG], R[SW_NDIAG];
    int64_t oI[SW_NDIAG], oI1[SW_NDIAG];   // offsets[I], offsets[I + 1] of each cut (clamped)
    int cnt[SW_NDIAG];
    int64_t o0, oS;
};
static_assert(sizeof(SearchSmem) <= SW_SMEM, "search scratch fits");
// Offsets arrays up to this size are copied whole into shared memory (behind
// the search scratch) and searched there.
constexpr uint32_t SW_SEARCH_BYTES = ((sizeof(SearchSmem) + 127) / 128) * 128;
constexpr uint32_t SW_SMALL_OFFS = 96 * 1024;
static_assert(SW_SEARCH_BYTES + SW_SMALL_OFFS <= SW_SMEM, "the offsets fit beside the search scratch");

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
    a.v.w = 0ull;
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
        b.v.w = __shfl_down_sync(0xffffffffu, a.v.w, o);
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
    using CO = ScalarCarry<T, OP>;
    using C = typename CO::C;
    constexpr uint32_t OSZ = sizeof(OffT);
    constexpr bool kFloatSum = OP == OP_SUM && kIsFloat<T>;
    constexpr unsigned FULL = 0xffffffffu;

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
    // Weighted merge path: end s sits at key(s) = (offsets[s+1] - o0) + SW_CW s.
    // A cut at D takes the I(D) = #{s : key(s) < D} ends before it and the rows
    // before both D - SW_CW I and the start of segment I.  The first probe round reads a
    // fixed grid of SW_GRID keys that every CTA shares (so it hits L2); then
    // each boundary narrows its bracket with SW_PROBES probes per round.
    // A small offsets array is copied whole into shared memory and each
    // boundary is a binary search there: no probe rounds.
    SearchSmem* ss = reinterpret_cast<SearchSmem*>(smem);
    OffT* soffs = reinterpret_cast<OffT*>(smem + SW_SEARCH_BYTES);
    const bool small = static_cast<uint64_t>(S + 1) * OSZ <= SW_SMALL_OFFS;
    if (small) {
        for (int64_t i = tid; i <= S; i += SW_NTHREADS) cp_async_small<OSZ>(soffs + i, offs + i);
        cp_async_commit();
        cp_async_wait_all();
    } else {
        // the grid's loads go out first, then the L2 prefetch of this CTA's
        // slice of the offsets (which the probe rounds and tiles read later)
        if (tid == 0) ss->o0 = clamp_off(__ldg(&offs[0]), N);
        if (tid == 1) ss->oS = clamp_off(__ldg(&offs[S]), N);
        for (int m = tid; m < SW_GRID; m += SW_NTHREADS) {
            const int64_t sm = static_cast<int64_t>(m) * S / SW_GRID;
            ss->graw[m] = clamp_off(__ldg(&offs[sm + 1]), N);
        }
        prefetch_offsets_slice(p.offsets, static_cast<uint64_t>(S + 1) * OSZ, cta, p.P, tid, SW_NTHREADS);
    }
    __syncthreads();
    const int64_t o0 = small ? clamp_off(soffs[0], N) : ss->o0;
    const int64_t oS_raw = small ? clamp_off(soffs[S], N) : ss->oS;
    const int64_t oS = oS_raw < o0 ? o0 : oS_raw;
    const int64_t nrows = oS - o0;
    const int64_t total = nrows + SW_CW * S;
    const int64_t Wu = (total + U - 1) / U;
    if (tid < SW_NDIAG) {
        const int64_t u = static_cast<int64_t>(cta) * SW_NW + tid;
        const int64_t D = u * Wu < total ? u * Wu : total;
        int64_t lo = D > nrows ? (D - nrows + SW_CW - 1) / SW_CW : 0;
        int64_t hi = (D + SW_CW - 1) / SW_CW;
        hi = hi < S ? hi : S;
        if (small) {
            // I = #{s : key(s) < D}: the first s in [lo, hi) with key(s) >= D
            while (lo < hi) {
                const int64_t mid = (lo + hi) >> 1;
                if (clamp_off(soffs[mid + 1], N) - o0 + SW_CW * mid < D)
                    lo = mid + 1;
                else
                    hi = mid;
            }
            hi = lo;
        } else {
            int a = 0, b = SW_GRID;   // c = #{m : key(s_m) < D}
            while (a < b) {
                const int mid = (a + b) >> 1;
                const int64_t sm = static_cast<int64_t>(mid) * S / SW_GRID;
                if (ss->graw[mid] - o0 + SW_CW * sm < D)
                    a = mid + 1;
                else
                    b = mid;
            }
            const int64_t lower = a > 0 ? static_cast<int64_t>(a - 1) * S / SW_GRID + 1 : 0;
            const int64_t upper = a < SW_GRID ? static_cast<int64_t>(a) * S / SW_GRID : S;
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
        for (int u = 0; u < SW_PROBE_PASSES; ++u) {
            const int pidx = tid + u * SW_NTHREADS;
            const int k = pidx / SW_PROBES;
            const int mm = pidx - k * SW_PROBES;
            if (k < SW_NDIAG) {
                const int64_t lo = ss->lo[k], hi = ss->hi[k];
                const int64_t len = hi - lo;
                if (len > 0) {
                    const int64_t step = (len + SW_PROBES - 1) / SW_PROBES;
                    const int64_t s = lo + mm * step;
                    if (s < hi && clamp_off(__ldg(&offs[s + 1]), N) - o0 + SW_CW * s < ss->D[k])
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
    if (tid < SW_NDIAG) {
        // rows before the cut: D - SW_CW I, but never fewer than segment I's
        // start; offsets[I] and offsets[I + 1] load together and stay for the
        // warps' cut-crossing segments
        const int64_t I = ss->lo[tid];
        const int64_t vI = clamp_off(small ? soffs[I] : __ldg(&offs[I]), N);
        const int64_t vI1 = I < S ? clamp_off(small ? soffs[I + 1] : __ldg(&offs[I + 1]), N) : 0;
        const int64_t oI = I > 0 ? vI - o0 : 0;
        int64_t R = ss->D[tid] - SW_CW * I;
        R = R < oI ? oI : R;
        R = R < 0 ? 0 : (R > nrows ? nrows : R);
        ss->R[tid] = o0 + R;
        ss->oI[tid] = vI;
        ss->oI1[tid] = vI1;
    }
    __syncthreads();
    // my unit: weighted positions [Dlo, Dhi), ends [Iu, Iu2), rows [Ru, Ru2)
    const int64_t u_me = static_cast<int64_t>(cta) * SW_NW + warp;
    const int64_t Dlo = ss->D[warp], Dhi = ss->D[warp + 1];
    const int64_t Iu = ss->lo[warp];
    const int64_t Iu2 = ss->lo[warp + 1] > Iu ? ss->lo[warp + 1] : Iu;
    const int64_t Rc = ss->R[warp];                              // the cuts' rows
    const int64_t Rc2 = ss->R[warp + 1] > Rc ? ss->R[warp + 1] : Rc;
    // Offsets of the segment that crosses each cut (the head and tail logic
    // needs them), as the search left them (Iu2 is cut warp + 1's I, or Iu
    // itself when offsets decrease)
    const int j2 = ss->lo[warp + 1] > Iu ? warp + 1 : warp;
    const int64_t off_Iu = ss->oI[warp];
    const int64_t off_Iu1 = Iu < S ? ss->oI1[warp] : 0;
    const int64_t off_Iu2 = Iu2 < S ? ss->oI[j2] : 0;
    const int64_t off_Iu21 = Iu2 < S ? ss->oI1[j2] : 0;
    __syncthreads();   // the search scratch is dead from here on
    if (Dlo >= Dhi) return;
    // A segment that crosses just one cut, with at most SW_ADOPT rows before
    // it, is adopted whole by the unit that holds its end: that unit starts
    // at the segment's first row and the unit before it stops there, so no
    // partial and no ticket are needed.  Both sides decide it from the same
    // cut and the same offsets.
    bool adopt_head = false, give_tail = false;
    if (Iu < Iu2 && off_Iu < Rc && Rc - off_Iu <= SW_ADOPT && u_me > 0)
        adopt_head = (off_Iu - o0 + SW_CW * Iu) / Wu == u_me - 1;
    if (Iu2 < S && off_Iu2 < Rc2 && Rc2 - off_Iu2 <= SW_ADOPT) {
        const int64_t f = off_Iu2 - o0 + SW_CW * Iu2;
        const int64_t e = (off_Iu21 > off_Iu2 ? off_Iu21 : off_Iu2) - o0 + SW_CW * Iu2;
        give_tail = f / Wu == u_me && e / Wu == u_me + 1;
    }
    const int64_t Ru = adopt_head ? off_Iu : Rc;
    const int64_t Ru2 = give_tail ? (off_Iu2 > Ru ? off_Iu2 : Ru) : Rc2;

    // ---- per-warp state ----------------------------------------------------------
    unsigned char* wbase = smem + warp * WarpSmem::bytes;
    unsigned char* vst = wbase + WarpSmem::vstage;
    unsigned char* obuf = wbase + WarpSmem::obuf;
    uint32_t* xs = reinterpret_cast<uint32_t*>(wbase + WarpSmem::xs);
    int32_t* xr = reinterpret_cast<int32_t*>(wbase + WarpSmem::xr);
    int16_t* argr = reinterpret_cast<int16_t*>(wbase + WarpSmem::argr);
    // Start flags (one byte per chunk row) share argr's bytes: a tile reads
    // them before it writes argr, and clears them once it is done with argr.
    unsigned char* flg = wbase + WarpSmem::argr;
    uint64_t* fv = reinterpret_cast<uint64_t*>(wbase + WarpSmem::bars);
    T* out = static_cast<T*>(p.out);
    PartElem* tails = static_cast<PartElem*>(p.ws_parts);
    PartElem* heads = tails + U;
    const int mean = p.mean;
    const bool want_arg = (OP != OP_SUM) && p.out_arg != nullptr;

    const uint64_t vbase = reinterpret_cast<uint64_t>(p.values);
    const Stream vs = make_stream(vbase, static_cast<uint64_t>(N) * 4, vbase + Ru * 4, vbase + Ru2 * 4,
                                  SW_VCHUNK);
    const int32_t nR = static_cast<int32_t>(Ru2 - Ru);
    // chunk 0's first row, relative to Ru (in [-3, 0]: chunks start 16-byte aligned)
    const int32_t cb0 = static_cast<int32_t>(static_cast<int64_t>(vs.A0 - vbase) / 4 - Ru);
    const uint64_t policy = policy_evict_first();

    // Value chunk k into its stage (lane 0).  Chunks inside the buffer's
    // 16-byte-aligned interior take one bulk copy; the first and last may
    // need plain loads for their edges.
    auto issue_v = [&](int64_t k) {
        unsigned char* dst = vst + (k % SW_NSV) * SW_VCHUNK;
        uint64_t* bar = &fv[k % SW_NSV];
        const uint64_t cs = vs.A0 + static_cast<uint64_t>(k) * SW_VCHUNK;
        if (cs >= vs.TA && cs + SW_VCHUNK <= vs.TE && cs + SW_VCHUNK <= vs.AE) {
            mbar_arrive_expect_tx(bar, SW_VCHUNK);
            bulk_load(dst, reinterpret_cast<const void*>(cs), SW_VCHUNK, bar, policy);
        } else {
            issue_chunk_to(vs, k, SW_VCHUNK, dst, bar, policy);
        }
    };

    if (lane == 0) {
        for (int k = 0; k < SW_NSV; ++k) mbar_init(&fv[k], 1);
        fence_mbarrier_init();
    }
    // clear my flag bytes
#pragma unroll
    for (int q = 0; q < SW_Q; ++q) reinterpret_cast<uint32_t*>(flg + lane * SW_KR)[q] = 0u;
    __syncwarp();
    // counters below are kept identical in every lane; lane 0 issues the copies
    int64_t v_issued = SW_NSV < vs.nch ? SW_NSV : vs.nch;
    if (lane == 0) {
        for (int64_t k = 0; k < v_issued; ++k) issue_v(k);
    }

    // Segment ends: half `h` of the offsets buffer holds offsets[Iu + i0 + 1 ..
    // Iu + i0 + n] for the tile that starts at end i0; lane l copies entries
    // l, l + 32, ...
    constexpr int NG = SW_EMAXT / 32;
    auto load_ends = [&](int32_t i0, int n, int h) {
        OffT* dst = reinterpret_cast<OffT*>(obuf) + h * SW_EMAXT;
        const OffT* src = offs + Iu + i0 + 1;
#pragma unroll
        for (int g = 0; g < NG; ++g) {
            const int idx = 32 * g + lane;
            if (idx < n) cp_async_small<OSZ>(dst + idx, src + idx);
        }
        cp_async_commit();
    };
    // an absolute offset as a row relative to Ru, clamped to [-1, nR + 1]
    // (which also keeps malformed offsets inside the unit)
    // (in 32 bits: a unit spans fewer than 2^31 rows, so a valid offset is
    // exact; a malformed one wraps, and the clamp still keeps it in the unit)
    const uint32_t Ru_lo = static_cast<uint32_t>(Ru);
    auto rel_off = [&](OffT raw) -> int32_t {
        const int32_t x = static_cast<int32_t>(static_cast<uint32_t>(raw) - Ru_lo);
        return x < -1 ? -1 : (x > nR + 1 ? nR + 1 : x);
    };
    bool ok = true;

    C carry = CO::ident();
    bool head_pending = (Iu < S) && off_Iu < Ru;
    bool head_taken = false;                 // the head ticket was taken ...
    unsigned long long head_ticket = 0;      // ... and returned this (lane 0)
    int64_t m = 0;            // current value chunk
    bool m_ready = false;
    int32_t ie = 0;           // next segment end, relative to Iu
    const int32_t nE = static_cast<int32_t>(Iu2 - Iu);
    int oh = 0;               // offsets buffer half of the current tile
    load_ends(0, nE < SW_EMAXT ? nE : SW_EMAXT, 0);
    int32_t b_es = off_Iu - Ru < -1 ? -1 : static_cast<int32_t>(off_Iu - Ru);   // offsets[Iu + ie]
    int32_t jj = 0;           // next row

    while (ok) {
        const bool lastc = m + 1 >= vs.nch;
        const int32_t cb = cb0 + static_cast<int32_t>(m) * SW_TROWS;   // chunk m's first row
        const int32_t rl = lastc ? nR : (cb + SW_TROWS < nR ? cb + SW_TROWS : nR);
        if (m < vs.nch && !m_ready) {
            ok = __all_sync(FULL, wait_bounded(&fv[m % SW_NSV], static_cast<uint32_t>((m / SW_NSV) & 1),
                                               p.status, STATUS_CONSUMER_TIMEOUT));
            m_ready = true;
            if (!ok) break;
        }
        const int32_t rem = nE - ie;
        const int ncand = rem < SW_EMAXT ? rem : SW_EMAXT;
        // This tile's ends: the prefix of the candidates whose segment ends by
        // row rl (all of them on the unit's last chunk).  Lane l keeps
        // E[g] = offsets[s + 1] of end s = Iu + ie + 32 g + l.  The same pass
        // sets the start flag of each row inside the chunk where a segment
        // starts (for valid offsets those are exactly this tile's ends).
        cp_async_wait_all();
        __syncwarp();
        const OffT* ob_cur = reinterpret_cast<const OffT*>(obuf) + oh * SW_EMAXT;
        int32_t E[NG];
        int n_e = 0;
        bool more = true;
#pragma unroll
        for (int g = 0; g < NG; ++g) {
            E[g] = INT32_MAX;
            if (more && 32 * g < ncand) {
                const int idx = 32 * g + lane;
                if (idx < ncand) E[g] = rel_off(ob_cur[idx]);
                if (E[g] >= jj && E[g] < rl && m < vs.nch) flg[E[g] - cb] = 1;
                const unsigned b = __ballot_sync(FULL, idx < ncand && (lastc || E[g] <= rl));
                if (b != FULL) {
                    n_e += __ffs(~b) - 1;
                    more = false;
                } else {
                    n_e += 32;
                }
            }
        }
        n_e = n_e < ncand ? n_e : ncand;
        const bool capped = n_e == SW_EMAXT && ie + n_e < nE;
        // the segment left open after this tile starts at offsets[Iu + ie + n_e],
        // the E of the tile's last end (read back from the buffer: selecting it
        // from E[] would index the array at run time)
        const int32_t bo = n_e == 0 ? b_es : rel_off(ob_cur[n_e - 1]);
        if (n_e > 0) {
            // the next tile's candidate ends go to the other half now
            __syncwarp();
            oh ^= 1;
            const int32_t rem2 = nE - (ie + n_e);
            load_ends(ie + n_e, rem2 < SW_EMAXT ? rem2 : SW_EMAXT, oh);
        }

        const int32_t tr1 = capped ? (bo < jj ? jj : (bo > rl ? rl : bo)) : rl;

        // ---- one tile: rows [jj, tr1) of chunk m, ends [ie, ie + n_e) ---------------
        if (n_e > 0 || jj < tr1) {
            unsigned char* stage = vst + (m % SW_NSV) * SW_VCHUNK;
            const int32_t jr = jj - cb;       // rows relative to the chunk
            const int32_t tr = tr1 - cb;
            const bool has_rows = tr1 > jj && m < vs.nch;
            const int32_t lrow0 = lane * SW_KR;   // my first row, relative to the chunk
            unsigned char* mine = stage + lane * (SW_KR * 4);
            if (has_rows && n_e == 0 && jr == 0 && tr == SW_TROWS) {
                // The whole chunk lies inside one segment: fold it.
                Acc<T> a = RD::ident();
#pragma unroll
                for (int q = 0; q < SW_Q; ++q) {
                    const uint4 u4 = *reinterpret_cast<const uint4*>(mine + 16 * q);
                    if constexpr (OP == OP_SUM) {
                        const T s01 = add_wrap(from_bits<T>(u4.x), from_bits<T>(u4.y));
                        const T s23 = add_wrap(from_bits<T>(u4.z), from_bits<T>(u4.w));
                        a.v = add_wrap(a.v, add_wrap(s01, s23));
                    } else {
                        const uint32_t xb[4] = {u4.x, u4.y, u4.z, u4.w};
#pragma unroll
                        for (int t = 0; t < 4; ++t) RD::add(a, from_bits<T>(xb[t]), lrow0 + 4 * q + t);
                    }
                }
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) {
                    Acc<T> b;
                    b.v = from_bits<T>(__shfl_xor_sync(FULL, bits_of(a.v), o));
                    b.row = OP == OP_SUM ? -1 : __shfl_xor_sync(FULL, a.row, o);
                    a = (lane & o) ? RD::comb(b, a) : RD::comb(a, b);
                }
                if constexpr (OP != OP_SUM) a.row += cb;
                carry = b_es < jj ? CO::then(carry, a) : CO::from(a);
            } else {
                if (has_rows) {
                    // start flags: the tile's first row (the ends' were set above)
                    if (lane == 0) flg[jr] = 1;
                    __syncwarp();
                    uint32_t fw[SW_Q];
#pragma unroll
                    for (int q = 0; q < SW_Q; ++q) fw[q] = reinterpret_cast<const uint32_t*>(flg + lane * SW_KR)[q];
                    __syncwarp();
                    if constexpr (OP == OP_SUM) {
                        // sum writes no argr: clear my flags at once
#pragma unroll
                        for (int q = 0; q < SW_Q; ++q) reinterpret_cast<uint32_t*>(flg + lane * SW_KR)[q] = 0u;
                    }
                    // inclusive segmented scan of my rows, a quad at a time
                    const int32_t hi = tr - lrow0;        // my rows below tr1
                    const bool full_tail = tr == SW_TROWS;    // the same in every lane
                    Acc<T> acc = RD::ident();
                    bool fi = false;
#pragma unroll
                    for (int q = 0; q < SW_Q; ++q) {
                        const uint4 u4 = *reinterpret_cast<const uint4*>(mine + 16 * q);
                        uint32_t xb[4] = {u4.x, u4.y, u4.z, u4.w};
                        int16_t rr[4];
                        fi = fi || fw[q] != 0u;
#pragma unroll
                        for (int t = 0; t < 4; ++t) {
                            const int k = 4 * q + t;
                            const T x = from_bits<T>(xb[t]);
                            const bool reset = (fw[q] >> (8 * t)) & 1u;
                            if constexpr (OP == OP_SUM) {
                                acc.v = reset ? x : add_wrap(acc.v, x);
                            } else {
                                const bool better = (OP == OP_MIN) ? (x < acc.v) : (x > acc.v);
                                if (reset || acc.row < 0 || better) {
                                    acc.v = x;
                                    acc.row = lrow0 + k;
                                }
                                rr[t] = static_cast<int16_t>(acc.row);
                            }
                            xb[t] = bits_of(acc.v);
                        }
                        // running values back over rows < tr1 (later rows are the
                        // next tile's input; earlier rows are finished); a tile
                        // that runs to the chunk's end writes every quad
                        if (full_tail || 4 * q + 4 <= hi) {
                            *reinterpret_cast<uint4*>(mine + 16 * q) = make_uint4(xb[0], xb[1], xb[2], xb[3]);
                            if constexpr (OP != OP_SUM)
                                *reinterpret_cast<uint2*>(&argr[lrow0 + 4 * q]) = make_uint2(
                                    (static_cast<uint32_t>(static_cast<uint16_t>(rr[1])) << 16) |
                                        static_cast<uint16_t>(rr[0]),
                                    (static_cast<uint32_t>(static_cast<uint16_t>(rr[3])) << 16) |
                                        static_cast<uint16_t>(rr[2]));
                        } else if (4 * q < hi) {
#pragma unroll
                            for (int t = 0; t < 4; ++t) {
                                if (4 * q + t < hi) {
                                    *reinterpret_cast<uint32_t*>(mine + 16 * q + 4 * t) = xb[t];
                                    if constexpr (OP != OP_SUM) argr[lrow0 + 4 * q + t] = rr[t];
                                }
                            }
                        }
                    }
                    // segmented scan of the lane totals; the exclusive prefix of
                    // each lane goes to shared memory
                    Acc<T> inc = acc;
#pragma unroll
                    for (int o = 1; o < 32; o <<= 1) {
                        Acc<T> pv;
                        pv.v = from_bits<T>(__shfl_up_sync(FULL, bits_of(inc.v), o));
                        if constexpr (OP != OP_SUM) pv.row = __shfl_up_sync(FULL, inc.row, o);
                        else pv.row = -1;
                        const bool pf = __shfl_up_sync(FULL, fi, o);
                        if (lane >= o) {
                            if (!fi) inc = RD::comb(pv, inc);
                            fi = fi || pf;
                        }
                    }
                    const uint32_t xv = __shfl_up_sync(FULL, bits_of(inc.v), 1);
                    xs[lane] = xv;
                    if constexpr (OP != OP_SUM) {
                        const int32_t xrow = __shfl_up_sync(FULL, inc.row, 1);
                        xr[lane] = lane == 0 ? -1 : xrow;
                    }
                    __syncwarp();
                }
                // Running value at chunk row k (jr <= k < tr) of the run that
                // starts at chunk row st: the stored running value, joined with
                // the owning lane's prefix when the run began in an earlier
                // lane.  min / max rows come back relative to Ru.
                auto running_at = [&](int32_t k, int32_t st) -> Acc<T> {
                    if (!has_rows) return RD::ident();
                    k = k < jr ? jr : (k >= tr ? tr - 1 : k);
                    const int o = k / SW_KR;
                    Acc<T> P;
                    P.v = *reinterpret_cast<const T*>(stage + k * 4);
                    P.row = OP == OP_SUM ? -1 : static_cast<int32_t>(argr[k]) + cb;
                    if (st < o * SW_KR) {
                        Acc<T> Xo;
                        Xo.v = from_bits<T>(xs[o]);
                        Xo.row = -1;
                        if constexpr (OP != OP_SUM) {
                            const int32_t r = xr[o];
                            Xo.row = r < 0 ? -1 : r + cb;
                        }
                        P = RD::comb(Xo, P);
                    }
                    return P;
                };
                bool skip_first = false;
                if (head_pending && n_e > 0) {
                    // end Iu began in an earlier unit: leave the head partial and
                    // take the ticket; its answer is read when the unit is done
                    const int32_t oe = __shfl_sync(FULL, E[0], 0);
                    const bool rows_here = has_rows && oe - 1 >= jj;
                    const Acc<T> P = running_at(oe - 1 - cb, jr);
                    const C R = rows_here ? CO::then(carry, P) : carry;
                    if (lane == 0) {
                        if constexpr (kFloatSum) heads[u_me] = to_part(R);
                        else heads[u_me] = to_part<T, OP>(R, Ru);
                        head_ticket = ticket_take(p.ws_tickets, static_cast<int>(u_me), p.gen);
                    }
                    head_taken = true;
                    skip_first = true;   // lane 0 of the first group skips end Iu below
                }
                // the ends, 32 at a time: E = offsets[s + 1], B = offsets[s]
                T* const out_t = out + (Iu + ie);
                int64_t* const arg_t = want_arg ? p.out_arg + (Iu + ie) : nullptr;
                int32_t prevE = b_es;
#pragma unroll
                for (int g = 0; g < NG; ++g) {
                    if (32 * g < n_e) {
                        const int idx = 32 * g + lane;
                        const bool valid = idx < n_e && !(g == 0 && lane == 0 && skip_first);
                        const int32_t oe = E[g];
                        const int32_t up = __shfl_up_sync(FULL, oe, 1);
                        const int32_t ob = lane == 0 ? prevE : up;
                        prevE = __shfl_sync(FULL, oe, 31);
                        if (valid) {
                            const int32_t len = oe > ob ? oe - ob : 0;
                            T v;
                            int64_t a;
                            if (len == 0) {
                                v = T(0);
                                a = -1;
                            } else if (ob >= jj) {
                                finish_acc<T, OP>(running_at(oe - 1 - cb, ob - cb), len, mean, Ru, v, a);
                            } else {
                                const bool rows_here = has_rows && oe - 1 >= jj;
                                const C R = rows_here ? CO::then(carry, running_at(oe - 1 - cb, jr)) : carry;
                                if constexpr (kFloatSum) {
                                    finish_carry(R, len, mean, v);
                                    a = -1;
                                } else {
                                    finish_acc<T, OP>(R, len, mean, Ru, v, a);
                                }
                            }
                            out_t[idx] = v;
                            if (want_arg) arg_t[idx] = a;
                        }
                    }
                }
                // carry of the segment left open, which starts at bo
                const int32_t sto = bo > jj ? bo : jj;
                if (has_rows && sto < tr1) {
                    const Acc<T> P = running_at(tr - 1, sto - cb);
                    carry = bo < jj ? CO::then(carry, P) : CO::from(P);
                } else if (!(bo < jj)) {
                    carry = CO::ident();
                }
                if constexpr (OP != OP_SUM) {
                    if (has_rows) {
                        // done with argr: clear my flag bytes for the next tile
                        __syncwarp();
#pragma unroll
                        for (int q = 0; q < SW_Q; ++q) reinterpret_cast<uint32_t*>(flg + lane * SW_KR)[q] = 0u;
                    }
                }
            }
            if (n_e > 0) head_pending = false;
            b_es = bo;
            jj = tr1;
            ie += n_e;
            __syncwarp();
        }
        // The chunk is finished once its rows are done and no further end
        // falls in it (the tile was not cut short by the ends cap).
        if (jj >= rl && !capped) {
            if (lastc) {
                if (ie >= nE) break;
                continue;   // malformed offsets only: drain the remaining ends
            }
            // the stage is refilled by the async proxy: order this warp's
            // reads and write-backs of it first
            fence_proxy_async_smem();
            __syncwarp();
            if (v_issued < vs.nch) {
                if (lane == 0) issue_v(v_issued);
                ++v_issued;
            }
            ++m;
            m_ready = false;
        }
    }

    // ---- a6: the segment still open at the end of the unit -------------------------
    // Its partial and ticket go out first; while that atomic is in flight the
    // head ticket taken earlier is read, and its segment combined if this
    // unit arrived last.
    bool tail_taken = false;
    unsigned long long tail_ticket = 0;
    int tpc = 0, tqc = 0;
    int64_t tob = 0;
    if (ok && Iu2 < S) {
        tob = off_Iu2;
        if (tob < Ru2) {
            if (lane == 0) {
                if constexpr (kFloatSum) tails[u_me] = to_part(carry);
                else tails[u_me] = to_part<T, OP>(carry, Ru);
                const int64_t oe = off_Iu21;
                const int64_t f = tob - o0 + SW_CW * Iu2;
                const int64_t e = (oe > tob ? oe : tob) - o0 + SW_CW * Iu2;
                tpc = static_cast<int>(f / Wu);
                tqc = static_cast<int>(e / Wu);
                tpc = tpc < 0 ? 0 : (tpc > u_me ? static_cast<int>(u_me) : tpc);
                tqc = tqc <= u_me ? static_cast<int>(u_me) + 1 : tqc;
                if (tqc < U) tail_ticket = ticket_take(p.ws_tickets, tqc, p.gen);
            }
            tqc = __shfl_sync(FULL, tqc, 0);
            tpc = __shfl_sync(FULL, tpc, 0);
            tail_taken = tqc < U;
        }
    }
    if (head_taken) {
        int pc = static_cast<int>((off_Iu - o0 + SW_CW * Iu) / Wu);
        pc = pc < 0 ? 0 : (pc > u_me ? static_cast<int>(u_me) : pc);
        const bool last = __shfl_sync(
            FULL, lane == 0 && ticket_last(head_ticket, p.gen, static_cast<int>(u_me) - pc + 1), 0);
        if (last) {
            fence_acq_rel_gpu();
            warp_combine_store<T, OP>(p, tails, heads, pc, static_cast<int>(u_me), Iu,
                                      off_Iu1 > off_Iu ? off_Iu1 - off_Iu : 0, lane);
        }
    }
    if (tail_taken) {
        const bool last = __shfl_sync(FULL, lane == 0 && ticket_last(tail_ticket, p.gen, tqc - tpc + 1), 0);
        if (last) {
            fence_acq_rel_gpu();
            warp_combine_store<T, OP>(p, tails, heads, tpc, tqc, Iu2, off_Iu21 > tob ? off_Iu21 - tob : 0, lane);
        }
    }
    // every copy this warp started must land before it exits
    if (lane == 0) {
        for (int64_t k = m + (m_ready ? 1 : 0); k < v_issued; ++k)
            wait_bounded(&fv[k % SW_NSV], static_cast<uint32_t>((k / SW_NSV) & 1), p.status,
                         STATUS_DRAIN_TIMEOUT);
    }
    cp_async_wait_all();
}

}  // namespace segred
