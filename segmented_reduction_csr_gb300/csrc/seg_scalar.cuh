// seg_scalar.cuh -- the scalar kernel: F == 1 vectors of uint32, int32 or
// float32 (GPUSegmentedReduction's "packed scalar values").
//
// Each CTA walks its merge range in tiles of up to SC_ROWS rows.  A tile is
// processed in three branch-free passes so that every row costs a couple of
// instructions whatever the segment lengths:
//
//  1. Segment pass (threads stride over the tile's segment ends): mark in
//     `keep` (one 32-bit mask per row) every row where a segment starts.
//  2. Row pass: thread t owns SC_KR consecutive rows of a 16-byte-aligned
//     block; it loads them with 128-bit shared loads (SC_KR / 4 is odd, so
//     the loads are bank-conflict free), runs an inclusive segmented scan in
//     registers (sum: acc = (acc & keep) + x, so a reset never multiplies a
//     NaN or an Inf; min / max: strict compare, restart at a mark) and
//     writes the running values back over the rows.  The thread totals are
//     combined by a segmented scan across the warp (shuffles) and then
//     across warps in order, giving each thread the running value of the
//     rows before its block.
//  3. Segment pass again: the result of segment s is the running value at its
//     last row, joined with the running value before that row's thread when
//     the segment started in an earlier thread, and with the carry of
//     earlier tiles when it started in an earlier tile.  Consecutive threads
//     write consecutive segments, so the stores coalesce.  The same pass
//     clears the marks and computes the carry for the segment left open.
//
// Shared memory: the value ring (rows are rewritten in place with running
// values), the offsets ring, the row marks, the running rows of min / max.
#pragma once
#include "seg_common.cuh"

namespace segred {

constexpr int SC_NT = 256;                  // consumer threads (8 warps)
constexpr int SC_NTHREADS = SC_NT + 32;     // + one producer warp
constexpr int SC_KR = 36;                   // rows per thread per tile (SC_KR / 4 odd)
constexpr int SC_ROWS = SC_NT * SC_KR;      // rows a tile's blocks can hold
constexpr int64_t SC_TILE_ITEMS = SC_ROWS - 3;  // merge items per tile (block alignment slack)
constexpr uint32_t SC_VRING = 128u * 1024u;
constexpr uint32_t SC_VCHUNK = 8u * 1024u;
constexpr int SC_NSV = SC_VRING / SC_VCHUNK;
constexpr uint32_t SC_ORING = 16u * 1024u;
constexpr uint32_t SC_OCHUNK = 1024u;
constexpr int SC_NSO = SC_ORING / SC_OCHUNK;
static_assert((SC_KR / 4) % 2 == 1, "conflict-free 128-bit row loads need SC_KR / 4 odd");
// Ring stages are handed back one tile late, so each ring holds two tiles.
static_assert(2 * SC_ROWS * 4 + 2 * SC_VCHUNK <= SC_VRING, "value ring too small for two tiles");

// Largest number of segment ends one tile may hold: two windows of
// (max_ends + 1) offsets plus two partial chunks fit the offsets ring.
__host__ __device__ constexpr int scalar_max_ends(int offset_bytes) {
    return static_cast<int>((SC_ORING - 2 * SC_OCHUNK) / (2u * offset_bytes)) - 2;
}

template <int OP>
struct ScalarSmem {
    static constexpr uint32_t vring = 0;
    static constexpr uint32_t oring = SC_VRING;
    static constexpr uint32_t keep = oring + SC_ORING;
    static constexpr uint32_t argr = keep + SC_ROWS * 4;
    static constexpr uint32_t argr_bytes = OP == OP_SUM ? 0 : SC_ROWS * 4;
    static constexpr uint32_t bars = argr + argr_bytes;
    static constexpr uint32_t misc = bars + 2 * (SC_NSV + SC_NSO) * 8;   // search counts, tile message
    static constexpr uint32_t carry = misc + 128;                        // [2] x 16 bytes
    static constexpr uint32_t xv = carry + 32;                           // [SC_NT] thread prefixes
    static constexpr uint32_t xr = xv + SC_NT * 4;
    static constexpr uint32_t wv = xr + SC_NT * 4;                       // [8] warp totals
    static constexpr uint32_t wr = wv + 32;
    static constexpr uint32_t wf = wr + 32;
    static constexpr uint32_t total = wf + 32;
};

struct TileMsg {
    int64_t d_end, i_end, j_end;
};

template <class T, int OP, class OffT>
__global__ void __launch_bounds__(SC_NTHREADS, 1) seg_scalar_kernel(const Params p) {
    using RD = Red<T, OP>;
    using CO = Carry<T, OP>;
    using C = typename CO::C;
    using L = ScalarSmem<OP>;
    constexpr uint32_t OSZ = sizeof(OffT);
    static_assert(sizeof(C) <= 16, "carry slot");

    extern __shared__ __align__(1024) unsigned char smem[];
    unsigned char* vring = smem + L::vring;
    unsigned char* oring = smem + L::oring;
    uint32_t* keep = reinterpret_cast<uint32_t*>(smem + L::keep);
    int32_t* argr = reinterpret_cast<int32_t*>(smem + L::argr);
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::bars);
    uint64_t* full_v = bars;
    uint64_t* empty_v = full_v + SC_NSV;
    uint64_t* full_o = empty_v + SC_NSV;
    uint64_t* empty_o = full_o + SC_NSO;
    int* counts = reinterpret_cast<int*>(smem + L::misc);
    TileMsg* tm = reinterpret_cast<TileMsg*>(smem + L::misc + 32);
    C* carry_buf = reinterpret_cast<C*>(smem + L::carry);
    T* xv = reinterpret_cast<T*>(smem + L::xv);
    int32_t* xr = reinterpret_cast<int32_t*>(smem + L::xr);
    T* wv = reinterpret_cast<T*>(smem + L::wv);
    int32_t* wr = reinterpret_cast<int32_t*>(smem + L::wr);
    int* wf = reinterpret_cast<int*>(smem + L::wf);

    const int tid = threadIdx.x;
    const int64_t N = p.N;
    const int64_t S = p.S;
    const OffT* offs = static_cast<const OffT*>(p.offsets);

    if (tid < 6) counts[tid] = 0;
    if (tid == 0) {
        init_ring_barriers(bars, SC_NSV, SC_NSO);
        carry_buf[0] = CO::ident();
    }
    if (tid < SC_NT) {
#pragma unroll
        for (int q = 0; q < SC_KR / 4; ++q)
            *reinterpret_cast<uint4*>(&keep[tid * SC_KR + 4 * q]) = make_uint4(~0u, ~0u, ~0u, ~0u);
    }
    __syncthreads();
    CtaRange cr;
    if (!cta_range<SC_NTHREADS, OffT>(p, counts, cr)) return;
    const int64_t o0 = cr.o0, W = cr.W, Dlo = cr.Dlo, Dhi = cr.Dhi;
    const int64_t Ilo = cr.Ilo, Ihi = cr.Ihi, Rlo = cr.Rlo, Rhi = cr.Rhi;
    const int cta = blockIdx.x;

    const uint64_t vbase = reinterpret_cast<uint64_t>(p.values);
    const uint64_t obase = reinterpret_cast<uint64_t>(p.offsets);
    const Stream vs = make_stream(vbase, static_cast<uint64_t>(N) * 4, vbase + Rlo * 4,
                                  vbase + Rhi * 4, SC_VCHUNK);
    const Stream os = make_stream(obase, static_cast<uint64_t>(S + 1) * OSZ, obase + Ilo * OSZ,
                                  obase + (Ihi + 1) * OSZ, SC_OCHUNK);
    if (tid >= SC_NT) {
        if (tid == SC_NT)
            producer_loop<SC_VRING, SC_VCHUNK, SC_ORING, SC_OCHUNK>(vs, os, vring, oring, full_v,
                                                                    empty_v, full_o, empty_o, p.status);
        return;
    }

    // ---- consumers ------------------------------------------------------------
    const int lane = tid & 31;
    const int warp = tid >> 5;
    T* out = static_cast<T*>(p.out);
    PartElem* tails = static_cast<PartElem*>(p.ws_parts);
    PartElem* heads = tails + static_cast<int64_t>(p.P);
    const int mean = p.mean;
    const bool want_arg = (OP != OP_SUM) && p.out_arg != nullptr;

    auto off_r = [&](int64_t s) -> int64_t {
        const uint32_t at = static_cast<uint32_t>((obase + static_cast<uint64_t>(s) * OSZ) - os.A0) &
                            (SC_ORING - 1);
        return clamp_off(*reinterpret_cast<const OffT*>(oring + at), N);
    };
    auto key_r = [&](int64_t s) -> int64_t { return off_r(s + 1) - o0 + s; };
    auto ring_at = [&](int64_t row) -> uint32_t {
        return static_cast<uint32_t>((vbase + static_cast<uint64_t>(row) * 4) - vs.A0) & (SC_VRING - 1);
    };

    bool head_pending = (Ilo < S) && (clamp_off(__ldg(&offs[Ilo]), N) < Rlo);
    int64_t d = Dlo, i = Ilo, j = Rlo;
    int64_t vw = 0, vrel = 0, ow = 0, orel = 0;
    int par = 0;

    while (d < Dhi) {
        // (A)-(C), warp 0: wait for the offsets window, find the tile's end,
        // wait for its rows.
        bool ok = true;
        if (warp == 0) {
            const int64_t cap_i = i + p.max_ends < Ihi ? i + p.max_ends : Ihi;
            const int64_t need_o =
                static_cast<int64_t>((obase + static_cast<uint64_t>(cap_i + 1) * OSZ - 1 - os.A0) / SC_OCHUNK);
            for (; ok && ow <= need_o && ow < os.nch; ++ow)
                ok = wait_bounded(&full_o[ow % SC_NSO], static_cast<uint32_t>((ow / SC_NSO) & 1), p.status,
                                  STATUS_CONSUMER_TIMEOUT);
            int64_t d_end = d + SC_TILE_ITEMS < Dhi ? d + SC_TILE_ITEMS : Dhi;
            int64_t i_end = i;
            if (ok) {
                if (cap_i < Ihi && key_r(cap_i - 1) < d_end) {
                    i_end = cap_i;
                    d_end = key_r(cap_i - 1) + 1;
                } else {
                    int64_t a = i, b = cap_i;
                    while (a < b) {
                        const int64_t mid = a + ((b - a) >> 1);
                        if (key_r(mid) < d_end)
                            a = mid + 1;
                        else
                            b = mid;
                    }
                    i_end = a;
                }
            }
            // Valid offsets give i <= i_end <= cap_i and d < d_end; the clamps
            // only keep malformed offsets from stalling the loop.
            i_end = i_end < i ? i : (i_end > cap_i ? cap_i : i_end);
            if (d_end <= d) d_end = d + 1;
            int64_t j_end = d_end - i_end + o0;
            j_end = j_end < j ? j : (j_end > Rhi ? Rhi : j_end);
            if (j_end - j > SC_TILE_ITEMS) j_end = j + SC_TILE_ITEMS;
            if (j_end > j) {
                const int64_t need_v =
                    static_cast<int64_t>((vbase + static_cast<uint64_t>(j_end) * 4 - 1 - vs.A0) / SC_VCHUNK);
                for (; ok && vw <= need_v && vw < vs.nch; ++vw)
                    ok = wait_bounded(&full_v[vw % SC_NSV], static_cast<uint32_t>((vw / SC_NSV) & 1),
                                      p.status, STATUS_CONSUMER_TIMEOUT);
            }
            if (lane == 0) {
                tm->d_end = d_end;
                tm->i_end = i_end;
                tm->j_end = j_end;
            }
        }
        // (D) every consumer: data is in, the previous tile is finished.
        if (!named_bar_and<SC_NT>(ok)) return;
        const int64_t d_end = tm->d_end, i_end = tm->i_end, j_end = tm->j_end;
        if (tid == 0) {
            // Stages that hold only rows before j and offsets before entry i.
            const uint64_t vlimit = vbase + static_cast<uint64_t>(j) * 4;
            while (vrel < vw && vs.A0 + static_cast<uint64_t>(vrel + 1) * SC_VCHUNK <= vlimit) {
                mbar_arrive(&empty_v[vrel % SC_NSV]);
                ++vrel;
            }
            const uint64_t olimit = obase + static_cast<uint64_t>(i) * OSZ;
            while (orel < ow && os.A0 + static_cast<uint64_t>(orel + 1) * SC_OCHUNK <= olimit) {
                mbar_arrive(&empty_o[orel % SC_NSO]);
                ++orel;
            }
        }
        // rb: the 16-byte-aligned row at or just before j; thread t owns rows
        // [rb + t * SC_KR, rb + (t + 1) * SC_KR).
        const int64_t rb = j - static_cast<int64_t>(((vbase >> 2) + static_cast<uint64_t>(j)) & 3);
        const int nE = static_cast<int>(i_end - i);

        // ---- pass 1: mark segment starts (and j) ------------------------------
        for (int q = tid; q <= nE; q += SC_NT) {
            const int64_t b = off_r(i + q);
            if (b >= j && b < j_end) keep[b - rb] = 0u;
        }
        if (tid == 0 && j < j_end) keep[j - rb] = 0u;
        named_bar_sync<SC_NT>();

        // ---- pass 2: segmented scan of my rows --------------------------------
        const int64_t blk = rb + static_cast<int64_t>(tid) * SC_KR;
        const int32_t row0 = static_cast<int32_t>(blk - Rlo);    // CTA-relative row of my first row
        uint32_t xb[SC_KR];
        uint32_t kp[SC_KR];
        {
            const uint32_t at0 = ring_at(blk);
#pragma unroll
            for (int q = 0; q < SC_KR / 4; ++q) {
                const uint4 u = *reinterpret_cast<const uint4*>(vring + ((at0 + 16u * q) & (SC_VRING - 1)));
                xb[4 * q + 0] = u.x;
                xb[4 * q + 1] = u.y;
                xb[4 * q + 2] = u.z;
                xb[4 * q + 3] = u.w;
                const uint4 k4 = *reinterpret_cast<const uint4*>(&keep[tid * SC_KR + 4 * q]);
                kp[4 * q + 0] = k4.x;
                kp[4 * q + 1] = k4.y;
                kp[4 * q + 2] = k4.z;
                kp[4 * q + 3] = k4.w;
            }
        }
        Acc<T> acc = RD::ident();
        bool fl = false;
        int32_t rr[OP == OP_SUM ? 1 : SC_KR];
#pragma unroll
        for (int k = 0; k < SC_KR; ++k) {
            const T x = from_bits<T>(xb[k]);
            if constexpr (OP == OP_SUM) {
                acc.v = add_wrap(from_bits<T>(bits_of(acc.v) & kp[k]), x);
            } else {
                const bool better = (OP == OP_MIN) ? (x < acc.v) : (x > acc.v);
                if (kp[k] == 0u || acc.row < 0 || better) {
                    acc.v = x;
                    acc.row = row0 + k;
                }
                rr[k] = acc.row;
            }
            xb[k] = bits_of(acc.v);
            fl = fl || (kp[k] == 0u);
        }
        {
            // Write running values back over rows < j_end (rows >= j_end belong
            // to the next tile; rows < j were finished by the previous tile).
            const int64_t hi = j_end - blk;
            const uint32_t at0 = ring_at(blk);
            if (hi >= SC_KR) {
#pragma unroll
                for (int q = 0; q < SC_KR / 4; ++q) {
                    *reinterpret_cast<uint4*>(vring + ((at0 + 16u * q) & (SC_VRING - 1))) =
                        make_uint4(xb[4 * q], xb[4 * q + 1], xb[4 * q + 2], xb[4 * q + 3]);
                    if constexpr (OP != OP_SUM)
                        *reinterpret_cast<int4*>(&argr[tid * SC_KR + 4 * q]) =
                            make_int4(rr[4 * q], rr[4 * q + 1], rr[4 * q + 2], rr[4 * q + 3]);
                }
            } else if (hi > 0) {
#pragma unroll
                for (int k = 0; k < SC_KR; ++k) {
                    if (k < hi) {
                        *reinterpret_cast<uint32_t*>(vring + ((at0 + 4u * k) & (SC_VRING - 1))) = xb[k];
                        if constexpr (OP != OP_SUM) argr[tid * SC_KR + k] = rr[k];
                    }
                }
            }
        }
        // segmented scan of the thread totals across the warp
        Acc<T> inc = acc;
        bool fi = fl;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            Acc<T> pv;
            pv.v = from_bits<T>(__shfl_up_sync(0xffffffffu, bits_of(inc.v), o));
            pv.row = __shfl_up_sync(0xffffffffu, inc.row, o);
            const bool pf = __shfl_up_sync(0xffffffffu, fi, o);
            if (lane >= o) {
                if (!fi) inc = RD::comb(pv, inc);
                fi = fi || pf;
            }
        }
        Acc<T> ex;
        ex.v = from_bits<T>(__shfl_up_sync(0xffffffffu, bits_of(inc.v), 1));
        ex.row = __shfl_up_sync(0xffffffffu, inc.row, 1);
        bool exf = __shfl_up_sync(0xffffffffu, fi, 1);
        if (lane == 0) {
            ex = RD::ident();
            exf = false;
        }
        if (lane == 31) {
            wv[warp] = inc.v;
            wr[warp] = inc.row;
            wf[warp] = fi ? 1 : 0;
        }
        named_bar_sync<SC_NT>();
        {
            Acc<T> pre = RD::ident();
            for (int w2 = 0; w2 < warp; ++w2) {
                Acc<T> a;
                a.v = wv[w2];
                a.row = wr[w2];
                pre = wf[w2] ? a : RD::comb(pre, a);
            }
            const Acc<T> X = exf ? ex : RD::comb(pre, ex);
            xv[tid] = X.v;
            xr[tid] = X.row;
        }
        named_bar_sync<SC_NT>();

        // ---- pass 3: one result per segment end; clear the marks --------------
        const C carry_in = carry_buf[par];
        auto running_at = [&](int64_t row, int64_t start) -> Acc<T> {
            // running value at `row` of the run that starts at `start` (>= j);
            // valid offsets give j <= row < j_end, the clamp only guards
            // shared-memory indexing against malformed offsets
            row = row < j ? j : (row >= j_end ? j_end - 1 : row);
            const int64_t k = row - rb;
            Acc<T> P;
            P.v = *reinterpret_cast<const T*>(vring + ring_at(row));
            if constexpr (OP == OP_SUM) {
                P.row = -1;
            } else {
                P.row = argr[k];
            }
            const int t2 = static_cast<int>(k / SC_KR);
            if (start < rb + static_cast<int64_t>(t2) * SC_KR) {
                Acc<T> X;
                X.v = xv[t2];
                X.row = xr[t2];
                P = RD::comb(X, P);
            }
            return P;
        };
        for (int q = tid; q <= nE; q += SC_NT) {
            const int64_t s = i + q;
            const int64_t b = off_r(s);
            if (b >= j && b < j_end) keep[b - rb] = ~0u;
            if (q == 0 && j < j_end) keep[j - rb] = ~0u;
            if (q < nE) {
                const int64_t e = off_r(s + 1);
                C R = CO::ident();
                if (e > b) {
                    if (e - 1 < j) {
                        R = carry_in;    // ended exactly at the tile start
                    } else {
                        const Acc<T> P = running_at(e - 1, b > j ? b : j);
                        R = b < j ? CO::then(carry_in, P) : CO::from(P);
                    }
                }
                const int64_t len = e > b ? e - b : 0;
                if (head_pending && s == Ilo) {
                    // began in an earlier CTA: leave the head partial, join the ticket
                    if constexpr (OP == OP_SUM && kIsFloat<T>) heads[cta] = to_part(R);
                    else heads[cta] = to_part<T, OP>(R, Rlo);
                    __threadfence();
                    const int64_t f = b - o0 + Ilo;
                    int pc = static_cast<int>(f / W);
                    pc = pc < 0 ? 0 : (pc > cta ? cta : pc);
                    if (ticket_arrive(p.ws_tickets, cta, cta - pc + 1, p.gen)) {
                        __threadfence();
                        combine_store<T, OP>(p, tails, heads, pc, cta, s, len, 0, 1);
                    }
                } else {
                    T v;
                    int64_t a;
                    if constexpr (OP == OP_SUM && kIsFloat<T>) {
                        finish_carry(R, len, mean, v);
                        a = -1;
                    } else {
                        finish_acc<T, OP>(R, len, mean, Rlo, v, a);
                    }
                    out[s] = v;
                    if (want_arg) p.out_arg[s] = a;
                }
            } else {
                // the segment left open (i_end): its running value into the carry
                C nc = CO::ident();
                if (i_end < S) {
                    const int64_t st = b > j ? b : j;
                    if (st < j_end) {
                        const Acc<T> P = running_at(j_end - 1, st);
                        nc = b < j ? CO::then(carry_in, P) : CO::from(P);
                    } else {
                        nc = b < j ? carry_in : CO::ident();
                    }
                }
                carry_buf[par ^ 1] = nc;
            }
        }
        if (i_end > i) head_pending = false;
        par ^= 1;
        d = d_end;
        i = i_end;
        j = j_end;
    }

    // ---- a6: the segment still open at the end of the range ------------------
    named_bar_sync<SC_NT>();
    if (tid == 0 && Ihi < S) {
        const int64_t ob = clamp_off(__ldg(&offs[Ihi]), N);
        if (ob < Rhi) {
            const C cf = carry_buf[par];
            if constexpr (OP == OP_SUM && kIsFloat<T>) tails[cta] = to_part(cf);
            else tails[cta] = to_part<T, OP>(cf, Rlo);
            __threadfence();
            const int64_t oe = clamp_off(__ldg(&offs[Ihi + 1]), N);
            const int64_t f = ob - o0 + Ihi;
            const int64_t e = (oe > ob ? oe : ob) - o0 + Ihi;
            int pc = static_cast<int>(f / W);
            int qc = static_cast<int>(e / W);
            pc = pc < 0 ? 0 : (pc > cta ? cta : pc);
            qc = qc <= cta ? cta + 1 : qc;
            if (qc < p.P && ticket_arrive(p.ws_tickets, qc, qc - pc + 1, p.gen)) {
                __threadfence();
                combine_store<T, OP>(p, tails, heads, pc, qc, Ihi, oe > ob ? oe - ob : 0, 0, 1);
            }
        }
    }
}

}  // namespace segred
