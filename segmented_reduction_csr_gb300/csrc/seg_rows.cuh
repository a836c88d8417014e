// seg_rows.cuh -- the row kernel: [N, F] values, any F up to 2048 (and F == 1
// when the scalar kernel's shape does not apply).
//
// The consumer warps walk the CTA's merge range in tiles.  A tile is split
// into slots of G threads; each slot owns K consecutive merge items and its
// threads own disjoint columns of a row (float4 lanes when rows are 16-byte
// aligned).  A slot reduces its rows in registers in row order and writes
// every segment that starts and ends inside it; segments that cross slots are
// finished by a segmented scan of the slot tails (warp shuffles, then the
// warps in order); a segment still open at a tile boundary keeps a running
// carry per column (float sums in double).  So a short segment is finished by
// one slot, a medium one by the CTA's scan and a long one by several CTAs.
#pragma once
#include "seg_common.cuh"

namespace segred {

constexpr int NT = 256;              // consumer threads (8 warps)
constexpr int NTHREADS = NT + 32;    // + one producer warp
constexpr uint32_t VRING = 128u * 1024u;
constexpr uint32_t VCHUNK = 8u * 1024u;
constexpr int NSV = VRING / VCHUNK;
constexpr uint32_t ORING = 16u * 1024u;
constexpr uint32_t OCHUNK = 1024u;
constexpr int NSO = ORING / OCHUNK;

struct SmemLayout {
    static constexpr uint32_t vring = 0;
    static constexpr uint32_t oring = VRING;
    static constexpr uint32_t bars = VRING + ORING;
    static constexpr uint32_t nbars = 2 * (NSV + NSO);
    static constexpr uint32_t misc = bars + nbars * 8;
    static constexpr uint32_t misc_bytes = 128;
    static constexpr uint32_t scan = misc + misc_bytes;
    __host__ __device__ static constexpr uint32_t scan_plane(int nvec) { return NT * nvec * 4; }
    __host__ __device__ static constexpr uint32_t total(int nvec) {
        return scan + 2 * scan_plane(nvec) + 64;
    }
};


template <class T, int OP, class OffT, int VEC, int NV>
__global__ void __launch_bounds__(NTHREADS, 1) seg_rows_kernel(const Params p) {
    constexpr int NVEC = NV * VEC;
    using RD = Red<T, OP>;
    using CO = Carry<T, OP>;
    using C = typename CO::C;
    constexpr uint32_t OSZ = sizeof(OffT);

    extern __shared__ __align__(1024) unsigned char smem[];
    unsigned char* vring = smem + SmemLayout::vring;
    unsigned char* oring = smem + SmemLayout::oring;
    uint64_t* full_v = reinterpret_cast<uint64_t*>(smem + SmemLayout::bars);
    uint64_t* empty_v = full_v + NSV;
    uint64_t* full_o = empty_v + NSV;
    uint64_t* empty_o = full_o + NSO;
    int* counts = reinterpret_cast<int*>(smem + SmemLayout::misc);             // [3][2]
    volatile int* bcast = reinterpret_cast<volatile int*>(smem + SmemLayout::misc + 32);
    T* scan_v = reinterpret_cast<T*>(smem + SmemLayout::scan);
    int32_t* scan_r = reinterpret_cast<int32_t*>(smem + SmemLayout::scan + SmemLayout::scan_plane(NVEC));
    int* scan_f = reinterpret_cast<int*>(smem + SmemLayout::scan + 2 * SmemLayout::scan_plane(NVEC));

    const int tid = threadIdx.x;
    const int cta = blockIdx.x;
    const int64_t N = p.N;
    const int64_t S = p.S;
    const OffT* offs = static_cast<const OffT*>(p.offsets);

    // ---- a1/a2: this CTA's share of the merge path --------------------------
    if (tid < 6) counts[tid] = 0;
    if (tid == 0) init_ring_barriers(full_v, NSV, NSO);
    __syncthreads();
    CtaRange cr;
    if (!cta_range<NTHREADS, OffT>(p, counts, cr)) return;
    const int64_t o0 = cr.o0, W = cr.W, Dlo = cr.Dlo, Dhi = cr.Dhi;
    const int64_t Ilo = cr.Ilo, Ihi = cr.Ihi, Rlo = cr.Rlo, Rhi = cr.Rhi;

    // ---- streams -------------------------------------------------------------
    const uint64_t esz = static_cast<uint64_t>(p.F) * sizeof(T);
    const uint64_t vbase = reinterpret_cast<uint64_t>(p.values);
    const uint64_t obase = reinterpret_cast<uint64_t>(p.offsets);
    const Stream vs = make_stream(vbase, static_cast<uint64_t>(N) * esz, vbase + Rlo * esz,
                                  vbase + Rhi * esz, VCHUNK);
    const Stream os = make_stream(obase, static_cast<uint64_t>(S + 1) * OSZ, obase + Ilo * OSZ,
                                  obase + (Ihi + 1) * OSZ, OCHUNK);

    if (tid >= NT) {
        if (tid == NT)
            producer_loop<VRING, VCHUNK, ORING, OCHUNK>(vs, os, vring, oring, full_v, empty_v, full_o,
                                                        empty_o, p.status);
        return;
    }

    // ---- consumers -------------------------------------------------------------
    const int G = p.G;
    const int K = p.K;
    const int sl = tid / G;
    const int g = tid - sl * G;
    const int lane = tid & 31;
    const int warp = tid >> 5;
    const int64_t T_items = static_cast<int64_t>(NT / G) * K;
    const int F = p.F;
    const int mean = p.mean;
    const bool want_arg = (OP != OP_SUM) && p.out_arg != nullptr;
    T* out = static_cast<T*>(p.out);
    PartElem* tails = static_cast<PartElem*>(p.ws_parts);
    PartElem* heads = tails + static_cast<int64_t>(p.P) * F;

    // offsets / keys from the ring (entries Ilo .. Ihi only)
    auto off_r = [&](int64_t s) -> int64_t {
        const uint32_t at = static_cast<uint32_t>((obase + static_cast<uint64_t>(s) * OSZ) - os.A0) &
                            (ORING - 1);
        return clamp_off(*reinterpret_cast<const OffT*>(oring + at), N);
    };
    auto key_r = [&](int64_t s) -> int64_t { return off_r(s + 1) - o0 + s; };
    // #{s in [a, b) : key(s) < x}
    auto count_ends = [&](int64_t a, int64_t b, int64_t x) -> int64_t {
        while (a < b) {
            const int64_t mid = a + ((b - a) >> 1);
            if (key_r(mid) < x)
                a = mid + 1;
            else
                b = mid;
        }
        return a;
    };
    // column of (thread g, element e); < F when valid
    auto col_of = [&](int e) -> int { return (g + (e / VEC) * G) * VEC + (e % VEC); };

    const bool cta_head_spans = (Ilo < S) && (clamp_off(__ldg(&offs[Ilo]), N) < Rlo);
    bool head_pending = cta_head_spans;

    C carry[NVEC];
#pragma unroll
    for (int e = 0; e < NVEC; ++e) carry[e] = CO::ident();

    int64_t d = Dlo, i = Ilo, j = Rlo;
    int64_t vw = 0, vrel = 0, ow = 0, orel = 0;
    bool ok = true;

    while (d < Dhi) {
        // (A) offsets window [i, cap_i]
        const int64_t cap_i = i + p.max_ends < Ihi ? i + p.max_ends : Ihi;
        {
            const int64_t need =
                static_cast<int64_t>((obase + static_cast<uint64_t>(cap_i + 1) * OSZ - 1 - os.A0) / OCHUNK);
            for (; ok && ow <= need && ow < os.nch; ++ow)
                ok = wait_bounded(&full_o[ow % NSO], static_cast<uint32_t>((ow / NSO) & 1), p.status,
                                  STATUS_CONSUMER_TIMEOUT);
        }
        // (B) end of this tile
        int64_t d_end = d + T_items < Dhi ? d + T_items : Dhi;
        int64_t i_end;
        if (ok && cap_i < Ihi && key_r(cap_i - 1) < d_end) {
            i_end = cap_i;
            d_end = key_r(cap_i - 1) + 1;
        } else {
            i_end = ok ? count_ends(i, cap_i, d_end) : i;
        }
        // Valid offsets always give i <= i_end <= cap_i and d < d_end; the
        // clamps only keep malformed offsets from stalling the loop.
        i_end = i_end < i ? i : (i_end > cap_i ? cap_i : i_end);
        if (d_end <= d) d_end = d + 1;
        int64_t j_end = d_end - i_end + o0;
        j_end = j_end < j ? j : (j_end > Rhi ? Rhi : j_end);
        // (C) values window [j, j_end)
        if (j_end > j) {
            const int64_t need = static_cast<int64_t>((vbase + static_cast<uint64_t>(j_end) * esz - 1 - vs.A0) / VCHUNK);
            for (; ok && vw <= need && vw < vs.nch; ++vw)
                ok = wait_bounded(&full_v[vw % NSV], static_cast<uint32_t>((vw / NSV) & 1), p.status,
                                  STATUS_CONSUMER_TIMEOUT);
        }
        // (D) all consumers agree the data is there; previous tile fully read
        if (!named_bar_and<NT>(ok)) return;

        // (E) this slot's K items
        const int64_t x0 = d + static_cast<int64_t>(sl) * K;
        const int64_t x1 = x0 + K < d_end ? x0 + K : d_end;
        bool has_end = false;
        int64_t head_seg = -1, head_len = 0;
        Acc<T> acc[NVEC], head[NVEC];
#pragma unroll
        for (int e = 0; e < NVEC; ++e) {
            acc[e] = RD::ident();
            head[e] = RD::ident();
        }
        if (x0 < d_end) {
            int64_t s = count_ends(i, i_end, x0);
            const int64_t r0 = x0 - s + o0;
            const int n_items = static_cast<int>(x1 - x0);
            // tile-relative 32-bit row coordinates
            int32_t rr = static_cast<int32_t>(r0 - j);
            int64_t ne64 = s < i_end ? off_r(s + 1) - j : INT32_MAX;
            int32_t ne = static_cast<int32_t>(ne64 < INT32_MAX ? ne64 : INT32_MAX);
            int64_t seg_start = off_r(s);
            const int32_t row_cta0 = static_cast<int32_t>(j - Rlo);
            const uint32_t vb0 = static_cast<uint32_t>((vbase + static_cast<uint64_t>(j) * esz) - vs.A0);
            for (int k = 0; k < n_items; ++k) {
                if (rr < ne) {
                    const uint32_t rowb = vb0 + static_cast<uint32_t>(rr) * static_cast<uint32_t>(esz);
#pragma unroll
                    for (int v = 0; v < NV; ++v) {
                        const int cg = g + v * G;
                        if (cg * VEC < F) {
                            const uint32_t at = (rowb + static_cast<uint32_t>(cg * VEC) * 4u) & (VRING - 1);
                            if constexpr (VEC == 4) {
                                const uint4 u4 = *reinterpret_cast<const uint4*>(vring + at);
                                RD::add(acc[v * 4 + 0], from_bits<T>(u4.x), row_cta0 + rr);
                                RD::add(acc[v * 4 + 1], from_bits<T>(u4.y), row_cta0 + rr);
                                RD::add(acc[v * 4 + 2], from_bits<T>(u4.z), row_cta0 + rr);
                                RD::add(acc[v * 4 + 3], from_bits<T>(u4.w), row_cta0 + rr);
                            } else {
                                RD::add(acc[v], *reinterpret_cast<const T*>(vring + at), row_cta0 + rr);
                            }
                        }
                    }
                    ++rr;
                } else {
                    const int64_t seg_end = ne64 + j;
                    if (!has_end) {
#pragma unroll
                        for (int e = 0; e < NVEC; ++e) head[e] = acc[e];
                        head_seg = s;
                        head_len = seg_end - seg_start;
                        has_end = true;
                    } else {
                        const int64_t len = seg_end - seg_start;
#pragma unroll
                        for (int e = 0; e < NVEC; ++e) {
                            const int col = col_of(e);
                            if (col < F) {
                                T v;
                                int64_t a;
                                finish_acc<T, OP>(acc[e], len, mean, Rlo, v, a);
                                out[s * F + col] = v;
                                if (want_arg) p.out_arg[s * F + col] = a;
                            }
                        }
                    }
#pragma unroll
                    for (int e = 0; e < NVEC; ++e) acc[e] = RD::ident();
                    seg_start = seg_end;
                    ++s;
                    ne64 = s < i_end ? off_r(s + 1) - j : INT32_MAX;
                    ne = static_cast<int32_t>(ne64 < INT32_MAX ? ne64 : INT32_MAX);
                }
            }
        }

        // (F) segmented scan of the slot tails (flag = slot holds a segment end)
        bool fl = has_end;
        Acc<T> inc[NVEC];
#pragma unroll
        for (int e = 0; e < NVEC; ++e) inc[e] = acc[e];
        if (G < 32) {
            for (int o = G; o < 32; o <<= 1) {
                const bool pf = __shfl_up_sync(0xffffffffu, fl, o);
                Acc<T> pv[NVEC];
#pragma unroll
                for (int e = 0; e < NVEC; ++e) {
                    pv[e].v = from_bits<T>(__shfl_up_sync(0xffffffffu, bits_of(inc[e].v), o));
                    pv[e].row = __shfl_up_sync(0xffffffffu, inc[e].row, o);
                }
                if (lane >= o) {
#pragma unroll
                    for (int e = 0; e < NVEC; ++e)
                        if (!fl) inc[e] = RD::comb(pv[e], inc[e]);
                    fl = fl || pf;
                }
            }
        }
        const int NB = G <= 32 ? NT / 32 : NT / G;
        const int b = G <= 32 ? warp : sl;
        if (G <= 32 ? (lane >= 32 - G) : true) {
#pragma unroll
            for (int e = 0; e < NVEC; ++e) {
                scan_v[(b * G + g) * NVEC + e] = inc[e].v;
                scan_r[(b * G + g) * NVEC + e] = inc[e].row;
            }
            if (g == 0) scan_f[b] = fl ? 1 : 0;
        }
        // exclusive prefix of the warp (in-warp part)
        bool ef = false;
        Acc<T> ev[NVEC];
#pragma unroll
        for (int e = 0; e < NVEC; ++e) ev[e] = RD::ident();
        if (G < 32) {
            const bool pf = __shfl_up_sync(0xffffffffu, fl, G);
            Acc<T> pv[NVEC];
#pragma unroll
            for (int e = 0; e < NVEC; ++e) {
                pv[e].v = from_bits<T>(__shfl_up_sync(0xffffffffu, bits_of(inc[e].v), G));
                pv[e].row = __shfl_up_sync(0xffffffffu, inc[e].row, G);
            }
            if (lane >= G) {
#pragma unroll
                for (int e = 0; e < NVEC; ++e) ev[e] = pv[e];
                ef = pf;
            }
        }
        named_bar_sync<NT>();
        // Neither ring is read again for this tile: hand back the stages that
        // hold only rows before j_end and offsets entries before i_end.
        if (tid == 0) {
            const uint64_t vlimit = vbase + static_cast<uint64_t>(j_end) * esz;
            while (vrel < vw && vs.A0 + static_cast<uint64_t>(vrel + 1) * VCHUNK <= vlimit) {
                mbar_arrive(&empty_v[vrel % NSV]);
                ++vrel;
            }
            const uint64_t olimit = obase + static_cast<uint64_t>(i_end) * OSZ;
            while (orel < ow && os.A0 + static_cast<uint64_t>(orel + 1) * OCHUNK <= olimit) {
                mbar_arrive(&empty_o[orel % NSO]);
                ++orel;
            }
        }
        // blocks before mine, and the whole tile
        bool bf_pre = false, tf = false;
        Acc<T> bv_pre[NVEC], tv[NVEC];
#pragma unroll
        for (int e = 0; e < NVEC; ++e) {
            tv[e] = RD::ident();
            bv_pre[e] = RD::ident();
        }
        for (int bb = 0; bb < NB; ++bb) {
            if (bb == b) {
                bf_pre = tf;
#pragma unroll
                for (int e = 0; e < NVEC; ++e) bv_pre[e] = tv[e];
            }
            const bool f = scan_f[bb] != 0;
#pragma unroll
            for (int e = 0; e < NVEC; ++e) {
                Acc<T> a;
                a.v = scan_v[(bb * G + g) * NVEC + e];
                a.row = scan_r[(bb * G + g) * NVEC + e];
                tv[e] = f ? a : RD::comb(tv[e], a);
            }
            tf = tf || f;
        }
        // full exclusive prefix = blocks before, then the in-warp part
        if (!ef) {
#pragma unroll
            for (int e = 0; e < NVEC; ++e) ev[e] = RD::comb(bv_pre[e], ev[e]);
            ef = bf_pre;
        }

        // (F') the slot's first segment end: prefix + head
        const bool resolve_cta_head = head_pending && i_end > i;
        if (has_end) {
            const bool to_scratch = head_pending && head_seg == Ilo;
            const int64_t len = head_len;
#pragma unroll
            for (int e = 0; e < NVEC; ++e) {
                const int col = col_of(e);
                if (col >= F) continue;
                const Acc<T> hv = RD::comb(ev[e], head[e]);
                if (!ef) {
                    const C hc = CO::then(carry[e], hv);
                    if (to_scratch) {
                        if constexpr (OP == OP_SUM && kIsFloat<T>) heads[static_cast<int64_t>(cta) * F + col] = to_part(hc);
                        else heads[static_cast<int64_t>(cta) * F + col] = to_part<T, OP>(hc, Rlo);
                    } else {
                        T v;
                        int64_t a;
                        if constexpr (OP == OP_SUM && kIsFloat<T>) {
                            finish_carry(hc, len, mean, v);
                            a = -1;
                        } else {
                            finish_acc<T, OP>(hc, len, mean, Rlo, v, a);
                        }
                        out[head_seg * F + col] = v;
                        if (want_arg) p.out_arg[head_seg * F + col] = a;
                    }
                } else {
                    T v;
                    int64_t a;
                    finish_acc<T, OP>(hv, len, mean, Rlo, v, a);
                    out[head_seg * F + col] = v;
                    if (want_arg) p.out_arg[head_seg * F + col] = a;
                }
            }
        }
        // carry into the next tile
#pragma unroll
        for (int e = 0; e < NVEC; ++e) carry[e] = tf ? CO::from(tv[e]) : CO::then(carry[e], tv[e]);

        // (G) the CTA's first segment began in an earlier CTA: join the ticket
        if (resolve_cta_head) {
            __threadfence();
            named_bar_sync<NT>();
            if (tid == 0) {
                const int64_t f = clamp_off(__ldg(&offs[Ilo]), N) - o0 + Ilo;
                int pc = static_cast<int>(f / W);
                pc = pc < 0 ? 0 : (pc > cta ? cta : pc);
                bcast[0] = ticket_arrive(p.ws_tickets, cta, cta - pc + 1, p.gen) ? 1 : 0;
                bcast[1] = pc;
            }
            named_bar_sync<NT>();
            if (bcast[0]) {
                __threadfence();
                const int64_t len = clamp_off(__ldg(&offs[Ilo + 1]), N) - clamp_off(__ldg(&offs[Ilo]), N);
                combine_store<T, OP>(p, tails, heads, bcast[1], cta, Ilo, len, tid, NT);
            }
            head_pending = false;
        }

        d = d_end;
        i = i_end;
        j = j_end;
    }

    // ---- a6: the segment still open at the end of the range ------------------
    if (Ihi < S && clamp_off(__ldg(&offs[Ihi]), N) < Rhi) {
        if (sl == 0) {
#pragma unroll
            for (int e = 0; e < NVEC; ++e) {
                const int col = col_of(e);
                if (col >= F) continue;
                if constexpr (OP == OP_SUM && kIsFloat<T>) tails[static_cast<int64_t>(cta) * F + col] = to_part(carry[e]);
                else tails[static_cast<int64_t>(cta) * F + col] = to_part<T, OP>(carry[e], Rlo);
            }
        }
        __threadfence();
        named_bar_sync<NT>();
        if (tid == 0) {
            const int64_t ob = clamp_off(__ldg(&offs[Ihi]), N);
            const int64_t oe = clamp_off(__ldg(&offs[Ihi + 1]), N);
            const int64_t f = ob - o0 + Ihi;
            const int64_t e = (oe > ob ? oe : ob) - o0 + Ihi;
            int pc = static_cast<int>(f / W);
            int qc = static_cast<int>(e / W);
            pc = pc < 0 ? 0 : (pc > cta ? cta : pc);
            qc = qc <= cta ? cta + 1 : qc;
            const bool last = qc < p.P && ticket_arrive(p.ws_tickets, qc, qc - pc + 1, p.gen);
            bcast[0] = last ? 1 : 0;
            bcast[1] = pc;
            bcast[2] = qc;
        }
        named_bar_sync<NT>();
        if (bcast[0]) {
            __threadfence();
            const int64_t len = clamp_off(__ldg(&offs[Ihi + 1]), N) - clamp_off(__ldg(&offs[Ihi]), N);
            combine_store<T, OP>(p, tails, heads, bcast[1], bcast[2], Ihi, len, tid, NT);
        }
    }
}

}  // namespace segred
