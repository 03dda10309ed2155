// dgt_r4esc.cuh -- R4 escape handling shared by the matrix-vector kernels
// (batch-1 product and MoE expert gather): the row-segment escape counts of a
// window of 512-column rounds, and the exponent table with its rank-15 entry
// replaced by an escaped weight's exponent.
//
// R4 layout (Binade README, "Runtime layout"): a rank >= 15 is stored as
// nibble 15 and its rank appended to the escape list in flat order;
// seg[row * nseg + j] counts the escapes before column 512 j of the row.  A
// 512-column round of one row therefore holds seg[.. + j + 1] - seg[.. + j]
// escapes, and the i-th of them, in column order, is esc[seg[.. + j] + i].
//
// The helpers take any argument block A with the fields esc, n_esc, seg and
// nseg.
#pragma once
#include "dgt_device.cuh"

namespace dgt {

// Escape information of up to 32 rounds [jbase, jbase + 32) of one row:
// lane t holds round jbase + t.
struct SegInfo {
    uint32_t cnt, base, fexp, fexp1, emask;
};

template <class A>
__device__ __forceinline__ SegInfo load_seginfo(const A &a, const uint8_t *table_s, uint64_t row,
                                                uint32_t jbase, uint32_t j1, uint32_t lane) {
    SegInfo g;
    g.cnt = g.base = g.fexp = g.fexp1 = 0;
    const uint32_t j = jbase + lane;
    if (j < j1) {
        const uint32_t *sp = a.seg + row * a.nseg + j;
        g.base = sp[0];
        g.cnt = sp[1] - g.base;
        if (g.cnt && g.base < a.n_esc) g.fexp = table_s[a.esc[g.base]];
        if (g.cnt >= 2 && (uint64_t)g.base + 1 < a.n_esc) g.fexp1 = table_s[a.esc[g.base + 1]];
    }
    g.emask = __ballot_sync(DGT_FULL, g.cnt != 0);
    return g;
}

// Escape counts of the next unit's first 32 rounds (lane t: round j0 + t) and
// the ranks of their first two escapes, loaded ahead of use.
struct SegPre {
    uint32_t cnt, base, e0, e1;
};

template <class A>
__device__ __forceinline__ void seg_issue(const A &a, uint64_t row, uint32_t jb, uint32_t j1,
                                          uint32_t lane, SegPre &p) {
    p.cnt = p.base = 0;
    const uint32_t j = jb + lane;
    if (j < j1) {
        const uint32_t *sp = a.seg + row * a.nseg + j;
        p.base = sp[0];
        p.cnt = sp[1] - p.base;
    }
}

template <class A>
__device__ __forceinline__ void seg_issue_esc(const A &a, SegPre &p) {
    p.e0 = (p.cnt >= 1 && p.base < a.n_esc) ? a.esc[p.base] : 0u;
    p.e1 = (p.cnt >= 2 && (uint64_t)p.base + 1 < a.n_esc) ? a.esc[p.base + 1] : 0u;
}

__device__ __forceinline__ SegInfo seg_finish(const SegPre &p, const uint8_t *table_s) {
    SegInfo g;
    g.cnt = p.cnt;
    g.base = p.base;
    g.fexp = table_s[p.e0];
    g.fexp1 = table_s[p.e1];
    g.emask = __ballot_sync(DGT_FULL, p.cnt != 0);
    return g;
}

// A copy of v the compiler cannot trace back to its source.
__device__ __forceinline__ uint32_t opaque(uint32_t v) {
    uint32_t r;
    asm volatile("mov.b32 %0, %1;" : "=r"(r) : "r"(v));
    return r;
}

// The exponent table with the rank-15 entry replaced by exponent e.
__device__ __forceinline__ R4Lut lut15(const R4Lut &L, uint32_t e) {
    R4Lut o = L;
    o.h3 = prmt(L.h3, e >> 1, 0x4210u);
    o.l1 = (L.l1 & 0x7FFFFFFFu) | ((e & 1u) << 31);
    return o;
}

// Per round of a seg window (lane t: round jbase + t): the two table words
// of the round's decode (rank 15 -> the exponent of its first escape when it
// has one) and a mask of rounds with two or more escapes.
struct RoundLut {
    uint32_t h3, l1, multi;
};

__device__ __forceinline__ RoundLut round_luts(const SegInfo &g, const R4Lut &L) {
    RoundLut o;
    const R4Lut m = lut15(L, g.fexp);
    o.h3 = g.cnt ? m.h3 : L.h3;
    o.l1 = g.cnt ? m.l1 : L.l1;
    o.multi = __ballot_sync(DGT_FULL, g.cnt >= 2);
    return o;
}

// The same per piece from the round summaries (lane r: round r's word,
// min(c, 255) | x0 << 8 | x1 << 16 | x2 << 24): rank 15 -> x0 where c >= 1.
__device__ __forceinline__ RoundLut round_luts_rec(uint32_t rec, const R4Lut &L) {
    RoundLut o;
    const uint32_t c = rec & 0xFFu;
    const R4Lut m = lut15(L, (rec >> 8) & 0xFFu);
    o.h3 = c ? m.h3 : L.h3;
    o.l1 = c ? m.l1 : L.l1;
    o.multi = __ballot_sync(DGT_FULL, c >= 2);
    return o;
}

// A round with two or three escapes, each in a different lane: this lane's
// escape exponent from the round's summary word (its place among the escaped
// lanes picks x0, x1 or x2).  Returns false (the general patch is needed)
// for more escapes, a lane with two, or counts that disagree.
__device__ __forceinline__ bool rec_exponent(uint32_t rec, uint2 nv, uint32_t lane, uint32_t &e) {
    const uint32_t c = rec & 0xFFu;
    const uint32_t k = __popc(nib15_mask(nv.x)) + __popc(nib15_mask(nv.y));
    const uint32_t bal = __ballot_sync(DGT_FULL, k != 0);
    if (c > 3 || __any_sync(DGT_FULL, k > 1) || (uint32_t)__popc(bal) != c) return false;
    const uint32_t q = __popc(bal & ((1u << lane) - 1u));
    e = k ? (rec >> (8 + 8 * q)) & 0xFFu : 0u;
    return true;
}

// The same when a lane may hold two of the round's (at most three) escapes:
// e1 = this lane's first escape exponent, and for a lane with two, e2 = the
// second's and i2 = its weight index (0..15) in the lane's 16-weight chunk
// (i2 = 16 otherwise).  The lane decodes with the rank-15 entry set to e1 and
// then rewrites weight i2's exponent to e2.  Returns false for more than
// three escapes, three in one lane, or counts that disagree.
__device__ __forceinline__ bool rec_exponent2(uint32_t rec, uint2 nv, uint32_t lane, uint32_t &e1, uint32_t &e2,
                                              uint32_t &i2) {
    const uint32_t c = rec & 0xFFu;
    const uint32_t m0 = nib15_mask(nv.x), m1 = nib15_mask(nv.y);
    const uint32_t k = __popc(m0) + __popc(m1);
    const uint32_t b1 = __ballot_sync(DGT_FULL, k == 1), b2 = __ballot_sync(DGT_FULL, k == 2);
    if (c > 3 || __any_sync(DGT_FULL, k > 2) || (uint32_t)(__popc(b1) + 2 * __popc(b2)) != c) return false;
    const uint32_t lt = (1u << lane) - 1u;
    const uint32_t q = __popc(b1 & lt) + 2u * __popc(b2 & lt);   // escapes in the lanes before this one
    e1 = k ? (rec >> (8 + 8 * q)) & 0xFFu : 0u;
    e2 = 0;
    i2 = 16;
    if (k == 2) {
        e2 = (rec >> (16 + 8 * q)) & 0xFFu;   // q <= 1: the two fit in x0..x2
        const uint32_t lo_rest = m0 & (m0 - 1u);   // m0 without its first escape
        i2 = m0 == 0 ? 8 + ((__ffs(m1 & (m1 - 1u)) - 1) >> 2)
                     : (lo_rest ? (__ffs(lo_rest) - 1) >> 2 : 8 + ((__ffs(m1) - 1) >> 2));
    }
    return true;
}

// A round whose segment holds two or more escapes, when every lane holds at
// most one of them: the exponent of this lane's escape (its place among the
// round's escaped lanes; the first two come prefetched).  Returns false when
// a lane holds more than one, or the counts disagree.
template <class A>
__device__ __forceinline__ bool multi_exponent(const A &a, const SegInfo &g, uint32_t bit, uint2 nv,
                                               const uint8_t *table_s, uint32_t lane, uint32_t &e) {
    const uint32_t c = __shfl_sync(DGT_FULL, g.cnt, bit);
    const uint32_t e0 = __shfl_sync(DGT_FULL, g.fexp, bit);
    const uint32_t e1 = __shfl_sync(DGT_FULL, g.fexp1, bit);
    const uint32_t b = __shfl_sync(DGT_FULL, g.base, bit);
    const uint32_t k = __popc(nib15_mask(nv.x)) + __popc(nib15_mask(nv.y));
    const uint32_t bal = __ballot_sync(DGT_FULL, k != 0);
    if (__any_sync(DGT_FULL, k > 1) || (uint32_t)__popc(bal) != c) return false;
    const uint32_t q = __popc(bal & ((1u << lane) - 1u));
    e = q == 0 ? e0 : e1;
    if (k && q >= 2) e = (uint64_t)b + q < a.n_esc ? table_s[a.esc[b + q]] : 0u;
    return true;
}

// Any R4 round with escapes, in line: decode, then patch every escaped weight
// from the segment's escape ranks (staged in shared memory); c escapes from
// index b on.
template <class A>
__device__ __forceinline__ void r4_round_general_cb(const A &a, const R4Lut &L, uint2 nv, uint4 sv, uint32_t c,
                                                    uint32_t b, uint8_t *escb, const uint8_t *table_s,
                                                    uint32_t lane, bool act, uint32_t p[8]) {
    r4_dec16(nv, sv, L, p);
    const uint32_t m0 = act ? nib15_mask(nv.x) : 0u;
    const uint32_t m1 = act ? nib15_mask(nv.y) : 0u;
    const uint32_t cc = c > DGT_SEG ? DGT_SEG : c;
    for (uint32_t i = lane; i < cc; i += 32) escb[i] = (uint64_t)b + i < a.n_esc ? a.esc[b + i] : 0;
    __syncwarp();
    patch_escapes(p, m0, m1, cc, escb, table_s);
    __syncwarp();
}

template <class A>
__device__ __forceinline__ void r4_round_general(const A &a, const R4Lut &L, uint2 nv, uint4 sv,
                                                 const SegInfo &g, uint32_t bit, uint8_t *escb,
                                                 const uint8_t *table_s, uint32_t lane, bool act, uint32_t p[8]) {
    const uint32_t c = __shfl_sync(DGT_FULL, g.cnt, bit);
    const uint32_t b = __shfl_sync(DGT_FULL, g.base, bit);
    r4_round_general_cb(a, L, nv, sv, c, b, escb, table_s, lane, act, p);
}

}  // namespace dgt
