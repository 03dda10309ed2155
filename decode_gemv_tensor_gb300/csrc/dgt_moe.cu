// dgt_moe.cu -- mixture-of-experts expert-gather products with R4 (or BF16)
// expert weights, in the batch-1 product's fixed summation order.
//
// Binade README, "How it works" (Exactness: "the matvec, the MoE expert
// gather and the GEMM" follow one order) and "Limitations" (the fused kernels
// cover "every expert product").  The experts of one projection are stacked
// as one tensor [E * Ne, K] with one rank table.  For token t and slot j,
// y[t, j, :] = W[ids[t, j]] x_t in the order of dgt_gemv (plan S(Ne, K));
// with routing weights p, out[t, :] = fmaf chain over j = 0..topk-1 of
// p[t, j] * y[t, j, :], starting from +0.
//
// Three launches:
//  1. k_moe_route (one CTA): counts the pairs per expert, lists the experts
//     in use, and places every pair (t, j) in its expert's list in (t, j)
//     order -- deterministic, no atomics in the placement.
//  2. k_moe: the rows of the experts in use are split over one CTA per SM by
//     cost (row passes and token chains); a producer warp streams each consumer warp's rows into shared
//     memory with bulk copies, and the consumer decodes each 16-weight lane
//     chunk once and runs one fmaf chain per routed token (up to 4 per pass
//     over the row), x read through L1; at each slice end the chains are
//     butterfly-reduced into the workspace.
//  3. k_moe_combine: adds each pair's slices left to right (y) and applies
//     the routing weights in slot order (out).
// With few (token, slot) pairs (a decode step: one token, or one slot per
// token) each pair instead runs as a block of the batch-1 product's bulk-copy
// kernel, then the combine over its results if routing weights are given.
#include <cuda_runtime.h>

#include "../../include/dgt.h"
#include "dgt_device.cuh"
#include "dgt_internal.h"
#include "dgt_launch.h"
#include "dgt_r4esc.cuh"

namespace dgt {

constexpr uint32_t MOE_MAX_EXPERTS = 4096;
constexpr uint32_t MOE_MAX_PAIRS = 1u << 16;

struct MoeArgs {
    const uint8_t *sm, *nib, *esc;
    const uint32_t *seg;
    const uint32_t *rsum;   // per-round escape summaries (second part of seg)
    const uint16_t *W;
    const int32_t *ids;
    const float *p;
    const uint16_t *x;
    float *y32;
    uint16_t *out;
    float *out32;
    uint64_t cols, nseg, n_esc, ne;
    uint32_t n_experts, tokens, topk, J, S;
    int bulk;          // rows stream through bulk copies (else direct loads)
    uint32_t xs_slots; // tokens whose x fits in shared memory
    R4Lut L;
    uint8_t table[256];
    // workspace
    uint32_t *eoff;    // n_experts + 1
    uint32_t *elist;   // pairs: t << 8 | j
    uint32_t *active;  // experts in use, then the count at active[pairs]
    uint32_t *rbound;  // CTA b takes active rows [rbound[b], rbound[b + 1])
    uint32_t grid;     // CTAs of the gather kernel
    float *partial;    // pairs * ne * S
    int32_t *status;
    uint32_t spin;     // polls a consumer waits for a piece before it gives up
};

static inline size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

constexpr uint32_t MOE_MAX_CTAS = 1024;
constexpr uint32_t MAXT = 4;     // tokens per pass over a row (more stream the row again)

struct WsLayout {
    size_t eoff, elist, active, rbound, partial, total;
};

static inline WsLayout moe_ws_layout(uint32_t n_experts, uint64_t ne, uint64_t cols, uint32_t tokens,
                                     uint32_t topk) {
    const uint64_t pairs = (uint64_t)tokens * topk;
    const int S = dgt_plan_slices(ne, cols);
    WsLayout l;
    l.eoff = 0;
    l.elist = align256(l.eoff + 4ull * (n_experts + 1));
    l.active = align256(l.elist + 4ull * pairs);
    l.rbound = align256(l.active + 4ull * (pairs + 1));
    l.partial = align256(l.rbound + 4ull * (MOE_MAX_CTAS + 1));
    l.total = align256(l.partial + 4ull * pairs * ne * (uint64_t)S);
    return l;
}

// Exclusive prefix sum over a 1024-thread block of one 64-bit value per
// thread; *total gets the block sum.
__device__ __forceinline__ uint64_t block_excl_scan64(uint64_t v, uint64_t *sw, uint64_t *total) {
    const uint32_t lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    uint64_t x = v;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        const uint64_t y = __shfl_up_sync(DGT_FULL, x, d);
        if (lane >= (uint32_t)d) x += y;
    }
    if (lane == 31) sw[w] = x;
    __syncthreads();
    if (w == 0) {
        uint64_t t = sw[lane];
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
            const uint64_t y = __shfl_up_sync(DGT_FULL, t, d);
            if (lane >= (uint32_t)d) t += y;
        }
        sw[lane] = t;
    }
    __syncthreads();
    const uint64_t before = (w ? sw[w - 1] : 0ull) + x - v;
    *total = sw[31];
    __syncthreads();
    return before;
}

// Cost of one row of an expert with nt routed pairs: its passes over the row
// (each a stream of the row, weighted as ROW_COST token chains) and its chains.
constexpr uint64_t ROW_COST = 2;
__device__ __forceinline__ uint64_t moe_row_cost(uint32_t nt) {
    return ((nt + MAXT - 1) / MAXT) * ROW_COST + nt;
}

// One CTA: count the pairs per expert, list the experts in use, place every
// pair (t, j) in its expert's list in (t, j) order (deterministic, no
// atomics in the placement), and split the rows of the experts in use over
// the gather kernel's CTAs by cost (passes and token chains), so that a CTA
// whose rows belong to an expert with many tokens gets fewer rows.
__global__ void __launch_bounds__(1024) k_moe_route(MoeArgs a) {
    // cnt (per expert) and, once every thread has read it, the cost prefix
    // (per active expert) share one array
    __shared__ uint64_t cost[MOE_MAX_EXPERTS + 1];
    __shared__ uint64_t sw[32];
    pdl_trigger();
    pdl_wait();
    uint32_t *cnt = reinterpret_cast<uint32_t *>(cost);
    const uint32_t P = a.tokens * a.topk, tid = threadIdx.x;
    for (uint32_t e = tid; e < a.n_experts; e += blockDim.x) cnt[e] = 0;
    __syncthreads();
    for (uint32_t q = tid; q < P; q += blockDim.x) {
        const int32_t e = a.ids[q];
        if (e < 0 || (uint32_t)e >= a.n_experts) {
            set_status(a.status, DGT_ERR_ARG);
            continue;
        }
        atomicAdd(&cnt[e], 1u);
    }
    __syncthreads();
    // eoff (pairs before each expert) and the active list, four experts per thread
    constexpr uint32_t PER = MOE_MAX_EXPERTS / 1024;
    uint32_t c4[PER], f4[PER];
    uint64_t cs = 0, fs = 0;
#pragma unroll
    for (uint32_t i = 0; i < PER; i++) {
        const uint32_t e = tid * PER + i;
        c4[i] = e < a.n_experts ? cnt[e] : 0u;
        f4[i] = c4[i] != 0;
        cs += c4[i];
        fs += f4[i];
    }
    uint64_t ptot, atot;
    uint64_t o = block_excl_scan64(cs, sw, &ptot);
    uint64_t na = block_excl_scan64(fs, sw, &atot);
    const uint32_t nact = (uint32_t)atot;
#pragma unroll
    for (uint32_t i = 0; i < PER; i++) {
        const uint32_t e = tid * PER + i;
        if (e < a.n_experts) {
            a.eoff[e] = (uint32_t)o;
            if (c4[i]) {
                a.active[na] = e;
                cost[na] = a.ne * moe_row_cost(c4[i]);
            }
        }
        o += c4[i];
        na += f4[i];
    }
    if (tid == 0) {
        a.eoff[a.n_experts] = (uint32_t)ptot;
        a.active[P] = nact;
    }
    __syncthreads();
    // cost prefix over the active experts (in active[] order)
    uint64_t cv[PER], csum = 0;
#pragma unroll
    for (uint32_t i = 0; i < PER; i++) {
        const uint32_t k = tid * PER + i;
        cv[i] = k < nact ? cost[k] : 0ull;
        csum += cv[i];
    }
    uint64_t ctot;
    uint64_t cb = block_excl_scan64(csum, sw, &ctot);
#pragma unroll
    for (uint32_t i = 0; i < PER; i++) {
        const uint32_t k = tid * PER + i;
        if (k < nact) cost[k] = cb;
        cb += cv[i];
    }
    if (tid == 0) cost[nact] = ctot;
    __syncthreads();
    // CTA b starts at the row where the cost b * ctot / grid falls
    for (uint32_t b = tid; b <= a.grid; b += blockDim.x) {
        uint64_t row = (uint64_t)nact * a.ne;
        if (b < a.grid && nact) {
            const uint64_t c = ctot * b / a.grid;
            uint32_t lo = 0, hi = nact - 1;   // largest k with cost[k] <= c
            while (lo < hi) {
                const uint32_t mid = (lo + hi + 1) / 2;
                if (cost[mid] <= c) lo = mid;
                else hi = mid - 1;
            }
            const uint64_t rc = (cost[lo + 1] - cost[lo]) / a.ne;
            uint64_t r = rc ? (c - cost[lo]) / rc : 0;
            if (r > a.ne) r = a.ne;
            row = (uint64_t)lo * a.ne + r;
        }
        a.rbound[b] = (uint32_t)row;
    }
    // placement
    for (uint32_t q = tid; q < P; q += blockDim.x) {
        const int32_t e = a.ids[q];
        if (e < 0 || (uint32_t)e >= a.n_experts) continue;
        uint32_t before = 0;
        for (uint32_t q2 = 0; q2 < q; q2++) before += a.ids[q2] == e;
        a.elist[a.eoff[e] + before] = ((q / a.topk) << 8) | (q % a.topk);
    }
}

// ---------------------------------------------------------------------------
// Expert rows streamed through shared memory.  The rows of the experts in use
// (active[] order, expert by expert) are split over one CTA per SM by cost;
// consumer warp w of a CTA takes its rows w, w + MNW, ...  A producer warp
// keeps each consumer's ring of stages full with 1-D bulk copies of pieces of
// MCV rounds (R4: 6 in two stages, BF16: 4 in two stages; polling the rings'
// "empty" barriers without blocking).  For each
// row a warp decodes every 16-weight lane chunk once and runs one fmaf chain
// per routed token (up to MAXT per pass over the row; more tokens stream the
// row again), x read through L1.  At every slice end the chains are
// butterfly-reduced into the workspace.
// ---------------------------------------------------------------------------
#ifndef DGT_MOE_MNW
#define DGT_MOE_MNW 15
#endif
#ifndef DGT_MOE_MPW
#define DGT_MOE_MPW 1
#endif
constexpr int MNW = DGT_MOE_MNW;  // consumer warps
constexpr int MPW = DGT_MOE_MPW;  // producer warps (producer warp p serves consumers p, p + MPW, ...)
template <bool R4>
constexpr uint32_t MCV = R4 ? 6u : 4u;   // rounds per piece (R4: a 2816-column expert row in one piece)
constexpr uint32_t MNS_MAX = 2;  // stages per consumer
constexpr uint32_t XS_BYTES = 64 * 1024;   // x of the CTA's tokens staged in shared memory
constexpr uint32_t XS_TOKENS = 1024;       // token bitmap / slot map size

template <bool R4>
struct MoeStage {
    static constexpr uint32_t BYTES = R4 ? MCV<R4> * 768 + 64 : MCV<R4> * 1024;   // R4: sm, nibbles, round summaries
    static constexpr uint32_t NS = 2;
};

// Row gi of the active rows: the expert's flat row and its routed pairs.
struct MoeRow {
    uint64_t grow;     // row of the stacked weight tensor
    uint32_t r;        // row inside the expert
    uint32_t l0, nt;   // the expert's pairs: elist[l0 .. l0 + nt)
    uint32_t li;       // the expert's place in the CTA's expert table (or XT_MAX)
};

// The experts a CTA's rows belong to (consecutive in active[] order), with
// their first routed pairs, staged in shared memory once per CTA.
constexpr uint32_t XT_MAX = 64;    // experts per CTA table
constexpr uint32_t XT_ENT = 16;    // pairs kept per expert
struct MoeTable {
    uint64_t ai0;                  // first expert (index into active[])
    uint32_t n;                    // experts in the table
    uint32_t e[XT_MAX], l0[XT_MAX], nt[XT_MAX];
    uint32_t ent[XT_MAX][XT_ENT];
};

// Place of an active row: expert ai (index into active[]) and row r in it,
// stepped without division.
struct RowPos {
    uint64_t ai;
    uint32_t r;
};

__device__ __forceinline__ RowPos row_pos(const MoeArgs &a, uint64_t gi) {
    RowPos p;
    p.ai = gi / a.ne;
    p.r = (uint32_t)(gi - p.ai * a.ne);
    return p;
}

__device__ __forceinline__ void row_step(const MoeArgs &a, RowPos &p, uint32_t d) {
    p.r += d;
    while (p.r >= a.ne) {
        p.r -= (uint32_t)a.ne;
        p.ai++;
    }
}

__device__ __forceinline__ MoeRow moe_row(const MoeArgs &a, const MoeTable &T, RowPos pos) {
    MoeRow m;
    const uint64_t ai = pos.ai;
    m.r = pos.r;
    const uint64_t li = ai - T.ai0;
    uint32_t e;
    if (li < T.n) {
        m.li = (uint32_t)li;
        e = T.e[li];
        m.l0 = T.l0[li];
        m.nt = T.nt[li];
    } else {
        const uint32_t P = a.tokens * a.topk;
        m.li = XT_MAX;
        e = a.active[ai] % a.n_experts;
        m.l0 = min(a.eoff[e], P);
        m.nt = min(max(a.eoff[e + 1], m.l0), P) - m.l0;
    }
    m.grow = (uint64_t)e * a.ne + m.r;
    return m;
}

// Pair k of a row's expert (t << 8 | slot).
__device__ __forceinline__ uint32_t moe_pair(const MoeArgs &a, const MoeTable &T, const MoeRow &m, uint32_t k) {
    return (m.li < XT_MAX && k < XT_ENT) ? T.ent[m.li][k] : a.elist[m.l0 + k];
}

// The next piece a producer lane copies.
struct MoeCursor {
    uint64_t i;        // CTA-local row index (warp w: w, w + MNW, ...)
    RowPos pos;
    uint64_t grow;
    uint32_t pass, npass, j;
};

__device__ __forceinline__ void moe_cursor_load(const MoeArgs &a, const MoeTable &T, MoeCursor &c, uint64_t nrows) {
    c.pass = 0;
    c.j = 0;
    if (c.i < nrows) {
        const MoeRow m = moe_row(a, T, c.pos);
        c.grow = m.grow;
        c.npass = (m.nt + MAXT - 1) / MAXT;
    }
}

template <bool R4>
__device__ __forceinline__ void moe_issue(const MoeArgs &a, uint64_t grow, uint32_t j, uint32_t stage, uint32_t bar) {
    const uint32_t n = min(MCV<R4>, a.J - j);
    const uint32_t k0 = j * 512;
    const uint32_t cols = min((j + n) * 512, (uint32_t)a.cols) - k0;
    const uint64_t f = grow * a.cols + k0;
    fence_proxy_async_smem();
    if (R4) {
        // the piece's round summaries (words x .. x + n), as the aligned run of
        // 16-byte chunks that covers them; word x lands at slot offset 4 (x & 3)
        const uint64_t x = grow * a.nseg + j, s0 = x & ~3ull, s1 = (x + n + 3) & ~3ull;
        const uint32_t rb = (uint32_t)(s1 - s0) * 4;
        mbar_arrive_expect_tx(bar, cols + cols / 2 + rb);
        bulk_g2s(stage, a.sm + f, cols, bar);
        bulk_g2s(stage + MCV<R4> * 512, a.nib + f / 2, cols / 2, bar);
        bulk_g2s(stage + MCV<R4> * 768, a.rsum + s0, rb, bar);
    } else {
        mbar_arrive_expect_tx(bar, cols * 2);
        bulk_g2s(stage, a.W + f, cols * 2, bar);
    }
}

// x of token t for lane chunk (round j, lane): two uint4 of bf16 pairs; zero
// past K.
__device__ __forceinline__ void moe_x(const MoeArgs &a, uint32_t t, uint32_t j, uint32_t lane, bool act, uint4 &xa,
                                      uint4 &xb) {
    if (act) {
        const uint4 *xp = reinterpret_cast<const uint4 *>(a.x + (size_t)t * a.cols + 512 * j + 16 * lane);
        xa = __ldg(xp);
        xb = __ldg(xp + 1);
    } else {
        xa = xb = make_uint4(0, 0, 0, 0);
    }
}

__device__ __forceinline__ float fma_chunk16_x(const uint32_t p[8], uint4 xa, uint4 xb, float acc) {
    acc = fma2_bf16(p[0], xa.x, acc);
    acc = fma2_bf16(p[1], xa.y, acc);
    acc = fma2_bf16(p[2], xa.z, acc);
    acc = fma2_bf16(p[3], xa.w, acc);
    acc = fma2_bf16(p[4], xb.x, acc);
    acc = fma2_bf16(p[5], xb.y, acc);
    acc = fma2_bf16(p[6], xb.z, acc);
    acc = fma2_bf16(p[7], xb.w, acc);
    return acc;
}

// A consumer warp's ring state.
struct MoeRing {
    const uint8_t *ring;
    uint32_t full_a, empty_a;
    uint32_t st, phases, waited;
    bool ok;
    int *abort;        // tells the producer to stop after a timeout
};

// One pass over one row for NT token chains (the first ntp of them are real;
// the others repeat token 0 and store nothing): pieces from the ring, each
// 16-weight lane chunk decoded once, one fmaf chain per token, slice partials
// butterfly-reduced into the workspace.
template <bool R4, bool BK, int NT>
__device__ __forceinline__ void moe_row_pass(const MoeArgs &a, MoeRing &rg, const MoeRow &m, uint32_t ent,
                                             uint32_t ntp, const R4Lut &L, SegInfo &g, RoundLut &rl,
                                             const uint8_t *table_s, uint8_t *escb, uint32_t lane, bool act_last,
                                             uint32_t S, uint32_t log2S, const uint16_t *xslot, const uint16_t *xsm) {
    constexpr uint32_t STAGE = MoeStage<R4>::BYTES;
    const uint32_t J = a.J, Jm1 = J - 1;
    const uint4 *xr[NT];
    uint32_t en[NT];
#pragma unroll
    for (int t = 0; t < NT; t++) {
        en[t] = __shfl_sync(DGT_FULL, ent, (uint32_t)t < ntp ? t : 0);
        const uint32_t tk = (en[t] >> 8) % a.tokens;
        const uint32_t slot = (xslot && tk < XS_TOKENS) ? xslot[tk] : 0xFFFFu;
        xr[t] = (slot != 0xFFFFu ? reinterpret_cast<const uint4 *>(xsm + (size_t)slot * a.cols)
                                 : reinterpret_cast<const uint4 *>(a.x + (size_t)tk * a.cols)) + 2 * lane;
    }
    float acc[NT];
#pragma unroll
    for (int t = 0; t < NT; t++) acc[t] = 0.0f;
    uint32_t s = 0, send = J >> log2S, jbase = 0;
    for (uint32_t jp = 0; jp < J; jp += MCV<R4>) {
        if (rg.ok && BK) {
            if (mbar_wait_n(rg.full_a + 8 * rg.st, (rg.phases >> rg.st) & 1u, a.spin)) {
                rg.waited++;
            } else {
                rg.ok = false;
                if (lane == 0) {
                    set_status(a.status, DGT_ERR_TIMEOUT);
                    atomicExch(rg.abort, 1);
                }
            }
            if (*(volatile int *)rg.abort) rg.ok = false;
        }
        rg.ok = __all_sync(DGT_FULL, rg.ok);
        rg.phases ^= 1u << rg.st;
        const uint32_t n = min(MCV<R4>, J - jp);
        const uint8_t *stg = rg.ring + rg.st * STAGE;
        // escape tables of the piece's rounds: from the round summaries that
        // came with the piece (bulk), else from the row's seg window
        uint32_t rec = 0, wb = 0;
        RoundLut prl = rl;
        if (R4) {
            if (BK) {
                const uint32_t *recs =
                    reinterpret_cast<const uint32_t *>(stg + MCV<R4> * 768) + ((m.grow * a.nseg + jp) & 3u);
                rec = lane < n ? recs[lane] : 0u;
                prl = round_luts_rec(rec, L);
                wb = jp;
            } else {
                if (jp - jbase >= 32) {
                    jbase = jp;
                    g = load_seginfo(a, table_s, m.grow, jbase, J, lane);
                    rl = round_luts(g, L);
                }
                prl = rl;
                wb = jbase;
            }
        }
        const uint4 *xp[NT];
#pragma unroll
        for (int t = 0; t < NT; t++) xp[t] = xr[t] + 64 * jp;
#pragma unroll
        for (uint32_t r = 0; r < MCV<R4>; r++) {
            if (r >= n) break;
            const uint32_t j = jp + r;
            const bool act = j != Jm1 || act_last;
            uint32_t p[8];
            if (R4) {
                uint4 sv;
                uint2 nv;
                if (BK) {
                    sv = *reinterpret_cast<const uint4 *>(stg + r * 512 + 16 * lane);
                    nv = *reinterpret_cast<const uint2 *>(stg + MCV<R4> * 512 + r * 256 + 8 * lane);
                } else {
                    // rows whose nibbles are not 16-byte aligned: direct loads
                    const uint64_t f = m.grow * a.cols + 512 * j + 16 * lane;
                    sv = act ? ldg_stream16(a.sm + f) : make_uint4(0, 0, 0, 0);
                    nv = act ? ldg_stream8(a.nib + f / 2) : make_uint2(0, 0);
                }
                const uint32_t bit = j - wb;
                R4Lut Lr = L;
                Lr.h3 = __shfl_sync(DGT_FULL, prl.h3, bit);
                Lr.l1 = __shfl_sync(DGT_FULL, prl.l1, bit);
                if ((prl.multi >> bit) & 1u) {
                    uint32_t e;
                    const uint2 nva = act ? nv : make_uint2(0, 0);
                    const bool one_each = BK ? rec_exponent(__shfl_sync(DGT_FULL, rec, bit), nva, lane, e)
                                                 : multi_exponent(a, g, bit, nva, table_s, lane, e);
                    if (one_each) {
                        r4_dec16(nv, sv, lut15(L, e), p);
                    } else if (BK) {
                        // a rare round: its escape index straight from seg
                        const uint64_t sx = m.grow * a.nseg + j;
                        const uint32_t b = a.seg[sx], c = a.seg[sx + 1] - b;
                        r4_round_general_cb(a, L, nv, sv, c, b, escb, table_s, lane, act, p);
                    } else {
                        r4_round_general(a, L, nv, sv, g, bit, escb, table_s, lane, act, p);
                    }
                } else {
                    r4_dec16(nv, sv, Lr, p);
                }
            } else {
                const uint4 lo = *reinterpret_cast<const uint4 *>(stg + r * 1024 + 32 * lane);
                const uint4 hi = *reinterpret_cast<const uint4 *>(stg + r * 1024 + 32 * lane + 16);
                p[0] = lo.x; p[1] = lo.y; p[2] = lo.z; p[3] = lo.w;
                p[4] = hi.x; p[5] = hi.y; p[6] = hi.z; p[7] = hi.w;
            }
            if (act) {
#pragma unroll
                for (int t = 0; t < NT; t++) {
                    const uint4 xa = xp[t][64 * r], xb = xp[t][64 * r + 1];
                    acc[t] = fma_chunk16_x(p, xa, xb, acc[t]);
                }
            }
            if (j + 1 == send) {
                // end of slice s: reduce and store; the next slice starts from +0
#pragma unroll
                for (int t = 0; t < NT; t++) {
                    float v = acc[t];
#pragma unroll
                    for (int d = 16; d >= 1; d >>= 1) v += __shfl_xor_sync(DGT_FULL, v, d);
                    const uint64_t q = (uint64_t)(en[t] >> 8) * a.topk + (en[t] & 0xFF);
                    if (lane == 0 && rg.ok && (uint32_t)t < ntp) a.partial[(q * a.ne + m.r) * S + s] = v;
                    acc[t] = 0.0f;
                }
                s++;
                send = ((s + 1) * J) >> log2S;
            }
        }
        __syncwarp();
        if (BK) {
            if (rg.ok && lane == 0) mbar_arrive(rg.empty_a + 8 * rg.st);
            rg.st = rg.st + 1 == MoeStage<R4>::NS ? 0 : rg.st + 1;
        }
    }
}

template <bool R4, bool BK>
__global__ void __launch_bounds__((MNW + MPW) * 32, 1) k_moe(MoeArgs a) {
    constexpr uint32_t STAGE = MoeStage<R4>::BYTES, MNS = MoeStage<R4>::NS;
    extern __shared__ __align__(128) uint8_t dsm[];
    __shared__ __align__(8) uint64_t full[MNW][MNS_MAX];
    __shared__ __align__(8) uint64_t empty[MNW][MNS_MAX];
    __shared__ uint32_t tok_bits[XS_TOKENS / 32];
    __shared__ uint16_t xslot[XS_TOKENS];
    __shared__ uint8_t table_s[256];
    __shared__ uint8_t escb[R4 ? MNW : 1][R4 ? DGT_SEG : 1];
    __shared__ int abort_flag;
    __shared__ uint32_t stop_word[MNW];   // producer lane of ring w: pieces issued, bit 31 once stopped
    __shared__ MoeTable T;
    pdl_trigger();
    pdl_wait();
    const uint32_t tid = threadIdx.x, w = tid >> 5, lane = tid & 31;
    const uint32_t P = a.tokens * a.topk;
    const uint64_t rb = a.rbound[blockIdx.x], nrows = a.rbound[blockIdx.x + 1] - rb;
    (void)P;
    const uint32_t J = a.J, K = (uint32_t)a.cols;
    // the experts of rows [rb, rb + nrows) and their first pairs
    if (nrows) {
        const uint64_t ai0 = rb / a.ne, ai1 = (rb + nrows - 1) / a.ne;
        const uint32_t n = (uint32_t)min(ai1 - ai0 + 1, (uint64_t)XT_MAX);
        if (tid == 0) {
            T.ai0 = ai0;
            T.n = n;
        }
        for (uint32_t li = tid; li < n; li += blockDim.x) {
            const uint32_t e = a.active[ai0 + li] % a.n_experts;
            const uint32_t l0 = min(a.eoff[e], P), l1 = min(max(a.eoff[e + 1], l0), P);
            T.e[li] = e;
            T.l0[li] = l0;
            T.nt[li] = l1 - l0;
        }
        __syncthreads();
        for (uint32_t k = tid; k < n * XT_ENT; k += blockDim.x) {
            const uint32_t li = k / XT_ENT, kk = k % XT_ENT;
            if (kk < T.nt[li]) T.ent[li][kk] = a.elist[T.l0[li] + kk];
        }
    } else if (tid == 0) {
        T.ai0 = 0;
        T.n = 0;
    }
    // x of the tokens routed to those experts, in shared memory (as many as fit)
    const bool xstage = a.tokens <= XS_TOKENS && a.xs_slots > 0;
    uint16_t *xsm = reinterpret_cast<uint16_t *>(dsm + (size_t)MNW * MoeStage<R4>::NS * MoeStage<R4>::BYTES);
    if (xstage) {
        for (uint32_t i = tid; i < XS_TOKENS / 32; i += blockDim.x) tok_bits[i] = 0;
        __syncthreads();
        for (uint32_t k = tid; k < T.n * XT_ENT; k += blockDim.x) {
            const uint32_t li = k / XT_ENT, kk = k % XT_ENT;
            if (kk < T.nt[li]) {
                const uint32_t tk = (T.ent[li][kk] >> 8) % a.tokens;
                atomicOr(&tok_bits[tk >> 5], 1u << (tk & 31));
            }
        }
        __syncthreads();
        if (w == 0) {
            // slots in token order, up to xs_slots
            uint32_t base = 0;
            for (uint32_t c = 0; c < XS_TOKENS / 32; c += 32) {
                const uint32_t bits = c + lane < XS_TOKENS / 32 ? tok_bits[c + lane] : 0u;
                uint32_t tot;
                const uint32_t pre = warp_excl_scan(__popc(bits), &tot);
                uint32_t b = bits, o = base + pre;
                while (b) {
                    const uint32_t i = __ffs(b) - 1;
                    b &= b - 1;
                    xslot[32 * (c + lane) + i] = o < a.xs_slots ? (uint16_t)o : (uint16_t)0xFFFFu;
                    o++;
                }
                for (uint32_t i = 0; i < 32; i++)
                    if (!((bits >> i) & 1u) && 32 * (c + lane) + i < XS_TOKENS) xslot[32 * (c + lane) + i] = 0xFFFFu;
                base += tot;
            }
        }
        __syncthreads();
        const uint32_t kv = K / 8;   // uint4 per token row
        for (uint32_t i = tid; i < a.tokens * kv; i += blockDim.x) {
            const uint32_t tk = i / kv, c = i - tk * kv;
            const uint32_t slot = xslot[tk];
            if (slot != 0xFFFFu)
                reinterpret_cast<uint4 *>(xsm + (size_t)slot * K)[c] =
                    reinterpret_cast<const uint4 *>(a.x + (size_t)tk * K)[c];
        }
    }
    const uint16_t *xslot_p = xstage ? xslot : nullptr;

    for (uint32_t i = tid; i < MNW * MNS_MAX; i += blockDim.x) {
        mbar_init(smem_u32(&full[0][0]) + 8 * i, 1);
        mbar_init(smem_u32(&empty[0][0]) + 8 * i, 1);
    }
    if (tid == 0) abort_flag = 0;
    if (tid < MNW) stop_word[tid] = 0;
    if (R4 && tid < 256) table_s[tid] = a.table[tid];
    fence_mbarrier_init();
    __syncthreads();

    if (w >= MNW) {
        // ---- producer warps: lane l of producer warp p keeps consumer
        // c = p + MPW l's ring full
        const uint32_t c = (w - MNW) + MPW * lane;
        if (c < MNW && BK) {
            const uint32_t ring_a = smem_u32(dsm + (size_t)c * MNS * STAGE);
            const uint32_t full_a = smem_u32(&full[c][0]), empty_a = smem_u32(&empty[c][0]);
            MoeCursor cur;
            cur.i = c;
            cur.pos = row_pos(a, rb + c);
            moe_cursor_load(a, T, cur, nrows);
            uint32_t q = 0, idle = 0;
            while (cur.i < nrows && !*(volatile int *)&abort_flag) {
                const uint32_t st = q % MNS;
                if (q < MNS || mbar_test_wait(empty_a + 8 * st, ((q / MNS) - 1) & 1u)) {
                    moe_issue<R4>(a, cur.grow, cur.j, ring_a + st * STAGE, full_a + 8 * st);
                    q++;
                    idle = 0;
                    cur.j += MCV<R4>;
                    if (cur.j >= J) {
                        cur.j = 0;
                        if (++cur.pass >= cur.npass) {
                            cur.i += MNW;
                            row_step(a, cur.pos, MNW);
                            moe_cursor_load(a, T, cur, nrows);
                        }
                    }
                } else if (++idle >= MBAR_SPIN_LIMIT) {
                    set_status(a.status, DGT_ERR_TIMEOUT);
                    atomicExch(&abort_flag, 1);
                    break;
                }
            }
            ring_publish_stop(&stop_word[c], q);
        }
        return;
    }

    // ---- consumer warps
    R4Lut L;
    L.h0 = opaque(a.L.h0);
    L.h1 = opaque(a.L.h1);
    L.h2 = opaque(a.L.h2);
    L.h3 = opaque(a.L.h3);
    L.l0 = opaque(a.L.l0);
    L.l1 = opaque(a.L.l1);
    const uint8_t *ring = dsm + (size_t)w * MNS * STAGE;
    const uint32_t full_a = smem_u32(&full[w][0]), empty_a = smem_u32(&empty[w][0]);
    const uint32_t Jm1 = J - 1;
    const bool act_last = 16 * lane < K - 512 * Jm1;
    const uint32_t S = a.S, log2S = __ffs(S) - 1;
    uint32_t st = 0, phases = 0, waited = 0;
    bool ok = true;
    // escape metadata runs two rows ahead: the segment counts of the row
    // after next, and the first escape ranks of the next row, are requested
    // while this row streams, so no load is waited for at a row start
    SegPre pre = {0, 0, 0, 0}, nxt = {0, 0, 0, 0};
    RowPos pos = row_pos(a, rb + w);
    // (bulk rows take their escape tables from the round summaries instead)
    const bool segpre = R4 && !BK;
    if (segpre && (uint64_t)w < nrows) {
        seg_issue(a, moe_row(a, T, pos).grow, 0, J, lane, pre);
        seg_issue_esc(a, pre);
        if ((uint64_t)w + MNW < nrows) {
            RowPos pn = pos;
            row_step(a, pn, MNW);
            seg_issue(a, moe_row(a, T, pn).grow, 0, J, lane, nxt);
        }
    }
    for (uint64_t i = w; i < nrows; i += MNW, row_step(a, pos, MNW)) {
        const MoeRow m = moe_row(a, T, pos);
        SegInfo g = {0, 0, 0, 0, 0};
        RoundLut rl = {0, 0, 0};
        if (segpre) {
            g = seg_finish(pre, table_s);
            rl = round_luts(g, L);
            pre = nxt;
            if (i + MNW < nrows) seg_issue_esc(a, pre);
            nxt = SegPre{0, 0, 0, 0};
            if (i + 2 * MNW < nrows) {
                RowPos pn = pos;
                row_step(a, pn, 2 * MNW);
                seg_issue(a, moe_row(a, T, pn).grow, 0, J, lane, nxt);
            }
        }
        for (uint32_t tg = 0; tg < m.nt; tg += MAXT) {
            const uint32_t ntp = min(MAXT, m.nt - tg);
            const uint32_t ent = lane < ntp ? moe_pair(a, T, m, tg + lane) : 0u;
            MoeRing rg{ring, full_a, empty_a, st, phases, waited, ok, &abort_flag};
            if (ntp == 1)
                moe_row_pass<R4, BK, 1>(a, rg, m, ent, ntp, L, g, rl, table_s, escb[R4 ? w : 0], lane, act_last, S, log2S,
                                     xslot_p, xsm);
            else if (ntp == 2)
                moe_row_pass<R4, BK, 2>(a, rg, m, ent, ntp, L, g, rl, table_s, escb[R4 ? w : 0], lane, act_last, S, log2S,
                                     xslot_p, xsm);
            else
                moe_row_pass<R4, BK, 4>(a, rg, m, ent, ntp, L, g, rl, table_s, escb[R4 ? w : 0], lane, act_last, S, log2S,
                                     xslot_p, xsm);
            st = rg.st;
            phases = rg.phases;
            waited = rg.waited;
            ok = rg.ok;
        }
    }
    // after a timeout: the ring's producer stops, and the copies it issued
    // that this warp did not take land before exit
    if (!ok && BK) ring_drain(&stop_word[w], full_a, waited, MNS);
}

__global__ void __launch_bounds__(256) k_moe_combine(MoeArgs a) {
    pdl_trigger();
    pdl_wait();
    const float *__restrict__ part = a.partial;
    const float *__restrict__ pw = a.p;
    float *__restrict__ y32 = a.y32;
    const uint64_t n_out = (uint64_t)a.tokens * a.ne;
    for (uint64_t i = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n_out;
         i += (uint64_t)gridDim.x * blockDim.x) {
        const uint32_t t = (uint32_t)(i / a.ne);
        const uint64_t n = i - (uint64_t)t * a.ne;
        float acc = 0.0f;
        for (uint32_t j = 0; j < a.topk; j++) {
            const uint64_t q = (uint64_t)t * a.topk + j;
            const float *pp = part + (q * a.ne + n) * a.S;
            float y = pp[0];
            for (uint32_t s = 1; s < a.S; s++) y = y + pp[s];
            if (y32) y32[q * a.ne + n] = y;
            if (pw) acc = fmaf(pw[q], y, acc);
        }
        if (pw) {
            if (a.out32) a.out32[i] = acc;
            if (a.out) a.out[i] = f32_to_bf16_rne(acc);
        }
    }
}

template <bool R4>
int launch_moe(MoeArgs &a, void *d_ws, size_t ws_bytes, cudaStream_t st) {
    const WsLayout l = moe_ws_layout(a.n_experts, a.ne, a.cols, a.tokens, a.topk);
    if (!d_ws || ws_bytes < l.total || ((uintptr_t)d_ws & 255)) return DGT_ERR_ARG;
    uint8_t *ws = static_cast<uint8_t *>(d_ws);
    a.eoff = reinterpret_cast<uint32_t *>(ws + l.eoff);
    a.elist = reinterpret_cast<uint32_t *>(ws + l.elist);
    a.active = reinterpret_cast<uint32_t *>(ws + l.active);
    a.rbound = reinterpret_cast<uint32_t *>(ws + l.rbound);
    a.partial = reinterpret_cast<float *>(ws + l.partial);
    DeviceInfo di;
    if (device_info(&di) != DGT_OK) return DGT_ERR_CUDA;
    a.grid = (uint32_t)min(di.sms, (int)MOE_MAX_CTAS);
    if (launch_pdl(k_moe_route, dim3(1), dim3(1024), 0, st, a) != cudaSuccess) return DGT_ERR_CUDA;
    a.xs_slots = a.tokens <= XS_TOKENS ? (uint32_t)min((uint64_t)a.tokens, (uint64_t)(XS_BYTES / (2 * a.cols))) : 0u;
    const size_t smem = (size_t)MNW * MoeStage<R4>::NS * MoeStage<R4>::BYTES + (size_t)a.xs_slots * a.cols * 2;
    int bps = 0;
    const void *fn = a.bulk ? (const void *)k_moe<R4, true> : (const void *)k_moe<R4, false>;
    if (prepare_kernel(fn, smem, (MNW + MPW) * 32, &bps) != DGT_OK) return DGT_ERR_CUDA;
    const cudaError_t e = a.bulk ? launch_pdl(k_moe<R4, true>, dim3(a.grid), dim3((MNW + MPW) * 32), smem, st, a)
                                 : launch_pdl(k_moe<R4, false>, dim3(a.grid), dim3((MNW + MPW) * 32), smem, st, a);
    if (e != cudaSuccess) return DGT_ERR_CUDA;
    const uint64_t n_out = (uint64_t)a.tokens * a.ne;
    uint64_t cgrid = (n_out + 255) / 256;
    if (cgrid > (uint64_t)di.sms * 8) cgrid = (uint64_t)di.sms * 8;
    if (cgrid < 1) cgrid = 1;
    if (launch_pdl(k_moe_combine, dim3((unsigned)cgrid), dim3(256), 0, st, a) != cudaSuccess)
        return DGT_ERR_CUDA;
    return cudaPeekAtLastError() == cudaSuccess ? DGT_OK : DGT_ERR_CUDA;
}

// Few (token, slot) pairs -- a decode step's gather: every pair as a block of
// the batch-1 product's bulk-copy kernel (dgt_gemv.cu), its own group of CTAs
// streaming its expert's rows with its token's x, in the same order and slice
// plan; no routing lists and no slice workspace.  Reading the experts' rows
// once per pair instead of once per expert costs nothing when every pair has
// its own expert (one token, or one slot per token).  The routing weights, if
// given, are applied by the combine kernel over those results (one slice
// each).  DGT_ERR_UNSUPPORTED (nothing launched) hands the call to the
// gather kernels.
constexpr uint64_t MOE_FEW_PAIRS = 32;

template <bool R4>
static int moe_few_pairs(MoeArgs &a, const dgt_r4 *W, const uint16_t *d_W, void *d_ws, size_t ws_bytes,
                         cudaStream_t st) {
    if ((uint64_t)a.tokens * a.topk > MOE_FEW_PAIRS) return DGT_ERR_UNSUPPORTED;
    const WsLayout l = moe_ws_layout(a.n_experts, a.ne, a.cols, a.tokens, a.topk);
    if (!d_ws || ws_bytes < l.total || ((uintptr_t)d_ws & 255)) return DGT_ERR_ARG;
    float *y = a.y32 ? a.y32 : reinterpret_cast<float *>(static_cast<uint8_t *>(d_ws) + l.partial);
    const int rc = R4 ? dgt_gemv_expert_blocks(W, a.n_experts, a.ids, a.tokens, a.topk, a.x, y, a.status, a.spin, st)
                      : dgt_gemv_expert_blocks_bf16(d_W, a.ne * a.n_experts, a.cols, a.n_experts, a.ids, a.tokens,
                                                    a.topk, a.x, y, a.status, a.spin, st);
    if (rc != DGT_OK || !a.p) return rc;
    MoeArgs c = a;
    c.partial = y;
    c.S = 1;
    c.y32 = nullptr;
    DeviceInfo di;
    if (device_info(&di) != DGT_OK) return DGT_ERR_CUDA;
    const uint64_t n_out = (uint64_t)a.tokens * a.ne;
    uint64_t cgrid = (n_out + 255) / 256;
    if (cgrid > (uint64_t)di.sms * 8) cgrid = (uint64_t)di.sms * 8;
    if (cgrid < 1) cgrid = 1;
    if (launch_pdl(k_moe_combine, dim3((unsigned)cgrid), dim3(256), 0, st, c) != cudaSuccess) return DGT_ERR_CUDA;
    return cudaPeekAtLastError() == cudaSuccess ? DGT_OK : DGT_ERR_CUDA;
}

static int moe_common(MoeArgs &a, uint64_t rows, uint64_t cols, uint32_t n_experts, uint32_t tokens, uint32_t topk,
                      const int32_t *d_ids, const uint16_t *d_x, const void *w_ptr, int32_t *d_status,
                      cudaStream_t st) {
    if (n_experts == 0 || n_experts > MOE_MAX_EXPERTS || rows % n_experts) return DGT_ERR_SHAPE;
    if (topk == 0 || topk > 255 || (uint64_t)tokens * topk > MOE_MAX_PAIRS || tokens >= (1u << 24))
        return DGT_ERR_SHAPE;
    if (cols == 0 || cols % 16 || cols >= (1ull << 31)) return DGT_ERR_SHAPE;
    if (!d_ids || !d_x || !w_ptr || !aligned16(d_x) || !aligned16(w_ptr)) return DGT_ERR_ARG;
    if (rows == 0) return DGT_ERR_SHAPE;
    a.cols = cols;
    a.ne = rows / n_experts;
    a.n_experts = n_experts;
    a.tokens = tokens;
    a.topk = topk;
    a.J = (uint32_t)((cols + 511) / 512);
    a.S = (uint32_t)dgt_plan_slices(a.ne, cols);
    a.ids = d_ids;
    a.x = d_x;
    a.status = d_status;
    a.spin = MBAR_SPIN_LIMIT;
    if (d_status && cudaMemsetAsync(d_status, 0, 4, st) != cudaSuccess) return DGT_ERR_CUDA;
    return DGT_OK;
}

}  // namespace dgt

using namespace dgt;

extern "C" size_t dgt_moe_workspace_bytes(uint32_t n_experts, uint64_t expert_rows, uint64_t cols, uint32_t tokens,
                                          uint32_t topk) {
    return moe_ws_layout(n_experts, expert_rows, cols, tokens, topk).total;
}

extern "C" int dgt_moe_gemv_ex(const dgt_r4 *W, uint32_t n_experts, const int32_t *d_ids, const float *d_p,
                               uint32_t tokens, uint32_t topk, const uint16_t *d_x, float *d_y32, uint16_t *d_out,
                               float *d_out32, void *d_ws, size_t ws_bytes, int32_t *d_status, unsigned flags,
                               void *stream) {
    if (!W) return DGT_ERR_ARG;
    if ((flags & ~(DGT_TEST_SHORT_WAITS | 0xFFFF0000u)) || (!(flags & DGT_TEST_SHORT_WAITS) && (flags >> 16)))
        return DGT_ERR_ARG;
    if (tokens == 0) return DGT_OK;
    cudaStream_t st = (cudaStream_t)stream;
    MoeArgs a = {};
    int rc = moe_common(a, W->rows, W->cols, n_experts, tokens, topk, d_ids, d_x, W->sm, d_status, st);
    if (rc != DGT_OK) return rc;
    a.spin = wait_limit_from_flags(flags);
    if (!W->nib || !W->seg || (W->n_esc && !W->esc) || !aligned16(W->nib)) return DGT_ERR_ARG;
    a.sm = W->sm;
    a.nib = W->nib;
    a.esc = W->esc;
    a.seg = W->seg;
    a.nseg = dgt_r4_nseg(W->cols);
    a.n_esc = W->n_esc;
    a.L = make_r4lut(W->table, W->n_table);
    for (int i = 0; i < 256; i++) a.table[i] = W->table[i];
    a.bulk = W->cols % 32 == 0 && aligned16(W->sm) && aligned16(W->nib) && aligned16(W->seg);
    a.rsum = W->seg + dgt_rsum_offset(W->rows, a.nseg);
    a.p = d_p;
    a.y32 = d_y32;
    a.out = d_out;
    a.out32 = d_out32;
    const int frc = moe_few_pairs<true>(a, W, nullptr, d_ws, ws_bytes, st);
    if (frc != DGT_ERR_UNSUPPORTED) return frc;
    return launch_moe<true>(a, d_ws, ws_bytes, st);
}

extern "C" int dgt_moe_gemv(const dgt_r4 *W, uint32_t n_experts, const int32_t *d_ids, const float *d_p,
                            uint32_t tokens, uint32_t topk, const uint16_t *d_x, float *d_y32, uint16_t *d_out,
                            float *d_out32, void *d_ws, size_t ws_bytes, int32_t *d_status, void *stream) {
    return dgt_moe_gemv_ex(W, n_experts, d_ids, d_p, tokens, topk, d_x, d_y32, d_out, d_out32, d_ws, ws_bytes,
                           d_status, 0u, stream);
}

extern "C" int dgt_moe_gemv_bf16(const uint16_t *d_W, uint64_t rows, uint64_t cols, uint32_t n_experts,
                                 const int32_t *d_ids, const float *d_p, uint32_t tokens, uint32_t topk,
                                 const uint16_t *d_x, float *d_y32, uint16_t *d_out, float *d_out32, void *d_ws,
                                 size_t ws_bytes, int32_t *d_status, void *stream) {
    if (tokens == 0) return DGT_OK;
    cudaStream_t st = (cudaStream_t)stream;
    MoeArgs a = {};
    int rc = moe_common(a, rows, cols, n_experts, tokens, topk, d_ids, d_x, d_W, d_status, st);
    if (rc != DGT_OK) return rc;
    a.W = d_W;
    a.bulk = 1;
    a.p = d_p;
    a.y32 = d_y32;
    a.out = d_out;
    a.out32 = d_out32;
    const int frc = moe_few_pairs<false>(a, nullptr, d_W, d_ws, ws_bytes, st);
    if (frc != DGT_ERR_UNSUPPORTED) return frc;
    return launch_moe<false>(a, d_ws, ws_bytes, st);
}

// ---------------------------------------------------------------------------
// Allocation-free variant of dgt_moe_gemv.
//
// Some callers cannot allocate device memory when they call: a plugin running
// inside a host framework that owns the whole device memory pool, or a
// latency-critical decode loop where a cudaMalloc (which may synchronise the
// device) is not allowed.  This entry point keeps its workspace in a fixed
// array that lives in the library's own device image, so it never calls
// cudaMalloc, cudaFree or any allocating routine.
//
// The array is DGT_MOE_NOALLOC_SCRATCH_BYTES large and every GPU that loads
// the library holds it until the process exits.  Host code cannot use the
// array's name as a device address (it is only a host-side stand-in), so the
// first call on each device, with that device current, looks the address up
// with cudaGetSymbolAddress and caches it; make that first call before any
// stream capture.  All calls share the one array and it keeps the last call's
// contents: nothing in it needs to start at zero (the routing kernel rewrites
// every list and count, and every partial sum is written before it is read),
// but calls that overlap on the GPU -- on different streams, or on
// different host threads at once -- race on it.
// ---------------------------------------------------------------------------
static __device__ __align__(256) uint8_t g_moe_scratch[DGT_MOE_NOALLOC_SCRATCH_BYTES];

static int moe_scratch_address(void **out) {
    static std::atomic<void *> cached[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return DGT_ERR_CUDA;
    void *p = cached[dev].load(std::memory_order_acquire);
    if (!p) {
        // Two threads may both look the address up; they store the same value.
        if (cudaGetSymbolAddress(&p, g_moe_scratch) != cudaSuccess || !p) return DGT_ERR_CUDA;
        cached[dev].store(p, std::memory_order_release);
    }
    *out = p;
    return DGT_OK;
}

extern "C" int dgt_moe_gemv_noalloc(const dgt_r4 *W, uint32_t n_experts, const int32_t *d_ids, const float *d_p,
                                    uint32_t tokens, uint32_t topk, const uint16_t *d_x, float *d_y32,
                                    uint16_t *d_out, float *d_out32, int32_t *d_status, void *stream) {
    if (!W || n_experts == 0) return DGT_ERR_ARG;
    if (W->rows % n_experts) return DGT_ERR_SHAPE;
    if (tokens == 0) return DGT_OK;
    const size_t need = dgt_moe_workspace_bytes(n_experts, W->rows / n_experts, W->cols, tokens, topk);
    if (need > DGT_MOE_NOALLOC_SCRATCH_BYTES) return DGT_ERR_SHAPE;
    void *ws = nullptr;
    const int rc = moe_scratch_address(&ws);
    if (rc != DGT_OK) return rc;
    return dgt_moe_gemv(W, n_experts, d_ids, d_p, tokens, topk, d_x, d_y32, d_out, d_out32, ws,
                        DGT_MOE_NOALLOC_SCRATCH_BYTES, d_status, stream);
}
