// dgt_gemv.cu -- batch-1 products y = W x, with W in R4 (decoded in
// registers) or in plain BF16, both in one fixed summation order.
//
// Binade README, "Results" (Matvec kernel: batch-1 matvec at BF16's bandwidth
// efficiency, 1.33x BF16 per token) and "How it works" (Runtime layout: R4's
// matvec streams at full bandwidth; Exactness: the kernels add in the order
// of the BF16 kernels, so the outputs are bit-identical).
//
// Order (both kernels): rounds of 512 columns; in round j lane u owns the 16
// columns [512j + 16u, 512j + 16u + 16); fmaf from +0 over its columns in
// increasing order, round after round; butterfly acc += shfl_xor(acc, d) for
// d = 16, 8, 4, 2, 1; with S slices (dgt_plan_slices) slice s owns rounds
// [sJ/S, (s+1)J/S) and the slice results are added left to right.
//
// GB300 design: a persistent grid of one CTA per SM; CTA b owns a contiguous,
// even share of the rows and walks its (row, slice) units warp by warp, so no
// SM waits on a second wave.  x is copied once per CTA into shared memory as
// bf16 pairs in a [round][half][lane] uint4 layout (two conflict-free LDS.128
// per lane and round), and the products use the mixed-precision
// fma.rn.f32.bf16, which takes the bf16 halves directly; the exponent comes
// from register byte-permutes.  Three kernels: the bulk-copy kernel
// (k_gemv_tma, the default, described below); a register-streaming kernel
// (k_gemv) when a row's length is a multiple of 16 but not of 32, or the
// bulk-copy kernel's rings and x do not fit shared memory (16-byte
// sign/mantissa and 8-byte nibble loads per lane and round, double-buffered;
// a ballot gives a warp-uniform mask of the rounds with escapes, which go out
// of line); and an any-shape kernel (k_gemv_any) for unaligned arrays, other
// lengths and rows longer than 160 rounds.
#include <cuda_runtime.h>

#include "../../include/dgt.h"
#include "dgt_device.cuh"
#include "dgt_internal.h"
#include "dgt_launch.h"
#include "dgt_r4esc.cuh"

namespace dgt {

constexpr int GW = 8;        // warps per CTA of the any-shape kernel
constexpr int CHUNK = 128;   // (row, slice) units per CTA chunk
constexpr uint32_t MAX_FAST_ROUNDS = 160;  // x staged in shared memory, 1 KB per round

struct GemvArgs {
    const uint8_t *sm;
    const uint8_t *nib;
    const uint8_t *esc;
    const uint32_t *seg;
    const uint32_t *rsum;   // per-round escape summaries (second part of seg)
    const uint16_t *W;
    const uint16_t *x;
    uint16_t *y;
    float *y32;
    uint64_t rows, cols, nseg, n_esc;
    uint32_t J;
    int S;
    uint32_t early;   // DGT_GEMV_STATIC_WEIGHTS: stream W before the grid dependency wait
    uint32_t spin;    // polls a consumer waits for a piece before it gives up
    R4Lut L;
    uint8_t table[256];
    int32_t *status;
    // expert blocks (the expert gather with few (token, slot) pairs): pair i
    // takes a contiguous group of CTAs, which compute y32[i * ne + n] =
    // W[ids[i] * ne + n] . x[i / topk] for n < ne; ids == nullptr otherwise
    const int32_t *ids;
    uint32_t pairs, topk, n_experts;
    uint64_t ne;
};

template <bool R4, int U>
struct Batch {
    uint4 s[U];   // R4: sign/mantissa bytes; BF16: first 8 weights
    uint2 n[U];   // R4: nibbles
    uint4 v[U];   // BF16: last 8 weights
};

template <bool R4, int U>
__device__ __forceinline__ void load_batch(Batch<R4, U> &B, const uint8_t *smp, const uint8_t *nbp,
                                           const uint16_t *wp, uint32_t jb, uint32_t j1, uint32_t Jm1,
                                           bool last_ok) {
#pragma unroll
    for (int t = 0; t < U; t++) {
        const uint32_t j = jb + t;
        if (j < j1 && (j != Jm1 || last_ok)) {
            if (R4) {
                B.s[t] = ldg_stream16(smp + (size_t)j * 512);
                B.n[t] = ldg_stream8(nbp + (size_t)j * 256);
            } else {
                ldg_stream32(wp + (size_t)j * 512, B.s[t], B.v[t]);
            }
        }
    }
}

// A round of an R4 row that holds escapes: decode, patch, multiply-add.
// Kept out of line so that the common path stays small in the instruction
// cache.  Called by all 32 lanes; c = escapes in the round, b = the first
// escape's index, e = its exponent.
__device__ __noinline__ float round_with_escapes(const uint8_t *esc, uint64_t n_esc, R4Lut L, uint2 n,
                                                 uint4 s, const uint4 *xs,
                                                 uint8_t *escb, const uint8_t *table_s, uint32_t j,
                                                 uint32_t lane, bool act, uint32_t c, uint32_t b, uint32_t e,
                                                 float acc) {
    uint32_t p[8];
    r4_dec16(n, s, L, p);
    const uint32_t m0 = act ? nib15_mask(n.x) : 0u;
    const uint32_t m1 = act ? nib15_mask(n.y) : 0u;
    if (c == 1) {
        if (m0 | m1) {
            const uint32_t pos = m0 ? (__ffs(m0) - 1) >> 2 : 8 + ((__ffs(m1) - 1) >> 2);
#pragma unroll
            for (int i = 0; i < 8; i++) {
                if ((pos >> 1) == (uint32_t)i) {
                    const uint32_t sh = (pos & 1) * 16;
                    p[i] = (p[i] & ~(0x7F80u << sh)) | (e << (7 + sh));
                }
            }
        }
    } else {
        const uint32_t cc = c > DGT_SEG ? DGT_SEG : c;
        for (uint32_t i = lane; i < cc; i += 32) escb[i] = (uint64_t)b + i < n_esc ? esc[b + i] : 0;
        __syncwarp();
        patch_escapes(p, m0, m1, cc, escb, table_s);
        __syncwarp();
    }
    if (act) acc = fma_chunk16(p, xs, j, lane, acc);
    return acc;
}

template <bool R4, int U>
__device__ __forceinline__ float compute_batch(const GemvArgs &a, const Batch<R4, U> &B, const uint4 *xs,
                                               uint8_t *escb, const uint8_t *table_s, const SegInfo &g,
                                               uint32_t jb, uint32_t jbase, uint32_t j1, uint32_t Jm1,
                                               bool last_ok, uint32_t lane, float acc) {
#pragma unroll
    for (int t = 0; t < U; t++) {
        const uint32_t j = jb + t;
        if (j >= j1) break;
        const bool act = j != Jm1 || last_ok;
        uint32_t p[8];
        if (R4) {
            const uint32_t bit = j - jbase;
            if ((g.emask >> bit) & 1u) {
                const uint32_t c = __shfl_sync(DGT_FULL, g.cnt, bit);
                const uint32_t b = __shfl_sync(DGT_FULL, g.base, bit);
                const uint32_t e = __shfl_sync(DGT_FULL, g.fexp, bit);
                acc = round_with_escapes(a.esc, a.n_esc, a.L, B.n[t], B.s[t], xs, escb, table_s, j, lane, act, c, b,
                                         e, acc);
                continue;
            }
            r4_dec16(B.n[t], B.s[t], a.L, p);
        } else {
            p[0] = B.s[t].x; p[1] = B.s[t].y; p[2] = B.s[t].z; p[3] = B.s[t].w;
            p[4] = B.v[t].x; p[5] = B.v[t].y; p[6] = B.v[t].z; p[7] = B.v[t].w;
        }
        if (act) acc = fma_chunk16(p, xs, j, lane, acc);
    }
    return acc;
}

// One (row, slice) unit: the lane's fmaf chain over rounds [j0, j1).
template <bool R4, int U>
__device__ __forceinline__ float unit_dot(const GemvArgs &a, const uint4 *xs, uint8_t *escb, const uint8_t *table_s,
                                          uint64_t row, uint32_t j0, uint32_t j1, uint32_t lane, bool last_ok) {
    const uint64_t rb = row * a.cols + 16 * lane;
    const uint8_t *smp = R4 ? a.sm + rb : nullptr;
    const uint8_t *nbp = R4 ? a.nib + rb / 2 : nullptr;
    const uint16_t *wp = R4 ? nullptr : a.W + rb;
    const uint32_t Jm1 = a.J - 1;
    SegInfo g = {0, 0, 0, 0, 0};
    uint32_t jbase = j0;
    if (R4) g = load_seginfo(a, table_s, row, jbase, j1, lane);
    float acc = 0.0f;
    Batch<R4, U> A, B;
    load_batch<R4, U>(A, smp, nbp, wp, j0, j1, Jm1, last_ok);
    for (uint32_t jb = j0; jb < j1; jb += 2 * U) {
        if (R4 && jb - jbase >= 32) {
            jbase = jb;
            g = load_seginfo(a, table_s, row, jbase, j1, lane);
        }
        load_batch<R4, U>(B, smp, nbp, wp, jb + U, j1, Jm1, last_ok);
        acc = compute_batch<R4, U>(a, A, xs, escb, table_s, g, jb, jbase, j1, Jm1, last_ok, lane, acc);
        load_batch<R4, U>(A, smp, nbp, wp, jb + 2 * U, j1, Jm1, last_ok);
        acc = compute_batch<R4, U>(a, B, xs, escb, table_s, g, jb + U, jbase, j1, Jm1, last_ok, lane, acc);
    }
    return acc;
}

// Streaming kernel: one CTA of 16 warps per SM; CTA b owns rows
// [b*N/G, (b+1)*N/G) and walks their (row, slice) units in chunks of 128,
// warp w taking units w, w+16, ...; slice partials meet in shared memory and
// are added left to right.
template <bool R4, int PW, int U>
__global__ void __launch_bounds__(PW * 32, 1) k_gemv(GemvArgs a) {
    extern __shared__ uint4 xs[];
    __shared__ uint8_t table_s[256];
    __shared__ uint8_t escb[PW][DGT_SEG];
    __shared__ float part[CHUNK];
    const uint32_t tid = threadIdx.x, w = tid >> 5, lane = tid & 31;
    const uint32_t K = (uint32_t)a.cols;
    for (uint32_t i = tid; i < K / 8; i += PW * 32) {
        const uint32_t k = 8 * i, j = k >> 9, u = (k >> 4) & 31, h = (k >> 3) & 1;
        xs[(2 * j + h) * 32 + u] = *reinterpret_cast<const uint4 *>(a.x + k);
    }
    if (R4 && tid < 256) table_s[tid] = a.table[tid];
    __syncthreads();
    const int S = a.S;
    const uint64_t G = gridDim.x;
    const uint64_t r0 = (uint64_t)blockIdx.x * a.rows / G, r1 = (uint64_t)(blockIdx.x + 1) * a.rows / G;
    const uint64_t units = (r1 - r0) * S;
    const bool last_ok = 16 * lane < K - 512 * (a.J - 1);
    for (uint64_t c0 = 0; c0 < units; c0 += CHUNK) {
        const uint32_t cu = (uint32_t)min((uint64_t)CHUNK, units - c0);
        for (uint32_t u = w; u < cu; u += PW) {
            const uint64_t uu = c0 + u;
            const uint64_t row = r0 + uu / S;
            const uint32_t s = (uint32_t)(uu % S);
            const uint32_t j0 = (uint32_t)((uint64_t)s * a.J / S), j1 = (uint32_t)((uint64_t)(s + 1) * a.J / S);
            float acc = unit_dot<R4, U>(a, xs, escb[w], table_s, row, j0, j1, lane, last_ok);
#pragma unroll
            for (int d = 16; d >= 1; d >>= 1) acc += __shfl_xor_sync(DGT_FULL, acc, d);
            if (lane == 0) part[u] = acc;
        }
        __syncthreads();
        for (uint32_t t = tid; t < cu / S; t += PW * 32) {
            float y = part[t * S];
            for (int s = 1; s < S; s++) y = y + part[t * S + s];
            const uint64_t row = r0 + c0 / S + t;
            if (a.y32) a.y32[row] = y;
            if (a.y) a.y[row] = f32_to_bf16_rne(y);
        }
        __syncthreads();
    }
}

// ---------------------------------------------------------------------------
// Bulk-copy streaming kernel (the default when cols % 32 == 0). One CTA per SM
// of TNW = 18 consumer warps and TPW = 2 producer warps; CTA b owns rows
// [b*N/G, (b+1)*N/G) and consumer warp w takes the (row, slice) units w, w+18,
// ...; or (CONTIG, R4 units of one or two rounds) the w-th of 18 even
// contiguous stretches of them, streamed as pieces that run across unit ends
// (and across row ends when a row is whole rounds): a unit that ends inside a
// piece leaves its sum there (fin) and the next unit's sum starts at 0, in the
// same order as unit by unit. Each consumer owns a ring of NS shared-memory
// stages; one lane of a producer warp keeps it full, issuing the 1-D bulk
// copies (cp.async.bulk) of the next piece as soon as the consumer has released
// a stage (its "empty" mbarrier, polled without blocking), the arrival counted
// on the stage's "full" mbarrier. No consumer waits on another consumer. A bulk
// copy takes warp-uniform operands, so a producer warp issues its lanes' copies
// one after another: two producer warps halve that queue (BF16 streams about 7%
// faster; R4, bound by its decode, is unchanged). A piece is C rounds (fewer at
// a unit's end), decoded from shared memory with no branch between its rounds,
// so that one round's decode overlaps the previous round's multiply-adds. R4
// pieces are 4 rounds in three stages, or 6 rounds in two stages when a unit's
// round count is a multiple of 6 (a 3072-column row, say): a short last piece
// costs nearly as much as a full one, so 6-round units as 4 + 2 rounds ran
// about 15% slower. An R4 round whose segment holds one escape decodes with the
// rank-15 entry of the exponent table replaced by that escape's exponent (only
// the escaped weight has nibble 15); two or three escapes do the same per lane,
// a lane holding two of them rewriting its second escaped weight's exponent;
// other cases take a general patch from the escape list. Every wait is bounded:
// one that runs out sets the status word, and the warp stops, lets its copies
// in flight land and exits.
// ---------------------------------------------------------------------------
#ifndef DGT_GEMV_TNW
#define DGT_GEMV_TNW 18
#endif
#ifndef DGT_GEMV_NS_R4
#define DGT_GEMV_NS_R4 3
#endif
#ifndef DGT_GEMV_C_R4
#define DGT_GEMV_C_R4 4   // rounds per R4 piece (at most 13: the summary slot holds C + 6 words)
#endif
#ifndef DGT_GEMV_NS_BF16
#define DGT_GEMV_NS_BF16 4
#endif
#ifndef DGT_GEMV_TCHUNK
#define DGT_GEMV_TCHUNK 864
#endif
#ifndef DGT_GEMV_TPW
#define DGT_GEMV_TPW 2
#endif
#ifndef DGT_GEMV_SMEM_KB
#define DGT_GEMV_SMEM_KB 212   // dynamic shared memory of the bulk-copy kernel (rings + x), at most
#endif
constexpr int TNW = DGT_GEMV_TNW;    // consumer warps per CTA
constexpr int TPW = DGT_GEMV_TPW;    // producer warps (producer warp p serves consumers p, p + TPW, ...)
constexpr uint32_t TNS_MAX = DGT_GEMV_NS_R4 > DGT_GEMV_NS_BF16 ? DGT_GEMV_NS_R4 : DGT_GEMV_NS_BF16;
constexpr uint32_t TCHUNK = DGT_GEMV_TCHUNK;  // (row, slice) units per combine chunk
// a chunk holds whole rows for every slice count (S <= 8); consumer warp w
// takes the w-th of TNW even, contiguous stretches of each chunk's units
static_assert(TCHUNK % TNW == 0 && TCHUNK % 8 == 0, "chunk size");
static_assert(TNW <= 32 * TPW, "one producer lane per consumer warp");
static_assert(DGT_GEMV_C_R4 >= 1 && DGT_GEMV_C_R4 <= 13, "R4 piece rounds");

// R4 rings: pieces of DGT_GEMV_C_R4 rounds in NS_R4 stages, or (CR = 6, for
// units whose round count is a multiple of 6: 6-round rows, and longer rows
// split into such slices) pieces of 6 rounds in two stages of the same total
// size, so that such a unit is whole pieces.
template <bool R4, uint32_t CR = DGT_GEMV_C_R4>
struct TmaCfg {
    static constexpr uint32_t C = CR;                                   // rounds per piece
    static constexpr uint32_t NS = CR == DGT_GEMV_C_R4 ? DGT_GEMV_NS_R4 : 2;   // stages per warp
    static constexpr uint32_t STAGE = C * 768 + 64;   // sm bytes, nibbles, then round summaries
};
template <uint32_t CR>
struct TmaCfg<false, CR> {
    static constexpr uint32_t C = 2;
    static constexpr uint32_t NS = DGT_GEMV_NS_BF16;
    static constexpr uint32_t STAGE = 2 * 1024;
};
constexpr uint32_t GEMV_C6 = 6;   // the second R4 piece length

// A piece: n rounds from round j of row `row` (flat weight index f = row * K
// + 512 j), cols weights.  R4: the piece's round summaries (words x .. x + n
// of rsum, x = row * nseg + j) travel with it, as the aligned run of 16-byte
// chunks that covers them (at most 48 bytes); word x lands at offset
// 4 * (x & 3) of the summary slot.
template <bool R4, uint32_t CR>
__device__ __forceinline__ void issue_piece(const GemvArgs &a, uint64_t f, uint64_t x, uint32_t n, uint32_t cols,
                                            uint32_t stage, uint32_t bar) {
    constexpr uint32_t C = TmaCfg<R4, CR>::C;
    fence_proxy_async_smem();
    if (R4) {
        const uint64_t s0 = x & ~3ull, s1 = (x + n + 3) & ~3ull;
        const uint32_t rb = (uint32_t)(s1 - s0) * 4;
        mbar_arrive_expect_tx(bar, cols + cols / 2 + rb);
        bulk_g2s(stage, a.sm + f, cols, bar);
        bulk_g2s(stage + C * 512, a.nib + f / 2, cols / 2, bar);
        bulk_g2s(stage + C * 768, a.rsum + s0, rb, bar);
    } else {
        mbar_arrive_expect_tx(bar, cols * 2);
        bulk_g2s(stage, a.W + f, cols * 2, bar);
    }
}

// First round of unit uu in its row, and its round count.
__device__ __forceinline__ uint32_t unit_j0(uint32_t uu, uint32_t log2S, uint32_t J) {
    return ((uu & ((1u << log2S) - 1u)) * J) >> log2S;
}
__device__ __forceinline__ uint32_t unit_len(uint32_t uu, uint32_t log2S, uint32_t J) {
    const uint32_t s = uu & ((1u << log2S) - 1u);
    return (((s + 1) * J) >> log2S) - ((s * J) >> log2S);
}

// A stretch: units [ua, ub) of the CTA (row-major: a row's slices in order,
// then the next row's), whose rounds follow one another in memory.  The
// cursor is at round j of its row, x = row * nseg + j (the round's index in
// the round summaries; nseg = J), f = row * K + 512 j (its first weight),
// with left rounds to go.  x0 = r0 * J and f0 = r0 * K for the CTA's first
// row r0.
struct Stretch {
    uint64_t x, f;
    uint32_t j, left;
};

__device__ __forceinline__ Stretch stretch_start(uint32_t ua, uint32_t ub, uint64_t x0, uint64_t f0, uint32_t log2S,
                                                 uint32_t J, uint32_t K) {
    Stretch c;
    const uint32_t rowl = ua >> log2S;
    c.j = unit_j0(ua, log2S, J);
    c.x = x0 + (rowl * J + c.j);
    c.f = f0 + (uint64_t)rowl * K + c.j * 512;
    c.left = ((ub >> log2S) - rowl) * J + unit_j0(ub, log2S, J) - c.j;
    return c;
}

// The next piece's round count: C at most, and within the row unless rows
// are whole rounds and at least C of them (then a piece may run on into the
// next row).
template <uint32_t C>
__device__ __forceinline__ uint32_t piece_len(const Stretch &c, uint32_t J, bool span) {
    return min(min(C, c.left), span ? C : J - c.j);
}

__device__ __forceinline__ void stretch_advance(Stretch &c, uint32_t n, uint32_t J) {
    c.x += n;
    c.j += n;
    c.left -= n;
    if (c.j >= J) c.j -= J;
}

// Warp w's stretch of chunk ch (CONTIG): the w-th of TNW even contiguous
// shares of the chunk's units, [ua, ub).  (A CTA's units number below 2^31:
// its rows are at most 2^35 / G.)
struct ChunkWalk {
    uint32_t ua, ub;
};
__device__ __forceinline__ ChunkWalk chunk_walk(uint32_t ch, uint32_t units, uint32_t w) {
    const uint32_t c0 = ch * TCHUNK, nu = min(c0 + TCHUNK, units) - c0;
    ChunkWalk k;
    k.ua = c0 + (w * nu) / TNW;
    k.ub = c0 + ((w + 1) * nu) / TNW;
    return k;
}

template <bool R4, uint32_t CR = DGT_GEMV_C_R4, bool CONTIG = false>
__global__ void __launch_bounds__((TNW + TPW) * 32, 1) k_gemv_tma(GemvArgs a) {
    constexpr uint32_t C = TmaCfg<R4, CR>::C, TNS = TmaCfg<R4, CR>::NS, STAGE = TmaCfg<R4, CR>::STAGE;
    // longer pieces keep their rare paths (multi-escape set-up, general
    // patch) as rolled loops: unrolled over 6 rounds they overflow the
    // instruction cache on escape-rich tensors
    constexpr bool ROLL = R4 && C > DGT_GEMV_C_R4;
    extern __shared__ __align__(128) uint8_t dsm[];
    __shared__ __align__(8) uint64_t full[TNW][TNS_MAX];
    __shared__ __align__(8) uint64_t empty[TNW][TNS_MAX];
    __shared__ uint8_t table_s[256];
    __shared__ uint8_t escb[R4 ? TNW : 1][R4 ? DGT_SEG : 1];
    __shared__ float part[TCHUNK];
    __shared__ int abort_flag;
    __shared__ uint32_t stop_word[TNW];   // producer lane of ring w: pieces issued, bit 31 once stopped
    const uint32_t tid = threadIdx.x, w = tid >> 5, lane = tid & 31;
    uint4 *xs = reinterpret_cast<uint4 *>(dsm + (size_t)TNW * TNS * STAGE);
    const uint64_t G = gridDim.x;
    uint64_t r0 = (uint64_t)blockIdx.x * a.rows / G, nrows = (uint64_t)(blockIdx.x + 1) * a.rows / G - r0;
    uint64_t o0 = r0;           // output index of row r0
    const uint16_t *xv = a.x;   // this CTA's x
    if (a.ids) {
        // expert blocks: CTAs [ceil(iG/P), ceil((i+1)G/P)) take pair i, each an
        // even share of the expert's rows.  The pair's expert id may come from
        // the previous kernel, so everything here waits for it first.
        pdl_wait();
        const uint32_t P = a.pairs;
        const uint32_t i = (uint32_t)(((uint64_t)blockIdx.x * P) / G);
        const uint64_t g0 = ((uint64_t)i * G + P - 1) / P, g1 = ((uint64_t)(i + 1) * G + P - 1) / P;
        const uint64_t c = blockIdx.x - g0, ng = g1 - g0;
        const int32_t e = a.ids[i];
        const uint64_t lr0 = c * a.ne / ng, lr1 = (c + 1) * a.ne / ng;
        if (e < 0 || (uint32_t)e >= a.n_experts) {
            if (threadIdx.x == 0) set_status(a.status, DGT_ERR_ARG);
            nrows = 0;
        } else {
            r0 = (uint64_t)e * a.ne + lr0;
            nrows = lr1 - lr0;
        }
        o0 = (uint64_t)i * a.ne + lr0;
        xv = a.x + (uint64_t)(i / a.topk) * a.cols;
    }
    const uint32_t log2S = __ffs(a.S) - 1;
    const uint64_t units = nrows << log2S;
    const uint64_t nchunks = (units + TCHUNK - 1) / TCHUNK;
    const uint32_t J = a.J;
    const uint32_t K = (uint32_t)a.cols;
    // pieces may run on from one row into the next when rows are whole rounds
    const bool span = (K & 511u) == 0 && J >= C;
    const uint64_t x0 = r0 * J, f0 = r0 * K;   // the CTA's first row: its first round and weight

    for (uint32_t i = tid; i < TNW * TNS_MAX; i += blockDim.x) {
        mbar_init(smem_u32(&full[0][0]) + 8 * i, 1);
        mbar_init(smem_u32(&empty[0][0]) + 8 * i, 1);
    }
    if (tid == 0) abort_flag = 0;
    if (tid < TNW) stop_word[tid] = 0;
    fence_mbarrier_init();
    __syncthreads();
    // the next kernel may start as SMs free up.  With static weights they
    // stream from here on; otherwise, and for everything else the previous
    // kernel may write (x, y), only after the grid dependency wait
    pdl_trigger();

    if (w >= TNW) {
        if (!a.early) pdl_wait();
        // ---- producer warps: lane l of producer warp p keeps consumer warp
        // c = p + TPW l's ring full.  It polls the ring's "empty" barriers
        // without blocking, so no consumer waits for another.
        const uint32_t c = (w - TNW) + TPW * lane;
        if (c < TNW) {
            const uint32_t ring_a = smem_u32(dsm + (size_t)c * TNS * STAGE);
            const uint32_t full_a = smem_u32(&full[c][0]), empty_a = smem_u32(&empty[c][0]);
            // ring c's pieces in consumer c's order
            uint32_t q = 0, idle = 0;
            uint64_t ch = 0, uu = c, rowf = 0, rowx = 0;   // CONTIG: chunk; else unit, its row's first weight and round
            uint32_t j = 0, j1 = 0;
            Stretch cs = {0, 0, 0, 0};
            bool more;
            auto next_stretch = [&]() {
                for (; ch < nchunks; ch++) {
                    const ChunkWalk k = chunk_walk((uint32_t)ch, (uint32_t)units, c);
                    if (k.ua < k.ub) {
                        cs = stretch_start(k.ua, k.ub, x0, f0, log2S, J, K);
                        return true;
                    }
                }
                return false;
            };
            auto unit_start = [&]() {
                if (uu >= units) return false;
                rowf = f0 + (uu >> log2S) * K;
                rowx = x0 + (uu >> log2S) * J;
                j = unit_j0((uint32_t)uu, log2S, J);
                j1 = j + unit_len((uint32_t)uu, log2S, J);
                return true;
            };
            if constexpr (CONTIG) more = next_stretch();
            else more = unit_start();
            while (more && !*(volatile int *)&abort_flag) {
                const uint32_t st = q % TNS;
                if (q < TNS || mbar_test_wait(empty_a + 8 * st, ((q / TNS) - 1) & 1u)) {
                    if constexpr (CONTIG) {
                        const uint32_t n = piece_len<C>(cs, J, span);
                        // a piece within the row stops at K (the row's last piece
                        // ends where the next row starts); one running on into the
                        // next row only exists when K is whole rounds
                        const uint32_t cols = span ? n * 512 : min(n * 512, K - cs.j * 512);
                        issue_piece<R4, CR>(a, cs.f, cs.x, n, cols, ring_a + st * STAGE, full_a + 8 * st);
                        cs.f += cols;
                        stretch_advance(cs, n, J);
                        if (cs.left == 0) {
                            ch++;
                            more = next_stretch();
                        }
                    } else {
                        const uint32_t n = min(C, j1 - j);
                        const uint32_t cols = min(n * 512, K - j * 512);
                        issue_piece<R4, CR>(a, rowf + j * 512, rowx + j, n, cols, ring_a + st * STAGE, full_a + 8 * st);
                        j += n;
                        if (j >= j1) {
                            uu += TNW;
                            more = unit_start();
                        }
                    }
                    q++;
                    idle = 0;
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
    pdl_wait();
    for (uint32_t i = tid; i < J * 64; i += TNW * 32) {
        const uint32_t k = 8 * i, j = k >> 9, u = (k >> 4) & 31, h = (k >> 3) & 1;
        xs[(2 * j + h) * 32 + u] = k < K ? *reinterpret_cast<const uint4 *>(xv + k) : make_uint4(0, 0, 0, 0);
    }
    if (R4 && tid < 256) table_s[tid] = a.table[tid];
    asm volatile("bar.sync 1, %0;" ::"r"(TNW * 32) : "memory");

    // the exponent table, held in registers (opaque copies: never re-read from
    // the parameter space inside the loop)
    R4Lut L;
    L.h0 = opaque(a.L.h0);
    L.h1 = opaque(a.L.h1);
    L.h2 = opaque(a.L.h2);
    L.h3 = opaque(a.L.h3);
    L.l0 = opaque(a.L.l0);
    L.l1 = opaque(a.L.l1);
    const uint8_t *ring = dsm + (size_t)w * TNS * STAGE;
    const uint32_t full_a = smem_u32(&full[w][0]), empty_a = smem_u32(&empty[w][0]);
    const uint32_t Jm1 = J - 1;
    const bool act = 16 * lane < K - 512 * Jm1;
    const bool cut = (K & 511) != 0;
    uint32_t st = 0, phases = 0, waited = 0;
    bool ok = true;
    // one piece: n rounds from round jp of its row (px = row * nseg + jp in
    // the round summaries); inner: its rounds before the last that end a unit
    // (their sums leave through fin); rounds r >= jw belong to the next row
    uint64_t c0 = 0;
    uint32_t udone = 0;   // next unit to finish
    float acc = 0.0f;
    auto piece = [&](const uint32_t n, const uint32_t jp, const uint64_t px, const uint32_t inner, const uint32_t jw) {
        if (ok) {
            if (mbar_wait_n(full_a + 8 * st, (phases >> st) & 1u, a.spin)) {
                waited++;
            } else {
                ok = false;
                if (lane == 0) {
                    set_status(a.status, DGT_ERR_TIMEOUT);
                    atomicExch(&abort_flag, 1);
                }
            }
            if (*(volatile int *)&abort_flag) ok = false;
        }
        ok = __all_sync(DGT_FULL, ok);
        phases ^= 1u << st;
        const uint32_t rp = (cut && Jm1 - jp < n) ? Jm1 - jp : 0xFFFFFFFFu;
        const uint8_t *stg = ring + st * STAGE;
        // the piece's round summaries arrived with it: lane r < n holds
        // round jp + r's word, and its two table words for the decode
        uint32_t rec = 0;
        RoundLut rl = {0, 0, 0};
        if (R4) {
            const uint32_t *recs =
                reinterpret_cast<const uint32_t *>(stg + C * 768) + (px & 3u);
            rec = lane < n ? recs[lane] : 0u;
            rl = round_luts_rec(rec, L);
        }
        const uint32_t pm = rl.multi;
        // BF16 pieces of fewer than C rounds take the general loop
        bool slow = !R4 && n != C;
        // rounds with two or three escapes: per-lane rank-15 entries (and,
        // for a lane holding two, its second escaped weight), worked out
        // before the multiply-adds; a round where that fails takes the
        // general patch from the escape list
        uint32_t mh3[C], ml1[C], mi2[C], me2[C];
        uint32_t pm2 = 0, pmok = 0;   // rounds with a second patch; rounds worked out
        if (R4 && ok && pm) {
#pragma unroll
            for (uint32_t r = 0; r < C; r++) mh3[r] = ml1[r] = 0, mi2[r] = 16, me2[r] = 0;
            // round r of the set bits of pm: its lane's values, placed by
            // compile-time index (a select per round when rolled)
            auto multi_round = [&](uint32_t r) {
                uint2 nv = *reinterpret_cast<const uint2 *>(stg + C * 512 + r * 256 + 8 * lane);
                if (r == rp && !act) nv = make_uint2(0, 0);   // bytes past K are not this row's
                uint32_t e, e2, i2;
                if (rec_exponent2(__shfl_sync(DGT_FULL, rec, r), nv, lane, e, e2, i2)) {
                    const R4Lut t = lut15(L, e);
#pragma unroll
                    for (uint32_t i = 0; i < C; i++) {
                        if (i == r) {
                            mh3[i] = t.h3;
                            ml1[i] = t.l1;
                            mi2[i] = i2;
                            me2[i] = e2;
                        }
                    }
                    pmok |= 1u << r;
                    if (__any_sync(DGT_FULL, i2 < 16)) pm2 |= 1u << r;
                } else {
                    slow = true;
                }
            };
            if constexpr (ROLL) {
                uint32_t bits = pm;
#pragma unroll 1
                while (bits) {
                    const uint32_t r = __ffs(bits) - 1;
                    bits &= bits - 1u;
                    multi_round(r);
                }
            } else {
#pragma unroll
                for (uint32_t r = 0; r < C; r++)
                    if ((pm >> r) & 1u) multi_round(r);
            }
        }
        // round r's weights into bf16 pairs: R4 decoded with the table
        // words h3, l1 (rank 15 -> an escape's exponent), or the BF16 words
        auto weights = [&](uint32_t r, uint32_t h3, uint32_t l1, uint32_t p[8]) {
            if (R4) {
                const uint4 sv = *reinterpret_cast<const uint4 *>(stg + r * 512 + 16 * lane);
                const uint2 nv = *reinterpret_cast<const uint2 *>(stg + C * 512 + r * 256 + 8 * lane);
                R4Lut Lr = L;
                Lr.h3 = h3;
                Lr.l1 = l1;
                r4_dec16(nv, sv, Lr, p);
            } else {
                const uint4 lo = *reinterpret_cast<const uint4 *>(stg + r * 1024 + 32 * lane);
                const uint4 hi = *reinterpret_cast<const uint4 *>(stg + r * 1024 + 32 * lane + 16);
                p[0] = lo.x; p[1] = lo.y; p[2] = lo.z; p[3] = lo.w;
                p[4] = hi.x; p[5] = hi.y; p[6] = hi.z; p[7] = hi.w;
            }
        };
        // the multiply-adds of round r (x round jp + r, or jp + r - J past
        // the row's end); in the row's last round cut by K (r == rp) a
        // lane past K adds fma(+0, +0) = +0 instead, its weights there
        // being the next row's.  fin[r] keeps the sum after round r; a
        // round that ends a unit starts the next unit's sum at 0
        float fin[C];
        auto fma_round = [&](uint32_t r, const uint32_t p[8]) {
            const uint32_t jx = jp + r - (r >= jw ? J : 0u);
            float t = fma_chunk16(p, xs, jx, lane, acc);
            t = (r == rp && !act) ? __fadd_rn(acc, 0.0f) : t;
            if constexpr (CONTIG) {
#pragma unroll
                for (uint32_t i = 0; i < C; i++)
                    if (i == r) fin[i] = t;
            }
            acc = ((inner >> r) & 1u) ? 0.0f : t;
        };
        // a lane holding two of the round's escapes: its second escaped
        // weight (index mi2[r]) gets exponent me2[r], without an indexed store
        // (index i2, exponent e2: mi2[r] and me2[r] of the round)
        auto second_escape = [&](uint32_t i2, uint32_t e2, uint32_t p[8]) {
            const uint32_t fm = 0x7F80u << (16 * (i2 & 1u));
            const uint32_t fv = e2 * 0x00800080u;
#pragma unroll
            for (uint32_t t = 0; t < 8; t++) {
                const uint32_t hit = (i2 >> 1) == t ? fm : 0u;
                p[t] = (p[t] & ~hit) | (fv & hit);
            }
        };
        // the piece's rounds, each decoded with its own table words
        // (multi-escape rounds with the lane's own); no branch between
        // the rounds of a full piece, so that one round's decode overlaps
        // the previous round's multiply-adds
        auto table_round = [&](uint32_t r) {
            uint32_t p[8];
            const uint32_t h3 = __shfl_sync(DGT_FULL, rl.h3, r);
            const uint32_t l1 = __shfl_sync(DGT_FULL, rl.l1, r);
            const bool own = (pm >> r) & 1u;
            weights(r, own ? mh3[r] : h3, own ? ml1[r] : l1, p);
            fma_round(r, p);
        };
        if (ok && !slow && pm == 0 && n == C && rp >= C - 1 && jw >= C && inner == 0) {
            // the common piece: full, one escape at most per round, within one
            // row and one unit (which may end at its last round); a cut row's
            // last round may be its last (rp == C - 1)
            const bool cutl = rp == C - 1 && !act;
#pragma unroll
            for (uint32_t r = 0; r < C; r++) {
                uint32_t p[8];
                weights(r, __shfl_sync(DGT_FULL, rl.h3, r), __shfl_sync(DGT_FULL, rl.l1, r), p);
                const float t = fma_chunk16(p, xs, jp + r, lane, acc);
                acc = (r == C - 1 && cutl) ? __fadd_rn(acc, 0.0f) : t;
            }
        } else if (ok && !slow && pm2 == 0 && n == C) {
#pragma unroll
            for (uint32_t r = 0; r < C; r++) table_round(r);
        } else if (ok && !slow && pm2 == 0) {
#pragma unroll
            for (uint32_t r = 0; r < C; r++) {
                if (r >= n) break;
                table_round(r);
            }
        } else if (ok) {
            // a round whose escapes need the general patch, a lane with two
            // escapes, or a short BF16 piece
            auto general_round = [&](uint32_t r) {
                uint32_t p[8];
                const uint32_t h3 = __shfl_sync(DGT_FULL, rl.h3, r);
                const uint32_t l1 = __shfl_sync(DGT_FULL, rl.l1, r);
                if (R4 && ((pm >> r) & 1u) && !((pmok >> r) & 1u)) {
                    // its escape index and ranks straight from memory
                    const uint64_t sx = px + r;
                    const uint32_t b = a.seg[sx], c = a.seg[sx + 1] - b;
                    const uint4 sv = *reinterpret_cast<const uint4 *>(stg + r * 512 + 16 * lane);
                    const uint2 nv = *reinterpret_cast<const uint2 *>(stg + C * 512 + r * 256 + 8 * lane);
                    r4_round_general_cb(a, L, nv, sv, c, b, escb[R4 ? w : 0], table_s, lane,
                                        r != rp || act, p);
                } else {
                    const bool own = (pm >> r) & 1u;
                    uint32_t oh3 = h3, ol1 = l1, oi2 = 16, oe2 = 0;
#pragma unroll
                    for (uint32_t i = 0; i < C; i++) {
                        if (i == r && own) {
                            oh3 = mh3[i];
                            ol1 = ml1[i];
                            oi2 = mi2[i];
                            oe2 = me2[i];
                        }
                    }
                    weights(r, oh3, ol1, p);
                    if ((pm2 >> r) & 1u) second_escape(oi2, oe2, p);
                }
                fma_round(r, p);
            };
            if constexpr (ROLL) {
#pragma unroll 1
                for (uint32_t r = 0; r < n; r++) general_round(r);
            } else {
#pragma unroll
                for (uint32_t r = 0; r < C; r++) {
                    if (r >= n) break;
                    general_round(r);
                }
            }
        }
        __syncwarp();
        // a stage is released only after a good wait: after a timeout the
        // producer stops, and the copies in flight are waited for below
        if (ok && lane == 0) mbar_arrive(empty_a + 8 * st);
        st = st + 1 == TNS ? 0 : st + 1;
        // the units that ended in this piece, in order: before its last
        // round (fin), then at it (acc)
        if (inner) {
#pragma unroll
            for (uint32_t r = 0; r + 1 < C; r++) {
                if ((inner >> r) & 1u) {
                    float v = fin[r];
#pragma unroll
                    for (int d = 16; d >= 1; d >>= 1) v += __shfl_xor_sync(DGT_FULL, v, d);
                    if (lane == 0) part[udone - c0] = v;
                    udone++;
                }
            }
        }
    };
    for (uint64_t ch = 0; ch < nchunks; ch++) {
        c0 = ch * TCHUNK;
        const uint64_t cend = min(c0 + TCHUNK, units);
        if constexpr (CONTIG) {
            // this warp's stretch of the chunk, walked piece by piece; a piece
            // may hold the ends of several units
            const ChunkWalk k = chunk_walk((uint32_t)ch, (uint32_t)units, w);
            if (k.ua < k.ub) {
                Stretch cs = stretch_start(k.ua, k.ub, x0, f0, log2S, J, K);
                udone = k.ua;
                uint32_t unext = k.ua + 1;                   // the unit after the current one
                uint32_t uleft = unit_len(k.ua, log2S, J);   // rounds of the current unit not yet taken
                acc = 0.0f;
                while (cs.left) {
                    const uint32_t n = piece_len<C>(cs, J, span);
                    // the piece's rounds that end a unit (bit r: round r)
                    uint32_t emask = 0, r = 0;
                    while (uleft <= n - r) {
                        r += uleft;
                        emask |= 1u << (r - 1);
                        uleft = unit_len(unext++, log2S, J);
                    }
                    uleft -= n - r;
                    piece(n, cs.j, cs.x, emask & ((1u << (n - 1)) - 1u), J - cs.j);
                    if (emask >> (n - 1)) {
#pragma unroll
                        for (int d = 16; d >= 1; d >>= 1) acc += __shfl_xor_sync(DGT_FULL, acc, d);
                        if (lane == 0) part[udone - c0] = acc;
                        udone++;
                        acc = 0.0f;
                    }
                    stretch_advance(cs, n, J);
                }
            }
        } else {
            // units w, w + TNW, ...: each its own pieces
            for (uint64_t uu = c0 + w; uu < cend; uu += TNW) {
                const uint32_t j0 = unit_j0((uint32_t)uu, log2S, J), j1 = j0 + unit_len((uint32_t)uu, log2S, J);
                const uint64_t xr = x0 + (uu >> log2S) * J;
                acc = 0.0f;
                for (uint32_t jp = j0; jp < j1; jp += C) piece(min(C, j1 - jp), jp, xr + jp, 0u, 0xFFFFFFFFu);
#pragma unroll
                for (int d = 16; d >= 1; d >>= 1) acc += __shfl_xor_sync(DGT_FULL, acc, d);
                if (lane == 0) part[uu - c0] = acc;
            }
        }
        asm volatile("bar.sync 1, %0;" ::"r"(TNW * 32) : "memory");
        const uint32_t S = 1u << log2S;
        for (uint32_t t = tid; t < (cend - c0) / S; t += TNW * 32) {
            float y = part[t * S];
            for (uint32_t s = 1; s < S; s++) y = y + part[t * S + s];
            const uint64_t orow = o0 + c0 / S + t;
            if (a.y32) a.y32[orow] = y;
            if (a.y) a.y[orow] = f32_to_bf16_rne(y);
        }
        asm volatile("bar.sync 1, %0;" ::"r"(TNW * 32) : "memory");
    }
    // after a timeout: the ring's producer stops, and the copies it issued
    // that this warp did not take land before exit
    if (!ok) ring_drain(&stop_word[w], full_a, waited, TNS);
}

// Any shape / alignment: one warp per (row, slice), element loads, x read
// from global memory.  Same order as k_gemv.
template <bool R4>
__global__ void __launch_bounds__(GW * 32) k_gemv_any(GemvArgs a, int S) {
    __shared__ float part[GW];
    const uint32_t w = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t RPB = GW / S;
    const uint32_t rl = w / S, s = w % S;
    const uint32_t j0 = (uint32_t)((uint64_t)s * a.J / S), j1 = (uint32_t)((uint64_t)(s + 1) * a.J / S);
    const uint64_t groups = (a.rows + RPB - 1) / RPB;
    for (uint64_t gi = blockIdx.x; gi < groups; gi += gridDim.x) {
        const uint64_t row = gi * RPB + rl;
        float acc = 0.0f;
        if (row < a.rows) {
            const uint64_t rbase = row * a.cols;
            for (uint32_t j = j0; j < j1; j++) {
                const uint64_t k0 = (uint64_t)j * 512 + 16 * lane;
                const uint32_t len = k0 < a.cols ? (uint32_t)min((uint64_t)16, a.cols - k0) : 0u;
                uint32_t idx = 0;
                if (R4) {
                    uint32_t c = 0;
                    for (uint32_t i = 0; i < len; i++) {
                        const uint64_t f = rbase + k0 + i;
                        c += ((a.nib[f >> 1] >> (4 * (f & 1))) & 15u) == 15u;
                    }
                    uint32_t tot;
                    const uint64_t su = row * a.nseg + j;
                    idx = a.seg[su] + warp_excl_scan(c, &tot);
                    if (tot != a.seg[su + 1] - a.seg[su] && lane == 0) set_status(a.status, DGT_ERR_CORRUPT);
                }
                for (uint32_t i = 0; i < len; i++) {
                    const uint64_t f = rbase + k0 + i;
                    uint32_t bits;
                    if (R4) {
                        uint32_t r = (a.nib[f >> 1] >> (4 * (f & 1))) & 15u;
                        if (r == 15u) {
                            r = idx < a.n_esc ? a.esc[idx] : 0u;
                            idx++;
                        }
                        const uint32_t smb = a.sm[f];
                        bits = ((smb & 0x80u) << 8) | ((uint32_t)a.table[r] << 7) | (smb & 0x7Fu);
                    } else {
                        bits = a.W[f];
                    }
                    const float xv = __uint_as_float((uint32_t)a.x[k0 + i] << 16);
                    acc = fmaf(__uint_as_float(bits << 16), xv, acc);
                }
            }
        }
        for (int d = 16; d >= 1; d >>= 1) acc += __shfl_xor_sync(DGT_FULL, acc, d);
        if (lane == 0) part[w] = acc;
        __syncthreads();
        if (s == 0 && lane == 0 && row < a.rows) {
            float y = part[w];
            for (int t = 1; t < S; t++) y = y + part[w + t];
            if (a.y32) a.y32[row] = y;
            if (a.y) a.y[row] = f32_to_bf16_rne(y);
        }
        __syncthreads();
    }
}

template <bool R4>
int launch_gemv(GemvArgs &a, int path, cudaStream_t st) {
    DeviceInfo di;
    if (device_info(&di) != DGT_OK) return DGT_ERR_CUDA;
    a.S = dgt_plan_slices(a.rows, a.cols);
    int bps = 0;
    if (path == 2) {
        // R4 units whose round count is a multiple of 6 stream as 6-round pieces
        constexpr uint32_t C6 = R4 ? GEMV_C6 : DGT_GEMV_C_R4;   // BF16 has one piece length
        using D = TmaCfg<R4>;
        using E = TmaCfg<R4, C6>;
        const bool c6 = R4 && a.J % a.S == 0 && (a.J / a.S) % GEMV_C6 == 0 &&
                        (size_t)TNW * E::NS * E::STAGE + (size_t)a.J * 1024 <= (size_t)DGT_GEMV_SMEM_KB * 1024;
        // R4 units of one or two rounds (fewer than two on average): each warp
        // streams a contiguous stretch of them, pieces running across their
        // ends.  (At two rounds each, 3840 x 4096, the stretches ran faster
        // back to back but slower inside a decode step.)
        const bool contig = R4 && a.J < 2u * (uint32_t)a.S;
        void (*fn)(GemvArgs) = c6 ? k_gemv_tma<R4, C6> : contig ? k_gemv_tma<R4, DGT_GEMV_C_R4, R4> : k_gemv_tma<R4>;
        const size_t smem = (size_t)TNW * (c6 ? E::NS * E::STAGE : D::NS * D::STAGE) + (size_t)a.J * 1024;
        if (prepare_kernel((const void *)fn, smem, (TNW + TPW) * 32, &bps) != DGT_OK) return DGT_ERR_CUDA;
        const unsigned grid = (unsigned)min((uint64_t)di.sms, a.rows);
        if (launch_pdl(fn, dim3(grid), dim3((TNW + TPW) * 32), smem, st, a) != cudaSuccess)
            return DGT_ERR_CUDA;
    } else if (path == 1) {
        const size_t smem = (size_t)a.J * 1024;
        if (prepare_kernel((const void *)k_gemv<R4, 16, 4>, smem, 16 * 32, &bps) != DGT_OK) return DGT_ERR_CUDA;
        const unsigned grid = (unsigned)min((uint64_t)di.sms, a.rows);
        k_gemv<R4, 16, 4><<<grid, 16 * 32, smem, st>>>(a);
    } else {
        const uint64_t groups = (a.rows + (GW / a.S) - 1) / (GW / a.S);
        if (prepare_kernel((const void *)k_gemv_any<R4>, 0, GW * 32, &bps) != DGT_OK) return DGT_ERR_CUDA;
        const uint64_t grid = min((uint64_t)di.sms * bps, groups);
        k_gemv_any<R4><<<(unsigned)grid, GW * 32, 0, st>>>(a, a.S);
    }
    return cudaPeekAtLastError() == cudaSuccess ? DGT_OK : DGT_ERR_CUDA;
}

// 2: bulk-copy kernel, 1: register-streaming kernel, 0: any-shape kernel.
template <bool R4>
int choose_path(uint64_t K, uint32_t J, bool aligned) {
    if (K == 0 || K % 16 != 0 || !aligned) return 0;
    const size_t tma_smem = (size_t)TNW * TmaCfg<R4>::NS * TmaCfg<R4>::STAGE + (size_t)J * 1024;
    if (K % 32 == 0 && tma_smem <= (size_t)DGT_GEMV_SMEM_KB * 1024) return 2;
    return J <= MAX_FAST_ROUNDS ? 1 : 0;
}

}  // namespace dgt

using namespace dgt;

// Flags the batch-1 products accept: the static-weights promise, and the
// failure-path test hook with its poll count in bits 16..31.
static inline bool gemv_flags_ok(unsigned flags) {
    const unsigned known = DGT_GEMV_STATIC_WEIGHTS | DGT_TEST_SHORT_WAITS;
    if (flags & ~(known | 0xFFFF0000u)) return false;
    return (flags & DGT_TEST_SHORT_WAITS) || !(flags >> 16);
}

extern "C" int dgt_gemv_ex(const dgt_r4 *W, const uint16_t *d_x, uint16_t *d_y, float *d_y32, int32_t *d_status,
                           unsigned flags, void *stream) {
    if (!W || !gemv_flags_ok(flags)) return DGT_ERR_ARG;
    const uint64_t N = W->rows, K = W->cols;
    if (K >= (1ull << 31) || (N && (N * K) / N != K)) return DGT_ERR_SHAPE;
    if (N == 0) return DGT_OK;
    if (!d_y && !d_y32) return DGT_ERR_ARG;
    if (K && (!d_x || !W->sm || !W->nib || !W->seg || (W->n_esc && !W->esc))) return DGT_ERR_ARG;
    GemvArgs a = {};
    a.sm = W->sm;
    a.nib = W->nib;
    a.esc = W->esc;
    a.seg = W->seg;
    a.rsum = W->seg + dgt_rsum_offset(N, dgt_r4_nseg(K));
    a.x = d_x;
    a.y = d_y;
    a.y32 = d_y32;
    a.rows = N;
    a.cols = K;
    a.nseg = dgt_r4_nseg(K);
    a.n_esc = W->n_esc;
    a.J = (uint32_t)((K + 511) / 512);
    a.L = make_r4lut(W->table, W->n_table);
    for (int i = 0; i < 256; i++) a.table[i] = W->table[i];
    a.status = d_status;
    a.early = flags & DGT_GEMV_STATIC_WEIGHTS;
    a.spin = wait_limit_from_flags(flags);
    const int path = choose_path<true>(K, a.J, aligned16(W->sm) && aligned16(W->nib) && aligned16(d_x));
    return launch_gemv<true>(a, path, (cudaStream_t)stream);
}

extern "C" int dgt_gemv(const dgt_r4 *W, const uint16_t *d_x, uint16_t *d_y, float *d_y32, int32_t *d_status,
                        void *stream) {
    return dgt_gemv_ex(W, d_x, d_y, d_y32, d_status, 0u, stream);
}

extern "C" int dgt_gemv_bf16_ex(const uint16_t *d_W, uint64_t rows, uint64_t cols, const uint16_t *d_x,
                                uint16_t *d_y, float *d_y32, int32_t *d_status, unsigned flags, void *stream) {
    if (!gemv_flags_ok(flags)) return DGT_ERR_ARG;
    const uint64_t N = rows, K = cols;
    if (K >= (1ull << 31) || (N && (N * K) / N != K)) return DGT_ERR_SHAPE;
    if (N == 0) return DGT_OK;
    if (!d_y && !d_y32) return DGT_ERR_ARG;
    if (K && (!d_x || !d_W)) return DGT_ERR_ARG;
    GemvArgs a = {};
    a.W = d_W;
    a.status = d_status;
    a.x = d_x;
    a.y = d_y;
    a.y32 = d_y32;
    a.rows = N;
    a.cols = K;
    a.J = (uint32_t)((K + 511) / 512);
    a.early = flags & DGT_GEMV_STATIC_WEIGHTS;
    a.spin = wait_limit_from_flags(flags);
    const int path = choose_path<false>(K, a.J, aligned16(d_W) && aligned16(d_x));
    return launch_gemv<false>(a, path, (cudaStream_t)stream);
}

extern "C" int dgt_gemv_bf16(const uint16_t *d_W, uint64_t rows, uint64_t cols, const uint16_t *d_x,
                             uint16_t *d_y, float *d_y32, int32_t *d_status, void *stream) {
    return dgt_gemv_bf16_ex(d_W, rows, cols, d_x, d_y, d_y32, d_status, 0u, stream);
}

// ---------------------------------------------------------------------------
// Expert blocks: the expert gather with few (token, slot) pairs runs as the
// bulk-copy kernel over the pairs' expert rows (GemvArgs.ids), each pair with
// its own group of CTAs and its token's x; no routing lists, no slice
// workspace.  Same order as the gather (the batch-1 order, plan S(ne, K)).
// ---------------------------------------------------------------------------
namespace dgt {

template <bool R4>
static int launch_expert_blocks(GemvArgs &a, cudaStream_t st) {
    const uint64_t pairs = a.pairs;
    if (pairs == 0) return DGT_OK;
    DeviceInfo di;
    if (device_info(&di) != DGT_OK) return DGT_ERR_CUDA;
    const size_t smem = (size_t)TNW * TmaCfg<R4>::NS * TmaCfg<R4>::STAGE + (size_t)a.J * 1024;
    if (a.cols % 32 || smem > (size_t)DGT_GEMV_SMEM_KB * 1024 || pairs > (uint64_t)di.sms)
        return DGT_ERR_UNSUPPORTED;
    a.S = dgt_plan_slices(a.ne, a.cols);
    void (*fn)(GemvArgs) = R4 && a.J < 2u * (uint32_t)a.S ? k_gemv_tma<R4, DGT_GEMV_C_R4, R4> : k_gemv_tma<R4>;
    int bps = 0;
    if (prepare_kernel((const void *)fn, smem, (TNW + TPW) * 32, &bps) != DGT_OK) return DGT_ERR_CUDA;
    const unsigned grid = (unsigned)min((uint64_t)di.sms, pairs * a.ne);
    if (launch_pdl(fn, dim3(grid), dim3((TNW + TPW) * 32), smem, st, a) != cudaSuccess)
        return DGT_ERR_CUDA;
    return cudaPeekAtLastError() == cudaSuccess ? DGT_OK : DGT_ERR_CUDA;
}

}  // namespace dgt

int dgt_gemv_expert_blocks(const dgt_r4 *W, uint32_t n_experts, const int32_t *d_ids, uint32_t tokens,
                           uint32_t topk, const uint16_t *d_x, float *d_y32, int32_t *d_status, uint32_t spin,
                           void *stream) {
    if (!W || !n_experts || W->rows % n_experts || !d_ids || !d_x || !d_y32) return DGT_ERR_ARG;
    if (!aligned16(W->sm) || !aligned16(W->nib) || !aligned16(W->seg) || !aligned16(d_x))
        return DGT_ERR_UNSUPPORTED;
    const uint64_t K = W->cols;
    GemvArgs a = {};
    a.sm = W->sm;
    a.nib = W->nib;
    a.esc = W->esc;
    a.seg = W->seg;
    a.rsum = W->seg + dgt_rsum_offset(W->rows, dgt_r4_nseg(K));
    a.x = d_x;
    a.y32 = d_y32;
    a.rows = W->rows;
    a.cols = K;
    a.nseg = dgt_r4_nseg(K);
    a.n_esc = W->n_esc;
    a.J = (uint32_t)((K + 511) / 512);
    a.L = make_r4lut(W->table, W->n_table);
    for (int i = 0; i < 256; i++) a.table[i] = W->table[i];
    a.status = d_status;
    a.spin = spin;
    a.ids = d_ids;
    a.pairs = tokens * topk;
    a.topk = topk;
    a.n_experts = n_experts;
    a.ne = W->rows / n_experts;
    return launch_expert_blocks<true>(a, (cudaStream_t)stream);
}

int dgt_gemv_expert_blocks_bf16(const uint16_t *d_W, uint64_t rows, uint64_t cols, uint32_t n_experts,
                                const int32_t *d_ids, uint32_t tokens, uint32_t topk, const uint16_t *d_x,
                                float *d_y32, int32_t *d_status, uint32_t spin, void *stream) {
    if (!d_W || !n_experts || rows % n_experts || !d_ids || !d_x || !d_y32) return DGT_ERR_ARG;
    if (!aligned16(d_W) || !aligned16(d_x)) return DGT_ERR_UNSUPPORTED;
    GemvArgs a = {};
    a.W = d_W;
    a.x = d_x;
    a.y32 = d_y32;
    a.rows = rows;
    a.cols = cols;
    a.J = (uint32_t)((cols + 511) / 512);
    a.status = d_status;
    a.spin = spin;
    a.ids = d_ids;
    a.pairs = tokens * topk;
    a.topk = topk;
    a.n_experts = n_experts;
    a.ne = rows / n_experts;
    return launch_expert_blocks<false>(a, (cudaStream_t)stream);
}
