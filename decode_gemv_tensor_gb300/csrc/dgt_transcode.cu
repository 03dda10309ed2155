// dgt_transcode.cu -- load transcode (format 2 / format 1 -> R4) and the
// R4 -> BF16 rebuild.
//
// Binade README, "How it works", "Runtime layout": at load a GPU kernel turns
// either file format into R4.  The decode organisation follows the "Best
// measured configuration" of the "Lossless BF16 weight compression" README
// (blocks of 64 symbols, an 8-bit length per block turned into offsets by a
// warp prefix sum, output staged in shared memory and written coalesced),
// re-designed for sm_103a:
//  - one warp per group of 32 blocks (format 2) or 32 tiles (format 1), one
//    lane per block/tile; a persistent grid;
//  - format 2: each lane decodes its Rice block two codes at a time through a
//    12-bit window table in shared memory, so a full block is exactly 32
//    table steps; windows the table does not finish take an out-of-line step;
//  - escapes (ranks >= 15) are collected per lane, placed by a warp prefix sum
//    from the group's escape base, and the row-segment escape index (seg) is
//    written for every segment that starts inside the group;
//  - every group checks its index against its neighbours and its decoded
//    length against its index bytes; a mismatch sets the status word.
#include <cuda_runtime.h>
#include <type_traits>

#include "../../include/dgt.h"
#include "dgt_device.cuh"
#include "dgt_internal.h"
#include "dgt_launch.h"

namespace dgt {


// ---------------------------------------------------------------------------
// segment starts inside a unit [B0, B0 + cnt): seg index and offset
// ---------------------------------------------------------------------------
struct SegWalk {
    uint64_t r, c;  // row and column of the next segment start
};

__device__ __forceinline__ SegWalk first_seg_start(uint64_t B0, uint64_t r0, uint64_t cols) {
    uint64_t local = B0 - r0 * cols;
    uint64_t dr = 0;
    if (local >= cols) dr = cols >= 8192 ? 1 : (uint64_t)((uint32_t)local / (uint32_t)cols);
    SegWalk s;
    s.r = r0 + dr;
    s.c = B0 - s.r * cols;
    if (s.c % DGT_SEG) {
        s.c = (s.c / DGT_SEG + 1) * DGT_SEG;
        if (s.c >= cols) { s.r++; s.c = 0; }
    }
    return s;
}

__device__ __forceinline__ void next_seg_start(SegWalk &s, uint64_t cols) {
    s.c += DGT_SEG;
    if (s.c >= cols) { s.r++; s.c = 0; }
}

// ---------------------------------------------------------------------------
// format 2 (Rice) -> R4
//
// Block layout (dgt.h): a Rice block holds its remainder field (the k low
// bits of every rank; in a full block with k = 1, 2 in nibble-slot order)
// and then every rank's unary part (q = r >> k zeros, a one).  One warp per
// group of 32 blocks, one lane per 64-rank block, a persistent grid.
//
// A full block with k <= 2 is decoded in exactly 16 steps of four ranks.  The
// next 14 bits of its unary parts index a table whose entry holds the four
// quotients as 4-bit fields min(q << k, 15), the bits they use and a flag for
// a field that may belong to an escape (rank >= 15).  A step is a window
// extract, one table load and a position update.  Two steps give the
// quotient fields of eight ranks; one shift and one mask of a remainder field
// word put the remainders under them, giving one 32-bit word of eight R4
// nibbles (nibble = min(rank, 15) since (q << k) | rem saturates exactly when
// the rank is 15 or more).  A window with fewer than four complete codes
// finishes its step code by code with find-first-set, in line.  The table is
// built at compile time (one per k) and bulk-copied into shared memory while
// the previous kernel of the stream finishes.  An output word whose fields
// may hold an escape records where its codes start; after the loop those
// words are decoded again code by code to get the escapes' exact ranks.  Raw
// and partial blocks, k >= 3 and groups too long to stage take a per-code
// path.  The next group's stream is copied to shared memory (cp.async) while
// this one decodes.
// ---------------------------------------------------------------------------
struct F2Args {
    const uint32_t *words;
    uint64_t n_words;
    const uint8_t *blkq;
    const uint32_t *grp;
    uint64_t n, cols, nseg, nblk, ngrp;
    int k;
    uint8_t *nib;
    uint8_t *esc;
    uint32_t *seg;
    uint64_t n_esc, seg_last;
    int32_t *status;
};

#ifndef DGT_RICE_RW
#define DGT_RICE_RW 32
#endif
constexpr int RW = DGT_RICE_RW;  // warps per CTA
constexpr int RWIN = 14;         // table window bits
constexpr int RCAP = 192;        // staged stream words per group (about 170 at 2.7 bits/rank)
constexpr int RPAD = 16;         // zero words after the staged stream
constexpr int RBUF = RCAP + RPAD;
constexpr int RESC = 16;         // escape ranks kept per lane; more re-walk the block
constexpr uint32_t R4_ESCF = 1u << 16;   // table entry: a field may belong to an escape

// Table entry for window v (bit 0 = next bit of the unary parts): bits 0..15
// the fields min(q << k, 15) of the first four codes, R4_ESCF if one of them
// is at least 16 - 2^k (the rank may be 15 or more), bits 28..31 the bits the
// four use.  A window with fewer than four complete codes has 0 in bits
// 28..31, the fields of its c complete codes, c in bits 17..19 and the bits
// they use in bits 20..23.
constexpr uint32_t rice4_entry(uint32_t v, int k) {
    uint32_t pos = 0, f = 0, fl = 0;
    for (uint32_t c = 0; c < 4; c++) {
        uint32_t q = 0;
        while (pos + q < (uint32_t)RWIN && !((v >> (pos + q)) & 1u)) q++;
        if (pos + q >= (uint32_t)RWIN) return f | fl | (c << 17) | (pos << 20);
        const uint32_t fq = (q << k) < 15u ? (q << k) : 15u;
        f |= fq << (4 * c);
        if (fq >= 16u - (1u << k)) fl = R4_ESCF;
        pos += q + 1;
    }
    return f | fl | (pos << 28);
}

struct RiceLut {
    uint32_t t[3][1 << RWIN];
};
constexpr RiceLut make_rice_lut() {
    RiceLut r{};
    for (int k = 0; k < 3; k++)
        for (uint32_t v = 0; v < (1u << RWIN); v++) r.t[k][v] = rice4_entry(v, k);
    return r;
}
// The three tables (k = 0, 1, 2) in the library's device image: 192 KB,
// built by the compiler.
__device__ __align__(16) const RiceLut g_rice_lut = make_rice_lut();

template <class Src>
struct WordReader {
    Src src;
    uint32_t nw;
    __device__ __forceinline__ uint32_t operator()(uint32_t i) const { return i < nw ? src[i] : 0u; }
};

// Zeros before the next one at bit pos (at most 255 counted; more set bad);
// pos moves past the one.
template <class Rd>
__device__ __forceinline__ uint32_t unary_at(const Rd &rd, uint32_t &pos, bool &bad) {
    const uint32_t win = __funnelshift_r(rd(pos >> 5), rd((pos >> 5) + 1), pos);
    if (win) {
        const uint32_t q = __ffs(win) - 1;
        pos += q + 1;
        return q;
    }
    uint32_t p = pos, q = 0;
    for (;;) {
        const uint32_t wv = rd(p >> 5) >> (p & 31);
        const uint32_t avail = 32 - (p & 31);
        if (wv) {
            const uint32_t f = __ffs(wv) - 1;
            q += f;
            p += f;
            break;
        }
        q += avail;
        p += avail;
        if (q > 255) {
            bad = true;
            break;
        }
    }
    pos = p + 1;
    return q;
}

// k bits at bit pos (k <= 8).
template <class Rd>
__device__ __forceinline__ uint32_t bits_at(const Rd &rd, uint32_t pos, int k) {
    return __funnelshift_r(rd(pos >> 5), rd((pos >> 5) + 1), pos) & ((1u << k) - 1u);
}

// Position, inside a block's remainder field, of the remainder of rank i
// (cnt ranks): nibble-slot order for a full block with k = 1, 2, else k bits
// per rank in order.
__device__ __forceinline__ uint32_t rem_field_pos(int k, uint32_t cnt, uint32_t i) {
    if (cnt == DGT_BLOCK && (k == 1 || k == 2)) {
        const uint32_t m = i >> 3, j = i & 7, per = 4u / (uint32_t)k;
        return 32u * (m / per) + 4u * j + (uint32_t)k * (m % per);
    }
    return (uint32_t)k * i;
}

// Rank i of a block starting at bit b0 (the per-code path); *up = the next
// unary part (advanced).
template <class Rd>
__device__ __forceinline__ uint32_t rice_rank_slow(const Rd &rd, uint32_t b0, uint32_t *up, uint32_t i, uint32_t cnt,
                                                   int k, bool raw, bool &bad) {
    if (raw) return bits_at(rd, b0 + 8 * i, 8);
    const uint32_t q = unary_at(rd, *up, bad);
    const uint32_t rem = k ? bits_at(rd, b0 + rem_field_pos(k, cnt, i), k) : 0u;
    uint32_t r = (q << k) | rem;
    if (r > 255) {
        bad = true;
        r = 255;
    }
    return r;
}

// Per-code path for one block: nibbles straight to nib (bytes).
struct SlowBlock {
    uint32_t ec, end, bad;
    uint64_t emask;   // bit s: rank s of the block is an escape
};
template <class Rd>
__device__ __noinline__ SlowBlock rice_block_slow(Rd rd, uint32_t b0, uint32_t cnt, bool raw, int k, uint8_t *nib) {
    bool bad = false;
    uint32_t up = b0 + cnt * (uint32_t)k, byte = 0, ec = 0;
    uint64_t em = 0;
    for (uint32_t s = 0; s < cnt; s++) {
        const uint32_t r = rice_rank_slow(rd, b0, &up, s, cnt, k, raw, bad);
        if (r >= 15) {
            ec++;
            em |= 1ull << s;
        }
        byte |= min(r, 15u) << (4 * (s & 1));
        if ((s & 1) || s + 1 == cnt) {
            nib[s >> 1] = (uint8_t)byte;
            byte = 0;
        }
    }
    SlowBlock o;
    o.ec = ec;
    o.end = raw ? b0 + 8 * cnt : up;
    o.bad = bad;
    o.emask = em;
    return o;
}

// The escapes of one block (per-code path) written to dst in order.
template <class Rd>
__device__ __noinline__ void rice_block_slow_escapes(Rd rd, uint32_t b0, uint32_t cnt, bool raw, int k, uint8_t *dst) {
    bool bad = false;
    uint32_t up = b0 + cnt * (uint32_t)k;
    for (uint32_t s = 0; s < cnt; s++) {
        const uint32_t r = rice_rank_slow(rd, b0, &up, s, cnt, k, raw, bad);
        if (r >= 15) *dst++ = (uint8_t)r;
    }
}

__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait1() { asm volatile("cp.async.wait_group 1;" ::: "memory"); }
__device__ __forceinline__ void cp_async16(uint32_t *dst, const uint32_t *src, uint32_t bytes) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(smem_u32(dst)), "l"(src), "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ void cp_async4(uint32_t *dst, const uint32_t *src, uint32_t bytes) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;" ::"r"(smem_u32(dst)), "l"(src), "r"(bytes)
                 : "memory");
}

// A group's index entries and this lane's block index byte, loaded one or
// two groups ahead of use.
struct RiceMeta {
    uint32_t w0, base;     // first stream word, escapes before the group
    uint32_t nextw, nexte; // the same for the following group (or the totals)
    uint32_t q;            // this lane's block index byte
};

template <class IX>
__device__ __forceinline__ RiceMeta rice_meta(const F2Args &a, IX g, uint32_t lane) {
    RiceMeta m = {0, 0, 0, 0, 0};
    const IX ngrp = (IX)a.ngrp;
    if (g < ngrp) {
        const uint32_t *gp = a.grp + 2 * (uint64_t)g;
        m.w0 = gp[0];
        m.base = gp[1];
        m.nextw = g + 1 < ngrp ? gp[2] : (uint32_t)a.n_words;
        m.nexte = g + 1 < ngrp ? gp[3] : (uint32_t)a.n_esc;
        const IX blk = g * DGT_GROUP + lane;
        m.q = blk < (IX)a.nblk ? a.blkq[blk] : 0u;
    }
    return m;
}

// Group g's stream in 16-byte pieces from the 16-byte boundary at or below
// its first word (the stream then starts 32 * (w0 % 4) bits into dst); bytes
// past the stream array's end, and past the buffer's need, are zero-filled.
// The stream array must start on a 16-byte boundary.
template <class IX>
__device__ __forceinline__ void rice_stage16(const F2Args &a, IX g, const RiceMeta &m, uint32_t *dst,
                                             uint32_t lane) {
    if (g < (IX)a.ngrp) {
        const uint32_t a0 = m.w0 & ~3u;
        const uint32_t need = m.nextw > a0 ? min(m.nextw - a0, (uint32_t)RBUF) : 0u;
        const uint32_t nw = (uint32_t)a.n_words;   // < 2^32 on this path
        for (uint32_t i = lane; i < RBUF / 4; i += 32) {
            const uint32_t wi = a0 + 4 * i;
            uint32_t bytes = 0;
            if (4 * i < need && wi < nw) bytes = min(16u, (nw - wi) * 4u);
            cp_async16(dst + 4 * i, bytes ? a.words + wi : a.words, bytes);
        }
    }
    cp_async_commit();
}

// Word by word copy for a stream array that is not 16-byte aligned (the
// stream starts at dst[0]).
__device__ __forceinline__ void rice_stage4(const F2Args &a, uint64_t g, const RiceMeta &m, uint32_t *dst,
                                            uint32_t lane) {
    if (g < a.ngrp) {
        const uint64_t w0 = m.w0, w1 = m.nextw;
        const uint64_t nw = (w1 > w0 && w1 <= a.n_words && w0 < a.n_words) ? w1 - w0 : 0;
        for (uint32_t i = lane; i < RBUF; i += 32) {
            const bool in = i < nw;
            cp_async4(dst + i, in ? a.words + w0 + i : a.words, in ? 4u : 0u);
        }
    }
    cp_async_commit();
}

struct RiceSmem {
    uint32_t lut[1 << RWIN];
    uint32_t buf[2][RW][RBUF];
    uint32_t rec[RW][8][32];      // per lane: where each flagged output word's codes start
    uint32_t recf[RW][8][32];     // and its quotient fields
    uint8_t escl[RW][RESC][32];   // per lane: escape ranks of the block, in order
    uint64_t lut_bar;
};

// FAST: 32-bit block indices (n < 2^31), blocks that never straddle rows
// (cols % 64 == 0, cols >= 2048), rows * nseg < 2^32 and a 16-byte aligned
// stream: the group bookkeeping takes a shorter path.  K = the tensor's Rice
// parameter for 0, 1, 2 (the table path); 3 for any larger k (per-code path).
template <bool FAST, int K>
__global__ void __launch_bounds__(RW * 32, 1) k_rice_to_r4(F2Args a) {
    extern __shared__ __align__(16) uint8_t rice_smem[];
    RiceSmem &S = *reinterpret_cast<RiceSmem *>(rice_smem);
    const uint32_t w = threadIdx.x >> 5, lane = threadIdx.x & 31;
    constexpr bool TAB = K <= 2;
    const int k = TAB ? K : a.k;
    const uint32_t bar = smem_u32(&S.lut_bar);
    if (TAB && threadIdx.x == 0) {
        // the table does not depend on the previous kernel: it is copied while
        // that kernel may still run
        mbar_init(bar, 1);
        fence_mbarrier_init();
        mbar_arrive_expect_tx(bar, sizeof(S.lut));
        bulk_g2s(smem_u32(S.lut), g_rice_lut.t[TAB ? K : 0], sizeof(S.lut), bar);
    }
    pdl_trigger();
    pdl_wait();
    if (blockIdx.x == 0 && threadIdx.x == 0) a.seg[a.seg_last] = (uint32_t)a.n_esc;
    __syncthreads();
    bool lut_ok = true;
    if (TAB) {
        lut_ok = mbar_wait(bar, 0);
        if (!lut_ok) {
            if (threadIdx.x == 0) set_status(a.status, DGT_ERR_TIMEOUT);
            mbar_wait(bar, 0);   // the copy lands before the CTA can exit
            return;
        }
    }
    // row / column of the group's first rank, stepped with the grid stride
    // (32-bit indices on the FAST path: n < 2^31)
    using IX = typename std::conditional<FAST, uint32_t, uint64_t>::type;
    const IX g0 = (IX)blockIdx.x * RW + w, G = (IX)gridDim.x * RW;
    const IX GS = (IX)DGT_GROUP * DGT_BLOCK;
    const IX cols = (IX)a.cols;
    IX r0 = (IX)(((uint64_t)g0 * GS) / cols), c0 = (IX)(((uint64_t)g0 * GS) % cols);
    const IX step_r = (IX)(((uint64_t)G * GS) / cols), step_c = (IX)(((uint64_t)G * GS) % cols);
    // index entries: group g in m0, g + G in m1 (its stream is copied while g
    // decodes), g + 2G loaded during g
    RiceMeta m0 = rice_meta(a, g0, lane);
    RiceMeta m1 = rice_meta(a, g0 + G, lane);
    if (FAST) rice_stage16(a, g0, m0, S.buf[0][w], lane);
    else rice_stage4(a, g0, m0, S.buf[0][w], lane);
    const uint32_t nfull = (uint32_t)(a.n / DGT_BLOCK), nblk32 = (uint32_t)a.nblk;
    uint32_t cur = 0;
    const IX ngrp = (IX)a.ngrp;
    for (IX g = g0; g < ngrp; g += G, cur ^= 1) {
        const uint32_t *buf = S.buf[cur][w];
        if (FAST) rice_stage16(a, g + G, m1, S.buf[cur ^ 1][w], lane);
        else rice_stage4(a, g + G, m1, S.buf[cur ^ 1][w], lane);
        const RiceMeta m2 = rice_meta(a, g + 2 * G, lane);
        const IX blk = g * DGT_GROUP + lane;
        const uint64_t B0 = (uint64_t)blk * DGT_BLOCK;
        uint32_t cnt;
        if (FAST) {
            const uint32_t b32 = (uint32_t)g * DGT_GROUP + lane;
            cnt = b32 < nfull ? DGT_BLOCK : (b32 < nblk32 ? (uint32_t)a.n - b32 * DGT_BLOCK : 0u);
        } else {
            cnt = blk < a.nblk ? (uint32_t)min((uint64_t)DGT_BLOCK, a.n - B0) : 0u;
        }
        const uint32_t boff = FAST ? 32u * (m0.w0 & 3u) : 0u;   // stream start inside the staged buffer
        const uint32_t q = cnt ? m0.q : 0u;
        const bool raw = q == 255;
        const uint32_t len = cnt == 0 ? 0u : (!raw ? cnt * (uint32_t)(k + 1) + q : 8u * cnt);
        uint32_t gbits;
        const uint32_t off = warp_excl_scan(len, &gbits);
        const uint32_t nw = (gbits + 31) / 32;
        const uint64_t gw0 = m0.w0, gbase = m0.base;
        const uint64_t next_w = m0.nextw, next_e = m0.nexte;
        m0 = m1;
        m1 = m2;
        // this lane's block: row and column of its first rank
        uint64_t br = r0, bc = c0 + (IX)DGT_BLOCK * lane;
        if (FAST) {
            uint32_t bc32 = (uint32_t)c0 + DGT_BLOCK * lane, br32 = (uint32_t)r0;
            if (bc32 >= (uint32_t)a.cols) {
                bc32 -= (uint32_t)a.cols;
                br32++;
            }
            br = br32;
            bc = bc32;
        } else if (bc >= a.cols) {
            if (a.cols >= GS) {
                bc -= a.cols;
                br++;
            } else {
                br += bc / a.cols;
                bc %= a.cols;
            }
        }
        c0 += step_c;
        r0 += step_r;
        if (c0 >= cols) {
            c0 -= cols;
            r0++;
        }
        cp_async_wait1();
        __syncwarp();
        if (gw0 + nw != next_w || next_w > a.n_words) {
            if (lane == 0) set_status(a.status, DGT_ERR_CORRUPT);
            __syncwarp();
            continue;
        }
        const bool staged = nw + (boff >> 5) <= RCAP;
        const uint32_t b0 = off + (staged ? boff : 0u);   // block start (bits) in the staged buffer or the stream
        const uint32_t end = b0 + len;
        bool bad = false;
        uint32_t ec = 0;
        uint64_t emask = 0;
        const bool fast = TAB && staged && cnt == DGT_BLOCK && !raw;
        if (TAB && fast) {
            constexpr uint32_t KK = TAB ? K : 0;
            constexpr uint32_t THR = 16u - (1u << KK);   // a field at least this may hold an escape
            uint32_t fw[4] = {0, 0, 0, 0};               // remainder field words
#pragma unroll
            for (int h = 0; h < 2 * (int)KK; h++) {
                const uint32_t p = b0 + 32 * h;
                fw[h] = __funnelshift_r(buf[p >> 5], buf[(p >> 5) + 1], p);
            }
            uint32_t p = b0 + 64 * KK;   // the unary parts
            uint32_t wi = p >> 5, lo = buf[wi], hi = buf[wi + 1];
            uint32_t out[8], nrec = 0, badw = 0;
#pragma unroll
            for (uint32_t m = 0; m < 8; m++) {
                const uint32_t pws = p;
                // two steps from one 32-bit window: a step uses at most 14 bits,
                // so the window shifted past the first step still covers the second
                uint32_t win = __funnelshift_r(lo, hi, p);
                uint32_t e2[2];
                bool inc = false;
#pragma unroll
                for (uint32_t h = 0; h < 2; h++) {
                    const uint32_t e = S.lut[win & ((1u << RWIN) - 1u)];
                    inc |= e < (1u << 28);
                    e2[h] = e;
                    win >>= e >> 28;
                }
                if (inc) {
                    // a window with fewer than four complete codes: each step again
                    // from its true start, the table's complete codes first, then
                    // the others one by one (find-first-set; long runs word by word)
#pragma unroll 1
                    for (uint32_t h = 0; h < 2; h++) {
                        uint32_t e = e2[0];
                        if (h) {
                            const uint32_t xi = p >> 5;
                            e = S.lut[__funnelshift_r(buf[xi], buf[xi + 1], p) & ((1u << RWIN) - 1u)];
                        }
                        if (e >= (1u << 28)) {
                            p += e >> 28;
                        } else {
                            uint32_t f = e & (0xFFFFu | R4_ESCF);
                            p += (e >> 20) & 15u;
                            for (uint32_t c = (e >> 17) & 7u; c < 4; c++) {
                                uint32_t qq = 0;
                                for (;;) {
                                    const uint32_t xi = p >> 5;
                                    const uint32_t x = __funnelshift_r(buf[xi], buf[xi + 1], p);
                                    if (x) {
                                        const uint32_t z = __ffs(x) - 1;
                                        qq += z;
                                        p += z + 1;
                                        break;
                                    }
                                    qq += 32;
                                    p += 32;
                                    if (qq > 255 || p > 32u * RCAP) break;
                                }
                                if (qq > 255 || p > 32u * RCAP) {
                                    badw = 1;
                                    p = 32u * RCAP;   // keeps every later buffer index in range
                                }
                                const uint32_t fq = min(qq << KK, 15u);
                                f |= fq << (4 * c);
                                if (fq >= THR) f |= R4_ESCF;
                            }
                            e = f;
                        }
                        e2[h] = e;
                    }
                    wi = p >> 5;
                    lo = buf[wi];
                    hi = buf[wi + 1];
                } else {
                    p += (e2[0] >> 28) + (e2[1] >> 28);
                    if ((p >> 5) != wi) {
                        lo = hi;
                        wi++;
                        hi = buf[wi + 1];
                    }
                }
                uint32_t x = __byte_perm(e2[0], e2[1], 0x5410u);
                if (KK == 1) x |= (fw[m >> 2] >> (m & 3)) & 0x11111111u;
                if (KK == 2) x |= (fw[m >> 1] >> (2 * (m & 1))) & 0x33333333u;
                out[m] = x;
                if ((e2[0] | e2[1]) & R4_ESCF) {
                    S.rec[w][nrec][lane] = pws << 3 | m;
                    S.recf[w][nrec][lane] = __byte_perm(e2[0], e2[1], 0x5410u);
                    nrec++;
                }
            }
            if (p != end || badw) bad = true;
            uint4 *dst = reinterpret_cast<uint4 *>(a.nib + B0 / 2);
            dst[0] = make_uint4(out[0], out[1], out[2], out[3]);
            dst[1] = make_uint4(out[4], out[5], out[6], out[7]);
            // flagged words: the exact rank of every field that may be an escape.
            // Code j of a word starts j + (sum of the earlier codes' quotients)
            // bits after the word's start; a field below the threshold is its
            // quotient << k exactly, a candidate's quotient is read from the stream.
            if (nrec) {
                const WordReader<const uint32_t *> rd{buf, RBUF};
                for (uint32_t i = 0; i < nrec; i++) {
                    const uint32_t rv = S.rec[w][i][lane];
                    const uint32_t ws = rv >> 3, mm = rv & 7u;
                    const uint32_t xw = mm < 4 ? (mm < 2 ? (mm == 0 ? out[0] : out[1]) : (mm == 2 ? out[2] : out[3]))
                                               : (mm < 6 ? (mm == 4 ? out[4] : out[5]) : (mm == 6 ? out[6] : out[7]));
                    // remainders from the field words (a saturated field reads 15 in
                    // the nibble whatever its remainder)
                    const uint32_t remw = KK == 1 ? ((mm >= 4 ? fw[1] : fw[0]) >> (mm & 3)) & 0x11111111u
                                        : KK == 2 ? ((mm >= 4 ? (mm >= 6 ? fw[3] : fw[2]) : (mm >= 2 ? fw[1] : fw[0])) >>
                                                     (2 * (mm & 1))) & 0x33333333u
                                                  : 0u;
                    // escapes are the nibbles 15.  One whose field is below 15 is
                    // exactly rank 15; a saturated field (15) is always an escape,
                    // and its quotient is read from the stream: its code starts j +
                    // (sum of the earlier quotients) bits after the word's start,
                    // where a field below 15 is its quotient << k exactly
                    const uint32_t F = S.recf[w][i][lane];
                    const uint32_t sat = nib15_mask(F);
                    uint32_t cand = nib15_mask(xw);
                    uint32_t fix = 0;   // saturated fields so far: exact quotient minus 15 >> k
                    while (cand) {
                        const uint32_t j = (__ffs(cand) - 1) >> 2;
                        cand &= cand - 1;
                        uint32_t r = 15;
                        if ((sat >> (4 * j)) & 1u) {
                            const uint32_t y = (F >> KK) & ((0xFu >> KK) * 0x11111111u) & ((1u << (4 * j)) - 1u);
                            const uint32_t before = __popc(y & 0x11111111u) + 2u * __popc(y & 0x22222222u) +
                                                    4u * __popc(y & 0x44444444u) + 8u * __popc(y & 0x88888888u);
                            uint32_t pp = ws + j + before + fix;
                            const uint32_t qq = unary_at(rd, pp, bad);
                            r = (qq << KK) | ((remw >> (4 * j)) & ((1u << KK) - 1u));
                            fix += qq - (15u >> KK);
                        }
                        if (ec < RESC) S.escl[w][ec][lane] = (uint8_t)min(r, 255u);
                        if (r > 255 || r < 15) bad = true;
                        ec++;
                    }
                }
            }
            if (!FAST && ec) {
                for (int mm = 0; mm < 8; mm++) {
                    const uint32_t msk = nib15_mask(out[mm]);
                    for (int j = 0; j < 8; j++)
                        if ((msk >> (4 * j)) & 1u) emask |= 1ull << (8 * mm + j);
                }
            }
        } else if (cnt) {
            const SlowBlock o = staged
                ? rice_block_slow(WordReader<const uint32_t *>{buf, RBUF}, b0, cnt, raw, k, a.nib + B0 / 2)
                : rice_block_slow(WordReader<const uint32_t *>{a.words + gw0, nw}, b0, cnt, raw, k, a.nib + B0 / 2);
            ec = o.ec;
            emask = o.emask;
            if (o.bad || o.end != end) bad = true;
        }
        // escapes, placed by a warp prefix sum from the group's escape base
        uint32_t etot;
        const uint32_t eb = warp_excl_scan(ec, &etot);
        if (gbase + etot != next_e || next_e > a.n_esc) bad = true;
        if (ec && !bad) {
            uint8_t *dst = a.esc + gbase + eb;
            if (fast && ec <= RESC) {
                for (uint32_t i = 0; i < ec; i++) dst[i] = S.escl[w][i][lane];
            } else if (staged) {
                rice_block_slow_escapes(WordReader<const uint32_t *>{buf, RBUF}, b0, cnt, raw, k, dst);
            } else {
                rice_block_slow_escapes(WordReader<const uint32_t *>{a.words + gw0, nw}, b0, cnt, raw, k, dst);
            }
        }
        // row-segment escape index for every segment that starts in this block
        if (FAST) {
            // the block lies in one row and starts on a multiple of 64: a segment
            // starts in it only at its first rank
            if (cnt && !bad && (bc & (DGT_SEG - 1)) == 0)
                a.seg[(uint32_t)br * (uint32_t)a.nseg + ((uint32_t)bc >> 9)] = (uint32_t)(gbase + eb);
        } else if (cnt && !bad) {
            uint32_t done = 0;
            uint64_t rr = br, cc = bc;
            while (done < cnt) {
                for (uint64_t s = (cc + DGT_SEG - 1) / DGT_SEG * DGT_SEG; s < a.cols && s - cc < cnt - done;
                     s += DGT_SEG) {
                    const uint32_t o = done + (uint32_t)(s - cc);
                    const uint64_t before = o ? (emask & ((~0ull) >> (64 - o))) : 0ull;
                    a.seg[rr * a.nseg + s / DGT_SEG] = (uint32_t)(gbase + eb + __popcll(before));
                }
                done += (uint32_t)min(a.cols - cc, (uint64_t)(cnt - done));
                rr++;
                cc = 0;
            }
        }
        if (bad) set_status(a.status, DGT_ERR_CORRUPT);
        __syncwarp();
    }
    asm volatile("cp.async.wait_all;" ::: "memory");
}

// ---------------------------------------------------------------------------
// format 1 -> R4
//
// One warp per group of 32 tiles, one lane per 128-rank tile.  A full tile of
// width w <= 4 is read with w 16-byte loads into registers.  Each run of eight
// w-bit codes becomes eight nibbles by three shift-and-add steps (the codes
// keep their order), and the codes equal to the escape code 2^w - 1 are found
// with one add and one mask.  The nibble words go to shared memory; each lane
// then patches its escaped nibbles from the group's escape bytes, in order,
// and records the ranks >= 15.  The group's nibbles leave with coalesced
// 16-byte stores.  Widths 5..8 and a short last tile take a per-code path.
// ---------------------------------------------------------------------------
struct F1Args {
    const uint8_t *payload;
    uint64_t payload_bytes;
    const uint8_t *tw;
    const uint8_t *tesc;
    const uint8_t *esc1;
    uint64_t n_esc1;
    const uint32_t *grp1;
    uint64_t n, cols, nseg, ntile, ngrp;
    uint8_t *nib;
    uint8_t *esc;
    uint32_t *seg;
    uint64_t n_esc, seg_last;
    int32_t *status;
};

constexpr int FW = 8;           // warps per CTA
constexpr int F1_E1CAP = 512;   // staged format-1 escape bytes per group
constexpr int F1_LIST = 16;     // ranks >= 15 kept per tile; more re-walk the tile
constexpr int F1_OSTR = 17;     // words per tile row of the staged output (16 + pad)

struct F1Smem {
    uint32_t out[FW][32 * F1_OSTR];
    uint8_t e1[FW][F1_E1CAP];
    uint16_t list[FW][32][F1_LIST];
};

// Eight w-bit codes (bits 0..8w-1 of x, first code lowest) -> eight nibbles.
template <int W>
__device__ __forceinline__ uint32_t f1_widen(uint32_t x) {
    if constexpr (W >= 4) {
        return x;
    } else {
    constexpr uint32_t fm = (1u << W) - 1u;
    constexpr uint32_t ma = ((1u << (4 * W)) - 1u) << (4 * W);
    constexpr uint32_t mb = (((1u << (2 * W)) - 1u) << (2 * W)) * 0x00010001u;
    constexpr uint32_t mc = (fm << W) * 0x01010101u;
    x &= (1u << (8 * W)) - 1u;
    x += (x & ma) * ((1u << (16 - 4 * W)) - 1u);  // codes 4..7 up to bit 16
    x += (x & mb) * ((1u << (8 - 2 * W)) - 1u);   // codes 2,3 / 6,7 up to bit 8 of their half
    x += (x & mc) * ((1u << (4 - W)) - 1u);       // odd codes up to bit 4 of their byte
    return x;
    }
}

// One marker bit inside every nibble that holds the escape code 2^w - 1.
template <int W>
__device__ __forceinline__ uint32_t f1_marks(uint32_t y) {
    if constexpr (W >= 4)
        return nib15_mask(y);
    else
        return (y + 0x11111111u) & (0x11111111u << W);
}

struct F1Lane {
    uint32_t ei;      // next format-1 escape of the group for this tile
    uint32_t rc;      // ranks >= 15 recorded
    bool bad;
};

__device__ __forceinline__ void f1_record(uint16_t *list, F1Lane &L, uint32_t s, uint32_t r) {
    if (L.rc < F1_LIST) list[L.rc] = (uint16_t)((s << 8) | r);
    L.rc++;
}

// Full tile of width W (1..4): nibble words to orow, escapes patched in order.
template <int W>
__device__ __forceinline__ void f1_tile(const uint8_t *tp, uint32_t *orow, const uint8_t *e1, uint32_t ge1,
                                        uint16_t *list, F1Lane &L) {
    uint32_t pw[4 * W];
#pragma unroll
    for (int i = 0; i < W; i++) {
        const uint4 v = ldg_stream16(tp + 16 * i);
        pw[4 * i] = v.x;
        pw[4 * i + 1] = v.y;
        pw[4 * i + 2] = v.z;
        pw[4 * i + 3] = v.w;
    }
    uint32_t clo = 0, chi = 0;  // escape count of word p in nibble p (words 0..7 / 8..15)
#pragma unroll
    for (int p = 0; p < 16; p++) {
        const int b = 8 * W * p, wi = b >> 5, sh = b & 31;
        uint32_t x;
        if (sh + 8 * W <= 32)
            x = pw[wi] >> sh;
        else
            x = __funnelshift_r(pw[wi], pw[wi + 1], sh);
        const uint32_t y = f1_widen<W>(x);
        const uint32_t c = __popc(f1_marks<W>(y));
        if (p < 8)
            clo += c << (4 * p);
        else
            chi += c << (4 * (p - 8));
        orow[p] = y;
    }
    // patch the escaped nibbles: the tile's escapes take the group's bytes in order
#pragma unroll
    for (int h = 0; h < 2; h++) {
        uint32_t m = h ? chi : clo;
        while (m) {
            const uint32_t z = __ffs(m) - 1;
            m &= ~(0xFu << (z & ~3u));
            const uint32_t p = (z >> 2) + 8 * h;
            uint32_t y = orow[p];
            uint32_t t = f1_marks<W>(y);
            while (t) {
                const uint32_t i = (__ffs(t) - 1) >> 2;
                t &= t - 1;
                uint32_t r = 0;
                if (L.ei < ge1) r = e1[L.ei];
                else L.bad = true;
                L.ei++;
                if constexpr (W < 4) y ^= ((min(r, 15u) ^ ((1u << W) - 1u)) << (4 * i));
                if (r >= 15) f1_record(list, L, 8 * p + i, r);
            }
            orow[p] = y;
        }
    }
}

// A group's index entries (and the next group's) and this lane's tile width
// and escape count, loaded one group ahead of use.  next_p16 = ~0 marks the
// last group (the totals stand in for the next entries).
struct F1Meta {
    uint32_t p16, e1, e15;
    uint32_t next_p16, next_e1, next_e15;
    uint32_t wd, te;
};

__device__ __forceinline__ F1Meta f1_meta(const F1Args &a, uint64_t g, uint32_t lane) {
    F1Meta m = {0, 0, 0, 0xFFFFFFFFu, 0, 0, 0, 0};
    if (g < a.ngrp) {
        m.p16 = a.grp1[3 * g];
        m.e1 = a.grp1[3 * g + 1];
        m.e15 = a.grp1[3 * g + 2];
        if (g + 1 < a.ngrp) {
            m.next_p16 = a.grp1[3 * g + 3];
            m.next_e1 = a.grp1[3 * g + 4];
            m.next_e15 = a.grp1[3 * g + 5];
        }
        const uint64_t t = g * DGT_GROUP + lane;
        if (t < a.ntile) {
            m.wd = a.tw[t];
            m.te = a.tesc[t];
        }
    }
    return m;
}

// Any width 0..8 and length: code by code from global memory.
__device__ __noinline__ F1Lane f1_tile_any(const uint8_t *tp, uint32_t wd, uint32_t cnt, uint32_t *orow,
                                           const uint8_t *e1, uint32_t ge1, uint16_t *list, F1Lane L,
                                           uint8_t *direct) {
    const uint32_t top = wd ? (1u << wd) - 1u : 0u;
    const uint32_t tbytes = 16 * wd;
    uint32_t word = 0;
    for (uint32_t s = 0; s < DGT_TILE; s++) {
        uint32_t r = 0;
        if (s < cnt && wd) {
            const uint32_t bit = s * wd, by = bit >> 3;
            const uint32_t v = tp[by] | ((by + 1 < tbytes ? (uint32_t)tp[by + 1] : 0u) << 8);
            const uint32_t c = (v >> (bit & 7)) & top;
            r = c;
            if (c == top) {
                r = 0;
                if (L.ei < ge1) r = e1[L.ei];
                else L.bad = true;
                L.ei++;
            }
        }
        if (r >= 15) {
            if (direct) *direct++ = (uint8_t)r;
            else f1_record(list, L, s, r);
        }
        word |= min(r, 15u) << (4 * (s & 7));
        if ((s & 7) == 7) {
            if (!direct) orow[s >> 3] = word;
            word = 0;
        }
    }
    return L;
}

// Escape bytes of the group: staged copy, or global memory.
struct E1Src {
    const uint8_t *p;
};

__global__ void __launch_bounds__(FW * 32) k_f1_to_r4(F1Args a) {
    extern __shared__ uint4 smem_raw[];
    F1Smem &S = *reinterpret_cast<F1Smem *>(smem_raw);
    pdl_trigger();
    pdl_wait();
    if (blockIdx.x == 0 && threadIdx.x == 0) a.seg[a.seg_last] = (uint32_t)a.n_esc;
    const uint32_t w = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint64_t nbytes = (a.n + 1) / 2;
    uint32_t *orow = &S.out[w][lane * F1_OSTR];
    uint16_t *list = S.list[w][lane];
    const uint64_t g0 = (uint64_t)blockIdx.x * FW + w, G = (uint64_t)gridDim.x * FW;
    const uint64_t GS = (uint64_t)DGT_GROUP * DGT_TILE;
    uint64_t r0 = (g0 * GS) / a.cols, c0 = (g0 * GS) % a.cols;
    const uint64_t step_r = (G * GS) / a.cols, step_c = (G * GS) % a.cols;
    F1Meta mnext = f1_meta(a, g0, lane);
    for (uint64_t g = g0; g < a.ngrp; g += G) {
        // this group's index entries (loaded one group ahead) and the next group's
        const F1Meta m = mnext;
        mnext = f1_meta(a, g + G, lane);
        const uint64_t t = g * DGT_GROUP + lane;
        const uint64_t B0 = t * DGT_TILE;
        const uint32_t cnt = t < a.ntile ? (uint32_t)min((uint64_t)DGT_TILE, a.n - B0) : 0u;
        const uint32_t wd = cnt ? m.wd : 0u;
        const uint32_t te = cnt ? m.te : 0u;
        uint32_t gsum;
        const uint32_t pre = warp_excl_scan((16 * min(wd, 9u)) | (te << 16), &gsum);
        const uint32_t toff = pre & 0xFFFFu, e1off = pre >> 16;
        const uint32_t gpay = gsum & 0xFFFFu, ge1 = gsum >> 16;
        const uint64_t p0 = (uint64_t)m.p16 * 16, e10 = m.e1, gbase = m.e15;
        const uint64_t next_p = m.next_p16 == 0xFFFFFFFFu ? a.payload_bytes : (uint64_t)m.next_p16 * 16;
        const uint64_t next_e1 = m.next_p16 == 0xFFFFFFFFu ? a.n_esc1 : (uint64_t)m.next_e1;
        const uint64_t next_e = m.next_p16 == 0xFFFFFFFFu ? a.n_esc : (uint64_t)m.next_e15;
        uint64_t br = r0, bc = c0 + (uint64_t)DGT_TILE * lane;
        if (bc >= a.cols) {
            if (a.cols >= GS) {
                bc -= a.cols;
                br++;
            } else {
                br += bc / a.cols;
                bc %= a.cols;
            }
        }
        c0 += step_c;
        r0 += step_r;
        if (c0 >= a.cols) {
            c0 -= a.cols;
            r0++;
        }
        const bool gbad = __any_sync(DGT_FULL, wd > 8) || p0 + gpay != next_p || next_p > a.payload_bytes ||
                          e10 + ge1 != next_e1 || next_e1 > a.n_esc1;
        if (gbad) {
            if (lane == 0) set_status(a.status, DGT_ERR_CORRUPT);
            continue;
        }
        const bool e1staged = ge1 <= F1_E1CAP;
        if (e1staged)
            for (uint32_t i = lane; i < ge1; i += 32) S.e1[w][i] = a.esc1[e10 + i];
        __syncwarp();
        const uint8_t *e1 = (e1staged ? S.e1[w] : a.esc1 + e10);
        F1Lane L{e1off, 0u, false};
        const uint8_t *tp = a.payload + p0 + toff;
        if (cnt == DGT_TILE && wd >= 1 && wd <= 4) {
            switch (wd) {
                case 1: f1_tile<1>(tp, orow, e1, ge1, list, L); break;
                case 2: f1_tile<2>(tp, orow, e1, ge1, list, L); break;
                case 3: f1_tile<3>(tp, orow, e1, ge1, list, L); break;
                default: f1_tile<4>(tp, orow, e1, ge1, list, L); break;
            }
        } else if (cnt == DGT_TILE && wd == 0) {
#pragma unroll
            for (int p = 0; p < 16; p++) orow[p] = 0;
        } else if (cnt) {
            L = f1_tile_any(tp, wd, cnt, orow, e1, ge1, list, L, nullptr);
        }
        bool bad = L.bad || (L.ei - e1off != te);
        __syncwarp();
        // the group's nibbles, coalesced
        const uint64_t b0 = g * (DGT_GROUP * DGT_TILE / 2);
        const uint32_t gbytes = (uint32_t)min((uint64_t)(DGT_GROUP * DGT_TILE / 2), nbytes - b0);
        const uint32_t *og = S.out[w];
        if (gbytes == DGT_GROUP * DGT_TILE / 2) {
            uint4 *dst = reinterpret_cast<uint4 *>(a.nib + b0);
#pragma unroll
            for (int m = 0; m < 4; m++) {
                const uint32_t v = lane + 32 * m, row = v >> 2, c = 4 * (v & 3);
                const uint32_t *src = og + row * F1_OSTR + c;
                dst[v] = make_uint4(src[0], src[1], src[2], src[3]);
            }
        } else {
            const uint8_t *ob = reinterpret_cast<const uint8_t *>(og);
            for (uint32_t i = lane; i < gbytes; i += 32) {
                const uint32_t row = i >> 6, o = i & 63;
                a.nib[b0 + i] = ob[row * F1_OSTR * 4 + o];
            }
        }
        // ranks >= 15, placed by a warp prefix sum from the group's escape base
        const uint32_t rc = L.rc;
        uint32_t etot;
        const uint32_t eb = warp_excl_scan(rc, &etot);
        if (gbase + etot != next_e || next_e > a.n_esc) bad = true;
        if (rc && !bad) {
            uint8_t *dst = a.esc + gbase + eb;
            if (rc <= F1_LIST) {
                for (uint32_t i = 0; i < rc; i++) dst[i] = (uint8_t)(list[i] & 0xFF);
            } else {
                f1_tile_any(tp, wd, cnt, orow, e1, ge1, list, F1Lane{e1off, 0u, false}, dst);
            }
        }
        // row-segment escape index for every segment that starts in this tile
        if (cnt && !bad) {
            uint32_t done = 0;
            uint64_t rr = br, cc = bc;
            while (done < cnt) {
                for (uint64_t s = (cc + DGT_SEG - 1) / DGT_SEG * DGT_SEG; s < a.cols && s - cc < cnt - done;
                     s += DGT_SEG) {
                    const uint32_t o = done + (uint32_t)(s - cc);
                    uint32_t before = 0;
                    if (o) {
                        if (rc <= F1_LIST) {
                            for (uint32_t i = 0; i < rc; i++) before += (uint32_t)((list[i] >> 8) < o);
                        } else {
                            // count again from the codes (more than F1_LIST of them)
                            uint32_t ej = e1off;
                            const uint32_t top = (1u << wd) - 1u;
                            for (uint32_t s2 = 0; s2 < o; s2++) {
                                const uint32_t bit = s2 * wd, by = bit >> 3;
                                const uint32_t v = tp[by] | ((by + 1 < 16 * wd ? (uint32_t)tp[by + 1] : 0u) << 8);
                                const uint32_t c = (v >> (bit & 7)) & top;
                                uint32_t r = c;
                                if (c == top) r = ej < ge1 ? e1[ej++] : 0u;
                                before += r >= 15;
                            }
                        }
                    }
                    a.seg[rr * a.nseg + s / DGT_SEG] = (uint32_t)(gbase + eb + before);
                }
                done += (uint32_t)min(a.cols - cc, (uint64_t)(cnt - done));
                rr++;
                cc = 0;
            }
        }
        if (bad) set_status(a.status, DGT_ERR_CORRUPT);
        __syncwarp();
    }
}

// ---------------------------------------------------------------------------
// R4 -> BF16
// ---------------------------------------------------------------------------
// Per-round escape summaries (the second part of the seg array): thread i
// reads the prefix counts of round i and i + 1 and the ranks of the round's
// first three escapes, and writes min(c, 255) | x0 << 8 | x1 << 16 | x2 << 24
// with x = table[rank].  Runs after the transcode that wrote seg and esc.
struct RsumArgs {
    const uint32_t *seg;
    const uint8_t *esc;
    uint64_t n_esc, nrounds;
    uint32_t *rsum;
    uint8_t table[256];
};

__global__ void __launch_bounds__(256) k_r4_rsum(RsumArgs a) {
    __shared__ uint8_t tb[256];
    pdl_trigger();
    tb[threadIdx.x] = a.table[threadIdx.x];
    pdl_wait();
    __syncthreads();
    for (uint64_t i = (uint64_t)blockIdx.x * 256 + threadIdx.x; i < a.nrounds; i += (uint64_t)gridDim.x * 256) {
        const uint32_t b = a.seg[i], c = a.seg[i + 1] - b;
        uint32_t w = c < 255u ? c : 255u;
#pragma unroll
        for (uint32_t q = 0; q < 3; q++)
            if (q < c && (uint64_t)b + q < a.n_esc) w |= (uint32_t)tb[a.esc[b + q]] << (8 + 8 * q);
        a.rsum[i] = w;
    }
}

struct R2BArgs {
    const uint8_t *sm;
    const uint8_t *nib;
    const uint8_t *esc;
    const uint32_t *seg;
    uint64_t rows, cols, nseg, n_esc;
    R4Lut L;
    uint8_t table[256];
    uint16_t *out;
    int32_t *status;
};

// Fast path: cols % 16 == 0, 16-byte aligned arrays.  One warp per
// row-segment of 512 columns; lane u owns columns [512j + 16u, +16).
__global__ void __launch_bounds__(256) k_r4_to_bf16(R2BArgs a) {
    pdl_trigger();
    pdl_wait();
    __shared__ uint8_t table_s[256];
    __shared__ uint8_t escb[8][DGT_SEG];
    table_s[threadIdx.x] = a.table[threadIdx.x];
    __syncthreads();
    const uint32_t w = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint64_t units = a.rows * a.nseg;
    for (uint64_t u = (uint64_t)blockIdx.x * 8 + w; u < units; u += (uint64_t)gridDim.x * 8) {
        const uint64_t row = u / a.nseg, j = u - row * a.nseg;
        const uint64_t k0 = j * DGT_SEG + 16 * lane;
        const bool act = k0 < a.cols;
        const uint64_t flat = row * a.cols + k0;
        uint4 s = make_uint4(0, 0, 0, 0);
        uint2 n = make_uint2(0, 0);
        if (act) {
            s = ldg_stream16(a.sm + flat);
            n = ldg_stream8(a.nib + flat / 2);
        }
        const uint32_t sb = a.seg[u], cnt = a.seg[u + 1] - sb;
        uint32_t p[8];
        r4_dec16(n, s, a.L, p);
        if (cnt) {
            if (cnt > DGT_SEG || (uint64_t)sb + cnt > a.n_esc) {
                if (lane == 0) set_status(a.status, DGT_ERR_CORRUPT);
            } else {
                for (uint32_t i = lane; i < cnt; i += 32) escb[w][i] = a.esc[sb + i];
                __syncwarp();
                const uint32_t m0 = act ? nib15_mask(n.x) : 0u, m1 = act ? nib15_mask(n.y) : 0u;
                if (!patch_escapes(p, m0, m1, cnt, escb[w], table_s) && lane == 0)
                    set_status(a.status, DGT_ERR_CORRUPT);
                __syncwarp();
            }
        }
        if (act) {
            uint4 *dst = reinterpret_cast<uint4 *>(a.out + flat);
            dst[0] = make_uint4(p[0], p[1], p[2], p[3]);
            dst[1] = make_uint4(p[4], p[5], p[6], p[7]);
        }
    }
}

// Any shape and alignment: one warp per row-segment, one element at a time per
// lane chunk, escapes located by a warp prefix sum of 15-nibbles.
__global__ void __launch_bounds__(256) k_r4_to_bf16_any(R2BArgs a) {
    pdl_trigger();
    pdl_wait();
    const uint32_t w = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint64_t units = a.rows * a.nseg;
    for (uint64_t u = (uint64_t)blockIdx.x * 8 + w; u < units; u += (uint64_t)gridDim.x * 8) {
        const uint64_t row = u / a.nseg, j = u - row * a.nseg;
        const uint64_t k0 = j * DGT_SEG + 16 * lane;
        const uint32_t len = k0 < a.cols ? (uint32_t)min((uint64_t)16, a.cols - k0) : 0u;
        const uint64_t flat = row * a.cols + k0;
        uint32_t nv[16], c = 0;
        for (uint32_t i = 0; i < 16; i++) {
            uint32_t v = 0;
            if (i < len) v = (a.nib[(flat + i) >> 1] >> (4 * ((flat + i) & 1))) & 15u;
            nv[i] = v;
            c += (i < len && v == 15);
        }
        uint32_t tot;
        uint32_t idx = a.seg[u] + warp_excl_scan(c, &tot);
        if (tot != a.seg[u + 1] - a.seg[u] && lane == 0) set_status(a.status, DGT_ERR_CORRUPT);
        for (uint32_t i = 0; i < len; i++) {
            uint32_t r = nv[i];
            if (r == 15) {
                r = idx < a.n_esc ? a.esc[idx] : 0u;
                idx++;
            }
            uint8_t sm = a.sm[flat + i];
            uint32_t e = a.table[r];
            a.out[flat + i] = (uint16_t)(((uint32_t)(sm & 0x80) << 8) | (e << 7) | (sm & 0x7F));
        }
    }
}

}  // namespace dgt

using namespace dgt;

extern "C" int dgt_load_r4(const dgt_packed_view *dev, dgt_r4 *r4, int32_t *d_status, void *stream) {
    if (!dev || !r4) return DGT_ERR_ARG;
    if (dev->format != 1 && dev->format != 2) return DGT_ERR_ARG;
    if (r4->rows != dev->rows || r4->cols != dev->cols) return DGT_ERR_SHAPE;
    const uint64_t n = dev->rows * dev->cols;
    if ((dev->rows && n / dev->rows != dev->cols) || n >= (1ull << 40)) return DGT_ERR_SHAPE;
    cudaStream_t st = (cudaStream_t)stream;
    if (!r4->seg) return DGT_ERR_ARG;
    if (d_status && cudaMemsetAsync(d_status, 0, 4, st) != cudaSuccess) return DGT_ERR_CUDA;
    const uint64_t nseg = dgt_r4_nseg(dev->cols);
    const uint64_t seg_last = dev->rows * nseg;
    if (n == 0) {
        return cudaMemsetAsync(r4->seg, 0, 4, st) == cudaSuccess ? DGT_OK : DGT_ERR_CUDA;
    }
    if (!r4->nib || !aligned16(r4->nib) || (dev->n_esc15 && !r4->esc)) return DGT_ERR_ARG;
    if (r4->n_esc != dev->n_esc15) return DGT_ERR_ARG;
    DeviceInfo di;
    if (device_info(&di) != DGT_OK) return DGT_ERR_CUDA;
    if (dev->format == 2) {
        if (!dev->words || !dev->blkq || !dev->grp || dev->rice_k < 0 || dev->rice_k > 7)
            return DGT_ERR_ARG;
        F2Args a;
        a.words = dev->words;
        a.n_words = dev->n_words;
        a.blkq = dev->blkq;
        a.grp = dev->grp;
        a.n = n;
        a.cols = dev->cols;
        a.nseg = nseg;
        a.nblk = (n + DGT_BLOCK - 1) / DGT_BLOCK;
        a.ngrp = (a.nblk + DGT_GROUP - 1) / DGT_GROUP;
        if (dev->n_blocks != a.nblk || dev->n_groups != a.ngrp) return DGT_ERR_CORRUPT;
        a.k = dev->rice_k;
        a.nib = r4->nib;
        a.esc = r4->esc;
        a.seg = r4->seg;
        a.n_esc = dev->n_esc15;
        a.seg_last = seg_last;
        a.status = d_status;
        const size_t smem = sizeof(RiceSmem);
        const bool fast = n < (1ull << 31) && dev->cols % 64 == 0 && dev->cols >= 2048 &&
                          dev->rows * nseg < (1ull << 32) && aligned16(dev->words) && dev->n_words < (1ull << 32);
        void (*fn)(F2Args) = nullptr;
        switch ((fast ? 4 : 0) + (a.k < 3 ? a.k : 3)) {
            case 0: fn = k_rice_to_r4<false, 0>; break;
            case 1: fn = k_rice_to_r4<false, 1>; break;
            case 2: fn = k_rice_to_r4<false, 2>; break;
            case 3: fn = k_rice_to_r4<false, 3>; break;
            case 4: fn = k_rice_to_r4<true, 0>; break;
            case 5: fn = k_rice_to_r4<true, 1>; break;
            case 6: fn = k_rice_to_r4<true, 2>; break;
            default: fn = k_rice_to_r4<true, 3>; break;
        }
        int bps = 0;
        if (prepare_kernel((const void *)fn, smem, RW * 32, &bps) != DGT_OK) return DGT_ERR_CUDA;
        uint64_t grid = min((uint64_t)di.sms * bps, (a.ngrp + RW - 1) / RW);
        if (launch_pdl(fn, dim3((unsigned)grid), dim3(RW * 32), smem, st, a) != cudaSuccess) return DGT_ERR_CUDA;
    } else {
        if (!dev->tw || !dev->tesc || !dev->grp1 || (dev->payload_bytes && !dev->payload) ||
            (dev->n_esc1 && !dev->esc1) || (dev->payload && !aligned16(dev->payload)))
            return DGT_ERR_ARG;
        F1Args a;
        a.payload = dev->payload;
        a.payload_bytes = dev->payload_bytes;
        a.tw = dev->tw;
        a.tesc = dev->tesc;
        a.esc1 = dev->esc1;
        a.n_esc1 = dev->n_esc1;
        a.grp1 = dev->grp1;
        a.n = n;
        a.cols = dev->cols;
        a.nseg = nseg;
        a.ntile = (n + DGT_TILE - 1) / DGT_TILE;
        a.ngrp = (a.ntile + DGT_GROUP - 1) / DGT_GROUP;
        if (dev->n_tiles != a.ntile || dev->n_groups1 != a.ngrp) return DGT_ERR_CORRUPT;
        a.nib = r4->nib;
        a.esc = r4->esc;
        a.seg = r4->seg;
        a.n_esc = dev->n_esc15;
        a.seg_last = seg_last;
        a.status = d_status;
        const size_t smem = sizeof(F1Smem);
        int bps = 0;
        if (prepare_kernel((const void *)k_f1_to_r4, smem, FW * 32, &bps) != DGT_OK) return DGT_ERR_CUDA;
        uint64_t grid = min((uint64_t)di.sms * bps, (a.ngrp + FW - 1) / FW);
        if (launch_pdl(k_f1_to_r4, dim3((unsigned)grid), dim3(FW * 32), smem, st, a) != cudaSuccess)
            return DGT_ERR_CUDA;
    }
    RsumArgs ra;
    ra.seg = r4->seg;
    ra.esc = r4->esc;
    ra.n_esc = dev->n_esc15;
    ra.nrounds = seg_last;
    ra.rsum = r4->seg + dgt_rsum_offset(dev->rows, nseg);
    for (int i = 0; i < 256; i++) ra.table[i] = r4->table[i];
    const uint64_t rgrid = min((uint64_t)di.sms * 8, (seg_last + 255) / 256);
    if (launch_pdl(k_r4_rsum, dim3((unsigned)rgrid), dim3(256), 0, st, ra) != cudaSuccess) return DGT_ERR_CUDA;
    return cudaPeekAtLastError() == cudaSuccess ? DGT_OK : DGT_ERR_CUDA;
}

extern "C" int dgt_r4_to_bf16(const dgt_r4 *r4, uint16_t *d_out, int32_t *d_status, void *stream) {
    if (!r4) return DGT_ERR_ARG;
    const uint64_t n = r4->rows * r4->cols;
    if ((r4->rows && n / r4->rows != r4->cols) || n >= (1ull << 40)) return DGT_ERR_SHAPE;
    cudaStream_t st = (cudaStream_t)stream;
    if (d_status && cudaMemsetAsync(d_status, 0, 4, st) != cudaSuccess) return DGT_ERR_CUDA;
    if (n == 0) return DGT_OK;
    if (!d_out || !r4->sm || !r4->nib || !r4->seg || (r4->n_esc && !r4->esc)) return DGT_ERR_ARG;
    DeviceInfo di;
    if (device_info(&di) != DGT_OK) return DGT_ERR_CUDA;
    R2BArgs a;
    a.sm = r4->sm;
    a.nib = r4->nib;
    a.esc = r4->esc;
    a.seg = r4->seg;
    a.rows = r4->rows;
    a.cols = r4->cols;
    a.nseg = dgt_r4_nseg(r4->cols);
    a.n_esc = r4->n_esc;
    a.L = make_r4lut(r4->table, r4->n_table);
    for (int i = 0; i < 256; i++) a.table[i] = r4->table[i];
    a.out = d_out;
    a.status = d_status;
    const uint64_t units = a.rows * a.nseg;
    const bool fast = r4->cols % 16 == 0 && aligned16(r4->sm) && aligned16(r4->nib) && aligned16(d_out);
    int bps = 0;
    const void *fn = fast ? (const void *)k_r4_to_bf16 : (const void *)k_r4_to_bf16_any;
    if (prepare_kernel(fn, 0, 256, &bps) != DGT_OK) return DGT_ERR_CUDA;
    uint64_t grid = min((uint64_t)di.sms * bps, (units + 7) / 8);
    if (launch_pdl(fast ? k_r4_to_bf16 : k_r4_to_bf16_any, dim3((unsigned)grid), dim3(256), 0, st, a) !=
        cudaSuccess)
        return DGT_ERR_CUDA;
    return cudaPeekAtLastError() == cudaSuccess ? DGT_OK : DGT_ERR_CUDA;
}

extern "C" int dgt_read_status(const int32_t *d_status, void *stream, int32_t *status) {
    if (!d_status || !status) return DGT_ERR_ARG;
    cudaStream_t st = (cudaStream_t)stream;
    if (cudaMemcpyAsync(status, d_status, 4, cudaMemcpyDeviceToHost, st) != cudaSuccess) return DGT_ERR_CUDA;
    if (cudaStreamSynchronize(st) != cudaSuccess) return DGT_ERR_CUDA;
    return DGT_OK;
}
