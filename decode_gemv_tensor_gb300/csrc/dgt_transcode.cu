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
//    lane per block/tile; a persistent grid of 256-thread CTAs;
//  - format 2: each lane decodes its Rice block with a 4096-entry shared
//    table indexed by the next 12 stream bits, which yields up to six ranks,
//    their bit count and their nibbles in one lookup; long codes and ranks
//    >= 15 take a short window decode;
//  - escapes (ranks >= 15) are collected per lane, placed by a warp prefix sum
//    from the group's escape base, and the row-segment escape index (seg) is
//    written for every segment that starts inside the group;
//  - every group checks its index against its neighbours and its decoded
//    length against its index bytes; a mismatch sets the status word.
#include <cuda_runtime.h>

#include "../../include/dgt.h"
#include "dgt_device.cuh"
#include "dgt_launch.h"

namespace dgt {

constexpr int TW = 8;           // warps per CTA
constexpr int K1_CAP = 384;     // staged stream words per group (else read from global)
constexpr int K2_E1CAP = 256;   // staged format-1 escapes per group
constexpr int LIST = 4;         // per-lane escape list (format 1), overflow re-walks

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

struct K1Smem {
    uint32_t lut[4096];
    uint32_t buf[TW][K1_CAP + 2];
    uint32_t outw[TW][256];
    uint8_t escr[TW][2048];
};

// Table entry for a 12-bit window v (bit 0 = next stream bit): the complete
// codes at its start, up to six, each of rank < 15.
// bits 0..2: count, 3..6: bits used, 7..30: ranks as nibbles.
__device__ __forceinline__ uint32_t rice_lut_entry(uint32_t v, int k) {
    uint32_t pos = 0, ns = 0, ranks = 0;
    while (ns < 6) {
        uint32_t q = 0;
        while (pos + q < 12 && !((v >> (pos + q)) & 1u)) q++;
        if (pos + q >= 12 || pos + q + 1 + (uint32_t)k > 12) break;
        uint32_t rem = (v >> (pos + q + 1)) & ((1u << k) - 1u);
        uint32_t r = (q << k) | rem;
        if (r >= 15) break;
        ranks |= r << (4 * ns);
        ns++;
        pos += q + 1 + k;
    }
    return ns | (pos << 3) | (ranks << 7);
}

template <class Src>
struct WordReader {
    Src src;
    uint32_t nw;
    __device__ __forceinline__ uint32_t operator()(uint32_t i) const { return i < nw ? src[i] : 0u; }
};

// Decode one block of cnt ranks starting at bit pos.  Nibble words go to
// out[0..], escape ranks to escr[position]; returns the escape count and the
// escape position mask; *end gets the bit position after the block.
template <class Rd>
__device__ __forceinline__ uint32_t rice_block(const Rd &rd, uint32_t pos, uint32_t cnt, uint32_t q,
                                               int k, const uint32_t *lut, uint32_t *out,
                                               uint8_t *escr, uint64_t &emask, uint32_t *end,
                                               bool &bad) {
    uint32_t wi = pos >> 5;
    uint32_t lo = rd(wi), hi = rd(wi + 1);
    uint64_t acc = 0;
    uint32_t fill = 0, wo = 0, sym = 0, ec = 0;
    const uint32_t kmask = (1u << k) - 1u;
    emask = 0;
    while (sym < cnt) {
        uint32_t win = __funnelshift_r(lo, hi, pos & 31);
        uint32_t add, nbits, nsym;
        if (q != 255) {
            uint32_t e = lut[win & 0xFFFu];
            nsym = e & 7u;
            if (nsym) {
                add = e >> 7;
                nbits = (e >> 3) & 15u;
                if (sym + nsym > cnt) {
                    // last lookup of the block: take only the codes that belong to it
                    uint32_t m = cnt - sym, t = win;
                    nbits = 0;
                    for (uint32_t i = 0; i < m; i++) {
                        uint32_t z = __ffs(t) - 1;
                        nbits += z + 1 + k;
                        t >>= z + 1 + k;
                    }
                    add &= (1u << (4 * m)) - 1u;
                    nsym = m;
                }
            } else {
                // one code that the table does not finish: a long code or rank >= 15
                uint32_t z;
                uint32_t r;
                if (win != 0 && (z = __ffs(win) - 1) + 1 + k <= 32) {
                    r = (z << k) | ((win >> (z + 1)) & kmask);
                    nbits = z + 1 + k;
                } else {
                    // more than 32 bits: walk word by word (bounded by 255 zeros)
                    uint32_t p = pos, zz = 0;
                    for (;;) {
                        uint32_t wv = rd(p >> 5) >> (p & 31);
                        uint32_t avail = 32 - (p & 31);
                        if (wv) {
                            uint32_t f = __ffs(wv) - 1;
                            zz += f;
                            p += f;
                            break;
                        }
                        zz += avail;
                        p += avail;
                        if (zz > 255) break;
                    }
                    p += 1;
                    uint32_t rem = __funnelshift_r(rd(p >> 5), rd((p >> 5) + 1), p & 31) & kmask;
                    r = (zz << k) | rem;
                    nbits = p + k - pos;
                    if (zz > 255) bad = true;
                }
                if (r > 255) { bad = true; r = 255; }
                if (r >= 15) {
                    escr[sym] = (uint8_t)r;
                    emask |= 1ull << sym;
                    ec++;
                    r = 15;
                }
                add = r;
                nsym = 1;
            }
        } else {
            uint32_t r = win & 0xFFu;
            if (r >= 15) {
                escr[sym] = (uint8_t)r;
                emask |= 1ull << sym;
                ec++;
                r = 15;
            }
            add = r;
            nbits = 8;
            nsym = 1;
        }
        acc |= (uint64_t)add << fill;
        fill += 4 * nsym;
        sym += nsym;
        pos += nbits;
        if (fill >= 32) {
            out[wo++] = (uint32_t)acc;
            acc >>= 32;
            fill -= 32;
        }
        uint32_t nwi = pos >> 5;
        if (nwi != wi) {
            if (nwi == wi + 1) {
                lo = hi;
                hi = rd(nwi + 1);
            } else {
                lo = rd(nwi);
                hi = rd(nwi + 1);
            }
            wi = nwi;
        }
    }
    if (fill) out[wo] = (uint32_t)acc;
    *end = pos;
    return ec;
}

__global__ void __launch_bounds__(TW * 32) k_rice_to_r4(F2Args a) {
    extern __shared__ uint4 smem_raw[];
    K1Smem &S = *reinterpret_cast<K1Smem *>(smem_raw);
    for (uint32_t v = threadIdx.x; v < 4096; v += blockDim.x) S.lut[v] = rice_lut_entry(v, a.k);
    if (blockIdx.x == 0 && threadIdx.x == 0) a.seg[a.seg_last] = (uint32_t)a.n_esc;
    __syncthreads();
    const uint32_t w = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint64_t nbytes = (a.n + 1) / 2;
    for (uint64_t g = (uint64_t)blockIdx.x * TW + w; g < a.ngrp; g += (uint64_t)gridDim.x * TW) {
        const uint64_t blk = g * DGT_GROUP + lane;
        const uint64_t B0 = blk * DGT_BLOCK;
        const uint32_t cnt = blk < a.nblk ? (uint32_t)min((uint64_t)DGT_BLOCK, a.n - B0) : 0u;
        const uint32_t q = cnt ? a.blkq[blk] : 0u;
        const uint32_t len = cnt == 0 ? 0u : (q != 255 ? cnt * (uint32_t)(a.k + 1) + q : 8u * cnt);
        uint32_t gbits;
        const uint32_t off = warp_excl_scan(len, &gbits);
        const uint32_t nw = (gbits + 31) / 32;
        const uint64_t gw0 = a.grp[2 * g], gbase = a.grp[2 * g + 1];
        const uint64_t next_w = g + 1 < a.ngrp ? (uint64_t)a.grp[2 * g + 2] : a.n_words;
        const uint64_t next_e = g + 1 < a.ngrp ? (uint64_t)a.grp[2 * g + 3] : a.n_esc;
        if (gw0 + nw != next_w || next_w > a.n_words) {
            if (lane == 0) set_status(a.status, DGT_ERR_CORRUPT);
            continue;
        }
        const bool staged = nw <= K1_CAP;
        if (staged) {
            for (uint32_t i = lane; i < nw + 2; i += 32) S.buf[w][i] = i < nw ? a.words[gw0 + i] : 0u;
            __syncwarp();
        }
        uint64_t emask = 0;
        uint32_t ec = 0, end = off;
        bool bad = false;
        if (cnt) {
            if (staged) {
                WordReader<const uint32_t *> rd{S.buf[w], nw + 2};
                ec = rice_block(rd, off, cnt, q, a.k, S.lut, &S.outw[w][8 * lane], &S.escr[w][64 * lane],
                                emask, &end, bad);
            } else {
                WordReader<const uint32_t *> rd{a.words + gw0, nw};
                ec = rice_block(rd, off, cnt, q, a.k, S.lut, &S.outw[w][8 * lane], &S.escr[w][64 * lane],
                                emask, &end, bad);
            }
            if (end != off + len) bad = true;
        }
        __syncwarp();
        // nibbles of the group, coalesced
        const uint64_t b0 = g * 1024;
        const uint32_t gbytes = (uint32_t)min((uint64_t)1024, nbytes - b0);
        const uint8_t *ob = reinterpret_cast<const uint8_t *>(S.outw[w]);
        if (gbytes == 1024) {
            uint4 *dst = reinterpret_cast<uint4 *>(a.nib + b0);
            const uint4 *src = reinterpret_cast<const uint4 *>(S.outw[w]);
            dst[lane] = src[lane];
            dst[lane + 32] = src[lane + 32];
        } else {
            for (uint32_t i = lane; i < gbytes; i += 32) a.nib[b0 + i] = ob[i];
        }
        // escapes and segment index
        uint32_t etot;
        const uint32_t eb = warp_excl_scan(ec, &etot);
        if (gbase + etot != next_e || next_e > a.n_esc) bad = true;
        if (ec && !bad) {
            uint64_t m = emask;
            uint64_t dst = gbase + eb;
            while (m) {
                uint32_t i = __ffsll((long long)m) - 1;
                m &= m - 1;
                a.esc[dst++] = S.escr[w][64 * lane + i];
            }
        }
        const uint64_t r0 = __shfl_sync(DGT_FULL, lane == 0 ? (g * 2048) / a.cols : 0ull, 0);
        if (cnt && !bad) {
            SegWalk s = first_seg_start(B0, r0, a.cols);
            for (uint64_t f = s.r * a.cols + s.c; f < B0 + cnt; f = s.r * a.cols + s.c) {
                uint32_t o = (uint32_t)(f - B0);
                uint64_t before = o ? (emask & ((~0ull) >> (64 - o))) : 0ull;
                a.seg[s.r * a.nseg + s.c / DGT_SEG] = (uint32_t)(gbase + eb + __popcll(before));
                next_seg_start(s, a.cols);
            }
        }
        if (bad) set_status(a.status, DGT_ERR_CORRUPT);
        __syncwarp();
    }
}

// ---------------------------------------------------------------------------
// format 1 -> R4
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

struct K2Smem {
    uint32_t pay[TW][1024 + 4];   // 32 tiles x up to 128 bytes, + guard
    uint32_t outw[TW][512];       // 4096 nibbles
    uint8_t e1[TW][K2_E1CAP];
    uint16_t list[TW][32][LIST];
};

__device__ __forceinline__ uint64_t load_bits64(const uint32_t *sw, uint32_t byteoff) {
    uint32_t wi = byteoff >> 2, sh = (byteoff & 3) * 8;
    uint32_t w0 = sw[wi], w1 = sw[wi + 1], w2 = sw[wi + 2];
    uint32_t lo = __funnelshift_r(w0, w1, sh), hi = __funnelshift_r(w1, w2, sh);
    return (uint64_t)lo | ((uint64_t)hi << 32);
}

__global__ void __launch_bounds__(TW * 32) k_f1_to_r4(F1Args a) {
    extern __shared__ uint4 smem_raw[];
    K2Smem &S = *reinterpret_cast<K2Smem *>(smem_raw);
    if (blockIdx.x == 0 && threadIdx.x == 0) a.seg[a.seg_last] = (uint32_t)a.n_esc;
    const uint32_t w = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint64_t nbytes = (a.n + 1) / 2;
    for (uint64_t g = (uint64_t)blockIdx.x * TW + w; g < a.ngrp; g += (uint64_t)gridDim.x * TW) {
        const uint64_t t = g * DGT_GROUP + lane;
        const uint64_t B0 = t * DGT_TILE;
        const uint32_t cnt = t < a.ntile ? (uint32_t)min((uint64_t)DGT_TILE, a.n - B0) : 0u;
        const uint32_t wd = cnt ? a.tw[t] : 0u;
        const uint32_t te = cnt ? a.tesc[t] : 0u;
        uint32_t gpay, ge1;
        const uint32_t toff = warp_excl_scan(16 * wd, &gpay);
        const uint32_t e1off = warp_excl_scan(te, &ge1);
        const uint64_t p0 = (uint64_t)a.grp1[3 * g] * 16, e10 = a.grp1[3 * g + 1], gbase = a.grp1[3 * g + 2];
        const uint64_t next_p = g + 1 < a.ngrp ? (uint64_t)a.grp1[3 * g + 3] * 16 : a.payload_bytes;
        const uint64_t next_e1 = g + 1 < a.ngrp ? (uint64_t)a.grp1[3 * g + 4] : a.n_esc1;
        const uint64_t next_e = g + 1 < a.ngrp ? (uint64_t)a.grp1[3 * g + 5] : a.n_esc;
        bool gbad = __any_sync(DGT_FULL, wd > 8) || p0 + gpay != next_p || next_p > a.payload_bytes ||
                    e10 + ge1 != next_e1 || next_e1 > a.n_esc1;
        if (gbad) {
            if (lane == 0) set_status(a.status, DGT_ERR_CORRUPT);
            continue;
        }
        // stage the group's payload (16-byte units) and its format-1 escapes
        {
            const uint4 *src = reinterpret_cast<const uint4 *>(a.payload + p0);
            uint4 *dst = reinterpret_cast<uint4 *>(S.pay[w]);
            for (uint32_t i = lane; i < gpay / 16; i += 32) dst[i] = src[i];
            if (lane < 4) S.pay[w][gpay / 4 + lane] = 0u;
            if (ge1 <= K2_E1CAP)
                for (uint32_t i = lane; i < ge1; i += 32) S.e1[w][i] = a.esc1[e10 + i];
        }
        __syncwarp();
        const bool e1staged = ge1 <= K2_E1CAP;
        const uint32_t top = wd ? (1u << wd) - 1u : 0u;
        uint32_t ei = e1off, ec = 0;
        uint64_t em0 = 0, em1 = 0;
        bool bad = false;
        if (cnt) {
            for (uint32_t p = 0; p < 16; p++) {
                uint64_t v = wd ? load_bits64(S.pay[w], toff + p * wd) : 0ull;
                uint32_t word = 0;
#pragma unroll
                for (uint32_t i = 0; i < 8; i++) {
                    uint32_t c = (uint32_t)(v >> (i * wd)) & top;
                    uint32_t r = c;
                    uint32_t s = p * 8 + i;
                    if (wd && c == top && s < cnt) {
                        if (ei < ge1) {
                            r = e1staged ? S.e1[w][ei] : a.esc1[e10 + ei];
                        } else {
                            r = 0;
                            bad = true;
                        }
                        ei++;
                    }
                    if (r >= 15 && s < cnt) {
                        if (ec < LIST) S.list[w][lane][ec] = (uint16_t)((s << 8) | r);
                        ec++;
                        if (s < 64) em0 |= 1ull << s; else em1 |= 1ull << (s - 64);
                    }
                    if (s >= cnt) r = 0;
                    word |= (r < 15 ? r : 15u) << (4 * i);
                }
                S.outw[w][16 * lane + p] = word;
            }
            if (ei - e1off != te) bad = true;
        }
        __syncwarp();
        const uint64_t b0 = g * 2048;
        const uint32_t gbytes = (uint32_t)min((uint64_t)2048, nbytes - b0);
        if (gbytes == 2048) {
            uint4 *dst = reinterpret_cast<uint4 *>(a.nib + b0);
            const uint4 *src = reinterpret_cast<const uint4 *>(S.outw[w]);
#pragma unroll
            for (int i = 0; i < 4; i++) dst[lane + 32 * i] = src[lane + 32 * i];
        } else {
            const uint8_t *ob = reinterpret_cast<const uint8_t *>(S.outw[w]);
            for (uint32_t i = lane; i < gbytes; i += 32) a.nib[b0 + i] = ob[i];
        }
        uint32_t etot;
        const uint32_t eb = warp_excl_scan(ec, &etot);
        if (gbase + etot != next_e || next_e > a.n_esc) bad = true;
        if (ec && !bad) {
            uint64_t dst = gbase + eb;
            if (ec <= LIST) {
                for (uint32_t i = 0; i < ec; i++) a.esc[dst + i] = (uint8_t)(S.list[w][lane][i] & 0xFF);
            } else {
                // more escapes than the list holds: walk the tile's codes again
                uint32_t ej = e1off;
                for (uint32_t s = 0; s < cnt; s++) {
                    uint64_t v = load_bits64(S.pay[w], toff + (s / 8) * wd);
                    uint32_t c = (uint32_t)(v >> ((s % 8) * wd)) & top;
                    uint32_t r = c;
                    if (c == top) {
                        r = 0;
                        if (ej < ge1) r = e1staged ? S.e1[w][ej] : a.esc1[e10 + ej];
                        ej++;
                    }
                    if (r >= 15) a.esc[dst++] = (uint8_t)r;
                }
            }
        }
        const uint64_t r0 = __shfl_sync(DGT_FULL, lane == 0 ? (g * 4096) / a.cols : 0ull, 0);
        if (cnt && !bad) {
            SegWalk s = first_seg_start(B0, r0, a.cols);
            for (uint64_t f = s.r * a.cols + s.c; f < B0 + cnt; f = s.r * a.cols + s.c) {
                uint32_t o = (uint32_t)(f - B0);
                uint32_t before;
                if (o <= 64) before = o ? __popcll(em0 & ((~0ull) >> (64 - o))) : 0u;
                else before = __popcll(em0) + __popcll(em1 & ((~0ull) >> (128 - o)));
                a.seg[s.r * a.nseg + s.c / DGT_SEG] = (uint32_t)(gbase + eb + before);
                next_seg_start(s, a.cols);
            }
        }
        if (bad) set_status(a.status, DGT_ERR_CORRUPT);
        __syncwarp();
    }
}

// ---------------------------------------------------------------------------
// R4 -> BF16
// ---------------------------------------------------------------------------
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
        const size_t smem = sizeof(K1Smem);
        int bps = 0;
        if (prepare_kernel((const void *)k_rice_to_r4, smem, TW * 32, &bps) != DGT_OK) return DGT_ERR_CUDA;
        uint64_t grid = min((uint64_t)di.sms * bps, (a.ngrp + TW - 1) / TW);
        k_rice_to_r4<<<(unsigned)grid, TW * 32, smem, st>>>(a);
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
        const size_t smem = sizeof(K2Smem);
        int bps = 0;
        if (prepare_kernel((const void *)k_f1_to_r4, smem, TW * 32, &bps) != DGT_OK) return DGT_ERR_CUDA;
        uint64_t grid = min((uint64_t)di.sms * bps, (a.ngrp + TW - 1) / TW);
        k_f1_to_r4<<<(unsigned)grid, TW * 32, smem, st>>>(a);
    }
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
    if (fast)
        k_r4_to_bf16<<<(unsigned)grid, 256, 0, st>>>(a);
    else
        k_r4_to_bf16_any<<<(unsigned)grid, 256, 0, st>>>(a);
    return cudaPeekAtLastError() == cudaSuccess ? DGT_OK : DGT_ERR_CUDA;
}

extern "C" int dgt_read_status(const int32_t *d_status, void *stream, int32_t *status) {
    if (!d_status || !status) return DGT_ERR_ARG;
    cudaStream_t st = (cudaStream_t)stream;
    if (cudaMemcpyAsync(status, d_status, 4, cudaMemcpyDeviceToHost, st) != cudaSuccess) return DGT_ERR_CUDA;
    if (cudaStreamSynchronize(st) != cudaSuccess) return DGT_ERR_CUDA;
    return DGT_OK;
}
