// dgt_host.cpp -- host side of libdgt: the packer (formats 1 and 2), host
// unpack, the safetensors container, status strings and the GEMV plan.
//
// Method: Binade project README -- title paragraphs (sign+mantissa byte,
// exponent frequency rank, Rice codes), "How it works" (one table per tensor,
// the two file formats, R4 at load) and "Use" (pack / unpack).  The per-block
// 8-bit index follows the "Best measured configuration" section of the
// "Lossless BF16 weight compression" README (BLOCK=64, 8-bit lengths).
//
// Everything here is multithreaded over independent groups / tiles with
// std::thread; results do not depend on the thread count.
#include <algorithm>
#include <atomic>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <new>
#include <string>
#include <thread>
#include <vector>

#include "../../include/dgt.h"
#include "dgt_internal.h"
#include "dgt_packed.h"

namespace {

int resolve_threads(int nthreads) {
    if (nthreads > 0) return nthreads;
    unsigned h = std::thread::hardware_concurrency();
    return h ? (int)h : 1;
}

// Run fn(begin, end) over [0, count) split into contiguous pieces.
template <class F>
void parallel_for(int nthreads, uint64_t count, F fn) {
    if (count == 0) return;
    uint64_t nt = std::min<uint64_t>((uint64_t)nthreads, count);
    if (nt <= 1 || count < 4) {
        fn((uint64_t)0, count);
        return;
    }
    std::vector<std::thread> th;
    th.reserve(nt);
    for (uint64_t t = 0; t < nt; t++) {
        uint64_t b = count * t / nt, e = count * (t + 1) / nt;
        th.emplace_back([=] { fn(b, e); });
    }
    for (auto &x : th) x.join();
}

// LSB-first bit writer into a word range that starts zeroed.
struct BitWriter {
    uint32_t *w;
    uint64_t acc = 0;
    int fill = 0;
    explicit BitWriter(uint32_t *dst) : w(dst) {}
    void put(uint64_t bits, int len) {  // len <= 32
        acc |= bits << fill;
        fill += len;
        if (fill >= 32) {
            *w++ = (uint32_t)acc;
            acc >>= 32;
            fill -= 32;
        }
    }
    void zeros(int len) {
        while (len > 32) { put(0, 32); len -= 32; }
        put(0, len);
    }
    void flush() {
        if (fill > 0) { *w++ = (uint32_t)acc; acc = 0; fill = 0; }
    }
};

// One Rice code at bit pos of an LSB-first word stream of limit bits, read
// through a 64-bit window (words past the end read as zero).  Returns the
// rank; a unary run that reaches the end of the stream, or runs past 255
// zeros, or a code that ends past the end, sets bad.
struct RiceReader {
    const uint32_t *w;
    uint64_t nw, pos, limit;
    bool bad = false;
    uint64_t word(uint64_t i) const { return i < nw ? w[i] : 0u; }
    uint64_t window() const {
        const uint64_t i = pos >> 5;
        const unsigned sh = (unsigned)(pos & 31);
        const uint64_t v = (word(i) | (word(i + 1) << 32)) >> sh;
        return sh ? v | (word(i + 2) << (64 - sh)) : v;
    }
    uint32_t code(int k, uint32_t *quo) {
        const uint64_t v = window();
        uint32_t q, r;
        if (v != 0 && (unsigned)__builtin_ctzll(v) + 1 + k <= 64) {
            q = (uint32_t)__builtin_ctzll(v);
            r = (q << k) | (uint32_t)((v >> (q + 1)) & ((1u << k) - 1u));
            pos += q + 1 + k;
        } else {
            // a unary run of 64 or more zeros: only valid data up to 255
            q = 0;
            while (pos < limit && !((word(pos >> 5) >> (pos & 31)) & 1u) && q <= 255) {
                q++;
                pos++;
            }
            pos++;
            const uint64_t rem = window() & ((1u << k) - 1u);
            r = (q << k) | (uint32_t)rem;
            pos += k;
        }
        if (pos > limit || q > 255) bad = true;
        *quo = q;
        return r;
    }
    uint32_t raw8() {
        const uint32_t r = (uint32_t)(window() & 0xFFu);
        pos += 8;
        if (pos > limit) bad = true;
        return r;
    }
};

// Format 2 block layout: a Rice block stores its remainder field (the k low
// bits of every rank) and then the unary parts.  Bit position, inside the
// remainder field, of the remainder of rank i of a block of cnt ranks: in a
// full block with k = 1 or 2 the field is in nibble-slot order (one 32-bit
// field word shifted right by k * (m mod 4/k) lines the remainders of ranks
// 8m..8m+7 up with their 4-bit R4 slots); otherwise k bits per rank in order.
inline uint32_t rem_field_pos(int k, uint64_t cnt, uint32_t i) {
    if (cnt == DGT_BLOCK && (k == 1 || k == 2)) {
        const uint32_t m = i >> 3, j = i & 7, per = 4u / (uint32_t)k;
        return 32u * (m / per) + 4u * j + (uint32_t)k * (m % per);
    }
    return (uint32_t)k * i;
}

inline uint8_t sm_of(uint16_t b) { return (uint8_t)(((b >> 8) & 0x80) | (b & 0x7F)); }
inline uint8_t exp_of(uint16_t b) { return (uint8_t)((b >> 7) & 0xFF); }
// The ranks of a tensor, read from its bf16 bits through the rank table
// (not stored as an array of their own).
struct Ranks {
    const uint16_t *b;
    uint8_t rank_of[256];
    uint8_t operator[](uint64_t i) const { return rank_of[exp_of(b[i])]; }
};

inline uint16_t bf16_of(uint8_t sm, uint8_t e) {
    return (uint16_t)(((uint16_t)(sm & 0x80) << 8) | ((uint16_t)e << 7) | (sm & 0x7F));
}

int pack_format2(dgt_packed *p, const Ranks &rk, int nt) {
    const uint64_t n = p->v.rows * p->v.cols;
    const uint64_t nblk = (n + DGT_BLOCK - 1) / DGT_BLOCK;
    const uint64_t ngrp = (nblk + DGT_GROUP - 1) / DGT_GROUP;
    // per group: bits for each k, and the number of ranks >= 15
    std::vector<uint64_t> gbits(ngrp * 8);
    std::vector<uint32_t> gesc(ngrp);
    parallel_for(nt, ngrp, [&](uint64_t g0, uint64_t g1) {
        for (uint64_t g = g0; g < g1; g++) {
            uint64_t bits[8] = {0, 0, 0, 0, 0, 0, 0, 0};
            uint32_t e15 = 0;
            uint64_t b_end = std::min(nblk, (g + 1) * DGT_GROUP);
            for (uint64_t b = g * DGT_GROUP; b < b_end; b++) {
                uint64_t i0 = b * DGT_BLOCK, cnt = std::min<uint64_t>(DGT_BLOCK, n - i0);
                uint32_t q[8] = {0, 0, 0, 0, 0, 0, 0, 0};
                for (uint64_t i = 0; i < cnt; i++) {
                    uint32_t r = rk[i0 + i];
                    e15 += r >= 15;
                    for (int k = 0; k < 8; k++) q[k] += r >> k;
                }
                for (int k = 0; k < 8; k++)
                    bits[k] += q[k] <= 254 ? cnt * (uint64_t)(k + 1) + q[k] : 8 * cnt;
            }
            for (int k = 0; k < 8; k++) gbits[g * 8 + k] = bits[k];
            gesc[g] = e15;
        }
    });
    int best_k = 0;
    uint64_t best_words = UINT64_MAX;
    for (int k = 0; k < 8; k++) {
        uint64_t words = 0;
        for (uint64_t g = 0; g < ngrp; g++) words += (gbits[g * 8 + k] + 31) / 32;
        if (words < best_words) { best_words = words; best_k = k; }
    }
    if (ngrp == 0) best_words = 0;
    if (best_words >= (1ull << 32)) return DGT_ERR_SHAPE;
    const int k = best_k;
    p->v.rice_k = k;
    p->words.assign(best_words, 0u);
    p->blkq.assign(nblk, 0);
    p->grp.assign(ngrp * 2, 0u);
    uint64_t off = 0, esc = 0;
    for (uint64_t g = 0; g < ngrp; g++) {
        p->grp[2 * g] = (uint32_t)off;
        p->grp[2 * g + 1] = (uint32_t)esc;
        off += (gbits[g * 8 + k] + 31) / 32;
        esc += gesc[g];
    }
    parallel_for(nt, ngrp, [&](uint64_t g0, uint64_t g1) {
        for (uint64_t g = g0; g < g1; g++) {
            BitWriter bw(p->words.data() + p->grp[2 * g]);
            uint64_t b_end = std::min(nblk, (g + 1) * DGT_GROUP);
            for (uint64_t b = g * DGT_GROUP; b < b_end; b++) {
                uint64_t i0 = b * DGT_BLOCK, cnt = std::min<uint64_t>(DGT_BLOCK, n - i0);
                uint32_t q = 0;
                for (uint64_t i = 0; i < cnt; i++) q += (uint32_t)rk[i0 + i] >> k;
                if (q <= 254) {
                    p->blkq[b] = (uint8_t)q;
                    // remainder field (at most 64 * 7 bits), then the unary parts
                    uint32_t fld[DGT_BLOCK * 7 / 32] = {0};
                    if (k) {
                        for (uint32_t i = 0; i < (uint32_t)cnt; i++) {
                            const uint32_t rem = (uint32_t)rk[i0 + i] & ((1u << k) - 1u);
                            const uint32_t at = rem_field_pos(k, cnt, i);
                            for (int t = 0; t < k; t++)
                                fld[(at + t) >> 5] |= ((rem >> t) & 1u) << ((at + t) & 31);
                        }
                        const uint32_t fbits = (uint32_t)cnt * (uint32_t)k;
                        for (uint32_t o = 0; o < fbits; o += 32) bw.put(fld[o >> 5], (int)std::min(32u, fbits - o));
                    }
                    for (uint64_t i = 0; i < cnt; i++) {
                        bw.zeros((int)((uint32_t)rk[i0 + i] >> k));
                        bw.put(1u, 1);
                    }
                } else {
                    p->blkq[b] = 255;
                    for (uint64_t i = 0; i < cnt; i++) bw.put(rk[i0 + i], 8);
                }
            }
            bw.flush();
        }
    });
    return DGT_OK;
}

inline int tile_width(const Ranks &rk, uint64_t i0, uint64_t cnt) {
    uint32_t hist[256];
    std::memset(hist, 0, sizeof(hist));
    bool nz = false;
    for (uint64_t i = 0; i < cnt; i++) {
        const uint8_t r = rk[i0 + i];
        hist[r]++;
        nz |= r != 0;
    }
    if (!nz) return 0;
    // ranks >= t for every threshold t, from the histogram
    uint32_t ge[257];
    ge[256] = 0;
    for (int t = 255; t >= 0; t--) ge[t] = ge[t + 1] + hist[t];
    int best = 1;
    uint64_t best_cost = UINT64_MAX;
    for (int w = 1; w <= 8; w++) {
        uint64_t cost = (uint64_t)DGT_TILE * w + 8ull * ge[(1 << w) - 1];
        if (cost < best_cost) { best_cost = cost; best = w; }
    }
    return best;
}

int pack_format1(dgt_packed *p, const Ranks &rk, int nt) {
    const uint64_t n = p->v.rows * p->v.cols;
    const uint64_t ntile = (n + DGT_TILE - 1) / DGT_TILE;
    const uint64_t ngrp = (ntile + DGT_GROUP - 1) / DGT_GROUP;
    p->tw.assign(ntile, 0);
    p->tesc.assign(ntile, 0);
    std::vector<uint8_t> te15(ntile);
    parallel_for(nt, ntile, [&](uint64_t t0, uint64_t t1) {
        for (uint64_t t = t0; t < t1; t++) {
            uint64_t i0 = t * DGT_TILE, cnt = std::min<uint64_t>(DGT_TILE, n - i0);
            int w = tile_width(rk, i0, cnt);
            uint32_t top = w ? (1u << w) - 1u : 0u;
            uint32_t e = 0, e15 = 0;
            for (uint64_t i = 0; i < cnt; i++) {
                e += w && rk[i0 + i] >= top;
                e15 += rk[i0 + i] >= 15;
            }
            p->tw[t] = (uint8_t)w;
            p->tesc[t] = (uint8_t)e;
            te15[t] = (uint8_t)e15;
        }
    });
    std::vector<uint64_t> poff(ntile + 1), eoff(ntile + 1);
    uint64_t e15 = 0;
    p->grp1.assign(ngrp * 3, 0u);
    poff[0] = eoff[0] = 0;
    for (uint64_t t = 0; t < ntile; t++) {
        if (t % DGT_GROUP == 0) {
            uint64_t g = t / DGT_GROUP;
            if (poff[t] / 16 >= (1ull << 32) || eoff[t] >= (1ull << 32)) return DGT_ERR_SHAPE;
            p->grp1[3 * g] = (uint32_t)(poff[t] / 16);
            p->grp1[3 * g + 1] = (uint32_t)eoff[t];
            p->grp1[3 * g + 2] = (uint32_t)e15;
        }
        poff[t + 1] = poff[t] + 16ull * p->tw[t];
        eoff[t + 1] = eoff[t] + p->tesc[t];
        e15 += te15[t];
    }
    p->payload.assign(poff[ntile], 0);
    p->esc1.assign(eoff[ntile], 0);
    parallel_for(nt, ntile, [&](uint64_t t0, uint64_t t1) {
        for (uint64_t t = t0; t < t1; t++) {
            int w = p->tw[t];
            if (!w) continue;
            uint64_t i0 = t * DGT_TILE, cnt = std::min<uint64_t>(DGT_TILE, n - i0);
            uint32_t top = (1u << w) - 1u;
            uint8_t *dst = p->payload.data() + poff[t];
            uint8_t *ed = p->esc1.data() + eoff[t];
            uint64_t acc = 0;
            int fill = 0;
            for (uint64_t i = 0; i < DGT_TILE; i++) {
                uint32_t r = i < cnt ? rk[i0 + i] : 0u;
                uint32_t c = r < top ? r : top;
                if (i < cnt && c == top) *ed++ = (uint8_t)r;
                acc |= (uint64_t)c << fill;
                fill += w;
                while (fill >= 8) { *dst++ = (uint8_t)acc; acc >>= 8; fill -= 8; }
            }
        }
    });
    return DGT_OK;
}

}  // namespace

extern "C" {

const char *dgt_status_string(int status) {
    switch (status) {
        case DGT_OK: return "ok";
        case DGT_ERR_ARG: return "invalid argument";
        case DGT_ERR_SHAPE: return "unsupported shape";
        case DGT_ERR_CORRUPT: return "corrupt packed data";
        case DGT_ERR_CUDA: return "CUDA error";
        case DGT_ERR_TIMEOUT: return "device wait timed out";
        case DGT_ERR_OOM: return "out of host memory";
        case DGT_ERR_IO: return "I/O error";
        case DGT_ERR_UNSUPPORTED: return "unsupported device or configuration";
        default: return "unknown status";
    }
}

int dgt_version(void) { return 100; }

int dgt_pack(const uint16_t *bf16, uint64_t rows, uint64_t cols, int format, int nthreads,
             dgt_packed **out) {
    if (!out || (format != 1 && format != 2)) return DGT_ERR_ARG;
    *out = nullptr;
    const uint64_t n = rows * cols;
    if ((rows && n / rows != cols) || n >= (1ull << 40)) return DGT_ERR_SHAPE;
    if (n && !bf16) return DGT_ERR_ARG;
    const int nt = resolve_threads(nthreads);
    dgt_packed *p = new (std::nothrow) dgt_packed();
    if (!p) return DGT_ERR_OOM;
    try {
        std::memset(&p->v, 0, sizeof(p->v));
        p->v.rows = rows;
        p->v.cols = cols;
        p->v.format = format;
        // exponent histogram and the sign/mantissa bytes, in one pass (sm is
        // first touched here, by the threads that fill it)
        p->sm.resize(n);
        const uint64_t chunks = std::min<uint64_t>((uint64_t)nt * 4, std::max<uint64_t>(1, n / 65536));
        std::vector<uint64_t> part(chunks * 256, 0);
        parallel_for(nt, chunks, [&](uint64_t c0, uint64_t c1) {
            // four sub-histograms, so that equal exponents in a row do not
            // wait on one another's counter
            std::vector<uint64_t> h4(4 * 256);
            for (uint64_t c = c0; c < c1; c++) {
                std::fill(h4.begin(), h4.end(), 0);
                const uint64_t lo = n * c / chunks, hi = n * (c + 1) / chunks;
                uint64_t i = lo;
                for (; i + 4 <= hi; i += 4) {
                    const uint16_t b0 = bf16[i], b1 = bf16[i + 1], b2 = bf16[i + 2], b3 = bf16[i + 3];
                    h4[exp_of(b0)]++;
                    h4[256 + exp_of(b1)]++;
                    h4[512 + exp_of(b2)]++;
                    h4[768 + exp_of(b3)]++;
                    p->sm[i] = sm_of(b0);
                    p->sm[i + 1] = sm_of(b1);
                    p->sm[i + 2] = sm_of(b2);
                    p->sm[i + 3] = sm_of(b3);
                }
                for (; i < hi; i++) {
                    h4[exp_of(bf16[i])]++;
                    p->sm[i] = sm_of(bf16[i]);
                }
                uint64_t *h = &part[c * 256];
                for (int e = 0; e < 256; e++) h[e] = h4[e] + h4[256 + e] + h4[512 + e] + h4[768 + e];
            }
        });
        uint64_t counts[256] = {0};
        for (uint64_t c = 0; c < chunks; c++)
            for (int e = 0; e < 256; e++) counts[e] += part[c * 256 + e];
        // rank table: count descending, exponent ascending
        int order[256], T = 0;
        for (int e = 0; e < 256; e++)
            if (counts[e]) order[T++] = e;
        std::stable_sort(order, order + T, [&](int a, int b) { return counts[a] > counts[b]; });
        Ranks rk;
        rk.b = bf16;
        std::memset(rk.rank_of, 0, sizeof(rk.rank_of));
        for (int r = 0; r < T; r++) {
            p->v.table[r] = (uint8_t)order[r];
            rk.rank_of[order[r]] = (uint8_t)r;
        }
        p->v.n_table = T;
        uint64_t e15 = 0;
        for (int r = 15; r < T; r++) e15 += counts[order[r]];
        p->v.n_esc15 = e15;
        int rc = format == 2 ? pack_format2(p, rk, nt) : pack_format1(p, rk, nt);
        if (rc != DGT_OK) {
            delete p;
            return rc;
        }
        p->refresh();
    } catch (const std::bad_alloc &) {
        delete p;
        return DGT_ERR_OOM;
    }
    *out = p;
    return DGT_OK;
}

void dgt_packed_free(dgt_packed *p) { delete p; }

int dgt_packed_get_view(const dgt_packed *p, dgt_packed_view *view) {
    if (!p || !view) return DGT_ERR_ARG;
    *view = p->v;
    return DGT_OK;
}

double dgt_packed_bits_per_weight(const dgt_packed *p) {
    if (!p) return 0.0;
    const uint64_t n = p->v.rows * p->v.cols;
    if (!n) return 0.0;
    uint64_t b = p->sm.size() + (uint64_t)p->v.n_table;
    if (p->v.format == 2)
        b += p->words.size() * 4 + p->blkq.size() + p->grp.size() * 4;
    else
        b += p->payload.size() + p->tw.size() + p->tesc.size() + p->esc1.size() + p->grp1.size() * 4;
    return (double)b * 8.0 / (double)n;
}

int dgt_unpack(const dgt_packed_view *v, uint16_t *out, int nthreads) {
    if (!v || (v->format != 1 && v->format != 2)) return DGT_ERR_ARG;
    const uint64_t n = v->rows * v->cols;
    if (n && (!out || !v->sm)) return DGT_ERR_ARG;
    const int nt = resolve_threads(nthreads);
    std::atomic<int> bad(0);
    if (v->format == 2) {
        const uint64_t nblk = (n + DGT_BLOCK - 1) / DGT_BLOCK;
        const uint64_t ngrp = (nblk + DGT_GROUP - 1) / DGT_GROUP;
        if (v->n_blocks != nblk || v->n_groups != ngrp || v->rice_k < 0 || v->rice_k > 7)
            return DGT_ERR_CORRUPT;
        const int k = v->rice_k;
        parallel_for(nt, ngrp, [&](uint64_t g0, uint64_t g1) {
            for (uint64_t g = g0; g < g1 && !bad.load(std::memory_order_relaxed); g++) {
                RiceReader br{v->words, v->n_words, (uint64_t)v->grp[2 * g] * 32, v->n_words * 32};
                uint64_t b_end = std::min(nblk, (g + 1) * DGT_GROUP);
                for (uint64_t b = g * DGT_GROUP; b < b_end; b++) {
                    uint64_t i0 = b * DGT_BLOCK, cnt = std::min<uint64_t>(DGT_BLOCK, n - i0);
                    uint8_t q = v->blkq[b];
                    if (q != 255) {
                        const uint64_t start = br.pos;
                        // the remainder field, read whole (at most 64 * 7 bits)
                        uint32_t fld[DGT_BLOCK * 7 / 32 + 1] = {0};
                        const uint32_t fbits = (uint32_t)cnt * (uint32_t)k;
                        for (uint32_t o = 0; o < fbits; o += 32) {
                            fld[o >> 5] = (uint32_t)br.window();
                            br.pos += std::min(32u, fbits - o);
                        }
                        if (fbits & 31) fld[fbits >> 5] &= (1u << (fbits & 31)) - 1u;
                        uint32_t qs = 0;
                        for (uint64_t i = 0; i < cnt; i++) {
                            uint32_t quo = 0;
                            br.code(0, &quo);
                            const uint32_t at = rem_field_pos(k, cnt, (uint32_t)i);
                            const uint64_t two = fld[at >> 5] | ((uint64_t)fld[(at >> 5) + 1] << 32);
                            const uint32_t rem = k ? (uint32_t)(two >> (at & 31)) & ((1u << k) - 1u) : 0u;
                            const uint32_t r = (quo << k) | rem;
                            if (r > 255) br.bad = true;
                            qs += quo;
                            out[i0 + i] = bf16_of(v->sm[i0 + i], v->table[r & 255]);
                        }
                        if (qs != q || br.pos - start != cnt * (uint64_t)(k + 1) + q || br.pos > br.limit)
                            br.bad = true;
                    } else {
                        for (uint64_t i = 0; i < cnt; i++)
                            out[i0 + i] = bf16_of(v->sm[i0 + i], v->table[br.raw8()]);
                    }
                    if (br.bad) { bad.store(1); break; }
                }
            }
        });
    } else {
        const uint64_t ntile = (n + DGT_TILE - 1) / DGT_TILE;
        const uint64_t ngrp = (ntile + DGT_GROUP - 1) / DGT_GROUP;
        if (v->n_tiles != ntile || v->n_groups1 != ngrp) return DGT_ERR_CORRUPT;
        parallel_for(nt, ngrp, [&](uint64_t g0, uint64_t g1) {
            for (uint64_t g = g0; g < g1 && !bad.load(std::memory_order_relaxed); g++) {
                uint64_t off = (uint64_t)v->grp1[3 * g] * 16, e = v->grp1[3 * g + 1];
                uint64_t t_end = std::min(ntile, (g + 1) * DGT_GROUP);
                for (uint64_t t = g * DGT_GROUP; t < t_end; t++) {
                    int w = v->tw[t];
                    uint64_t i0 = t * DGT_TILE, cnt = std::min<uint64_t>(DGT_TILE, n - i0);
                    if (w > 8 || off + 16ull * w > v->payload_bytes) { bad.store(1); break; }
                    uint32_t top = w ? (1u << w) - 1u : 0u, seen = 0;
                    for (uint64_t i = 0; i < cnt; i++) {
                        // w <= 8 bits from bit position off*8 + i*w: two bytes
                        // at most, the second only inside the payload
                        uint32_t c = 0;
                        if (w) {
                            const uint64_t bit = off * 8 + i * (uint64_t)w, by = bit >> 3;
                            uint32_t two = v->payload[by];
                            if (by + 1 < v->payload_bytes) two |= (uint32_t)v->payload[by + 1] << 8;
                            c = (two >> (bit & 7)) & top;
                        }
                        uint32_t r = c;
                        if (w && c == top) {
                            if (e >= v->n_esc1) { bad.store(1); break; }
                            r = v->esc1[e++];
                            seen++;
                        }
                        out[i0 + i] = bf16_of(v->sm[i0 + i], v->table[r]);
                    }
                    if (seen != v->tesc[t]) { bad.store(1); break; }
                    off += 16ull * w;
                }
            }
        });
    }
    return bad.load() ? DGT_ERR_CORRUPT : DGT_OK;
}

uint64_t dgt_r4_nseg(uint64_t cols) { return (cols + DGT_SEG - 1) / DGT_SEG; }

int dgt_r4_sizes(uint64_t rows, uint64_t cols, uint64_t n_esc, uint64_t *nib_bytes,
                 uint64_t *esc_bytes, uint64_t *seg_bytes) {
    uint64_t n = rows * cols;
    if (rows && n / rows != cols) return DGT_ERR_SHAPE;
    if (nib_bytes) *nib_bytes = (n + 1) / 2;
    if (esc_bytes) *esc_bytes = n_esc;
    if (seg_bytes) *seg_bytes = dgt_seg_words(rows, dgt_r4_nseg(cols)) * 4;
    return DGT_OK;
}

uint64_t dgt_r4_rsum_offset(uint64_t rows, uint64_t cols) { return dgt_rsum_offset(rows, dgt_r4_nseg(cols)); }

int dgt_r4_init_from_view(const dgt_packed_view *v, uint8_t *d_nib, uint8_t *d_esc,
                          uint32_t *d_seg, dgt_r4 *r4) {
    if (!v || !r4) return DGT_ERR_ARG;
    std::memset(r4, 0, sizeof(*r4));
    r4->rows = v->rows;
    r4->cols = v->cols;
    r4->n_table = v->n_table;
    std::memcpy(r4->table, v->table, 256);
    r4->n_esc = v->n_esc15;
    r4->sm = v->sm;
    r4->nib = d_nib;
    r4->esc = d_esc;
    r4->seg = d_seg;
    return DGT_OK;
}

int dgt_gemv_slices(uint64_t rows, uint64_t cols) { return dgt_plan_slices(rows, cols); }

}  // extern "C"
