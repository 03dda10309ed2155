/*
 * oracle.c -- plain, slow, obviously-correct CPU reference for the exponent-rank
 * BF16 weight codec and its fixed-order matrix products.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the library's product path may call,
 * link or load this file.  Only the tests, the smoke check and the bench's CPU
 * baseline use it.  It shares no code, header, table or constant generator with
 * the CUDA library.
 *
 * Sources (web pages; section names as printed there):
 *   [B]  "Binade" project README (pypi.org/project/binade), paragraphs under the
 *        title, "How it works" (No exponent locality, Two file formats, Runtime
 *        layout, Exactness) and "Limitations".
 *   [W]  "Lossless BF16 weight compression" README, "Best measured
 *        configuration" (BLOCK=64 blocks, 8-bit per-block index + warp prefix sum).
 *
 * Where the pages leave a byte layout or a rule open, the reading taken here is
 * stated beside the code.  Everything is sequential; no blocking, fusion or
 * reordering beyond the definitions.
 *
 * Floating point: compiled without fast-math and with -ffp-contract=off, so each
 * fmaf() below is one correctly rounded fused multiply-add and each '+' one
 * correctly rounded float addition; no flush-to-zero.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define OR_BLOCK 64      /* Rice block, after [W] BLOCK=64                 */
#define OR_GROUP 32      /* blocks (or tiles) per index group              */
#define OR_TILE 128      /* format-1 tile, [B] "per 128-weight tile"       */
#define OR_SEG 512       /* R4 escape-index segment (row-relative)         */
#define OR_CHUNK 16      /* GEMV: consecutive k per lane chunk             */
#define OR_LANES 32      /* GEMV: lanes per reduction                      */
#define OR_ROUND (OR_CHUNK * OR_LANES) /* k covered by one round = 512     */

/* ------------------------------------------------------------------------ */
/* bf16 <-> float                                                           */
/* ------------------------------------------------------------------------ */
static float or_bf16_to_f32(uint16_t b) {
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, 4);
    return f;
}

/* Round a float to bf16, nearest with ties to even; NaN -> 0x7FC0. */
uint16_t or_f32_to_bf16(float f) {
    uint32_t u;
    memcpy(&u, &f, 4);
    if ((u & 0x7F800000u) == 0x7F800000u && (u & 0x007FFFFFu) != 0) return 0x7FC0;
    uint32_t lsb = (u >> 16) & 1u;
    return (uint16_t)((u + 0x7FFFu + lsb) >> 16);
}

/* ------------------------------------------------------------------------ */
/* [B] title paragraph: sign and mantissa kept as one raw byte; the 8-bit     */
/* exponent replaced by a rank.  Reading: sign -> bit 7, mantissa -> 6..0.   */
/* ------------------------------------------------------------------------ */
void or_split(const uint16_t *b, uint64_t n, uint8_t *sm, uint8_t *e) {
    for (uint64_t i = 0; i < n; i++) {
        uint16_t v = b[i];
        uint8_t sign = (uint8_t)(v >> 15);
        uint8_t mant = (uint8_t)(v & 0x7F);
        uint8_t expo = (uint8_t)((v >> 7) & 0xFF);
        sm[i] = (uint8_t)((sign << 7) | mant);
        e[i] = expo;
    }
}

uint16_t or_join(uint8_t sm, uint8_t e) {
    uint16_t sign = (uint16_t)(sm >> 7);
    uint16_t mant = (uint16_t)(sm & 0x7F);
    return (uint16_t)((sign << 15) | ((uint16_t)e << 7) | mant);
}

/* ------------------------------------------------------------------------ */
/* [B] "No exponent locality": one frequency-rank table per tensor.          */
/* Reading: table holds only exponents that occur, sorted by count           */
/* descending, ties by exponent ascending; rank = position in the table.     */
/* Returns T (0 for an empty tensor).                                        */
/* ------------------------------------------------------------------------ */
int or_rank_table(const uint16_t *b, uint64_t n, uint64_t *counts,
                  uint8_t *table, uint8_t *rank_of) {
    for (int i = 0; i < 256; i++) counts[i] = 0;
    for (uint64_t i = 0; i < n; i++) counts[(b[i] >> 7) & 0xFF]++;
    int used[256];
    for (int i = 0; i < 256; i++) used[i] = 0;
    int T = 0;
    for (;;) {
        /* pick the unused present exponent with the largest count, smallest exponent on ties */
        int best = -1;
        for (int ex = 0; ex < 256; ex++) {
            if (used[ex] || counts[ex] == 0) continue;
            if (best < 0 || counts[ex] > counts[best]) best = ex;
        }
        if (best < 0) break;
        used[best] = 1;
        table[T] = (uint8_t)best;
        rank_of[best] = (uint8_t)T;
        T++;
    }
    for (int i = T; i < 256; i++) table[i] = 0;
    for (int ex = 0; ex < 256; ex++)
        if (counts[ex] == 0) rank_of[ex] = 0xFF;
    return T;
}

void or_ranks(const uint16_t *b, uint64_t n, const uint8_t *rank_of, uint8_t *ranks) {
    for (uint64_t i = 0; i < n; i++) ranks[i] = rank_of[(b[i] >> 7) & 0xFF];
}

/* Exponent entropy in bits per weight (the quantity [W] quotes as 2.65 of 8). */
double or_entropy(const uint64_t *counts) {
    uint64_t n = 0;
    for (int i = 0; i < 256; i++) n += counts[i];
    if (n == 0) return 0.0;
    double h = 0.0;
    for (int i = 0; i < 256; i++) {
        if (counts[i] == 0) continue;
        double p = (double)counts[i] / (double)n;
        h -= p * log2(p);
    }
    return h;
}

/* Rebuild bf16 from sign/mantissa bytes, ranks and the table. */
void or_rebuild(const uint8_t *sm, const uint8_t *ranks, const uint8_t *table,
                uint64_t n, uint16_t *out) {
    for (uint64_t i = 0; i < n; i++) out[i] = or_join(sm[i], table[ranks[i]]);
}

/* ------------------------------------------------------------------------ */
/* Bit stream: bit j lives in bit (j & 31) of little-endian 32-bit word j>>5.  */
/* ------------------------------------------------------------------------ */
static void put_bit(uint32_t *w, uint64_t pos, int bit) {
    if (bit) w[pos >> 5] |= (uint32_t)1u << (pos & 31);
}
static int get_bit(const uint32_t *w, uint64_t pos) {
    return (int)((w[pos >> 5] >> (pos & 31)) & 1u);
}

/* ------------------------------------------------------------------------ */
/* Format 2, [B] "Two file formats": Rice codes of the ranks.                 */
/* Block = 64 ranks ([W] BLOCK=64), group = 32 blocks.                       */
/* A block with Q = sum(r >> k) <= 254 is Rice coded; its index byte is Q,   */
/* so its length is count*(k+1) + Q bits.  Reading (the pages fix no bit     */
/* layout): the block first holds every rank's k low bits (the remainder     */
/* field, count*k bits), then every rank's unary part, q = r >> k zero bits  */
/* and one 1 bit, in rank order.  Remainders are stored least significant   */
/* bit first, in rank order, except in a full block with k = 1 or 2: there   */
/* bit i of the remainder of rank 8m + j sits at field bit                   */
/* 32*floor(m*k/4) + 4j + k*(m mod 4/k) + i ("nibble-slot order": one       */
/* 32-bit field word, shifted right by k*(m mod 4/k), puts the remainders   */
/* of ranks 8m..8m+7 under their 4-bit output slots).                        */
/* A block with Q >= 255 stores 8-bit raw ranks and index byte 255.          */
/* Every group starts on a 32-bit word boundary.                              */
/* ------------------------------------------------------------------------ */
/* Position, inside a block's remainder field, of bit t of the remainder of
   the block's rank i (cnt ranks in the block). */
static uint64_t rem_bit_pos(int k, uint64_t cnt, uint64_t i, int t) {
    if (cnt == OR_BLOCK && (k == 1 || k == 2)) {
        uint64_t m = i / 8, j = i % 8, per = (uint64_t)(4 / k);   /* output words per field word */
        return 32 * (m / per) + 4 * j + (uint64_t)k * (m % per) + (uint64_t)t;
    }
    return (uint64_t)k * i + (uint64_t)t;
}

static uint64_t rice_block_q(const uint8_t *r, uint64_t cnt, int k) {
    uint64_t q = 0;
    for (uint64_t i = 0; i < cnt; i++) q += (uint64_t)(r[i] >> k);
    return q;
}

static uint64_t rice_block_bits(const uint8_t *r, uint64_t cnt, int k) {
    uint64_t q = rice_block_q(r, cnt, k);
    if (q <= 254) return cnt * (uint64_t)(k + 1) + q;
    return 8 * cnt;
}

/* Total stream bits (whole 32-bit words) for parameter k. */
uint64_t or_f2_stream_bits(const uint8_t *ranks, uint64_t n, int k) {
    uint64_t total = 0;
    uint64_t per_group = (uint64_t)OR_BLOCK * OR_GROUP;
    for (uint64_t g0 = 0; g0 < n; g0 += per_group) {
        uint64_t gbits = 0;
        for (uint64_t b0 = g0; b0 < n && b0 < g0 + per_group; b0 += OR_BLOCK) {
            uint64_t cnt = (n - b0 < OR_BLOCK) ? n - b0 : OR_BLOCK;
            gbits += rice_block_bits(ranks + b0, cnt, k);
        }
        total += (gbits + 31) / 32 * 32;
    }
    return total;
}

/* Reading: one k per tensor, 0..7, the one with the fewest stream bits;
   ties go to the smaller k. */
int or_f2_choose_k(const uint8_t *ranks, uint64_t n) {
    int best = 0;
    uint64_t best_bits = or_f2_stream_bits(ranks, n, 0);
    for (int k = 1; k <= 7; k++) {
        uint64_t b = or_f2_stream_bits(ranks, n, k);
        if (b < best_bits) { best_bits = b; best = k; }
    }
    return best;
}

/* Encode.  words must hold or_f2_stream_bits()/32 words (zeroed here).
   blkq: ceil(n/64) bytes.  grp: 2 words per group {first word, ranks >= 15
   before the group}.  Returns the number of words written. */
uint64_t or_f2_encode(const uint8_t *ranks, uint64_t n, int k, uint32_t *words,
                      uint64_t cap_words, uint8_t *blkq, uint32_t *grp) {
    memset(words, 0, cap_words * 4);
    uint64_t pos = 0;
    uint64_t esc15 = 0;
    uint64_t per_group = (uint64_t)OR_BLOCK * OR_GROUP;
    for (uint64_t g0 = 0; g0 < n; g0 += per_group) {
        uint64_t g = g0 / per_group;
        grp[2 * g] = (uint32_t)(pos / 32);
        grp[2 * g + 1] = (uint32_t)esc15;
        for (uint64_t b0 = g0; b0 < n && b0 < g0 + per_group; b0 += OR_BLOCK) {
            uint64_t cnt = (n - b0 < OR_BLOCK) ? n - b0 : OR_BLOCK;
            uint64_t q = rice_block_q(ranks + b0, cnt, k);
            uint64_t b = b0 / OR_BLOCK;
            if (q <= 254) {
                blkq[b] = (uint8_t)q;
                /* remainder field, then the unary parts */
                for (uint64_t i = 0; i < cnt; i++) {
                    uint32_t r = ranks[b0 + i];
                    for (int t = 0; t < k; t++)
                        put_bit(words, pos + rem_bit_pos(k, cnt, i, t), (int)((r >> t) & 1u));
                }
                pos += cnt * (uint64_t)k;
                for (uint64_t i = 0; i < cnt; i++) {
                    uint32_t quo = (uint32_t)ranks[b0 + i] >> k;
                    for (uint32_t z = 0; z < quo; z++) put_bit(words, pos++, 0);
                    put_bit(words, pos++, 1);
                }
            } else {
                blkq[b] = 255;
                for (uint64_t i = 0; i < cnt; i++) {
                    uint32_t r = ranks[b0 + i];
                    for (int t = 0; t < 8; t++) put_bit(words, pos++, (int)((r >> t) & 1u));
                }
            }
            for (uint64_t i = 0; i < cnt; i++) esc15 += (ranks[b0 + i] >= 15);
        }
        pos = (pos + 31) / 32 * 32;
    }
    return pos / 32;
}

/* Decode every group from its index entry.  Returns 0, or -1 when a block's
   decoded length disagrees with its index byte or runs past the stream. */
int or_f2_decode(const uint32_t *words, uint64_t n_words, const uint8_t *blkq,
                 const uint32_t *grp, uint64_t n, int k, uint8_t *ranks) {
    uint64_t per_group = (uint64_t)OR_BLOCK * OR_GROUP;
    uint64_t limit = n_words * 32;
    for (uint64_t g0 = 0; g0 < n; g0 += per_group) {
        uint64_t g = g0 / per_group;
        uint64_t pos = (uint64_t)grp[2 * g] * 32;
        for (uint64_t b0 = g0; b0 < n && b0 < g0 + per_group; b0 += OR_BLOCK) {
            uint64_t cnt = (n - b0 < OR_BLOCK) ? n - b0 : OR_BLOCK;
            uint8_t q = blkq[b0 / OR_BLOCK];
            uint64_t start = pos;
            if (q != 255) {
                uint64_t qsum = 0;
                uint64_t rem0 = pos;            /* remainder field */
                pos += cnt * (uint64_t)k;       /* unary parts */
                for (uint64_t i = 0; i < cnt; i++) {
                    uint32_t quo = 0;
                    for (;;) {
                        if (pos >= limit) return -1;
                        if (get_bit(words, pos++)) break;
                        quo++;
                        if (quo > 255) return -1;
                    }
                    uint32_t rem = 0;
                    for (int t = 0; t < k; t++) {
                        uint64_t bp = rem0 + rem_bit_pos(k, cnt, i, t);
                        if (bp >= limit) return -1;
                        rem |= (uint32_t)get_bit(words, bp) << t;
                    }
                    uint32_t r = (quo << k) | rem;
                    if (r > 255) return -1;
                    ranks[b0 + i] = (uint8_t)r;
                    qsum += quo;
                }
                if (qsum != q || pos - start != cnt * (uint64_t)(k + 1) + q) return -1;
            } else {
                for (uint64_t i = 0; i < cnt; i++) {
                    uint32_t r = 0;
                    for (int t = 0; t < 8; t++) {
                        if (pos >= limit) return -1;
                        r |= (uint32_t)get_bit(words, pos++) << t;
                    }
                    ranks[b0 + i] = (uint8_t)r;
                }
            }
        }
    }
    return 0;
}

/* ------------------------------------------------------------------------ */
/* Format 1, [B] "Two file formats": fixed width per 128-weight tile with     */
/* escapes.  Reading: width w in 1..8 minimising 128*w + 8*#{r >= 2^w - 1},   */
/* ties to the smaller w; w = 0 iff every rank of the tile is 0.  Codes       */
/* c = min(r, 2^w - 1), w bits each, least significant first, 16*w payload   */
/* bytes per tile (a partial last tile is padded with zero codes).  A code    */
/* equal to 2^w - 1 is an escape: the raw rank follows in the escape list.    */
/* ------------------------------------------------------------------------ */
int or_f1_tile_width(const uint8_t *r, uint64_t cnt) {
    int all_zero = 1;
    for (uint64_t i = 0; i < cnt; i++)
        if (r[i]) all_zero = 0;
    if (all_zero) return 0;
    int best = -1;
    uint64_t best_cost = 0;
    for (int w = 1; w <= 8; w++) {
        uint32_t top = (1u << w) - 1u;
        uint64_t esc = 0;
        for (uint64_t i = 0; i < cnt; i++) esc += (r[i] >= top);
        uint64_t cost = (uint64_t)OR_TILE * w + 8 * esc;
        if (best < 0 || cost < best_cost) { best = w; best_cost = cost; }
    }
    return best;
}

/* Payload bytes needed for format 1. */
uint64_t or_f1_payload_bytes(const uint8_t *ranks, uint64_t n) {
    uint64_t total = 0;
    for (uint64_t t0 = 0; t0 < n; t0 += OR_TILE) {
        uint64_t cnt = (n - t0 < OR_TILE) ? n - t0 : OR_TILE;
        total += 16 * (uint64_t)or_f1_tile_width(ranks + t0, cnt);
    }
    return total;
}

/* Encode.  tw, tesc: one byte per tile; grp1: 3 words per 32 tiles
   {payload offset in 16-byte units, escapes before the group, ranks >= 15
   before the group}.  Returns the number of escapes written to esc1. */
uint64_t or_f1_encode(const uint8_t *ranks, uint64_t n, uint8_t *payload,
                      uint64_t cap_bytes, uint8_t *tw, uint8_t *tesc, uint8_t *esc1,
                      uint32_t *grp1) {
    memset(payload, 0, cap_bytes);
    uint64_t off = 0, nesc = 0, esc15 = 0;
    for (uint64_t t0 = 0; t0 < n; t0 += OR_TILE) {
        uint64_t t = t0 / OR_TILE;
        uint64_t cnt = (n - t0 < OR_TILE) ? n - t0 : OR_TILE;
        if (t % OR_GROUP == 0) {
            uint64_t g = t / OR_GROUP;
            grp1[3 * g] = (uint32_t)(off / 16);
            grp1[3 * g + 1] = (uint32_t)nesc;
            grp1[3 * g + 2] = (uint32_t)esc15;
        }
        int w = or_f1_tile_width(ranks + t0, cnt);
        tw[t] = (uint8_t)w;
        uint64_t tile_esc = 0;
        if (w > 0) {
            uint32_t top = (1u << w) - 1u;
            for (uint64_t i = 0; i < OR_TILE; i++) {
                uint32_t r = (i < cnt) ? ranks[t0 + i] : 0;
                uint32_t c = r < top ? r : top;
                for (int b = 0; b < w; b++) {
                    uint64_t bit = off * 8 + i * (uint64_t)w + (uint64_t)b;
                    if ((c >> b) & 1u) payload[bit >> 3] |= (uint8_t)(1u << (bit & 7));
                }
                if (i < cnt && c == top) { esc1[nesc++] = (uint8_t)r; tile_esc++; }
            }
        }
        tesc[t] = (uint8_t)tile_esc;
        for (uint64_t i = 0; i < cnt; i++) esc15 += (ranks[t0 + i] >= 15);
        off += 16 * (uint64_t)w;
    }
    return nesc;
}

/* Decode; returns 0, or -1 when the tile escape counts disagree with the codes. */
int or_f1_decode(const uint8_t *payload, const uint8_t *tw, const uint8_t *tesc,
                 const uint8_t *esc1, const uint32_t *grp1, uint64_t n, uint8_t *ranks) {
    uint64_t ntiles = (n + OR_TILE - 1) / OR_TILE;
    uint64_t off = 0, e = 0;
    for (uint64_t t = 0; t < ntiles; t++) {
        if (t % OR_GROUP == 0) {
            uint64_t g = t / OR_GROUP;
            if ((uint64_t)grp1[3 * g] * 16 != off || grp1[3 * g + 1] != e) return -1;
        }
        uint64_t t0 = t * OR_TILE;
        uint64_t cnt = (n - t0 < OR_TILE) ? n - t0 : OR_TILE;
        int w = tw[t];
        if (w > 8) return -1;
        uint64_t seen = 0;
        for (uint64_t i = 0; i < cnt; i++) {
            uint32_t c = 0;
            for (int b = 0; b < w; b++) {
                uint64_t bit = off * 8 + i * (uint64_t)w + (uint64_t)b;
                c |= (uint32_t)((payload[bit >> 3] >> (bit & 7)) & 1u) << b;
            }
            if (w > 0 && c == (1u << w) - 1u) { ranks[t0 + i] = esc1[e++]; seen++; }
            else ranks[t0 + i] = (uint8_t)c;
        }
        if (seen != tesc[t]) return -1;
        off += 16 * (uint64_t)w;
    }
    return 0;
}

/* ------------------------------------------------------------------------ */
/* R4 runtime layout, [B] "Runtime layout": every rank in 4 bits with rare   */
/* escapes.  Reading: nibble = min(r, 15), element i in byte i >> 1, low     */
/* nibble when i is even; each r >= 15 is appended (flat order) to esc;      */
/* seg[row*nseg + j] = escapes at flat positions < row*K + 512*j, with       */
/* nseg = ceil(K/512), and seg[rows*nseg] = total escapes.                   */
/* ------------------------------------------------------------------------ */
uint64_t or_r4_nseg(uint64_t cols) { return (cols + OR_SEG - 1) / OR_SEG; }

uint64_t or_r4_encode(const uint8_t *ranks, uint64_t rows, uint64_t cols,
                      uint8_t *nib, uint8_t *esc, uint32_t *seg) {
    uint64_t n = rows * cols;
    uint64_t nseg = or_r4_nseg(cols);
    memset(nib, 0, (n + 1) / 2);
    uint64_t e = 0;
    for (uint64_t r = 0; r < rows; r++) {
        for (uint64_t c = 0; c < cols; c++) {
            if (c % OR_SEG == 0) seg[r * nseg + c / OR_SEG] = (uint32_t)e;
            uint64_t i = r * cols + c;
            uint8_t v = ranks[i] < 15 ? ranks[i] : 15;
            nib[i >> 1] |= (uint8_t)(v << (4 * (i & 1)));
            if (ranks[i] >= 15) esc[e++] = ranks[i];
        }
    }
    seg[rows * nseg] = (uint32_t)e;
    return e;
}

/* Decode; each escape's index is found from the row segment's base plus the
   count of 15-nibbles before it in the segment.  Returns 0 or -1 (index out of
   range / inconsistent). */
int or_r4_decode(const uint8_t *nib, const uint8_t *esc, const uint32_t *seg,
                 uint64_t rows, uint64_t cols, uint64_t n_esc, uint8_t *ranks) {
    uint64_t nseg = or_r4_nseg(cols);
    for (uint64_t r = 0; r < rows; r++) {
        for (uint64_t j = 0; j < nseg; j++) {
            uint64_t e = seg[r * nseg + j];
            for (uint64_t c = j * OR_SEG; c < cols && c < (j + 1) * OR_SEG; c++) {
                uint64_t i = r * cols + c;
                uint8_t v = (uint8_t)((nib[i >> 1] >> (4 * (i & 1))) & 0xF);
                if (v == 15) {
                    if (e >= n_esc) return -1;
                    ranks[i] = esc[e++];
                } else {
                    ranks[i] = v;
                }
            }
            uint64_t next = (j + 1 < nseg) ? seg[r * nseg + j + 1] : seg[(r + 1) * nseg];
            if (e != next) return -1;
        }
    }
    return 0;
}

/* Per-round escape summary of the R4 layout (the row-segment index, as the   */
/* product kernels read it): for row r and 512-column round j, the number of */
/* escaped elements c (15-nibbles among the round's columns, counted in the   */
/* nibbles themselves) and the exponents table[rank] of its first three      */
/* escapes in column order.  Word = min(c, 255) | x0 << 8 | x1 << 16 |       */
/* x2 << 24, absent escapes 0.  The ranks are taken from esc starting at     */
/* seg[r*nseg + j].  out: rows*nseg words.  Returns 0 or -1 (index out of    */
/* range).                                                                    */
int or_r4_round_summary(const uint8_t *nib, const uint8_t *esc, const uint32_t *seg,
                        const uint8_t *table, uint64_t rows, uint64_t cols, uint64_t n_esc,
                        uint32_t *out) {
    uint64_t nseg = or_r4_nseg(cols);
    for (uint64_t r = 0; r < rows; r++) {
        for (uint64_t j = 0; j < nseg; j++) {
            uint64_t e = seg[r * nseg + j];
            uint32_t c = 0, x[3] = {0, 0, 0};
            for (uint64_t col = j * OR_SEG; col < cols && col < (j + 1) * OR_SEG; col++) {
                uint64_t i = r * cols + col;
                if (((nib[i >> 1] >> (4 * (i & 1))) & 0xF) != 15) continue;
                if (c < 3) {
                    if (e + c >= n_esc) return -1;
                    x[c] = table[esc[e + c]];
                }
                c++;
            }
            out[r * nseg + j] = (c < 255 ? c : 255) | x[0] << 8 | x[1] << 16 | x[2] << 24;
        }
    }
    return 0;
}

/* ------------------------------------------------------------------------ */
/* Fixed summation order of the batch-1 product y = W x.                     */
/* [B] "Exactness": the compressed and the BF16 kernels add the products in  */
/* one and the same order, so their outputs are bit-identical.  The pages do */
/* not print the order; this is the documented one both kernels follow:      */
/*   rounds of 512 k; in round j lane u (0..31) owns k in                    */
/*   [512j + 16u, min(K, 512j + 16u + 16)); each lane starts at +0 and does  */
/*   acc = fmaf(w_k, x_k, acc) over its k in increasing order, round after   */
/*   round; then five butterfly steps acc_u += acc_(u xor d), d = 16..1; the */
/*   slice result is lane 0's value.  With S slices, slice s owns rounds     */
/*   [floor(sJ/S), floor((s+1)J/S)), J = ceil(K/512), and y = P_0 + P_1 +   */
/*   ... added left to right.                                                */
/* The plan S(N, K): the smallest power of two >= ceil(8192/N), capped at 8 */
/* and at the largest power of two <= J (S = 1 when J <= 1).                 */
/* ------------------------------------------------------------------------ */
int or_gemv_slices(uint64_t N, uint64_t K) {
    uint64_t J = (K + OR_ROUND - 1) / OR_ROUND;
    if (N == 0 || J <= 1) return 1;
    uint64_t want = (8192 + N - 1) / N;
    int S = 1;
    while ((uint64_t)S < want && S * 2 <= 8 && (uint64_t)(S * 2) <= J) S *= 2;
    return S;
}

static float gemv_row(const uint16_t *wrow, uint64_t K, const uint16_t *x, int S) {
    uint64_t J = (K + OR_ROUND - 1) / OR_ROUND;
    float y = 0.0f;
    for (int s = 0; s < S; s++) {
        uint64_t j0 = (uint64_t)s * J / (uint64_t)S;
        uint64_t j1 = (uint64_t)(s + 1) * J / (uint64_t)S;
        float acc[OR_LANES];
        for (int u = 0; u < OR_LANES; u++) acc[u] = 0.0f;
        for (uint64_t j = j0; j < j1; j++) {
            for (int u = 0; u < OR_LANES; u++) {
                uint64_t k0 = j * OR_ROUND + (uint64_t)u * OR_CHUNK;
                for (uint64_t k = k0; k < k0 + OR_CHUNK && k < K; k++)
                    acc[u] = fmaf(or_bf16_to_f32(wrow[k]), or_bf16_to_f32(x[k]), acc[u]);
            }
        }
        for (int d = 16; d >= 1; d /= 2) {
            float nxt[OR_LANES];
            for (int u = 0; u < OR_LANES; u++) nxt[u] = acc[u] + acc[u ^ d];
            for (int u = 0; u < OR_LANES; u++) acc[u] = nxt[u];
        }
        if (s == 0) y = acc[0];
        else y = y + acc[0];
    }
    return y;
}

/* y32[i] (and y16[i] if non-null) for rows rows_sel[i] (all rows if rows_sel
   is null and nsel == N). */
void or_gemv(const uint16_t *W, uint64_t N, uint64_t K, const uint16_t *x,
             const uint64_t *rows_sel, uint64_t nsel, float *y32, uint16_t *y16) {
    int S = or_gemv_slices(N, K);
    for (uint64_t i = 0; i < nsel; i++) {
        uint64_t r = rows_sel ? rows_sel[i] : i;
        float y = gemv_row(W + r * K, K, x, S);
        y32[i] = y;
        if (y16) y16[i] = or_f32_to_bf16(y);
    }
}

/* Same product for a row given as its own array (used when only a few rows of
   a large tensor are rebuilt), with the plan of the full N x K matrix. */
float or_gemv_one(const uint16_t *wrow, uint64_t N, uint64_t K, const uint16_t *x) {
    return gemv_row(wrow, K, x, or_gemv_slices(N, K));
}

/* ------------------------------------------------------------------------ */
/* Mixture-of-experts gather, [B] "Exactness" (the MoE expert gather) and    */
/* "Limitations" (every expert product).  Experts are stacked as one tensor */
/* [E*Ne, K].  y[t, j, :] = expert ids[t, j] applied to x_t in the order    */
/* above (plan of an Ne x K matrix).  Combine, when p is given: out[t, n] = */
/* fmaf chain over j = 0..topk-1 of p[t, j] * y[t, j, n], from +0.          */
/* ------------------------------------------------------------------------ */
int or_moe_gemv(const uint16_t *W, uint64_t n_experts, uint64_t Ne, uint64_t K,
                const int32_t *ids, const float *p, uint64_t T, uint64_t topk,
                const uint16_t *X, float *y32, float *out32, uint16_t *out16) {
    int S = or_gemv_slices(Ne, K);
    for (uint64_t t = 0; t < T; t++) {
        for (uint64_t j = 0; j < topk; j++) {
            int32_t e = ids[t * topk + j];
            if (e < 0 || (uint64_t)e >= n_experts) return -1;
            for (uint64_t n = 0; n < Ne; n++) {
                const uint16_t *wrow = W + ((uint64_t)e * Ne + n) * K;
                y32[(t * topk + j) * Ne + n] = gemv_row(wrow, K, X + t * K, S);
            }
        }
        if (p) {
            for (uint64_t n = 0; n < Ne; n++) {
                float acc = 0.0f;
                for (uint64_t j = 0; j < topk; j++)
                    acc = fmaf(p[t * topk + j], y32[(t * topk + j) * Ne + n], acc);
                out32[t * Ne + n] = acc;
                if (out16) out16[t * Ne + n] = or_f32_to_bf16(acc);
            }
        }
    }
    return 0;
}

/* ------------------------------------------------------------------------ */
/* Prompt product Y = X W^T, [B] "Results" (prompt matmuls) and "NVIDIA     */
/* GPUs".  The tensor-core order is the hardware's, so the oracle is the    */
/* exact-product fp64 sum over k in increasing order.                        */
/* ------------------------------------------------------------------------ */
void or_gemm_f64(const uint16_t *X, const uint16_t *W, uint64_t M, uint64_t N,
                 uint64_t K, const uint64_t *cols_sel, uint64_t ncols, double *Y) {
    for (uint64_t m = 0; m < M; m++) {
        for (uint64_t c = 0; c < ncols; c++) {
            uint64_t n = cols_sel ? cols_sel[c] : c;
            double acc = 0.0;
            for (uint64_t k = 0; k < K; k++)
                acc += (double)or_bf16_to_f32(X[m * K + k]) * (double)or_bf16_to_f32(W[n * K + k]);
            Y[m * ncols + c] = acc;
        }
    }
    (void)N;
}

/* Expert products at prompt length, [B] "Results" (the fused prompt kernels */
/* cover every expert product): for token t and slot j with expert e =       */
/* ids[t, j], y[t, j, n] = sum_k x[t, k] W[e*Ne + n, k] (exact products, fp64, */
/* k increasing) and out[t, n] = sum_j p[t, j] y[t, j, n] (fp64, slot order). */
/* tsel/nsel: the tokens and output columns computed (all when NULL);       */
/* y: ntok x topk x ncol, out: ntok x ncol (may be NULL).  -1 on a bad id.  */
/* ------------------------------------------------------------------------ */
int or_moe_gemm_f64(const uint16_t *W, uint64_t n_experts, uint64_t Ne, uint64_t K,
                    const int32_t *ids, const float *p, uint64_t T, uint64_t topk,
                    const uint16_t *X, const uint64_t *tsel, uint64_t ntok,
                    const uint64_t *nsel, uint64_t ncol, double *y, double *out) {
    for (uint64_t a = 0; a < ntok; a++) {
        uint64_t t = tsel ? tsel[a] : a;
        if (t >= T) return -1;
        for (uint64_t c = 0; c < ncol; c++) {
            uint64_t n = nsel ? nsel[c] : c;
            double o = 0.0;
            for (uint64_t j = 0; j < topk; j++) {
                int32_t e = ids[t * topk + j];
                if (e < 0 || (uint64_t)e >= n_experts || n >= Ne) return -1;
                const uint16_t *wrow = W + ((uint64_t)e * Ne + n) * K;
                double acc = 0.0;
                for (uint64_t k = 0; k < K; k++)
                    acc += (double)or_bf16_to_f32(X[t * K + k]) * (double)or_bf16_to_f32(wrow[k]);
                y[(a * topk + j) * ncol + c] = acc;
                if (p) o += (double)p[t * topk + j] * acc;
            }
            if (out) out[a * ncol + c] = o;
        }
    }
    return 0;
}

/* ------------------------------------------------------------------------ */
/* Decoder-layer glue at batch 1, [B] "Results" (decode speed: a model's    */
/* per-token time) -- the steps between the products, in fp64.              */
/* ------------------------------------------------------------------------ */

/* Round a double to the nearest bf16 (ties to even), returning its bits:
   scale the significand to 8 bits, round half-even, scale back. */
uint16_t or_f64_to_bf16(double v) {
    if (v != v) return 0x7FC0;
    if (v == 0.0) return signbit(v) ? 0x8000 : 0;
    int e;
    double m = frexp(fabs(v), &e);            /* |v| = m 2^e, m in [0.5, 1) */
    double q = nearbyint(ldexp(m, 8));        /* 8 significant bits, half-even */
    float f = (float)ldexp(q, e - 8);         /* exact: 8 bits, bf16 range */
    uint32_t u;
    memcpy(&u, &f, 4);
    uint16_t b = (uint16_t)(u >> 16);
    return v < 0 ? (uint16_t)(b | 0x8000) : b;
}

/* RMS norm: r = 1 / sqrt(mean(x^2) + eps); out[i] = x[i] r gamma[i]. */
void or_rmsnorm_f64(const double *x, const uint16_t *gamma, uint64_t n, double eps, double *out) {
    double ss = 0.0;
    for (uint64_t i = 0; i < n; i++) ss += x[i] * x[i];
    double r = 1.0 / sqrt(ss / (double)n + eps);
    for (uint64_t i = 0; i < n; i++) out[i] = x[i] * r * (double)or_bf16_to_f32(gamma[i]);
}

/* SiLU(g) * u = g / (1 + exp(-g)) * u. */
void or_silu_mul_f64(const double *g, const double *u, uint64_t n, double *out) {
    for (uint64_t i = 0; i < n; i++) out[i] = g[i] / (1.0 + exp(-g[i])) * u[i];
}


/* ------------------------------------------------------------------------ */
/* Exponent statistics, [B] "How it works" ("No exponent locality": per-tile */
/* palettes against a shuffled tensor).  Tile t (c weights, the last one     */
/* may be shorter) costs c * H_t bits, H_t the entropy of its own exponent   */
/* counts: the ideal code with the tile's own table, side information not    */
/* counted.                                                                  */
/* ------------------------------------------------------------------------ */
void or_exp_tile_bits(const uint16_t *b, uint64_t n, uint32_t tile, double *tile_bits) {
    uint64_t ntiles = (n + tile - 1) / tile;
    for (uint64_t t = 0; t < ntiles; t++) {
        uint64_t cnt[256];
        memset(cnt, 0, sizeof(cnt));
        uint64_t lo = t * (uint64_t)tile, hi = lo + tile < n ? lo + tile : n;
        for (uint64_t i = lo; i < hi; i++) cnt[(b[i] >> 7) & 0xFF]++;
        double c = (double)(hi - lo), bits = 0.0;
        for (int e = 0; e < 256; e++)
            if (cnt[e]) bits -= (double)cnt[e] * log2((double)cnt[e] / c);
        tile_bits[t] = bits;
    }
}
