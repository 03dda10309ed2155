// dgt_internal.h -- definitions shared by libdgt's host and CUDA sources.
#pragma once
#include <stdint.h>

// GEMV plan S(N, K): the number of K slices whose partial sums are added left
// to right (part of the documented summation order; see dgt.h).  Slices are
// added until the product has 8192 (row, slice) units -- about 3.4 for each of
// the 16 streaming warps on each of GB300's 152 SMs: enough for even work,
// while each unit stays long enough that its per-unit work (escape index,
// reduction) is small next to its rounds -- and never more than 8 or more
// than the 512-column rounds allow (largest power of two <= J).
static inline int dgt_plan_slices(uint64_t N, uint64_t K) {
    uint64_t J = (K + 511) / 512;
    if (N == 0 || J <= 1) return 1;
    uint64_t want = (8192 + N - 1) / N;
    int S = 1;
    while ((uint64_t)S < want && S * 2 <= 8 && (uint64_t)(S * 2) <= J) S *= 2;
    return S;
}

// R4 row-segment index, in one array of 32-bit words: rows*nseg + 1 prefix
// counts, padded to a multiple of 4 words, then rows*nseg per-round escape
// summaries, padded to a multiple of 4 words (so that 16-byte bulk copies of
// any run of summaries stay inside the array).
static inline uint64_t dgt_rsum_offset(uint64_t rows, uint64_t nseg) { return (rows * nseg + 1 + 3) & ~3ull; }
static inline uint64_t dgt_seg_words(uint64_t rows, uint64_t nseg) {
    return dgt_rsum_offset(rows, nseg) + ((rows * nseg + 3) & ~3ull);
}

// The expert gather's path for few (token, slot) pairs (dgt_moe.cu): each pair
// as a block of the batch-1 product's bulk-copy kernel (dgt_gemv.cu), which
// writes y32[(t * topk + j) * ne + n] = W[ids[t, j] * ne + n] . x[t] in the
// batch-1 order with the plan S(ne, K), and DGT_ERR_ARG into the status word
// for an id outside [0, n_experts).  DGT_ERR_UNSUPPORTED (nothing launched)
// when that kernel does not apply: row length not a multiple of 32, arrays
// not 16-byte aligned, x too long for its shared memory, or more pairs than
// the grid has CTAs.
struct dgt_r4;
int dgt_gemv_expert_blocks(const dgt_r4 *W, uint32_t n_experts, const int32_t *d_ids, uint32_t tokens,
                           uint32_t topk, const uint16_t *d_x, float *d_y32, int32_t *d_status, uint32_t spin,
                           void *stream);
int dgt_gemv_expert_blocks_bf16(const uint16_t *d_W, uint64_t rows, uint64_t cols, uint32_t n_experts,
                                const int32_t *d_ids, uint32_t tokens, uint32_t topk, const uint16_t *d_x,
                                float *d_y32, int32_t *d_status, uint32_t spin, void *stream);
