/*
 * dgt.h -- C ABI of libdgt: lossless BF16 exponent-rank weight compression,
 * decoded inside the matrix product, for one NVIDIA GB300 (sm_103a).
 *
 * The method (Binade project README, title paragraphs and "How it works"):
 * each BF16 weight keeps its sign and 7-bit mantissa as one raw byte; its 8-bit
 * exponent is replaced by its frequency rank in a per-tensor table.  On disk
 * the ranks are Rice coded (format 2) or stored at a fixed width per
 * 128-weight tile with escapes (format 1).  At load a GPU kernel turns either
 * format into R4 -- one 4-bit rank per weight plus rare escapes -- which the
 * matrix-vector, expert-gather and prompt GEMM kernels decode in registers
 * while they compute.  Every product adds in one fixed, documented order, so
 * the R4 kernels and the BF16-weight kernels of this library give
 * bit-identical results.
 *
 * Conventions for every entry point:
 *  - Return value: DGT_OK (0) or a negative DGT_ERR_* code; nothing throws
 *    across the ABI.  dgt_status_string() names a code.
 *  - "device" pointers are CUDA device addresses on the current device; the
 *    caller owns and allocates every device buffer (the library allocates no
 *    device memory).  "host" pointers are ordinary process memory.
 *  - stream is a cudaStream_t passed as void* (NULL = legacy default stream).
 *    Device entry points only enqueue work; they return after the launch.
 *    Errors detected by a kernel (corrupt stream, bounded wait ran out) are
 *    written to the caller's device status word (int32, may be NULL) and are
 *    read with dgt_read_status() once the stream has reached that point.
 *  - Matrices are row-major [rows, cols] = [N, K] (out x in, like a
 *    PyTorch Linear weight); the element count n = rows * cols.
 *  - BF16 values travel as uint16_t bit patterns.
 */
#ifndef DGT_H
#define DGT_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ------------------------------------------------------------------------ */
/* Status codes                                                             */
/* ------------------------------------------------------------------------ */
#define DGT_OK 0
#define DGT_ERR_ARG (-1)         /* null pointer, bad enum, misaligned buffer */
#define DGT_ERR_SHAPE (-2)       /* sizes outside the supported range          */
#define DGT_ERR_CORRUPT (-3)     /* packed data disagrees with its own index    */
#define DGT_ERR_CUDA (-4)        /* a CUDA runtime call or launch failed        */
#define DGT_ERR_TIMEOUT (-5)     /* a bounded device wait ran out               */
#define DGT_ERR_OOM (-6)         /* host allocation failed                      */
#define DGT_ERR_IO (-7)          /* file open / read / write failed             */
#define DGT_ERR_UNSUPPORTED (-8) /* no kernel for this device or configuration  */

/* Human-readable name of a status code (static storage, never NULL). */
const char *dgt_status_string(int status);

/* ABI version of this header (major * 100 + minor). */
int dgt_version(void);

/* ------------------------------------------------------------------------ */
/* Layout constants                                                         */
/* ------------------------------------------------------------------------ */
#define DGT_BLOCK 64   /* format 2: ranks per Rice block, one index byte each */
#define DGT_GROUP 32   /* format 2: blocks per group; format 1: tiles per group */
#define DGT_TILE 128   /* format 1: ranks per fixed-width tile                */
#define DGT_SEG 512    /* R4: row-relative escape-index segment (columns)     */

/* ------------------------------------------------------------------------ */
/* Packed tensor (host object, library-owned)                               */
/* ------------------------------------------------------------------------ */
typedef struct dgt_packed dgt_packed;

/*
 * A read-only view of one packed tensor's arrays.  dgt_packed_get_view() fills
 * it with HOST pointers into a dgt_packed.  To load on the GPU the caller
 * copies each array to device memory and passes a copy of the view whose
 * pointers are the DEVICE addresses of those copies (every array must start
 * on a 16-byte boundary).
 *
 * Format 2 (Binade README, "Two file formats"; block index after the
 * "Best measured configuration" of the "Lossless BF16 weight compression"
 * README): ranks are cut into blocks of 64 and groups of 32 blocks.  A block
 * whose quotient sum Q = sum(r >> k) is <= 254 is Rice coded -- per rank
 * (r >> k) zero bits, a one bit, then the k low bits of r, least significant
 * first -- and its index byte blkq is Q (length count*(k+1)+Q bits); a block
 * with Q >= 255 holds 8-bit raw ranks and index byte 255.  Stream bit j is
 * bit (j % 32) of little-endian word j / 32.  Each group starts on a word;
 * grp holds two words per group: {first word, ranks >= 15 before the group}.
 *
 * Format 1 (same section, "fixed width per 128-weight tile with escapes"):
 * per tile a width w in 0..8 (tw); 128 codes of w bits, least significant bit
 * first, 16*w bytes (payload); code 2^w - 1 is an escape whose rank follows in
 * esc1 (tile order); tesc counts a tile's escapes; grp1 holds three words per
 * 32 tiles: {payload offset / 16, esc1 entries before, ranks >= 15 before}.
 */
typedef struct dgt_packed_view {
    uint64_t rows, cols;      /* N, K                                        */
    int32_t format;           /* 1 or 2                                      */
    int32_t rice_k;           /* format 2: Rice parameter 0..7               */
    int32_t n_table;          /* T: distinct exponents (0..256)              */
    int32_t reserved;
    uint8_t table[256];       /* rank -> exponent, entries >= T are 0        */
    uint64_t n_esc15;         /* ranks >= 15 (R4 escapes)                    */
    const uint8_t *sm;        /* n bytes: sign << 7 | mantissa               */
    const uint32_t *words;    /* format 2: Rice stream, n_words words        */
    uint64_t n_words;
    const uint8_t *blkq;      /* format 2: ceil(n/64) index bytes            */
    uint64_t n_blocks;
    const uint32_t *grp;      /* format 2: 2 words per group                 */
    uint64_t n_groups;
    const uint8_t *payload;   /* format 1: tile codes                        */
    uint64_t payload_bytes;
    const uint8_t *tw;        /* format 1: width per tile                    */
    const uint8_t *tesc;      /* format 1: escapes per tile                  */
    uint64_t n_tiles;
    const uint8_t *esc1;      /* format 1: raw escaped ranks                 */
    uint64_t n_esc1;
    const uint32_t *grp1;     /* format 1: 3 words per 32 tiles              */
    uint64_t n_groups1;
} dgt_packed_view;

/*
 * Pack a BF16 matrix (Binade README: "binade pack"; title paragraph and
 * "How it works").  bf16: host, rows*cols values.  format: 1 or 2.
 * nthreads: host threads to use (<= 0: all hardware threads).  On success
 * *out owns a new object; free it with dgt_packed_free().  The rank table
 * sorts exponents by count (descending), ties by exponent (ascending); format
 * 2 takes the k in 0..7 with the fewest stream words, ties to the smaller k;
 * format 1 takes per tile the w minimising 128*w + 8*escapes, ties to the
 * smaller w, and w = 0 iff the tile is all rank 0.
 * Errors: DGT_ERR_ARG (null, bad format), DGT_ERR_SHAPE (n >= 2^40 or a group
 * index overflowing 32 bits), DGT_ERR_OOM.
 */
int dgt_pack(const uint16_t *bf16, uint64_t rows, uint64_t cols, int format, int nthreads,
             dgt_packed **out);

/* Free a packed object (NULL is ignored). */
void dgt_packed_free(dgt_packed *p);

/* Fill *view with host pointers into p (valid until p is freed). */
int dgt_packed_get_view(const dgt_packed *p, dgt_packed_view *view);

/* Bits per weight of every stored array (sm, table, stream, index). */
double dgt_packed_bits_per_weight(const dgt_packed *p);

/*
 * Host unpack (Binade README, "Use": "binade unpack ... rebuilds the original
 * BF16 checkpoint, bit for bit").  view: host pointers.  out_bf16: host,
 * rows*cols values, caller-owned.  Errors: DGT_ERR_ARG, DGT_ERR_CORRUPT (a
 * block or tile disagrees with its index byte; out is then unspecified).
 */
int dgt_unpack(const dgt_packed_view *view, uint16_t *out_bf16, int nthreads);

/*
 * File container (model cards: "the packed bytes are stored as uint8
 * tensors"): a safetensors file -- u64 little-endian header length, a JSON
 * header, then the data -- with, per tensor name X, arrays "X.sm", "X.rice",
 * "X.blkq", "X.grp" (format 2) or "X.f1", "X.tw", "X.tesc", "X.esc1",
 * "X.grp1" (format 1), and the metadata entry "X" = "format=..;rows=..;...".
 * dgt_write: tensors/names are host arrays of count entries.  The file is
 * written under a temporary name beside `path` and renamed to `path` when
 * complete; on an error nothing is left under either name.
 * dgt_read: *tensors and *names are library-allocated arrays of *count
 * entries; release them with dgt_read_free().  Each array is read from the
 * file straight into its tensor (host memory: the packed size, no second
 * copy of the file).
 * Errors: DGT_ERR_ARG, DGT_ERR_IO, DGT_ERR_CORRUPT (malformed header or
 * arrays whose sizes disagree with the metadata), DGT_ERR_OOM.
 */
int dgt_write(const char *path, const dgt_packed *const *tensors, const char *const *names,
              int count);
int dgt_read(const char *path, dgt_packed ***tensors, char ***names, int *count);
void dgt_read_free(dgt_packed **tensors, char **names, int count);

/* ------------------------------------------------------------------------ */
/* R4 runtime layout (device, caller-owned)                                 */
/* ------------------------------------------------------------------------ */
/*
 * Binade README, "Runtime layout": every rank in 4 bits, with rare escapes.
 * nib: ceil(n/2) bytes, element i in byte i/2, low nibble when i is even,
 *      value min(rank, 15).
 * esc: n_esc bytes, the rank of every element whose nibble is 15, flat order.
 * seg: the row-segment escape index, nseg = ceil(cols/512), in two parts:
 *      - words [0, rows*nseg]: seg[r*nseg + j] counts the escapes at flat
 *        positions < r*cols + 512*j; word rows*nseg is n_esc;
 *      - from word dgt_r4_rsum_offset(rows, cols) (rows*nseg + 1 rounded up
 *        to a multiple of 4): rows*nseg per-round summaries, word r*nseg + j =
 *        min(c, 255) | x0 << 8 | x1 << 16 | x2 << 24, where c is the number
 *        of escapes in round j of row r (its 512 columns) and x0..x2 are the
 *        exponents table[rank] of the first three, in column order (0 when
 *        absent).  The product kernels read these with the weights, so a
 *        round's escape exponents need no dependent lookup.
 *      Both parts are written by dgt_load_r4; the array is
 *      dgt_r4_sizes(...seg_bytes) long (the summaries padded to 4 words).
 * sm:  n bytes, sign << 7 | mantissa (the packed array itself, not a copy).
 * All four device arrays must start on 16-byte boundaries.
 */
typedef struct dgt_r4 {
    uint64_t rows, cols;
    int32_t n_table;
    int32_t reserved;
    uint8_t table[256];
    uint64_t n_esc;
    const uint8_t *sm;
    uint8_t *nib;
    uint8_t *esc;
    uint32_t *seg;
} dgt_r4;

/* nseg = ceil(cols / 512). */
uint64_t dgt_r4_nseg(uint64_t cols);

/* Word offset of the per-round escape summaries inside seg:
   rows*nseg + 1 rounded up to a multiple of 4. */
uint64_t dgt_r4_rsum_offset(uint64_t rows, uint64_t cols);

/* Byte sizes of the R4 arrays for a rows x cols tensor with n_esc escapes. */
int dgt_r4_sizes(uint64_t rows, uint64_t cols, uint64_t n_esc, uint64_t *nib_bytes,
                 uint64_t *esc_bytes, uint64_t *seg_bytes);

/*
 * Load transcode (Binade README, "Runtime layout": "At load a GPU kernel
 * turns either format into R4").  dev: a view with DEVICE pointers of a
 * format 1 or 2 tensor.  r4: rows, cols, n_table, table, n_esc and sm must
 * be set by the caller (dgt_r4_init_from_view does it); nib, esc and seg are
 * written.  d_status: device int32 set to 0 then to a DGT_ERR_* code if a
 * kernel finds the stream corrupt.  Asynchronous on stream.
 * Errors (immediate): DGT_ERR_ARG, DGT_ERR_SHAPE, DGT_ERR_CUDA.
 */
int dgt_load_r4(const dgt_packed_view *dev, dgt_r4 *r4, int32_t *d_status, void *stream);

/* Fill rows, cols, table, n_table, n_esc from a view and set the four array
   pointers (sm is taken from the view). */
int dgt_r4_init_from_view(const dgt_packed_view *view, uint8_t *d_nib, uint8_t *d_esc,
                          uint32_t *d_seg, dgt_r4 *r4);

/*
 * R4 -> BF16 rebuild (Binade README, "NVIDIA GPUs" and "Exactness": the
 * runtime "rebuilds the BF16 weight" where no fused kernel applies).
 * d_out: device, rows*cols uint16, 16-byte aligned.  Asynchronous.
 */
int dgt_r4_to_bf16(const dgt_r4 *r4, uint16_t *d_out, int32_t *d_status, void *stream);

/* Copy the device status word to the host after the stream reaches it. */
int dgt_read_status(const int32_t *d_status, void *stream, int32_t *status);

/* ------------------------------------------------------------------------ */
/* Batch-1 products                                                         */
/* ------------------------------------------------------------------------ */
/*
 * Summation order shared by dgt_gemv and dgt_gemv_bf16 (Binade README,
 * "Exactness": the kernels add in one order, so outputs are bit-identical):
 * rounds of 512 columns; in round j lane u (0..31) owns columns
 * [512j + 16u, 512j + 16u + 16) (clipped at K); each lane starts at +0 and
 * applies fmaf(w, x, acc) over its columns in increasing order, round after
 * round; five butterfly steps acc_u += acc_(u xor d), d = 16, 8, 4, 2, 1; the
 * slice result is lane 0's value.  With S slices, slice s owns rounds
 * [floor(s*J/S), floor((s+1)*J/S)), J = ceil(K/512), and
 * y = ((P_0 + P_1) + ...) + P_(S-1).  y_bf16 is y rounded to nearest-even
 * (NaN -> 0x7FC0).  dgt_gemv_slices() is the plan S(N, K): the smallest power
 * of two >= ceil(8192/N), capped at 8 and at the largest power of two <= J.
 */
int dgt_gemv_slices(uint64_t rows, uint64_t cols);

/*
 * y = W x with W in R4 (Binade README, "Results": "Matvec kernel"; "How it
 * works": "its matvec streams at full bandwidth").  d_x: device, cols bf16.
 * d_y: device, rows bf16 (may be NULL).  d_y32: device, rows float (may be
 * NULL; not both).  d_status: device int32 or NULL; a kernel whose bounded
 * wait for its streamed data runs out writes DGT_ERR_TIMEOUT there (the
 * word is never cleared by this call).  W must come from dgt_load_r4 (its
 * escape index is trusted).  Asynchronous.  Errors: DGT_ERR_ARG,
 * DGT_ERR_SHAPE (cols >= 2^31), DGT_ERR_CUDA.
 */
int dgt_gemv(const dgt_r4 *W, const uint16_t *d_x, uint16_t *d_y, float *d_y32, int32_t *d_status,
             void *stream);

/* The same product and order with plain BF16 weights d_W [rows, cols]. */
int dgt_gemv_bf16(const uint16_t *d_W, uint64_t rows, uint64_t cols, const uint16_t *d_x,
                  uint16_t *d_y, float *d_y32, int32_t *d_status, void *stream);

/*
 * Launch behaviour.  The streaming kernel (cols % 32 == 0, 16-byte aligned
 * arrays) is launched with programmatic stream serialization: it may start
 * while the previous kernel of the stream finishes, and reads x, writes y and
 * the status word only after that kernel has completed (its writes visible).
 * By default it also reads W only after then.  DGT_GEMV_STATIC_WEIGHTS
 * promises that no work queued before this call that may still be running
 * writes W: W was written before the stream last synchronised with the host
 * or waited on an event recorded after the writes (true for weights loaded
 * once and only read since, as in a decode loop).  Kernels of this library
 * start their setup while earlier kernels finish, so without that promise a
 * chain of them could overlap a write to W.  With it, the weights start
 * streaming into shared memory at once, overlapping the previous kernel's
 * tail.  Results are the same either way.  Other flags: DGT_ERR_ARG.
 */
#define DGT_GEMV_STATIC_WEIGHTS 1u

/*
 * Test hook for the failure path (accepted in the flags of dgt_gemv_ex,
 * dgt_gemv_bf16_ex and dgt_moe_gemv_ex, and in dgt_gemm_plan.test_flags).
 * Every wait of the streaming kernels is bounded: a wait for data that does
 * not arrive within the limit writes DGT_ERR_TIMEOUT to the status word, and
 * the kernel stops its producers, lets every bulk copy it issued land, frees
 * its tensor memory and returns, so the context stays usable.  With
 * DGT_TEST_SHORT_WAITS set, the waits for weights and operands give up after
 * DGT_TEST_WAIT_POLLS(n) polls (n = 0..65535; 0 gives up at once) instead of
 * the library's limit of 2^24 polls, so a test can drive that path without a
 * fault or a hang.  Outputs of such a call are unspecified; the status word
 * is the result.  The waits that drain copies already issued keep the full
 * limit.
 */
#define DGT_TEST_SHORT_WAITS (1u << 1)
#define DGT_TEST_WAIT_POLLS(n) (((uint32_t)(n) & 0xFFFFu) << 16)

int dgt_gemv_ex(const dgt_r4 *W, const uint16_t *d_x, uint16_t *d_y, float *d_y32, int32_t *d_status,
                unsigned flags, void *stream);
int dgt_gemv_bf16_ex(const uint16_t *d_W, uint64_t rows, uint64_t cols, const uint16_t *d_x, uint16_t *d_y,
                     float *d_y32, int32_t *d_status, unsigned flags, void *stream);

/* ------------------------------------------------------------------------ */
/* Mixture-of-experts expert gather                                         */
/* ------------------------------------------------------------------------ */
/*
 * Binade README, "How it works" (Exactness: "the matvec, the MoE expert
 * gather and the GEMM" follow one order) and "Limitations" ("every expert
 * product").  W stacks the experts of one projection as one R4 tensor
 * [n_experts * Ne, K] (one rank table).  For token t < tokens and slot
 * j < topk, y[t, j, :] = W[ids[t, j]] x_t in the order of dgt_gemv with the
 * plan S(Ne, K); with routing weights p (may be NULL),
 * out[t, :] = fmaf(p[t, topk-1], y[t, topk-1, :], ... fmaf(p[t, 0], y[t, 0, :], +0)).
 * d_ids: device int32 [tokens, topk], each in [0, n_experts) (others set
 * DGT_ERR_ARG in the status word and leave their outputs undefined).
 * d_p: device float [tokens, topk] or NULL.  d_x: device bf16 [tokens, K].
 * d_y32: device float [tokens, topk, Ne] or NULL.  d_out / d_out32: device
 * bf16 / float [tokens, Ne] or NULL (written only when d_p is given).
 * d_ws: device workspace of dgt_moe_workspace_bytes() bytes, 256-byte
 * aligned, caller-owned, contents need not be initialised.  d_status: device
 * int32, set to 0 then to an error code.  Limits: K % 16 == 0, topk <= 255,
 * tokens * topk <= 65536, n_experts <= 4096.  Asynchronous.
 */
size_t dgt_moe_workspace_bytes(uint32_t n_experts, uint64_t expert_rows, uint64_t cols, uint32_t tokens,
                               uint32_t topk);
int dgt_moe_gemv(const dgt_r4 *W, uint32_t n_experts, const int32_t *d_ids, const float *d_p, uint32_t tokens,
                 uint32_t topk, const uint16_t *d_x, float *d_y32, uint16_t *d_out, float *d_out32, void *d_ws,
                 size_t ws_bytes, int32_t *d_status, void *stream);

/* dgt_moe_gemv with launch flags: 0, or the failure-path test hook
   DGT_TEST_SHORT_WAITS | DGT_TEST_WAIT_POLLS(n); other bits: DGT_ERR_ARG. */
int dgt_moe_gemv_ex(const dgt_r4 *W, uint32_t n_experts, const int32_t *d_ids, const float *d_p, uint32_t tokens,
                    uint32_t topk, const uint16_t *d_x, float *d_y32, uint16_t *d_out, float *d_out32, void *d_ws,
                    size_t ws_bytes, int32_t *d_status, unsigned flags, void *stream);

/* The same gather and order with plain BF16 stacked weights d_W [rows, cols]. */
int dgt_moe_gemv_bf16(const uint16_t *d_W, uint64_t rows, uint64_t cols, uint32_t n_experts,
                      const int32_t *d_ids, const float *d_p, uint32_t tokens, uint32_t topk,
                      const uint16_t *d_x, float *d_y32, uint16_t *d_out, float *d_out32, void *d_ws,
                      size_t ws_bytes, int32_t *d_status, void *stream);

/* ------------------------------------------------------------------------ */
/* Prompt GEMM on tcgen05                                                   */
/* ------------------------------------------------------------------------ */
/*
 * Y[M, N] = X[M, K] W[N, K]^T on the tensor cores (Binade README, "Results":
 * prompt matmuls at 16..2048 rows; "NVIDIA GPUs": each output is a sequence
 * of tensor-core MMA steps along K and split-K partitions follow a fixed
 * rule; "How it works", Exactness).  The plan fixes the arithmetic: the X
 * tile height m_tile (16..256, multiple of 16; each W tile is 128 rows) and
 * the number of K slices split_k (added left to right after the MMAs).  The
 * R4 GEMM and the BF16 GEMM with the same plan issue the same MMA sequence on
 * byte-identical tiles, so their outputs are bit-identical.
 * dgt_gemm_default_plan: m_tile = round_up(M, 16) up to 256; split_k =
 * floor(152 / tiles) (one wave of one CTA per SM; 1 when tiles >= 152), at
 * most K/256 and 16; schedule 0 (auto).
 * d_X: device bf16 [M, K].  d_Y32 / d_Y: device float / bf16 [M, N] (either
 * may be NULL).  d_ws: device workspace of dgt_gemm_workspace_bytes() bytes
 * (split partials; NULL when split_k == 1).  Limits: N % 128 == 0,
 * K % 64 == 0, 16-byte aligned arrays.  Asynchronous; d_status receives
 * DGT_ERR_TIMEOUT if a bounded wait runs out, DGT_ERR_CORRUPT if an escape
 * index runs past the escape list.
 */
typedef struct dgt_gemm_plan {
    int32_t m_tile;
    int32_t split_k;
    uint32_t test_flags;   /* 0, or DGT_TEST_SHORT_WAITS | DGT_TEST_WAIT_POLLS(n) */
    int32_t schedule;      /* 0 auto, 1 one CTA per output tile, 2 persistent (see below) */
} dgt_gemm_plan;

/*
 * Schedules (the plan's arithmetic is the same under each, so the outputs are
 * bit-identical whichever runs).  One CTA per output tile (x split_k) is the
 * first.  The persistent schedule (split_k = 1 only) runs one CTA per SM that
 * walks the tiles b, b + G, ... with two accumulators in tensor memory: the
 * MMAs of a tile fill one while the epilogue drains the other, so a tile's
 * stores run under the next tile's loads and MMAs.  Auto (0) takes the
 * persistent schedule when split_k = 1 and there are more tiles than SMs.
 * schedule = 2 with split_k > 1, or a value outside 0..2: DGT_ERR_ARG.
 */

int dgt_gemm_default_plan(uint64_t M, uint64_t N, uint64_t K, dgt_gemm_plan *plan);
size_t dgt_gemm_workspace_bytes(uint64_t M, uint64_t N, const dgt_gemm_plan *plan);
int dgt_gemm(const dgt_r4 *W, const uint16_t *d_X, uint64_t M, float *d_Y32, uint16_t *d_Y,
             const dgt_gemm_plan *plan, void *d_ws, size_t ws_bytes, int32_t *d_status, void *stream);
int dgt_gemm_bf16(const uint16_t *d_W, uint64_t N, uint64_t K, const uint16_t *d_X, uint64_t M, float *d_Y32,
                  uint16_t *d_Y, const dgt_gemm_plan *plan, void *d_ws, size_t ws_bytes, int32_t *d_status,
                  void *stream);

/*
 * Long prompts from R4 weights by the rebuilt-weight path (Binade README,
 * "NVIDIA GPUs": the runtime rebuilds the BF16 weight where no fused kernel
 * applies): dgt_r4_to_bf16 of W into d_scratch (device, W->rows * W->cols
 * bf16, 16-byte aligned, caller-owned), then dgt_gemm_bf16 on it with the
 * same plan and workspace rules.  Its outputs are the bf16 GEMM's, and so
 * bit-identical to dgt_gemm's.  At 2048 rows of a 4096 x 3840 tensor it runs
 * at 0.88x the bf16 GEMM's speed where the fused dgt_gemm runs at 0.68x; at
 * 128 rows the fused product is faster.  d_status: reset once, then the
 * rebuild's and the product's errors.  Errors: as the two calls.
 */
int dgt_gemm_rebuild(const dgt_r4 *W, const uint16_t *d_X, uint64_t M, float *d_Y32, uint16_t *d_Y,
                     const dgt_gemm_plan *plan, uint16_t *d_scratch, void *d_ws, size_t ws_bytes, int32_t *d_status,
                     void *stream);

/*
 * Expert products at prompt length on the tensor cores (Binade README,
 * "Results": the fused prompt kernels cover every expert product).  W holds
 * n_experts stacked experts (rows = n_experts * Ne, expert e = rows
 * [e*Ne, (e+1)*Ne)); d_ids int32 [tokens, topk], d_p float32 [tokens, topk]
 * (or NULL), d_X bf16 [tokens, K], all device, row-major.
 *   y[t, j, n] = sum_k X[t, k] W[ids[t, j]*Ne + n, k]
 *   out[t, n]  = fmaf chain over j = 0..topk-1 of p[t, j] * y[t, j, n]
 * The pairs (t, j) are placed expert by expert in (t, j) order with their x
 * rows gathered; one CTA computes a 128-row tile of one expert against up to
 * m_tile of its pairs (m_tile = the mean pairs per expert in use rounded up
 * to 16, 16..128) with K in 64-wide steps of four K=16 tcgen05.mma, fp32
 * accumulation in tensor memory; no split-K.  The R4 and the bf16 calls
 * issue the same MMAs on byte-identical tiles, so y, out and out32 are
 * bit-identical.
 * d_y32: [tokens*topk, Ne] float32 or NULL (then it stays in the workspace);
 * d_out (bf16) and d_out32: [tokens, Ne], need d_p.  d_ws: device, 256-byte
 * aligned, dgt_moe_gemm_workspace_bytes(...) bytes (pair lists, job list,
 * gathered X, y when d_y32 is NULL).
 * Limits: K % 64 == 0, n_experts <= 4096, topk <= 255,
 * tokens * topk <= 65536.  Errors: DGT_ERR_SHAPE, DGT_ERR_ARG (also, on the
 * device status, an expert id out of range: that pair contributes nothing),
 * DGT_ERR_CUDA, DGT_ERR_TIMEOUT (status).  Asynchronous on stream.
 */
size_t dgt_moe_gemm_workspace_bytes(uint32_t n_experts, uint64_t expert_rows, uint64_t cols, uint32_t tokens,
                                    uint32_t topk);
int dgt_moe_gemm(const dgt_r4 *W, uint32_t n_experts, const int32_t *d_ids, const float *d_p, const uint16_t *d_X,
                 uint32_t tokens, uint32_t topk, float *d_y32, uint16_t *d_out, float *d_out32, void *d_ws,
                 size_t ws_bytes, int32_t *d_status, void *stream);
int dgt_moe_gemm_bf16(const uint16_t *d_W, uint64_t rows, uint64_t cols, uint32_t n_experts, const int32_t *d_ids,
                      const float *d_p, const uint16_t *d_X, uint32_t tokens, uint32_t topk, float *d_y32,
                      uint16_t *d_out, float *d_out32, void *d_ws, size_t ws_bytes, int32_t *d_status,
                      void *stream);

/*
 * Allocation-free expert gather.  The paper has no counterpart: this entry
 * point exists for callers that cannot allocate device memory when they call
 * -- a plugin inside a host framework that owns the whole device memory pool,
 * or a latency-critical decode loop where a cudaMalloc (which may synchronise
 * the device) is not allowed.  It computes exactly what dgt_moe_gemv computes,
 * with the same arguments minus the workspace, which it takes from a fixed
 * DGT_MOE_NOALLOC_SCRATCH_BYTES array inside the library's device image
 * (every GPU that loads the library holds that memory until the process
 * exits).  It never calls cudaMalloc, cudaFree or any allocating routine.
 * The first call on each device (with that device current) looks up the
 * array's device address; make that first call before any stream capture.
 * All calls share the array and it keeps the last call's contents; nothing in
 * it must start at zero, but calls that overlap on the GPU race on it.
 * Errors: as dgt_moe_gemv, plus DGT_ERR_SHAPE when the workspace this call
 * needs (dgt_moe_workspace_bytes) exceeds DGT_MOE_NOALLOC_SCRATCH_BYTES.
 */
#define DGT_MOE_NOALLOC_SCRATCH_BYTES (4u << 20)
int dgt_moe_gemv_noalloc(const dgt_r4 *W, uint32_t n_experts, const int32_t *d_ids, const float *d_p,
                         uint32_t tokens, uint32_t topk, const uint16_t *d_x, float *d_y32, uint16_t *d_out,
                         float *d_out32, int32_t *d_status, void *stream);

/* ------------------------------------------------------------------------ */
/* Decoder-layer glue (batch-1 decode step)                                 */
/* ------------------------------------------------------------------------ */
/*
 * The steps between the products of one decoder layer at batch 1 (Binade
 * README, "Results": decode speed, a model's per-token time with R4 weights
 * against BF16; "How it works": the format changes only the products).  Each
 * has one fixed order, so a step run with R4 weights and the same step with
 * the BF16 weights produce bit-identical outputs.  All asynchronous on
 * `stream`; device pointers; caller-owned buffers.
 *
 * dgt_add_rmsnorm: residual add and RMS norm in one kernel (one CTA of 1024
 * threads).  If d_y is not NULL, x[i] = x[i] + y[i] (fp32, in place).  Then
 * ss = sum of x[i]^2, where thread t accumulates i = t, t + 1024, ... in
 * increasing order with fmaf from +0, each warp adds its 32 lanes by the
 * butterfly 16, 8, 4, 2, 1, and warp 0 does the same over the 32 warp sums;
 * r = 1 / sqrt(ss / n + eps) (correctly rounded fp32 operations);
 * h[i] = bf16_rne((x[i] * r) * gamma[i]).  d_x: float[n] (in/out); d_y:
 * float[n] or NULL; d_gamma, d_h: bf16 bits [n].  n in 1..65536 (else
 * DGT_ERR_SHAPE); eps >= 0 (else DGT_ERR_ARG).
 *
 * dgt_silu_mul: out[i] = bf16_rne((g[i] / (1 + exp(-g[i]))) * u[i]) in fp32
 * (exp: CUDA's expf).  d_g, d_u: float[n]; d_out: bf16 bits [n].
 *
 * dgt_repeat: out[i] = v[i mod n_in] for i < n_out (bf16 bits): the grouped
 * query heads' copy of a key/value-sized vector.  n_in == 0 with n_out > 0 is
 * DGT_ERR_SHAPE.
 *
 * dgt_weighted_sum: out[i] = fmaf(p[S-1], y[S-1][i], ... fmaf(p[0], y[0][i],
 * +0)) with S = slots: the routed experts' outputs of one token combined in
 * slot order (the combine of dgt_moe_gemv, for outputs computed per slot).
 * d_y: float [slots, n]; d_p: float [slots]; d_out: float [n].  slots == 0
 * with n > 0 is DGT_ERR_SHAPE.
 */
int dgt_add_rmsnorm(float *d_x, const float *d_y, const uint16_t *d_gamma, uint64_t n, float eps, uint16_t *d_h,
                    void *stream);
int dgt_silu_mul(const float *d_g, const float *d_u, uint64_t n, uint16_t *d_out, void *stream);

/* The same for stacked pairs: row r of d_gu (float32 [rows, 2n]) holds
   [gate | up]; d_out (bf16 [rows, n]) row r = bf16(silu(gate) * up), the
   per-element arithmetic of dgt_silu_mul.  Used after a product whose rows
   stack each gate row block with its up block (one launch for both). */
int dgt_silu_mul_rows(const float *d_gu, uint32_t rows, uint64_t n, uint16_t *d_out, void *stream);
int dgt_repeat(const uint16_t *d_v, uint64_t n_in, uint64_t n_out, uint16_t *d_out, void *stream);
int dgt_weighted_sum(const float *d_y, const float *d_p, uint32_t slots, uint64_t n, float *d_out, void *stream);

/* ------------------------------------------------------------------------ */
/* Exponent statistics                                                      */
/* ------------------------------------------------------------------------ */
/*
 * Binade README, "How it works" ("No exponent locality": per-tile palettes
 * gain only 0.011 to 0.027 bits per weight over a shuffled tensor) and its
 * exponent-statistics scripts.  For a BF16 tensor of n weights (bits d_w,
 * device, flat order) and a tile size T (1..65536; the last tile may be
 * shorter):
 *   d_hist[e] = number of weights with exponent e ((b >> 7) & 0xFF), e < 256
 *     (device uint64 [256]; zeroed by the call);
 *   d_tile_bits[t] = c_t * H_t with H_t = -sum_e (c_te / c_t) log2(c_te / c_t)
 *     over tile t's own counts (c_t weights): the bits of coding the tile's
 *     exponents with its own ideal table, side information not counted
 *     (device double [ceil(n / T)]);
 *   d_total_bits[0] = the sum of d_tile_bits in one fixed order, and
 *   d_total_bits[1] = the tensor's exponent entropy -sum_e (h_e/n) log2(h_e/n)
 *     in bits per weight (device double [2]).
 * d_total_bits[0] / n against the same for a shuffled copy is the per-tile
 * palette gain.  Asynchronous.  Errors:
 * DGT_ERR_ARG (null), DGT_ERR_SHAPE (n == 0, T out of range), DGT_ERR_CUDA.
 */
int dgt_exponent_stats(const uint16_t *d_w, uint64_t n, uint32_t tile, uint64_t *d_hist, double *d_tile_bits,
                       double *d_total_bits, void *stream);

#ifdef __cplusplus
}
#endif
#endif /* DGT_H */
