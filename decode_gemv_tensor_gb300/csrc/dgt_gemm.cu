// dgt_gemm.cu -- prompt products Y = X W^T on the 5th-generation tensor cores
// (tcgen05, accumulators in tensor memory), with W in R4 decoded in the
// producer (or plain BF16 for the twin).
//
// Binade README, "Results" (prompt matmuls at 16 to 2048 rows), "NVIDIA GPUs"
// (each output is a sequence of tensor-core MMA steps along K; split-K
// partitions follow a fixed rule) and "How it works" (Exactness: the GEMM
// mirrors the BF16 kernel step for step).  The R4 GEMM and the BF16 GEMM of
// this file issue the same MMA instructions on byte-identical shared-memory
// tiles with the same split and the same reduction order, so their outputs
// are bit-identical; against exact arithmetic the fp32 result is checked
// normwise.
//
// Design (cta_group::1, one CTA of 20 warps per tile):
//  - Swap-AB: the 128-row W tile is operand A (M = 128), the X tile is operand
//    B (N = mt in 16..256), the fp32 accumulator D = W x X^T lives in tensor
//    memory: lane = W row, column = X row.
//  - Operands are K-major SWIZZLE_128B tiles of 64 bf16 along K.  X (and W
//    for the twin) arrive by 2-D TMA.  For R4, 2-D TMA stages the raw
//    sign/mantissa and nibble tiles and warps 4..19 (four threads per W row,
//    16 columns each, sharing the row's running escape index through
//    shuffles) decode them into the same swizzled layout the TMA would write.
//  - Warp 0 lane 0 issues TMA, warp 1 lane 0 issues tcgen05.mma (four K=16
//    steps per 64-wide stage) and commits each stage back to the producer;
//    warps 4..7 read the accumulator with tcgen05.ld and write Y (or the
//    split-K partial).  A second kernel adds the split partials in slice
//    order.
//  - Every mbarrier wait is bounded; on a timeout the CTA raises an abort
//    flag, records DGT_ERR_TIMEOUT, lets its copies land and frees its tensor
//    memory before returning.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include "../../include/dgt.h"
#include "dgt_device.cuh"
#include "dgt_launch.h"

namespace dgt {

constexpr uint32_t GT_N = 128;      // W rows per tile (MMA M)
constexpr uint32_t GT_K = 64;       // bf16 columns per stage (one 128-byte swizzle row)
constexpr uint32_t GT_MAXP = 12;    // pipeline stages, upper bound
constexpr uint32_t GT_SMEM_LIMIT = 200 * 1024;

struct GemmArgs {
    const uint8_t *nib, *esc;
    const uint32_t *seg;
    uint64_t n_esc, nseg;
    uint64_t M, N, K;
    uint32_t mt, kb_total, split, stages;
    float *y32;
    uint16_t *y;
    float *partial;
    int32_t *status;
    R4Lut L;
    uint8_t table[256];
    // grouped expert products: CTA (x, y) takes n-tile x of the expert and
    // m-tile of job gjob[y] (e << 16 | m-tile, or ~0 for no work); the X rows
    // are the expert's pairs, gathered in glist order starting at geoff[e]
    const uint32_t *gjob, *geoff, *glist;
    uint64_t ne;
    uint32_t grouped, topk;
    uint32_t spin;   // polls a wait for work in flight takes before it gives up
    uint32_t schedule;   // 0 auto, 1 one CTA per tile, 2 persistent (split_k = 1)
};

// ---- tcgen05 / TMA wrappers -------------------------------------------------
__device__ __forceinline__ void tmem_alloc(uint32_t slot_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(slot_smem), "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

__device__ __forceinline__ void mma_bf16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                         uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.u32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}
__device__ __forceinline__ void mma_commit(uint32_t mbar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(mbar)
                 : "memory");
}
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t r[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
        "%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
}
__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap *map, uint32_t mbar, int32_t x,
                                            int32_t y) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4}], "
        "[%2];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(mbar), "r"(x), "r"(y)
        : "memory");
}

// Shared-memory matrix descriptor: K-major, SWIZZLE_128B, 8-row core groups
// 1024 bytes apart (stride byte offset), leading byte offset unused (16),
// descriptor version 1 for tcgen05.
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr) {
    uint64_t d = 0;
    d |= (uint64_t)((saddr >> 4) & 0x3FFF);
    d |= (uint64_t)(16 >> 4) << 16;
    d |= (uint64_t)(1024 >> 4) << 32;
    d |= 1ull << 46;
    d |= 2ull << 61;
    return d;
}

// Instruction descriptor for kind::f16: D fp32, A and B bf16, both K-major,
// N = n columns, M = 128.
__host__ __device__ constexpr uint32_t idesc_bf16(uint32_t n) {
    return (1u << 4) | (1u << 7) | (1u << 10) | ((n >> 3) << 17) | ((128u >> 4) << 24);
}

// A wait for work in flight: true when the phase completed; false when the
// CTA aborted or `limit` polls ran out.
__device__ __forceinline__ bool wait_or_abort(uint32_t bar, uint32_t parity, volatile int *abort_flag,
                                              uint32_t limit) {
    for (uint32_t i = 0; i < limit; i++) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((i & 63) == 63 && *abort_flag) return false;
    }
    return false;
}

__host__ __device__ inline uint32_t gemm_stage_bytes(bool r4, uint32_t mt) {
    return GT_N * 128 + mt * 128 + (r4 ? GT_N * 64 + GT_N * 32 : 0);
}

__device__ __forceinline__ uint4 lds128(uint32_t addr) {
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr));
    return v;
}
__device__ __forceinline__ uint2 lds64(uint32_t addr) {
    uint2 v;
    asm volatile("ld.shared.v2.u32 {%0,%1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(addr));
    return v;
}
__device__ __forceinline__ void sts128(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
    asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d) : "memory");
}

// Escape ranks a decoder row keeps in shared memory: the row's next GT_EW
// escapes from where its pass over the tile starts, so that the decode of a
// stage reads no escape from global memory; escapes past them (rows with
// more than GT_EW in the tile's K range) are read from the list itself.
constexpr uint32_t GT_EW = 32;

// The window of row t: esc[wbase, wbase + GT_EW), the row's four chunk
// threads loading 8 bytes each (q: the thread's chunk).
__device__ __forceinline__ void load_esc_window(const GemmArgs &a, uint8_t *win, uint64_t wbase, uint32_t q) {
    uint32_t lo = 0, hi = 0;
#pragma unroll
    for (uint32_t b = 0; b < 8; b++) {
        const uint64_t e = wbase + 8 * q + b;
        const uint32_t v = e < a.n_esc ? a.esc[e] : 0u;
        if (b < 4) lo |= v << (8 * b);
        else hi |= v << (8 * (b - 4));
    }
    *reinterpret_cast<uint2 *>(win + 8 * q) = make_uint2(lo, hi);
}

// The rank of escape e of the row (its window starting at escape wbase).
__device__ __forceinline__ uint32_t esc_rank(const GemmArgs &a, const uint8_t *win, uint64_t wbase, uint64_t e,
                                             bool &bad) {
    if (e >= a.n_esc) {
        bad = true;
        return 0u;
    }
    const uint64_t rel = e - wbase;
    return rel < GT_EW ? win[rel] : a.esc[e];
}

// Decoder thread (row t, chunk q): the 16 weights [16q, 16q + 16) of W row t
// of a stage, from the raw tiles (shared addresses raw_sm, raw_nib of the
// row) into the row's swizzled bf16 chunks 2q and 2q+1 (arow).  The four
// chunk threads of a row are lanes 4j..4j+3 of one warp; they place their
// escapes by a prefix sum over the four and advance the row's running escape
// index eidx, the ranks coming from the row's window (win, from escape wbase
// on).  A chunk with one escape decodes with the exponent table's rank-15
// entry replaced by its exponent; more are patched weight by weight.  A
// stage where no lane of the warp holds an escape (most of them) skips all
// of that.
__device__ __forceinline__ void decode_chunk16(const GemmArgs &a, const R4Lut &L, uint32_t raw_sm,
                                               uint32_t raw_nib, uint32_t arow, uint32_t t, uint32_t q,
                                               uint64_t &eidx, const uint8_t *win, uint64_t wbase,
                                               const uint8_t *table_s, bool &bad) {
    const uint4 sv = lds128(raw_sm + q * 16);
    const uint2 nv = lds64(raw_nib + q * 8);
    const uint32_t m0 = nib15_mask(nv.x), m1 = nib15_mask(nv.y);
    uint32_t p[8];
    if (!__any_sync(DGT_FULL, (m0 | m1) != 0)) {
        r4_dec16(nv, sv, L, p);
    } else {
        const uint32_t c = __popc(m0) + __popc(m1);
        uint32_t incl = c;
        uint32_t y = __shfl_up_sync(DGT_FULL, incl, 1, 4);
        if (q >= 1) incl += y;
        y = __shfl_up_sync(DGT_FULL, incl, 2, 4);
        if (q >= 2) incl += y;
        const uint32_t total = __shfl_sync(DGT_FULL, incl, 3, 4);
        const uint32_t before = incl - c;
        R4Lut Lr = L;
        if (c == 1) {
            const uint32_t ex = table_s[esc_rank(a, win, wbase, eidx + before, bad)];
            Lr.h3 = prmt(L.h3, ex >> 1, 0x4210u);
            Lr.l1 = (L.l1 & 0x7FFFFFFFu) | ((ex & 1u) << 31);
        }
        r4_dec16(nv, sv, Lr, p);
        if (c > 1) {
            uint64_t e = eidx + before;
#pragma unroll
            for (int i = 0; i < 16; i++) {
                const uint32_t m = i < 8 ? m0 : m1;
                if ((m >> (4 * (i & 7))) & 1u) {
                    const uint32_t ex = table_s[esc_rank(a, win, wbase, e, bad)];
                    e++;
                    const uint32_t sh = 16 * (i & 1);
                    p[i >> 1] = (p[i >> 1] & ~(0x7F80u << sh)) | (ex << (7 + sh));
                }
            }
        }
        eidx += total;
    }
    const uint32_t c0 = (2 * q) ^ (t & 7), c1 = (2 * q + 1) ^ (t & 7);
    sts128(arow + c0 * 16, p[0], p[1], p[2], p[3]);
    sts128(arow + c1 * 16, p[4], p[5], p[6], p[7]);
}

constexpr uint32_t GT_THREADS = 640;   // 4 control/epilogue warps + 16 decoder warps

template <bool R4>
__global__ void __launch_bounds__(GT_THREADS, 1)
    k_gemm(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_w,
           const __grid_constant__ CUtensorMap tm_nib, GemmArgs a) {
    extern __shared__ uint8_t smem_raw[];
    __shared__ __align__(8) uint64_t bar_full[GT_MAXP], bar_raw[GT_MAXP], bar_w[GT_MAXP], bar_empty[GT_MAXP];
    __shared__ __align__(8) uint64_t bar_done;
    __shared__ uint32_t tmem_slot;
    __shared__ uint8_t table_s[256];
    __shared__ __align__(8) uint8_t escw[R4 ? GT_N : 1][GT_EW];
    __shared__ int abort_flag;
    uint8_t *base = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
    const uint32_t tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const uint32_t mt = a.mt, P = a.stages;
    const uint32_t SB = gemm_stage_bytes(R4, mt);
    uint32_t n0 = blockIdx.x * GT_N, m0 = blockIdx.y * mt;
    const uint32_t sl = blockIdx.z;
    const uint32_t kb0 = (uint32_t)((uint64_t)sl * a.kb_total / a.split);
    const uint32_t kb1 = (uint32_t)((uint64_t)(sl + 1) * a.kb_total / a.split);
    const uint32_t nkb = kb1 - kb0;
    const uint32_t ncols = mt <= 32 ? 32 : (mt <= 64 ? 64 : (mt <= 128 ? 128 : 256));
    auto A = [&](uint32_t s) { return base + (size_t)s * SB; };
    auto B = [&](uint32_t s) { return base + (size_t)s * SB + GT_N * 128; };
    auto RS = [&](uint32_t s) { return base + (size_t)s * SB + GT_N * 128 + mt * 128; };
    auto RN = [&](uint32_t s) { return base + (size_t)s * SB + GT_N * 128 + mt * 128 + GT_N * 64; };

    if (tid == 0) {
        for (uint32_t i = 0; i < P; i++) {
            mbar_init(smem_u32(&bar_full[i]), 1);
            mbar_init(smem_u32(&bar_raw[i]), 1);
            mbar_init(smem_u32(&bar_w[i]), 16);
            mbar_init(smem_u32(&bar_empty[i]), 1);
        }
        mbar_init(smem_u32(&bar_done), 1);
        abort_flag = 0;
        fence_mbarrier_init();
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(&tmem_slot), ncols);
        tmem_relinquish();
    }
    if (tid < 256) table_s[tid] = a.table[tid];
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    // barriers and tensor memory are set up while the previous kernel of the
    // stream may still run; nothing it writes or reads is touched before this
    pdl_trigger();
    pdl_wait();
    const uint32_t taddr = tmem_slot;
    volatile int *abortp = &abort_flag;
    // grouped: this CTA's expert, its first gathered X row, and how many of
    // the tile's rows (W) and columns (X) are real
    uint32_t nvalid = GT_N, mvalid = mt;
    if (a.grouped) {
        const uint32_t job = a.gjob[blockIdx.y];
        if (job == 0xFFFFFFFFu) {
            tc_fence_before();
            __syncthreads();
            tc_fence_after();
            if (warp == 1) tmem_dealloc(taddr, ncols);
            return;
        }
        const uint32_t e = job >> 16, mtile = job & 0xFFFFu;
        const uint32_t p0 = a.geoff[e] + mtile * mt;
        mvalid = min(mt, a.geoff[e + 1] - p0);
        m0 = p0;
        const uint64_t nt0 = (uint64_t)blockIdx.x * GT_N;
        nvalid = (uint32_t)min((uint64_t)GT_N, a.ne - nt0);
        n0 = (uint32_t)((uint64_t)e * a.ne + nt0);
    }

    if (warp == 0) {
        if (lane == 0) {
            // ---- TMA producer
            uint32_t issued = 0;
            for (uint32_t i = 0; i < nkb; i++) {
                const uint32_t s = i % P, use = i / P;
                if (use > 0 && !wait_or_abort(smem_u32(&bar_empty[s]), (use - 1) & 1u, abortp, a.spin)) {
                    set_status(a.status, DGT_ERR_TIMEOUT);
                    *abortp = 1;
                    break;
                }
                const int32_t k = (int32_t)((kb0 + i) * GT_K);
                mbar_arrive_expect_tx(smem_u32(&bar_full[s]), mt * 128 + (R4 ? 0 : GT_N * 128));
                tma_load_2d(smem_u32(B(s)), &tm_x, smem_u32(&bar_full[s]), k, (int32_t)m0);
                if (!R4) {
                    tma_load_2d(smem_u32(A(s)), &tm_w, smem_u32(&bar_full[s]), k, (int32_t)n0);
                } else {
                    mbar_arrive_expect_tx(smem_u32(&bar_raw[s]), GT_N * 64 + GT_N * 32);
                    tma_load_2d(smem_u32(RS(s)), &tm_w, smem_u32(&bar_raw[s]), k, (int32_t)n0);
                    tma_load_2d(smem_u32(RN(s)), &tm_nib, smem_u32(&bar_raw[s]), k / 2, (int32_t)n0);
                }
                issued++;
            }
            // let every copy issued land before the CTA can exit
            for (uint32_t i = issued > P ? issued - P : 0; i < issued; i++) {
                const uint32_t s = i % P, par = (i / P) & 1u;
                wait_or_abort(smem_u32(&bar_full[s]), par, abortp, a.spin) || mbar_wait(smem_u32(&bar_full[s]), par);
                if (R4) wait_or_abort(smem_u32(&bar_raw[s]), par, abortp, a.spin) || mbar_wait(smem_u32(&bar_raw[s]), par);
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            // ---- MMA issuer
            const uint32_t idesc = idesc_bf16(mt);
            for (uint32_t i = 0; i < nkb; i++) {
                const uint32_t s = i % P, par = (i / P) & 1u;
                if (!wait_or_abort(smem_u32(&bar_full[s]), par, abortp, a.spin) ||
                    (R4 && !wait_or_abort(smem_u32(&bar_w[s]), par, abortp, a.spin))) {
                    set_status(a.status, DGT_ERR_TIMEOUT);
                    *abortp = 1;
                    break;
                }
                tc_fence_after();
                const uint64_t ad = sw128_desc(smem_u32(A(s))), bd = sw128_desc(smem_u32(B(s)));
#pragma unroll
                for (uint32_t kk = 0; kk < GT_K / 16; kk++)
                    mma_bf16(taddr, ad + 2 * kk, bd + 2 * kk, idesc, (i > 0 || kk > 0) ? 1u : 0u);
                mma_commit(smem_u32(&bar_empty[s]));
            }
            mma_commit(smem_u32(&bar_done));
        }
    } else if (warp >= 4) {
        if (R4) {
            // ---- decoders: thread (t, q) owns chunk q of W row n0 + t
            const uint32_t d = tid - 128, t = d >> 2, q = d & 3;
            const uint64_t row = (uint64_t)n0 + t;
            const bool rin = row < a.N;   // rows past the tensor (grouped tail tiles) read zeros
            const uint64_t kstart = (uint64_t)kb0 * GT_K;
            const uint64_t j = kstart / DGT_SEG;
            uint64_t eidx = rin ? a.seg[row * a.nseg + j] : a.n_esc;
            if (rin) {
                // escapes of this row's segment before kstart: at most 448 nibbles,
                // read as up to 14 independent 16-byte loads
                const uint4 *np = reinterpret_cast<const uint4 *>(a.nib + (row * a.K + j * DGT_SEG) / 2);
                const uint32_t nv = (uint32_t)((kstart - j * DGT_SEG) / 32);
                uint32_t cnt = 0;
#pragma unroll
                for (uint32_t v = 0; v < DGT_SEG / 32 - 2; v++) {
                    if (v < nv) {
                        const uint4 qv = np[v];
                        cnt += __popc(nib15_mask(qv.x)) + __popc(nib15_mask(qv.y)) + __popc(nib15_mask(qv.z)) +
                               __popc(nib15_mask(qv.w));
                    }
                }
                eidx += cnt;
            }
            bool bad = false;
            R4Lut L;
            L.h0 = a.L.h0;
            L.h1 = a.L.h1;
            L.h2 = a.L.h2;
            L.h3 = a.L.h3;
            L.l0 = a.L.l0;
            L.l1 = a.L.l1;
            const uint64_t wbase = eidx;
            if (rin) load_esc_window(a, escw[t], wbase, q);
            __syncwarp();
            const uint32_t base_a = smem_u32(base);
            uint32_t s = 0, par = 0;
            for (uint32_t i = 0; i < nkb; i++) {
                if (!wait_or_abort(smem_u32(&bar_raw[s]), par, abortp, a.spin)) {
                    if (lane == 0) set_status(a.status, DGT_ERR_TIMEOUT);
                    *abortp = 1;
                    break;
                }
                const uint32_t st0 = base_a + s * SB;
                decode_chunk16(a, L, st0 + GT_N * 128 + mt * 128 + t * 64, st0 + GT_N * 128 + mt * 128 + GT_N * 64 + t * 32,
                               st0 + t * 128, t, q, eidx, escw[t], wbase, table_s, bad);
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_u32(&bar_w[s]));
                if (++s == P) {
                    s = 0;
                    par ^= 1u;
                }
            }
            if (bad) set_status(a.status, DGT_ERR_CORRUPT);
        }
        if (warp >= 8) {
            // decoder-only warps are done
        } else {
        const uint32_t t = tid - 128;  // accumulator row, TMEM lane
        // ---- epilogue: thread t holds accumulator row t (W row n0 + t)
        const bool ok = wait_or_abort(smem_u32(&bar_done), 0, abortp, a.spin) || mbar_wait(smem_u32(&bar_done), 0);
        tc_fence_after();
        if (ok && !*abortp) {
            const uint32_t lane_base = ((warp - 4) * 32) << 16;
            const uint64_t n = n0 + t;
            for (uint32_t c = 0; c < mt; c += 16) {
                uint32_t r[16];
                tmem_ld16(taddr + lane_base + c, r);
                tmem_wait_ld();
                if (a.grouped) {
                    // row t of the expert's n-tile for each of its pairs
#pragma unroll
                    for (int i = 0; i < 16; i++) {
                        if (c + i < mvalid && t < nvalid) {
                            const uint32_t pr = a.glist[m0 + c + i];
                            const uint64_t q = (uint64_t)(pr >> 8) * a.topk + (pr & 0xFFu);
                            a.y32[q * a.ne + (uint64_t)blockIdx.x * GT_N + t] = __uint_as_float(r[i]);
                        }
                    }
                    continue;
                }
#pragma unroll
                for (int i = 0; i < 16; i++) {
                    const uint64_t m = (uint64_t)m0 + c + i;
                    if (m < a.M) {
                        const float v = __uint_as_float(r[i]);
                        if (a.split == 1) {
                            if (a.y32) a.y32[m * a.N + n] = v;
                            if (a.y) a.y[m * a.N + n] = f32_to_bf16_rne(v);
                        } else {
                            a.partial[((uint64_t)sl * a.M + m) * a.N + n] = v;
                        }
                    }
                }
            }
        }
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(taddr, ncols);
}

// ---- persistent schedule: one CTA per SM --------------------------------------
// One CTA per SM walks the output tiles b, b + G, b + 2G, ... (G = grid size)
// with two accumulators in tensor memory: the MMA warp fills accumulator
// i & 1 for the CTA's i-th tile while the epilogue warps drain the other, so
// a tile's epilogue runs under the next tile's loads and MMAs.  The TMA
// producer, the MMA warp and (R4) the decoder warps walk one continuous
// sequence of pipeline stages across the tiles.  Each tile issues the same
// MMA sequence as k_gemm with split_k = 1, so the outputs are bit-identical
// to it.  Warps: 0 TMA, 1 MMA (and the tensor-memory allocation), 4..7 the
// epilogue (warp 4 + w reads accumulator lanes 32w..32w + 31), 8..23 the R4
// decoders (four threads per W row, as in k_gemm).
constexpr uint32_t PT_WARPS_R4 = 24, PT_WARPS_BF16 = 8;

template <bool R4>
__global__ void __launch_bounds__((R4 ? PT_WARPS_R4 : PT_WARPS_BF16) * 32, 1)
    k_gemm_pt(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_w,
              const __grid_constant__ CUtensorMap tm_nib, GemmArgs a) {
    extern __shared__ uint8_t smem_raw[];
    __shared__ __align__(8) uint64_t bar_full[GT_MAXP], bar_raw[GT_MAXP], bar_w[GT_MAXP], bar_empty[GT_MAXP];
    __shared__ __align__(8) uint64_t acc_full[2], acc_empty[2], bar_done;
    __shared__ uint32_t tmem_slot;
    __shared__ uint8_t table_s[256];
    __shared__ __align__(8) uint8_t escw[R4 ? GT_N : 1][GT_EW];
    __shared__ int abort_flag;
    uint8_t *base = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
    const uint32_t tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const uint32_t mt = a.mt, P = a.stages;
    const uint32_t SB = gemm_stage_bytes(R4, mt);
    const uint32_t ncols = mt <= 32 ? 32 : (mt <= 64 ? 64 : (mt <= 128 ? 128 : 256));   // per accumulator
    const uint32_t NT = (uint32_t)(a.N / GT_N), MTL = (uint32_t)((a.M + mt - 1) / mt), tiles = NT * MTL;
    const uint32_t nkb = a.kb_total;
    const uint32_t my_tiles = blockIdx.x < tiles ? (tiles - 1 - blockIdx.x) / gridDim.x + 1 : 0;
    auto A = [&](uint32_t s) { return base + (size_t)s * SB; };
    auto B = [&](uint32_t s) { return base + (size_t)s * SB + GT_N * 128; };
    auto RS = [&](uint32_t s) { return base + (size_t)s * SB + GT_N * 128 + mt * 128; };
    auto RN = [&](uint32_t s) { return base + (size_t)s * SB + GT_N * 128 + mt * 128 + GT_N * 64; };
    auto tile_of = [&](uint32_t i, uint32_t &n0, uint32_t &m0) {
        const uint32_t t = blockIdx.x + i * gridDim.x;
        n0 = (t % NT) * GT_N;
        m0 = (t / NT) * mt;
    };

    if (tid == 0) {
        for (uint32_t i = 0; i < P; i++) {
            mbar_init(smem_u32(&bar_full[i]), 1);
            mbar_init(smem_u32(&bar_raw[i]), 1);
            mbar_init(smem_u32(&bar_w[i]), 16);
            mbar_init(smem_u32(&bar_empty[i]), 1);
        }
        for (int i = 0; i < 2; i++) {
            mbar_init(smem_u32(&acc_full[i]), 1);
            mbar_init(smem_u32(&acc_empty[i]), 4);
        }
        mbar_init(smem_u32(&bar_done), 1);
        abort_flag = 0;
        fence_mbarrier_init();
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(&tmem_slot), 2 * ncols);
        tmem_relinquish();
    }
    if (tid < 256) table_s[tid] = a.table[tid];
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    pdl_trigger();
    pdl_wait();
    const uint32_t taddr = tmem_slot;
    volatile int *abortp = &abort_flag;

    if (warp == 0) {
        if (lane == 0) {
            // ---- TMA producer
            uint32_t g = 0;
            bool stop = false;
            for (uint32_t i = 0; i < my_tiles && !stop; i++) {
                uint32_t n0, m0;
                tile_of(i, n0, m0);
                for (uint32_t kb = 0; kb < nkb; kb++) {
                    const uint32_t s = g % P, use = g / P;
                    if (use > 0 && !wait_or_abort(smem_u32(&bar_empty[s]), (use - 1) & 1u, abortp, a.spin)) {
                        set_status(a.status, DGT_ERR_TIMEOUT);
                        *abortp = 1;
                        stop = true;
                        break;
                    }
                    const int32_t k = (int32_t)(kb * GT_K);
                    mbar_arrive_expect_tx(smem_u32(&bar_full[s]), mt * 128 + (R4 ? 0 : GT_N * 128));
                    tma_load_2d(smem_u32(B(s)), &tm_x, smem_u32(&bar_full[s]), k, (int32_t)m0);
                    if (!R4) {
                        tma_load_2d(smem_u32(A(s)), &tm_w, smem_u32(&bar_full[s]), k, (int32_t)n0);
                    } else {
                        mbar_arrive_expect_tx(smem_u32(&bar_raw[s]), GT_N * 64 + GT_N * 32);
                        tma_load_2d(smem_u32(RS(s)), &tm_w, smem_u32(&bar_raw[s]), k, (int32_t)n0);
                        tma_load_2d(smem_u32(RN(s)), &tm_nib, smem_u32(&bar_raw[s]), k / 2, (int32_t)n0);
                    }
                    g++;
                }
            }
            // let every copy issued land before the CTA can exit
            for (uint32_t j = g > P ? g - P : 0; j < g; j++) {
                const uint32_t s = j % P, par = (j / P) & 1u;
                wait_or_abort(smem_u32(&bar_full[s]), par, abortp, a.spin) || mbar_wait(smem_u32(&bar_full[s]), par);
                if (R4) wait_or_abort(smem_u32(&bar_raw[s]), par, abortp, a.spin) || mbar_wait(smem_u32(&bar_raw[s]), par);
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            // ---- MMA issuer
            const uint32_t idesc = idesc_bf16(mt);
            uint32_t g = 0;
            bool stop = false;
            for (uint32_t i = 0; i < my_tiles && !stop; i++) {
                const uint32_t ab = i & 1u;
                // the epilogue has drained this accumulator (its tile i - 2)
                if (i >= 2 && !wait_or_abort(smem_u32(&acc_empty[ab]), ((i >> 1) - 1) & 1u, abortp, a.spin)) {
                    set_status(a.status, DGT_ERR_TIMEOUT);
                    *abortp = 1;
                    break;
                }
                tc_fence_after();
                const uint32_t d = taddr + ab * ncols;
                for (uint32_t kb = 0; kb < nkb; kb++, g++) {
                    const uint32_t s = g % P, par = (g / P) & 1u;
                    if (!wait_or_abort(smem_u32(&bar_full[s]), par, abortp, a.spin) ||
                        (R4 && !wait_or_abort(smem_u32(&bar_w[s]), par, abortp, a.spin))) {
                        set_status(a.status, DGT_ERR_TIMEOUT);
                        *abortp = 1;
                        stop = true;
                        break;
                    }
                    tc_fence_after();
                    const uint64_t ad = sw128_desc(smem_u32(A(s))), bd = sw128_desc(smem_u32(B(s)));
#pragma unroll
                    for (uint32_t kk = 0; kk < GT_K / 16; kk++)
                        mma_bf16(d, ad + 2 * kk, bd + 2 * kk, idesc, (kb > 0 || kk > 0) ? 1u : 0u);
                    mma_commit(smem_u32(&bar_empty[s]));
                }
                if (!stop) mma_commit(smem_u32(&acc_full[ab]));
            }
            mma_commit(smem_u32(&bar_done));
        }
    } else if (warp >= 4 && warp < 8) {
        // ---- epilogue: thread t holds accumulator row t (W row n0 + t)
        const uint32_t t = tid - 128;
        const uint32_t lane_base = ((warp - 4) * 32) << 16;
        for (uint32_t i = 0; i < my_tiles; i++) {
            const uint32_t ab = i & 1u;
            const bool ok = wait_or_abort(smem_u32(&acc_full[ab]), (i >> 1) & 1u, abortp, a.spin);
            tc_fence_after();
            if (!ok) {
                if (lane == 0) set_status(a.status, DGT_ERR_TIMEOUT);
                *abortp = 1;
                break;
            }
            uint32_t n0, m0;
            tile_of(i, n0, m0);
            const uint64_t n = n0 + t;
            for (uint32_t c = 0; c < mt; c += 16) {
                uint32_t r[16];
                tmem_ld16(taddr + lane_base + ab * ncols + c, r);
                tmem_wait_ld();
#pragma unroll
                for (int j = 0; j < 16; j++) {
                    const uint64_t m = (uint64_t)m0 + c + j;
                    if (m < a.M) {
                        const float v = __uint_as_float(r[j]);
                        if (a.y32) a.y32[m * a.N + n] = v;
                        if (a.y) a.y[m * a.N + n] = f32_to_bf16_rne(v);
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&acc_empty[ab]));
        }
    } else if (R4 && warp >= 8) {
        // ---- decoders: thread (t, q) owns chunk q of W row n0 + t of every tile
        const uint32_t dd = tid - 256, t = dd >> 2, q = dd & 3;
        R4Lut L;
        L.h0 = a.L.h0;
        L.h1 = a.L.h1;
        L.h2 = a.L.h2;
        L.h3 = a.L.h3;
        L.l0 = a.L.l0;
        L.l1 = a.L.l1;
        const uint32_t base_a = smem_u32(base);
        uint32_t g = 0;
        bool bad = false, stop = false;
        for (uint32_t i = 0; i < my_tiles && !stop; i++) {
            uint32_t n0, m0;
            tile_of(i, n0, m0);
            const uint64_t row = (uint64_t)n0 + t;
            const bool rin = row < a.N;   // rows past the tensor read zeros
            uint64_t eidx = rin ? a.seg[row * a.nseg] : a.n_esc;
            const uint64_t wbase = eidx;
            __syncwarp();   // the previous tile's reads of the window are done
            if (rin) load_esc_window(a, escw[t], wbase, q);
            __syncwarp();
            for (uint32_t kb = 0; kb < nkb; kb++, g++) {
                const uint32_t s = g % P, par = (g / P) & 1u;
                if (!wait_or_abort(smem_u32(&bar_raw[s]), par, abortp, a.spin)) {
                    if (lane == 0) set_status(a.status, DGT_ERR_TIMEOUT);
                    *abortp = 1;
                    stop = true;
                    break;
                }
                const uint32_t st0 = base_a + s * SB;
                decode_chunk16(a, L, st0 + GT_N * 128 + mt * 128 + t * 64,
                               st0 + GT_N * 128 + mt * 128 + GT_N * 64 + t * 32, st0 + t * 128, t, q, eidx, escw[t], wbase,
                               table_s, bad);
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_u32(&bar_w[s]));
            }
        }
        if (bad) set_status(a.status, DGT_ERR_CORRUPT);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) {
        // every MMA this CTA issued has completed before its tensor memory goes
        wait_or_abort(smem_u32(&bar_done), 0, abortp, a.spin) || mbar_wait(smem_u32(&bar_done), 0);
        tc_fence_after();
        tmem_dealloc(taddr, 2 * ncols);
    }
}

__global__ void __launch_bounds__(256) k_gemm_reduce(GemmArgs a) {
    pdl_trigger();
    pdl_wait();
    const uint64_t total = a.M * a.N;
    for (uint64_t i = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total; i += (uint64_t)gridDim.x * blockDim.x) {
        float y = a.partial[i];
        for (uint32_t s = 1; s < a.split; s++) y = y + a.partial[(uint64_t)s * total + i];
        if (a.y32) a.y32[i] = y;
        if (a.y) a.y[i] = f32_to_bf16_rne(y);
    }
}

// ---- host side ---------------------------------------------------------------
static PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (!fn) {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    }
    return fn;
}

static bool make_map(CUtensorMap *m, CUtensorMapDataType dt, const void *ptr, uint64_t inner, uint64_t outer,
                     uint64_t stride_bytes, uint32_t box_inner, uint32_t box_outer, CUtensorMapSwizzle sw) {
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[2] = {inner, outer};
    cuuint64_t strides[1] = {stride_bytes};
    cuuint32_t box[2] = {box_inner, box_outer};
    cuuint32_t es[2] = {1, 1};
    return fn(m, dt, 2, const_cast<void *>(ptr), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, sw,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

static uint32_t gemm_stages(bool r4, uint32_t mt) {
    uint32_t p = GT_SMEM_LIMIT / gemm_stage_bytes(r4, mt);
    return p > GT_MAXP ? GT_MAXP : p;
}

template <bool R4>
static int launch_gemm(GemmArgs &a, const void *w_or_sm, const uint16_t *d_X, void *d_ws, size_t ws_bytes,
                       cudaStream_t st) {
    CUtensorMap tm_x, tm_w, tm_nib;
    if (!make_map(&tm_x, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, d_X, a.K, a.M, a.K * 2, GT_K, a.mt,
                  CU_TENSOR_MAP_SWIZZLE_128B))
        return DGT_ERR_CUDA;
    if (R4) {
        if (!make_map(&tm_w, CU_TENSOR_MAP_DATA_TYPE_UINT8, w_or_sm, a.K, a.N, a.K, GT_K, GT_N,
                      CU_TENSOR_MAP_SWIZZLE_NONE) ||
            !make_map(&tm_nib, CU_TENSOR_MAP_DATA_TYPE_UINT8, a.nib, a.K / 2, a.N, a.K / 2, GT_K / 2, GT_N,
                      CU_TENSOR_MAP_SWIZZLE_NONE))
            return DGT_ERR_CUDA;
    } else {
        if (!make_map(&tm_w, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, w_or_sm, a.K, a.N, a.K * 2, GT_K, GT_N,
                      CU_TENSOR_MAP_SWIZZLE_128B))
            return DGT_ERR_CUDA;
        tm_nib = tm_w;
    }
    if (a.split > 1) {
        const size_t need = (size_t)a.split * a.M * a.N * 4;
        if (!d_ws || ws_bytes < need || !aligned16(d_ws)) return DGT_ERR_ARG;
        a.partial = static_cast<float *>(d_ws);
    }
    const size_t smem = (size_t)a.stages * gemm_stage_bytes(R4, a.mt) + 1024;
    int bps = 0;
    DeviceInfo di;
    if (device_info(&di) != DGT_OK) return DGT_ERR_CUDA;
    const uint64_t tiles = (a.N / GT_N) * ((a.M + a.mt - 1) / a.mt);
    const bool persistent = a.split == 1 && (a.schedule == 2 || (a.schedule == 0 && tiles > (uint64_t)di.sms));
    if (persistent) {
        const uint32_t threads = (R4 ? PT_WARPS_R4 : PT_WARPS_BF16) * 32;
        if (prepare_kernel((const void *)k_gemm_pt<R4>, smem, threads, &bps) != DGT_OK) return DGT_ERR_CUDA;
        const unsigned grid = (unsigned)min(tiles, (uint64_t)di.sms);
        if (launch_pdl(k_gemm_pt<R4>, dim3(grid), dim3(threads), smem, st, tm_x, tm_w, tm_nib, a) != cudaSuccess)
            return DGT_ERR_CUDA;
        return cudaPeekAtLastError() == cudaSuccess ? DGT_OK : DGT_ERR_CUDA;
    }
    if (prepare_kernel((const void *)k_gemm<R4>, smem, GT_THREADS, &bps) != DGT_OK) return DGT_ERR_CUDA;
    dim3 grid((unsigned)(a.N / GT_N), (unsigned)((a.M + a.mt - 1) / a.mt), a.split);
    if (launch_pdl(k_gemm<R4>, grid, dim3(GT_THREADS), smem, st, tm_x, tm_w, tm_nib, a) != cudaSuccess)
        return DGT_ERR_CUDA;
    if (a.split > 1) {
        const uint64_t total = a.M * a.N;
        uint64_t g = (total + 255) / 256;
        if (g > (uint64_t)di.sms * 8) g = (uint64_t)di.sms * 8;
        if (launch_pdl(k_gemm_reduce, dim3((unsigned)g), dim3(256), 0, st, a) != cudaSuccess) return DGT_ERR_CUDA;
    }
    return cudaPeekAtLastError() == cudaSuccess ? DGT_OK : DGT_ERR_CUDA;
}

static int fill_common(GemmArgs &a, uint64_t M, uint64_t N, uint64_t K, const dgt_gemm_plan *plan, float *d_Y32,
                       uint16_t *d_Y, int32_t *d_status, cudaStream_t st, bool reset = true) {
    if (M == 0 || N == 0 || K == 0) return DGT_ERR_SHAPE;
    if (N % GT_N || K % GT_K || M >= (1ull << 31) || N >= (1ull << 31) || K >= (1ull << 31)) return DGT_ERR_SHAPE;
    if (!d_Y32 && !d_Y) return DGT_ERR_ARG;
    dgt_gemm_plan p;
    if (plan) p = *plan;
    else dgt_gemm_default_plan(M, N, K, &p);
    if (p.m_tile < 16 || p.m_tile > 256 || p.m_tile % 16 || p.split_k < 1 || (uint64_t)p.split_k > K / GT_K)
        return DGT_ERR_ARG;
    if ((p.test_flags & ~(DGT_TEST_SHORT_WAITS | 0xFFFF0000u)) ||
        (!(p.test_flags & DGT_TEST_SHORT_WAITS) && (p.test_flags >> 16)))
        return DGT_ERR_ARG;
    a.spin = wait_limit_from_flags(p.test_flags);
    if (p.schedule < 0 || p.schedule > 2 || (p.schedule == 2 && p.split_k != 1)) return DGT_ERR_ARG;
    a.schedule = (uint32_t)p.schedule;
    a.M = M;
    a.N = N;
    a.K = K;
    a.mt = (uint32_t)p.m_tile;
    a.kb_total = (uint32_t)(K / GT_K);
    a.split = (uint32_t)p.split_k;
    a.y32 = d_Y32;
    a.y = d_Y;
    a.status = d_status;
    if (reset && d_status && cudaMemsetAsync(d_status, 0, 4, st) != cudaSuccess) return DGT_ERR_CUDA;
    return DGT_OK;
}

// The bf16 GEMM; reset = false keeps the status word as an earlier call of
// the same stream left it.
static int gemm_bf16_impl(const uint16_t *d_W, uint64_t N, uint64_t K, const uint16_t *d_X, uint64_t M,
                          float *d_Y32, uint16_t *d_Y, const dgt_gemm_plan *plan, void *d_ws, size_t ws_bytes,
                          int32_t *d_status, cudaStream_t st, bool reset) {
    if (!d_W || !d_X) return DGT_ERR_ARG;
    GemmArgs a = {};
    int rc = fill_common(a, M, N, K, plan, d_Y32, d_Y, d_status, st, reset);
    if (rc != DGT_OK) return rc;
    if (!aligned16(d_W) || !aligned16(d_X)) return DGT_ERR_ARG;
    a.stages = gemm_stages(false, a.mt);
    return launch_gemm<false>(a, d_W, d_X, d_ws, ws_bytes, st);
}

// ---- grouped expert products ---------------------------------------------------
// Pairs (t, j) of tokens and their routed slots are placed expert by expert
// in (t, j) order by a three-kernel counting sort (per-block expert counts,
// one scan, placement), which also gathers each pair's x row; the tcgen05
// kernel then runs one CTA per (n-tile, expert m-tile) job, and a last kernel
// adds out[t] = sum_j p[t, j] y[t, j] in slot order.
constexpr uint32_t MG_MAX_EXPERTS = 4096;
constexpr uint32_t MG_MAX_PAIRS = 1u << 16;
constexpr uint32_t MG_BLOCK = 256;   // pairs per counting block

struct MgArgs {
    const int32_t *ids;
    const float *p;
    const uint16_t *x;
    uint16_t *xg;        // gathered x rows, pairs x K
    uint32_t *hist;      // n_experts x nb: counts, then exclusive prefixes over blocks
    uint32_t *geoff;     // n_experts + 1
    uint32_t *gjob;      // jobs (grid y of the product kernel)
    uint32_t *glist;     // pairs in expert order: t << 8 | j
    const float *y32;    // pairs x ne
    float *out32;
    uint16_t *out;
    uint64_t K, ne;
    uint32_t n_experts, tokens, topk, pairs, nb, mt, njobs_max;
    int32_t *status;
};

static inline uint32_t mg_mtile(uint32_t pairs, uint32_t n_experts) {
    const uint32_t used = pairs < n_experts ? pairs : n_experts;
    uint32_t mean = (pairs + used - 1) / used;
    uint32_t mt = (mean + 15) / 16 * 16;
    return mt < 16 ? 16u : (mt > 128 ? 128u : mt);
}

__global__ void __launch_bounds__(MG_BLOCK) k_mg_count(MgArgs a) {
    __shared__ uint32_t cnt[MG_MAX_EXPERTS];
    pdl_trigger();
    pdl_wait();
    for (uint32_t e = threadIdx.x; e < a.n_experts; e += MG_BLOCK) cnt[e] = 0;
    __syncthreads();
    const uint32_t q = blockIdx.x * MG_BLOCK + threadIdx.x;
    if (q < a.pairs) {
        const int32_t e = a.ids[q];
        if (e >= 0 && (uint32_t)e < a.n_experts) atomicAdd(&cnt[e], 1u);
        else set_status(a.status, DGT_ERR_ARG);
    }
    __syncthreads();
    for (uint32_t e = threadIdx.x; e < a.n_experts; e += MG_BLOCK) a.hist[(uint64_t)e * a.nb + blockIdx.x] = cnt[e];
}

// One CTA: per expert, exclusive prefixes of its block counts (in place) and
// its total; geoff = exclusive prefix of the totals; the job list (every
// m-tile of every expert in use, expert order), padded with ~0.
__global__ void __launch_bounds__(1024) k_mg_scan(MgArgs a) {
    __shared__ uint32_t tot[MG_MAX_EXPERTS];
    __shared__ uint32_t wsum[32];
    pdl_trigger();
    pdl_wait();
    const uint32_t tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
    for (uint32_t e = tid; e < a.n_experts; e += 1024) {
        uint32_t sacc = 0;
        for (uint32_t b = 0; b < a.nb; b++) {
            const uint32_t v = a.hist[(uint64_t)e * a.nb + b];
            a.hist[(uint64_t)e * a.nb + b] = sacc;
            sacc += v;
        }
        tot[e] = sacc;
    }
    __syncthreads();
    // two exclusive scans over the experts (pairs, then m-tiles), four per thread
    constexpr uint32_t PER = MG_MAX_EXPERTS / 1024;
    for (int pass = 0; pass < 2; pass++) {
        uint32_t v[PER], sum = 0;
#pragma unroll
        for (uint32_t i = 0; i < PER; i++) {
            const uint32_t e = tid * PER + i;
            const uint32_t c = e < a.n_experts ? tot[e] : 0u;
            v[i] = pass == 0 ? c : (c + a.mt - 1) / a.mt;
            sum += v[i];
        }
        uint32_t x = sum;
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
            const uint32_t y = __shfl_up_sync(DGT_FULL, x, d);
            if (lane >= (uint32_t)d) x += y;
        }
        if (lane == 31) wsum[w] = x;
        __syncthreads();
        if (w == 0) {
            uint32_t t = wsum[lane];
#pragma unroll
            for (int d = 1; d < 32; d <<= 1) {
                const uint32_t y = __shfl_up_sync(DGT_FULL, t, d);
                if (lane >= (uint32_t)d) t += y;
            }
            wsum[lane] = t;
        }
        __syncthreads();
        uint32_t run = (w ? wsum[w - 1] : 0u) + x - sum;
        const uint32_t all = wsum[31];
#pragma unroll
        for (uint32_t i = 0; i < PER; i++) {
            const uint32_t e = tid * PER + i;
            if (e < a.n_experts) {
                if (pass == 0) {
                    a.geoff[e] = run;
                } else {
                    for (uint32_t m = 0; m < v[i] && run + m < a.njobs_max; m++) a.gjob[run + m] = e << 16 | m;
                }
            }
            run += v[i];
        }
        if (tid == 0) {
            if (pass == 0) a.geoff[a.n_experts] = all;
        }
        if (pass == 1)
            for (uint32_t j = all + tid; j < a.njobs_max; j += 1024) a.gjob[j] = 0xFFFFFFFFu;
        __syncthreads();
    }
}

// Block b places its pairs: rank among the block's earlier pairs of the
// same expert.
__global__ void __launch_bounds__(MG_BLOCK) k_mg_place(MgArgs a) {
    __shared__ int32_t sid[MG_BLOCK];
    pdl_trigger();
    pdl_wait();
    const uint32_t tid = threadIdx.x, q = blockIdx.x * MG_BLOCK + tid;
    const int32_t e = q < a.pairs ? a.ids[q] : -1;
    sid[tid] = e;
    __syncthreads();
    if (e >= 0 && (uint32_t)e < a.n_experts) {
        uint32_t r = 0;
        for (uint32_t i = 0; i < tid; i++) r += sid[i] == e;
        const uint32_t pos = a.geoff[e] + a.hist[(uint64_t)e * a.nb + blockIdx.x] + r;
        a.glist[pos] = ((q / a.topk) << 8) | (q % a.topk);
    }
}

// The gathered matrix: row i = x of pair glist[i]'s token (16-byte pieces,
// grid-stride over every SM).  Rows of pairs with a bad id stay unwritten;
// no job reads them.
__global__ void __launch_bounds__(256) k_mg_gather(MgArgs a) {
    pdl_trigger();
    pdl_wait();
    const uint32_t kv = (uint32_t)(a.K / 8);   // uint4 per row
    const uint32_t placed = a.geoff[a.n_experts];
    const uint64_t total = (uint64_t)placed * kv;
    for (uint64_t i = (uint64_t)blockIdx.x * 256 + threadIdx.x; i < total; i += (uint64_t)gridDim.x * 256) {
        const uint32_t r = (uint32_t)(i / kv), c = (uint32_t)(i - (uint64_t)r * kv);
        const uint32_t tk = a.glist[r] >> 8;
        reinterpret_cast<uint4 *>(a.xg + (uint64_t)r * a.K)[c] = reinterpret_cast<const uint4 *>(a.x + (uint64_t)tk * a.K)[c];
    }
}

// out[t, n] = fmaf(p[t, topk-1], y[t, topk-1, n], ... fmaf(p[t, 0], y[t, 0, n], +0)).
__global__ void __launch_bounds__(256) k_mg_combine(MgArgs a) {
    pdl_trigger();
    pdl_wait();
    const uint64_t total = (uint64_t)a.tokens * a.ne;
    for (uint64_t i = (uint64_t)blockIdx.x * 256 + threadIdx.x; i < total; i += (uint64_t)gridDim.x * 256) {
        const uint64_t t = i / a.ne, n = i - t * a.ne;
        float acc = 0.0f;
        for (uint32_t j = 0; j < a.topk; j++) {
            const uint64_t q = t * a.topk + j;
            const int32_t e = a.ids[q];
            if (e < 0 || (uint32_t)e >= a.n_experts) continue;
            acc = fmaf(a.p[q], a.y32[q * a.ne + n], acc);
        }
        if (a.out32) a.out32[i] = acc;
        if (a.out) a.out[i] = f32_to_bf16_rne(acc);
    }
}

struct MgLayout {
    size_t hist, geoff, gjob, glist, xg, y, total;
    uint32_t nb, mt, njobs;
};

static inline size_t al256(size_t x) { return (x + 255) & ~(size_t)255; }

static MgLayout mg_layout(uint32_t n_experts, uint64_t ne, uint64_t K, uint32_t tokens, uint32_t topk) {
    MgLayout l;
    const uint32_t P = tokens * topk;
    l.nb = (P + MG_BLOCK - 1) / MG_BLOCK;
    l.mt = mg_mtile(P, n_experts);
    l.njobs = (P + l.mt - 1) / l.mt + (P < n_experts ? P : n_experts);
    l.hist = 0;
    l.geoff = al256(l.hist + 4ull * n_experts * l.nb);
    l.gjob = al256(l.geoff + 4ull * (n_experts + 1));
    l.glist = al256(l.gjob + 4ull * l.njobs);
    l.xg = al256(l.glist + 4ull * P);
    l.y = al256(l.xg + 2ull * P * K);
    l.total = al256(l.y + 4ull * P * ne);
    return l;
}

// The grouped product: route and gather, the tcgen05 kernel over the jobs,
// then the weighted sum (when p is given).
template <bool R4>
static int launch_moe_gemm(GemmArgs &g, MgArgs &m, const void *w_or_sm, void *d_ws, size_t ws_bytes, float *d_y32,
                           cudaStream_t st) {
    const MgLayout l = mg_layout(m.n_experts, m.ne, m.K, m.tokens, m.topk);
    if (!d_ws || ws_bytes < l.total || ((uintptr_t)d_ws & 255)) return DGT_ERR_ARG;
    uint8_t *ws = static_cast<uint8_t *>(d_ws);
    m.hist = reinterpret_cast<uint32_t *>(ws + l.hist);
    m.geoff = reinterpret_cast<uint32_t *>(ws + l.geoff);
    m.gjob = reinterpret_cast<uint32_t *>(ws + l.gjob);
    m.glist = reinterpret_cast<uint32_t *>(ws + l.glist);
    m.xg = reinterpret_cast<uint16_t *>(ws + l.xg);
    float *y = d_y32 ? d_y32 : reinterpret_cast<float *>(ws + l.y);
    m.y32 = y;
    m.nb = l.nb;
    m.mt = l.mt;
    m.njobs_max = l.njobs;
    if (launch_pdl(k_mg_count, dim3(l.nb), dim3(MG_BLOCK), 0, st, m) != cudaSuccess) return DGT_ERR_CUDA;
    if (launch_pdl(k_mg_scan, dim3(1), dim3(1024), 0, st, m) != cudaSuccess) return DGT_ERR_CUDA;
    if (launch_pdl(k_mg_place, dim3(l.nb), dim3(MG_BLOCK), 0, st, m) != cudaSuccess) return DGT_ERR_CUDA;
    {
        DeviceInfo di;
        if (device_info(&di) != DGT_OK) return DGT_ERR_CUDA;
        const uint64_t need = ((uint64_t)m.pairs * (m.K / 8) + 255) / 256;
        const uint64_t gg = need < (uint64_t)di.sms * 4 ? (need ? need : 1) : (uint64_t)di.sms * 4;
        if (launch_pdl(k_mg_gather, dim3((unsigned)gg), dim3(256), 0, st, m) != cudaSuccess) return DGT_ERR_CUDA;
    }
    g.M = m.pairs;
    g.K = m.K;
    g.mt = l.mt;
    g.kb_total = (uint32_t)(m.K / GT_K);
    g.split = 1;
    g.y32 = y;
    g.y = nullptr;
    g.status = m.status;
    g.grouped = 1;
    g.spin = MBAR_SPIN_LIMIT;
    g.gjob = m.gjob;
    g.geoff = m.geoff;
    g.glist = m.glist;
    g.ne = m.ne;
    g.topk = m.topk;
    g.stages = gemm_stages(R4, g.mt);
    CUtensorMap tm_x, tm_w, tm_nib;
    if (!make_map(&tm_x, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, m.xg, g.K, g.M, g.K * 2, GT_K, g.mt,
                  CU_TENSOR_MAP_SWIZZLE_128B))
        return DGT_ERR_CUDA;
    if (R4) {
        if (!make_map(&tm_w, CU_TENSOR_MAP_DATA_TYPE_UINT8, w_or_sm, g.K, g.N, g.K, GT_K, GT_N,
                      CU_TENSOR_MAP_SWIZZLE_NONE) ||
            !make_map(&tm_nib, CU_TENSOR_MAP_DATA_TYPE_UINT8, g.nib, g.K / 2, g.N, g.K / 2, GT_K / 2, GT_N,
                      CU_TENSOR_MAP_SWIZZLE_NONE))
            return DGT_ERR_CUDA;
    } else {
        if (!make_map(&tm_w, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, w_or_sm, g.K, g.N, g.K * 2, GT_K, GT_N,
                      CU_TENSOR_MAP_SWIZZLE_128B))
            return DGT_ERR_CUDA;
        tm_nib = tm_w;
    }
    const size_t smem = (size_t)g.stages * gemm_stage_bytes(R4, g.mt) + 1024;
    int bps = 0;
    if (prepare_kernel((const void *)k_gemm<R4>, smem, GT_THREADS, &bps) != DGT_OK) return DGT_ERR_CUDA;
    dim3 grid((unsigned)((m.ne + GT_N - 1) / GT_N), l.njobs, 1);
    if (launch_pdl(k_gemm<R4>, grid, dim3(GT_THREADS), smem, st, tm_x, tm_w, tm_nib, g) != cudaSuccess)
        return DGT_ERR_CUDA;
    if (m.p && (m.out || m.out32)) {
        DeviceInfo di;
        if (device_info(&di) != DGT_OK) return DGT_ERR_CUDA;
        const uint64_t total = (uint64_t)m.tokens * m.ne;
        uint64_t cg = (total + 255) / 256;
        if (cg > (uint64_t)di.sms * 8) cg = (uint64_t)di.sms * 8;
        if (launch_pdl(k_mg_combine, dim3((unsigned)cg), dim3(256), 0, st, m) != cudaSuccess) return DGT_ERR_CUDA;
    }
    return cudaPeekAtLastError() == cudaSuccess ? DGT_OK : DGT_ERR_CUDA;
}

static int mg_common(MgArgs &m, GemmArgs &g, uint64_t rows, uint64_t cols, uint32_t n_experts, uint32_t tokens,
                     uint32_t topk, const int32_t *d_ids, const float *d_p, const uint16_t *d_X, uint16_t *d_out,
                     float *d_out32, int32_t *d_status, cudaStream_t st) {
    if (n_experts == 0 || n_experts > MG_MAX_EXPERTS || rows % n_experts) return DGT_ERR_SHAPE;
    if (topk == 0 || topk > 255 || (uint64_t)tokens * topk > MG_MAX_PAIRS || tokens >= (1u << 24))
        return DGT_ERR_SHAPE;
    if (cols == 0 || cols % GT_K || cols >= (1ull << 31) || rows >= (1ull << 31)) return DGT_ERR_SHAPE;
    if (!d_ids || !d_X || !aligned16(d_X) || ((d_out || d_out32) && !d_p)) return DGT_ERR_ARG;
    m.ids = d_ids;
    m.p = d_p;
    m.x = d_X;
    m.out = d_out;
    m.out32 = d_out32;
    m.K = cols;
    m.ne = rows / n_experts;
    m.n_experts = n_experts;
    m.tokens = tokens;
    m.topk = topk;
    m.pairs = tokens * topk;
    m.status = d_status;
    g.N = rows;
    if (d_status && cudaMemsetAsync(d_status, 0, 4, st) != cudaSuccess) return DGT_ERR_CUDA;
    return DGT_OK;
}

}  // namespace dgt

using namespace dgt;

extern "C" size_t dgt_moe_gemm_workspace_bytes(uint32_t n_experts, uint64_t expert_rows, uint64_t cols,
                                               uint32_t tokens, uint32_t topk) {
    if (n_experts == 0 || tokens == 0 || topk == 0) return 0;
    return mg_layout(n_experts, expert_rows, cols, tokens, topk).total;
}

extern "C" int dgt_moe_gemm(const dgt_r4 *W, uint32_t n_experts, const int32_t *d_ids, const float *d_p,
                            const uint16_t *d_X, uint32_t tokens, uint32_t topk, float *d_y32, uint16_t *d_out,
                            float *d_out32, void *d_ws, size_t ws_bytes, int32_t *d_status, void *stream) {
    if (!W) return DGT_ERR_ARG;
    if (tokens == 0) return DGT_OK;
    cudaStream_t st = (cudaStream_t)stream;
    MgArgs m = {};
    GemmArgs g = {};
    int rc = mg_common(m, g, W->rows, W->cols, n_experts, tokens, topk, d_ids, d_p, d_X, d_out, d_out32, d_status, st);
    if (rc != DGT_OK) return rc;
    if (!W->sm || !W->nib || !W->seg || (W->n_esc && !W->esc) || !aligned16(W->sm) || !aligned16(W->nib))
        return DGT_ERR_ARG;
    g.nib = W->nib;
    g.esc = W->esc;
    g.seg = W->seg;
    g.n_esc = W->n_esc;
    g.nseg = dgt_r4_nseg(W->cols);
    g.L = make_r4lut(W->table, W->n_table);
    for (int i = 0; i < 256; i++) g.table[i] = W->table[i];
    return launch_moe_gemm<true>(g, m, W->sm, d_ws, ws_bytes, d_y32, st);
}

extern "C" int dgt_moe_gemm_bf16(const uint16_t *d_W, uint64_t rows, uint64_t cols, uint32_t n_experts,
                                 const int32_t *d_ids, const float *d_p, const uint16_t *d_X, uint32_t tokens,
                                 uint32_t topk, float *d_y32, uint16_t *d_out, float *d_out32, void *d_ws,
                                 size_t ws_bytes, int32_t *d_status, void *stream) {
    if (!d_W) return DGT_ERR_ARG;
    if (tokens == 0) return DGT_OK;
    cudaStream_t st = (cudaStream_t)stream;
    MgArgs m = {};
    GemmArgs g = {};
    int rc = mg_common(m, g, rows, cols, n_experts, tokens, topk, d_ids, d_p, d_X, d_out, d_out32, d_status, st);
    if (rc != DGT_OK) return rc;
    if (!aligned16(d_W)) return DGT_ERR_ARG;
    return launch_moe_gemm<false>(g, m, d_W, d_ws, ws_bytes, d_y32, st);
}

extern "C" int dgt_gemm_default_plan(uint64_t M, uint64_t N, uint64_t K, dgt_gemm_plan *plan) {
    if (!plan || M == 0 || N == 0 || K == 0) return DGT_ERR_ARG;
    uint32_t mt = M <= 256 ? (uint32_t)((M + 15) / 16 * 16) : 256u;
    const uint64_t tiles = ((N + GT_N - 1) / GT_N) * ((M + mt - 1) / mt);
    uint64_t split = tiles >= 152 ? 1 : 152 / tiles;   // one CTA per SM, one wave
    const uint64_t kb = K / GT_K;
    if (split > kb / 4) split = kb / 4;
    if (split > 16) split = 16;
    if (split < 1) split = 1;
    plan->m_tile = (int32_t)mt;
    plan->split_k = (int32_t)split;
    plan->test_flags = 0;
    plan->schedule = 0;
    return DGT_OK;
}

extern "C" size_t dgt_gemm_workspace_bytes(uint64_t M, uint64_t N, const dgt_gemm_plan *plan) {
    if (!plan || plan->split_k <= 1) return 0;
    return (size_t)plan->split_k * M * N * 4;
}

extern "C" int dgt_gemm(const dgt_r4 *W, const uint16_t *d_X, uint64_t M, float *d_Y32, uint16_t *d_Y,
                        const dgt_gemm_plan *plan, void *d_ws, size_t ws_bytes, int32_t *d_status, void *stream) {
    if (!W || !d_X) return DGT_ERR_ARG;
    cudaStream_t st = (cudaStream_t)stream;
    GemmArgs a = {};
    int rc = fill_common(a, M, W->rows, W->cols, plan, d_Y32, d_Y, d_status, st);
    if (rc != DGT_OK) return rc;
    if (!W->sm || !W->nib || !W->seg || (W->n_esc && !W->esc) || !aligned16(W->sm) || !aligned16(W->nib) ||
        !aligned16(d_X))
        return DGT_ERR_ARG;
    a.nib = W->nib;
    a.esc = W->esc;
    a.seg = W->seg;
    a.n_esc = W->n_esc;
    a.nseg = dgt_r4_nseg(W->cols);
    a.L = make_r4lut(W->table, W->n_table);
    for (int i = 0; i < 256; i++) a.table[i] = W->table[i];
    a.stages = gemm_stages(true, a.mt);
    return launch_gemm<true>(a, W->sm, d_X, d_ws, ws_bytes, st);
}

extern "C" int dgt_gemm_rebuild(const dgt_r4 *W, const uint16_t *d_X, uint64_t M, float *d_Y32, uint16_t *d_Y,
                                const dgt_gemm_plan *plan, uint16_t *d_scratch, void *d_ws, size_t ws_bytes,
                                int32_t *d_status, void *stream) {
    if (!W || !d_scratch) return DGT_ERR_ARG;
    int rc = dgt_r4_to_bf16(W, d_scratch, d_status, stream);   // resets d_status, then may set it
    if (rc != DGT_OK) return rc;
    return gemm_bf16_impl(d_scratch, W->rows, W->cols, d_X, M, d_Y32, d_Y, plan, d_ws, ws_bytes, d_status,
                          (cudaStream_t)stream, false);
}

extern "C" int dgt_gemm_bf16(const uint16_t *d_W, uint64_t N, uint64_t K, const uint16_t *d_X, uint64_t M,
                             float *d_Y32, uint16_t *d_Y, const dgt_gemm_plan *plan, void *d_ws, size_t ws_bytes,
                             int32_t *d_status, void *stream) {
    return gemm_bf16_impl(d_W, N, K, d_X, M, d_Y32, d_Y, plan, d_ws, ws_bytes, d_status, (cudaStream_t)stream, true);
}
