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
// GB300 design: 8 warps per CTA, (8/S) rows x S slices per CTA iteration, a
// persistent grid sized by occupancy.  x is converted once per CTA into
// shared memory as float32 in a [round][quad][lane] float4 layout, so each
// lane's four LDS.128 per round are conflict-free.  R4 weights stream with one
// 16-byte load of sign/mantissa bytes and one 8-byte load of nibbles per lane
// and round (L1 no-allocate), four rounds in flight; the exponent comes from
// register byte-permutes.  Escapes are found per round from the row-segment
// index (a warp-uniform count, so rounds without escapes pay one shuffle).
#include <cuda_runtime.h>

#include "../../include/dgt.h"
#include "dgt_device.cuh"
#include "dgt_internal.h"
#include "dgt_launch.h"

namespace dgt {

constexpr int GW = 8;       // warps per CTA
constexpr int UNROLL = 4;   // rounds in flight per lane
constexpr uint32_t MAX_FAST_ROUNDS = 104;  // x in shared memory: 104 * 2 KB

struct GemvArgs {
    const uint8_t *sm;
    const uint8_t *nib;
    const uint8_t *esc;
    const uint32_t *seg;
    const uint16_t *W;
    const uint16_t *x;
    uint16_t *y;
    float *y32;
    uint64_t rows, cols, nseg, n_esc;
    uint32_t J;
    R4Lut L;
    uint8_t table[256];
    int32_t *status;
};

// acc = fmaf(w_i, x_i, acc) over the chunk's 16 weights in column order.
__device__ __forceinline__ float fma_chunk(const uint32_t p[8], const float4 *xs, uint32_t j, uint32_t lane,
                                           float acc) {
#pragma unroll
    for (int q = 0; q < 4; q++) {
        const float4 xv = xs[(j * 4 + q) * 32 + lane];
        acc = fmaf(bf16lo(p[2 * q]), xv.x, acc);
        acc = fmaf(bf16hi(p[2 * q]), xv.y, acc);
        acc = fmaf(bf16lo(p[2 * q + 1]), xv.z, acc);
        acc = fmaf(bf16hi(p[2 * q + 1]), xv.w, acc);
    }
    return acc;
}

template <bool R4>
__device__ __forceinline__ float row_fast(const GemvArgs &a, const float4 *xs, uint8_t *escb,
                                          const uint8_t *table_s, uint64_t row, uint32_t j0, uint32_t j1,
                                          uint32_t lane) {
    const uint64_t rbase = row * a.cols;
    float acc = 0.0f;
    uint32_t segb = 0, segc = 0, jbat = j0;
    if (R4) {
        const uint32_t *segr = a.seg + row * a.nseg;
        const uint32_t jj = j0 + lane;
        if (jj < a.nseg) {
            segb = segr[jj];
            segc = segr[jj + 1] - segb;
        }
    }
    for (uint32_t jb = j0; jb < j1; jb += UNROLL) {
        if (R4 && jb - jbat == 32) {
            jbat = jb;
            const uint32_t *segr = a.seg + row * a.nseg;
            const uint32_t jj = jb + lane;
            segb = segc = 0;
            if (jj < a.nseg) {
                segb = segr[jj];
                segc = segr[jj + 1] - segb;
            }
        }
        uint4 sv[UNROLL], wv2[UNROLL];
        uint2 nv[UNROLL];
        uint32_t cnt[UNROLL], sb[UNROLL], ev[UNROLL];
#pragma unroll
        for (int t = 0; t < UNROLL; t++) {
            const uint32_t j = jb + t;
            const uint64_t k0 = (uint64_t)j * 512 + 16 * lane;
            const bool act = j < j1 && k0 < a.cols;
            sv[t] = make_uint4(0, 0, 0, 0);
            wv2[t] = make_uint4(0, 0, 0, 0);
            nv[t] = make_uint2(0, 0);
            cnt[t] = 0;
            sb[t] = 0;
            ev[t] = 0;
            if (R4) {
                if (act) {
                    sv[t] = ldg_stream16(a.sm + rbase + k0);
                    nv[t] = ldg_stream8(a.nib + (rbase + k0) / 2);
                }
                const uint32_t c = __shfl_sync(DGT_FULL, segc, (j - jbat) & 31);
                const uint32_t b = __shfl_sync(DGT_FULL, segb, (j - jbat) & 31);
                if (j < j1 && c) {
                    cnt[t] = c;
                    sb[t] = b;
                    if (lane < c && (uint64_t)b + lane < a.n_esc) ev[t] = a.esc[b + lane];
                }
            } else if (act) {
                const uint4 *src = reinterpret_cast<const uint4 *>(a.W + rbase + k0);
                sv[t] = ldg_stream16(src);
                wv2[t] = ldg_stream16(src + 1);
            }
        }
#pragma unroll
        for (int t = 0; t < UNROLL; t++) {
            const uint32_t j = jb + t;
            if (j >= j1) break;
            const bool act = (uint64_t)j * 512 + 16 * lane < a.cols;
            uint32_t p[8];
            if (R4) {
                r4_dec16(nv[t], sv[t], a.L, p);
                if (cnt[t]) {
                    const uint32_t c = cnt[t];
                    if (lane < c) escb[lane] = (uint8_t)ev[t];
                    for (uint32_t i = lane + 32; i < c && i < DGT_SEG; i += 32)
                        escb[i] = (uint64_t)sb[t] + i < a.n_esc ? a.esc[sb[t] + i] : 0;
                    __syncwarp();
                    const uint32_t m0 = act ? nib15_mask(nv[t].x) : 0u;
                    const uint32_t m1 = act ? nib15_mask(nv[t].y) : 0u;
                    if ((!patch_escapes(p, m0, m1, c > DGT_SEG ? DGT_SEG : c, escb, table_s) ||
                         c > DGT_SEG) && lane == 0)
                        set_status(a.status, DGT_ERR_CORRUPT);
                    __syncwarp();
                }
            } else {
                p[0] = sv[t].x; p[1] = sv[t].y; p[2] = sv[t].z; p[3] = sv[t].w;
                p[4] = wv2[t].x; p[5] = wv2[t].y; p[6] = wv2[t].z; p[7] = wv2[t].w;
            }
            if (act) acc = fma_chunk(p, xs, j, lane, acc);
        }
    }
    return acc;
}

template <bool R4, int S>
__global__ void __launch_bounds__(GW * 32) k_gemv(GemvArgs a) {
    extern __shared__ float4 xs[];
    __shared__ uint8_t table_s[256];
    __shared__ uint8_t escb[GW][DGT_SEG];
    __shared__ float part[GW];
    const uint32_t tid = threadIdx.x, w = tid >> 5, lane = tid & 31;
    const uint32_t K = (uint32_t)a.cols;
    for (uint32_t i = tid; i < K / 8; i += GW * 32) {
        const uint4 v = *reinterpret_cast<const uint4 *>(a.x + 8 * i);
        const uint32_t k = 8 * i, j = k >> 9, u = (k >> 4) & 31, q = (k >> 2) & 3;
        xs[(j * 4 + q) * 32 + u] = make_float4(bf16lo(v.x), bf16hi(v.x), bf16lo(v.y), bf16hi(v.y));
        xs[(j * 4 + q + 1) * 32 + u] = make_float4(bf16lo(v.z), bf16hi(v.z), bf16lo(v.w), bf16hi(v.w));
    }
    if (R4) table_s[tid] = a.table[tid];
    __syncthreads();
    constexpr uint32_t RPB = GW / S;
    const uint32_t rl = w / S, s = w % S;
    const uint32_t j0 = (uint32_t)((uint64_t)s * a.J / S), j1 = (uint32_t)((uint64_t)(s + 1) * a.J / S);
    const uint64_t groups = (a.rows + RPB - 1) / RPB;
    for (uint64_t gi = blockIdx.x; gi < groups; gi += gridDim.x) {
        const uint64_t row = gi * RPB + rl;
        float acc = 0.0f;
        if (row < a.rows) acc = row_fast<R4>(a, xs, escb[w], table_s, row, j0, j1, lane);
#pragma unroll
        for (int d = 16; d >= 1; d >>= 1) acc += __shfl_xor_sync(DGT_FULL, acc, d);
        if (S == 1) {
            if (lane == 0 && row < a.rows) {
                if (a.y32) a.y32[row] = acc;
                if (a.y) a.y[row] = f32_to_bf16_rne(acc);
            }
        } else {
            if (lane == 0) part[w] = acc;
            __syncthreads();
            if (s == 0 && lane == 0 && row < a.rows) {
                float y = part[w];
#pragma unroll
                for (int t = 1; t < S; t++) y = y + part[w + t];
                if (a.y32) a.y32[row] = y;
                if (a.y) a.y[row] = f32_to_bf16_rne(y);
            }
            __syncthreads();
        }
    }
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
int launch_gemv(GemvArgs &a, bool fast, cudaStream_t st) {
    DeviceInfo di;
    if (device_info(&di) != DGT_OK) return DGT_ERR_CUDA;
    const int S = dgt_plan_slices(a.rows, a.cols);
    const uint64_t groups = (a.rows + (GW / S) - 1) / (GW / S);
    int bps = 0;
    if (!fast) {
        if (prepare_kernel((const void *)k_gemv_any<R4>, 0, GW * 32, &bps) != DGT_OK) return DGT_ERR_CUDA;
        const uint64_t grid = min((uint64_t)di.sms * bps, groups);
        k_gemv_any<R4><<<(unsigned)grid, GW * 32, 0, st>>>(a, S);
    } else {
        const size_t smem = (size_t)a.J * 2048;
        const void *fn = S == 1   ? (const void *)k_gemv<R4, 1>
                         : S == 2 ? (const void *)k_gemv<R4, 2>
                         : S == 4 ? (const void *)k_gemv<R4, 4>
                                  : (const void *)k_gemv<R4, 8>;
        if (prepare_kernel(fn, smem, GW * 32, &bps) != DGT_OK) return DGT_ERR_CUDA;
        const unsigned grid = (unsigned)min((uint64_t)di.sms * bps, groups);
        switch (S) {
            case 1: k_gemv<R4, 1><<<grid, GW * 32, smem, st>>>(a); break;
            case 2: k_gemv<R4, 2><<<grid, GW * 32, smem, st>>>(a); break;
            case 4: k_gemv<R4, 4><<<grid, GW * 32, smem, st>>>(a); break;
            default: k_gemv<R4, 8><<<grid, GW * 32, smem, st>>>(a); break;
        }
    }
    return cudaPeekAtLastError() == cudaSuccess ? DGT_OK : DGT_ERR_CUDA;
}

}  // namespace dgt

using namespace dgt;

extern "C" int dgt_gemv(const dgt_r4 *W, const uint16_t *d_x, uint16_t *d_y, float *d_y32, void *stream) {
    if (!W) return DGT_ERR_ARG;
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
    a.status = nullptr;
    const bool fast = K > 0 && K % 16 == 0 && a.J <= MAX_FAST_ROUNDS && aligned16(W->sm) &&
                      aligned16(W->nib) && aligned16(d_x);
    return launch_gemv<true>(a, fast, (cudaStream_t)stream);
}

extern "C" int dgt_gemv_bf16(const uint16_t *d_W, uint64_t rows, uint64_t cols, const uint16_t *d_x,
                             uint16_t *d_y, float *d_y32, void *stream) {
    const uint64_t N = rows, K = cols;
    if (K >= (1ull << 31) || (N && (N * K) / N != K)) return DGT_ERR_SHAPE;
    if (N == 0) return DGT_OK;
    if (!d_y && !d_y32) return DGT_ERR_ARG;
    if (K && (!d_x || !d_W)) return DGT_ERR_ARG;
    GemvArgs a = {};
    a.W = d_W;
    a.x = d_x;
    a.y = d_y;
    a.y32 = d_y32;
    a.rows = N;
    a.cols = K;
    a.J = (uint32_t)((K + 511) / 512);
    const bool fast = K > 0 && K % 16 == 0 && a.J <= MAX_FAST_ROUNDS && aligned16(d_W) && aligned16(d_x);
    return launch_gemv<false>(a, fast, (cudaStream_t)stream);
}
